// launch.h -- internal: the table of compiled kernel variants and how to launch one.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "kernel.cuh"
#include "mslkb.h"

namespace mslkb {

struct LaunchArgs {
  GemmParams params;
  CUtensorMap tmA;   // activation tiles [rows, K], box (128 B, box_act)
  CUtensorMap tmB;   // weight tiles [G, N, K], box (128 B, box_w, 1)
  CUtensorMap tmC;   // output [rows, N] bf16, box (32, 32), 64-byte swizzle (128-row tiles)
  CUtensorMap tmB2;  // swap-AB weights as (128 B, N, K / 128, G), box (128 B, box_w, 2, 1)
  dim3 grid;
  cudaStream_t stream;
};

using LaunchFn = cudaError_t (*)(const LaunchArgs&);
using AttrFn = cudaError_t (*)();
using OccupancyFn = cudaError_t (*)(int* blocks_per_sm, int* regs_per_thread,
                                    int* cluster_ctas);

struct VariantInfo {
  const char* name;
  int tile_n;     // MMA N
  int stages;
  bool swap;
  bool tma;
  bool dynamic;
  int threads;
  int smem;
  int act_rows;   // activation rows per output tile
  int w_rows;     // weight rows (output columns) per output tile
  int box_act;    // activation rows one CTA loads per stage (TMA box height)
  int box_w;      // weight rows one CTA loads per stage
  int cluster;    // CTAs per cluster: 2 for CTA pairs (cta_group::2), else 1
  int ragged;     // 0 grouped rows (stacked / dynamic), 1 ragged N, 2 ragged K
  int block_scale;  // 1: block-scaled (groupwise) scales
  int partial_bytes;  // fp32 partial sums of one tile (a split tile's piece)
  int launch_regs;    // registers per thread the kernel must be built with (0: any)
  LaunchFn launch;
  AttrFn set_attr;
  OccupancyFn occupancy;
};

template <class Cfg>
cudaError_t launch_variant(const LaunchArgs& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = a.grid;
  cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = a.stream;
  // programmatic dependent launch: the kernel waits (griddepcontrol.wait) before touching
  // global memory, so it may start launching while the previous kernel on the stream ends
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if constexpr (Cfg::kPair) {  // CTA pairs: clusters of two along x
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<Cfg>, a.params, a.tmA, a.tmB, a.tmC,
                            a.tmB2);
}

template <class Cfg>
cudaError_t set_attr_variant() {
  return cudaFuncSetAttribute(grouped_gemm_kernel<Cfg>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
}

// CTAs of this variant that fit on one SM (needs the shared-memory attribute set first)
// and, for CTA pairs, how many CTAs of the device can run at once in whole clusters
// (SMs left over in a GPC hold no pair); 0 for single-CTA variants.
template <class Cfg>
cudaError_t occupancy_variant(int* blocks_per_sm, int* regs_per_thread, int* cluster_ctas) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, grouped_gemm_kernel<Cfg>);
  if (e != cudaSuccess) return e;
  *regs_per_thread = fa.numRegs;
  *cluster_ctas = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, grouped_gemm_kernel<Cfg>,
                                                    Cfg::kThreads, Cfg::kSmemBytes);
  if (e != cudaSuccess || !Cfg::kPair) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1), 1, 1);
  cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, grouped_gemm_kernel<Cfg>, &cfg);
  if (e != cudaSuccess) return e;
  *cluster_ctas = 2 * clusters;
  return cudaSuccess;
}

template <class Cfg>
constexpr VariantInfo make_variant(const char* name) {
  return VariantInfo{name,           Cfg::kTileN,   Cfg::kStages,  Cfg::kSwap,
                     Cfg::kTma,      Cfg::kDynamic, Cfg::kThreads, Cfg::kSmemBytes,
                     Cfg::kTileAct,  Cfg::kTileW,   Cfg::kActRows, Cfg::kWRows,
                     Cfg::kCtas,     Cfg::kRagN ? 1 : (Cfg::kRagK ? 2 : 0),
                     Cfg::kBlockScale ? 1 : 0,
                     Cfg::kEpiWarps * 32 * Cfg::kThreadCols * 4,
                     Cfg::kLaunchRegs, &launch_variant<Cfg>, &set_attr_variant<Cfg>,
                     &occupancy_variant<Cfg>};
}

// Defined in mslkb.cu, for the allocation-free entry point in mslkb_noalloc.cu.
mslkb_status stacked_precheck(const void* A, const void* B, const float* scale_a,
                              const float* scale_b, const int64_t* m_sizes, void* out,
                              int64_t total_M, int64_t G, int64_t N, int64_t K,
                              bool* nothing_to_do);
mslkb_status run_stacked_with_scratch(const void* A, const void* B, const float* scale_a,
                                      const float* scale_b, const int64_t* m_sizes, void* out,
                                      int64_t total_M, int64_t G, int64_t N, int64_t K,
                                      void* stream, float* partials, size_t partial_bytes,
                                      uint32_t* counters, size_t counter_count);
void record_cuda_error(cudaError_t e);

// Defined in the variants_*.cu translation units.
extern const VariantInfo kVariantsStackedTma[];
extern const int kNumVariantsStackedTma;
extern const VariantInfo kVariantsDynamicTma[];
extern const int kNumVariantsDynamicTma;
extern const VariantInfo kVariantsCpAsync[];
extern const int kNumVariantsCpAsync;
extern const VariantInfo kVariantsRaggedN[];
extern const int kNumVariantsRaggedN;
extern const VariantInfo kVariantsRaggedK[];
extern const int kNumVariantsRaggedK;
extern const VariantInfo kVariantsBlockScale[];
extern const int kNumVariantsBlockScale;
extern const VariantInfo kVariantsBlockScaleDynamic[];
extern const int kNumVariantsBlockScaleDynamic;

}  // namespace mslkb
