// mslkb.cu -- the C ABI of libmslkb.so (declared in include/mslkb.h): argument checks,
// variant selection, TMA descriptor encoding and the launch of one persistent kernel.
//
// Host-side counterpart of the op modules and dispatcher of MSLK #471 "Back the FP8
// rowwise grouped GEMM ops with FlyDSL on ROCm" (commits moving operand marshalling,
// grid extent and tile selection into one dispatcher; the K-tail variant selected on the
// host): every decision here uses host-known values only (sizes, alignments, SM count);
// the group metadata stays on the device and is read by the kernel's scheduler.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "launch.h"
#include "mslkb.h"
#include "mslkb_tuning.h"

namespace {

using mslkb::GemmParams;
using mslkb::LaunchArgs;
using mslkb::VariantInfo;

constexpr int kVersion = 10000;  // 1.0.0
constexpr int kMaxDevices = 64;
constexpr uint64_t kWaitTimeoutNs = 1000000000ull;  // one pipeline wait gives up after ~1 s
std::atomic<uint64_t> g_wait_timeout_ns{kWaitTimeoutNs};
std::atomic<int> g_test_stall{0};  // one-shot: the next launch withholds a stage
// one-shot: the next launch's speculative schedule reads this metadata instead
std::atomic<const void*> g_test_spec_meta{nullptr};

__device__ uint32_t g_device_status;  // MSLKB_DEV_* bits, per device

thread_local int t_last_cuda_error = 0;
std::atomic<int> g_forced_variant{-1};
// K blocks (of 128) the tensor core accumulates before the epilogue adds the partial sum
// into round-to-nearest fp32 registers; 0 = the whole K in the tensor core.
// GB300: the worst case -- partial sums that climb and cancel inside every chunk -- stays
// at 0.24 / 0.50 / 1.04 of the 1e-6 * sum|terms| tolerance for chunks of 4 / 8 / 16
// K-blocks; the llama405b shape runs 2777 / 2938 / 3060 (whole K) TFLOPS at full clock.
constexpr int kDefaultKbPerChunk = 8;
constexpr int kMaxKbPerChunk = 8;
std::atomic<int> g_kb_per_chunk{kDefaultKbPerChunk};
// swap-AB weight prefetch ahead of the dependency wait, in K blocks (16 KB of weights each)
// per CTA; -1 = the default.  Measured on GB300 (back-to-back calls, llama3-70b shapes):
// 14 blocks (224 KB per CTA, 34 MB over 152 SMs: about what HBM delivers while a CTA
// waits) beat 4-11 and 17-22 at total_M = 1 and tie the best at 16 and 128 rows.
constexpr int kDefaultPrefetchKb = 14;
std::atomic<int> g_prefetch_kb{-1};

int prefetch_kb_for(const VariantInfo* v) {
  const int pf = g_prefetch_kb.load();
  if (!v->swap || !v->tma || v->ragged) return 0;
  return pf < 0 ? kDefaultPrefetchKb : pf;
}
// Split policy: 0 whole tiles only; 1 split the last waves' tiles along K over all CTAs
// (stream-K) for swap-AB plans, where a piece's partial sums are small; 2 split every plan
std::atomic<int> g_split_k{1};

// ---------------------------------------------------------------------------------
// variant table: stacked TMA, dynamic TMA, cp.async (both layouts)
// ---------------------------------------------------------------------------------
int num_variants() {
  return mslkb::kNumVariantsStackedTma + mslkb::kNumVariantsDynamicTma +
         mslkb::kNumVariantsCpAsync + mslkb::kNumVariantsRaggedN + mslkb::kNumVariantsRaggedK +
         mslkb::kNumVariantsBlockScale + mslkb::kNumVariantsBlockScaleDynamic;
}

const VariantInfo* variant(int i) {
  if (i < 0) return nullptr;
  if (i < mslkb::kNumVariantsStackedTma) return &mslkb::kVariantsStackedTma[i];
  i -= mslkb::kNumVariantsStackedTma;
  if (i < mslkb::kNumVariantsDynamicTma) return &mslkb::kVariantsDynamicTma[i];
  i -= mslkb::kNumVariantsDynamicTma;
  if (i < mslkb::kNumVariantsCpAsync) return &mslkb::kVariantsCpAsync[i];
  i -= mslkb::kNumVariantsCpAsync;
  if (i < mslkb::kNumVariantsRaggedN) return &mslkb::kVariantsRaggedN[i];
  i -= mslkb::kNumVariantsRaggedN;
  if (i < mslkb::kNumVariantsRaggedK) return &mslkb::kVariantsRaggedK[i];
  i -= mslkb::kNumVariantsRaggedK;
  if (i < mslkb::kNumVariantsBlockScale) return &mslkb::kVariantsBlockScale[i];
  i -= mslkb::kNumVariantsBlockScale;
  if (i < mslkb::kNumVariantsBlockScaleDynamic) return &mslkb::kVariantsBlockScaleDynamic[i];
  return nullptr;
}

// Profiler ranges: every launch is enqueued inside a push/pop range of the NVTX domain
// "mslkb" whose message is the kernel variant's name and whose payload is the call's rows
// (rows of A), so that a profiler can pick out this library's launches, e.g. ncu --nvtx
// --nvtx-include "mslkb@stacked_pair256x256_tma/".  Without a tool attached the NVTX calls
// return at once.
constexpr int kMaxTracedVariants = 128;
nvtxDomainHandle_t g_nvtx_domain = nullptr;
nvtxStringHandle_t g_nvtx_names[kMaxTracedVariants] = {};
std::once_flag g_nvtx_once;

cudaError_t launch_traced(int vi, const LaunchArgs& la, int64_t rows) {
  std::call_once(g_nvtx_once, [] {
    g_nvtx_domain = nvtxDomainCreateA("mslkb");
    for (int i = 0; i < num_variants() && i < kMaxTracedVariants; ++i)
      g_nvtx_names[i] = nvtxDomainRegisterStringA(g_nvtx_domain, variant(i)->name);
  });
  nvtxEventAttributes_t a = {};
  a.version = NVTX_VERSION;
  a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
  a.messageType = NVTX_MESSAGE_TYPE_REGISTERED;
  a.message.registered = vi < kMaxTracedVariants ? g_nvtx_names[vi] : nullptr;
  a.payloadType = NVTX_PAYLOAD_TYPE_INT64;
  a.payload.llValue = rows;
  nvtxDomainRangePushEx(g_nvtx_domain, &a);
  const cudaError_t e = variant(vi)->launch(la);
  nvtxDomainRangePop(g_nvtx_domain);
  return e;
}

int find_variant(bool dynamic, bool tma, bool swap, int tile_n, int cluster = 1, int ragged = 0,
                 int block_scale = 0) {
  for (int i = 0; i < num_variants(); ++i) {
    const VariantInfo* v = variant(i);
    if (v->dynamic == dynamic && v->tma == tma && v->swap == swap && v->tile_n == tile_n &&
        v->cluster == cluster && v->ragged == ragged && v->block_scale == block_scale)
      return i;
  }
  return -1;
}

// ---------------------------------------------------------------------------------
// per-device state
// ---------------------------------------------------------------------------------
struct DeviceState {
  bool ready = false;
  bool supported = false;
  int sm_count = 0;
  uint32_t* status_ptr = nullptr;
  uint64_t attr_done[2] = {0, 0};  // one bit per variant
  int cluster_ctas[128] = {};       // CTA-pair variants: CTAs that run at once in pairs
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_encode_tried = false;

mslkb_status cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return MSLKB_ERR_CUDA;
}

// Device query, status-word address and driver entry point, once per device.
mslkb_status device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return MSLKB_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& st = g_devices[dev];
  if (!st.ready) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e);
    st.supported = (major == 10 && minor == 3);
    st.sm_count = sms;
    if (st.supported) {
      void* p = nullptr;
      if ((e = cudaGetSymbolAddress(&p, g_device_status)) != cudaSuccess) return cuda_fail(e);
      st.status_ptr = static_cast<uint32_t*>(p);
    }
    if (!g_encode_tried) {
      g_encode_tried = true;
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q);
      if (e == cudaSuccess && q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    st.ready = true;
  }
  if (!st.supported) return MSLKB_ERR_DEVICE;
  *out = &st;
  return MSLKB_OK;
}

// ---------------------------------------------------------------------------------
// split-tile workspace, one per (device, stream): 2 partial-sum slots per CTA and one
// arrival counter per (split tile, epilogue warp), then the two words of the CTA pairs'
// tile claim counter.  Calls on one stream run in order, so they can share it; calls on
// different streams get different workspaces.
// ---------------------------------------------------------------------------------
struct Workspace {
  float* partials = nullptr;
  uint32_t* counters = nullptr;
};
std::map<std::pair<int, uintptr_t>, Workspace> g_workspaces;

// Where the CTA pairs' tile claim counter sits in a workspace's counters.
size_t pair_counter_offset(const DeviceState* st) {
  return 2 * static_cast<size_t>(st->sm_count) * 8;
}

size_t max_partial_bytes() {
  size_t m = 0;
  for (int i = 0; i < num_variants(); ++i)
    if (static_cast<size_t>(variant(i)->partial_bytes) > m) m = variant(i)->partial_bytes;
  return m;
}

// Finds or creates the workspace of `stream`; leaves *ws empty (no splitting) when the
// stream is being captured and has none yet, since allocating is not allowed there.
mslkb_status stream_workspace(const DeviceState* st, cudaStream_t stream, Workspace* ws) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const auto key = std::make_pair(dev, reinterpret_cast<uintptr_t>(stream));
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    auto it = g_workspaces.find(key);
    if (it != g_workspaces.end()) {
      *ws = it->second;
      return MSLKB_OK;
    }
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if ((e = cudaStreamIsCapturing(stream, &cap)) != cudaSuccess) return cuda_fail(e);
  if (cap != cudaStreamCaptureStatusNone) {
    *ws = Workspace{};
    return MSLKB_OK;
  }
  Workspace w;
  const size_t slots = 2 * static_cast<size_t>(st->sm_count);
  if ((e = cudaMalloc(&w.partials, slots * max_partial_bytes())) != cudaSuccess)
    return cuda_fail(e);
  // split tiles < 2 x CTAs, 8 epilogue warps at most; then the pairs' claim counter
  const size_t ncnt = pair_counter_offset(st) + 2;
  if ((e = cudaMalloc(&w.counters, ncnt * sizeof(uint32_t))) != cudaSuccess) {
    cudaFree(w.partials);
    return cuda_fail(e);
  }
  if ((e = cudaMemsetAsync(w.counters, 0, ncnt * sizeof(uint32_t), stream)) != cudaSuccess) {
    cudaFree(w.partials);
    cudaFree(w.counters);
    return cuda_fail(e);
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  auto ins = g_workspaces.emplace(key, w);
  if (!ins.second) {  // another thread created it first
    cudaFree(w.partials);
    cudaFree(w.counters);
  }
  *ws = ins.first->second;
  return MSLKB_OK;
}

mslkb_status ensure_attr(DeviceState* st, int vi) {
  const uint64_t bit = 1ull << (vi & 63);
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (st->attr_done[vi >> 6] & bit) return MSLKB_OK;
  }
  cudaError_t e = variant(vi)->set_attr();
  if (e != cudaSuccess) return cuda_fail(e);
  // a variant that cannot place one CTA on an SM is reported here, not at launch
  int blocks = 0, regs = 0, cluster_ctas = 0;
  e = variant(vi)->occupancy(&blocks, &regs, &cluster_ctas);
  if (e != cudaSuccess) return cuda_fail(e);
  if (blocks < 1) return cuda_fail(cudaErrorLaunchOutOfResources);
  if (variant(vi)->cluster > 1 && cluster_ctas < variant(vi)->cluster)
    return cuda_fail(cudaErrorLaunchOutOfResources);
  // a kernel that moves registers between warpgroups must start with exactly the budget
  // its split adds up to; with fewer, the warps asking for more would never get them
  if (variant(vi)->launch_regs != 0 && regs != variant(vi)->launch_regs)
    return cuda_fail(cudaErrorInvalidConfiguration);
  std::lock_guard<std::mutex> lock(g_mutex);
  st->cluster_ctas[vi & 127] = cluster_ctas;
  st->attr_done[vi >> 6] |= bit;
  return MSLKB_OK;
}

// The planned grid, for CTA pairs cut to the CTAs that run at once in whole clusters (a
// persistent grid must not queue a second partial wave).
unsigned launch_grid(const DeviceState* st, int vi, int64_t planned) {
  const VariantInfo* v = variant(vi);
  if (v->cluster > 1) {
    const int64_t fit = st->cluster_ctas[vi & 127];
    if (planned > fit) planned = (fit / v->cluster) * v->cluster;
  }
  return static_cast<unsigned>(planned);
}

// ---------------------------------------------------------------------------------
// planning (pure host)
// ---------------------------------------------------------------------------------
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int copy_width_for(int64_t K, int64_t a_align, int64_t b_align) {
  const int64_t al = a_align < b_align ? a_align : b_align;
  for (int w : {16, 8, 4})
    if (K % w == 0 && al % w == 0) return w;
  return 1;
}

// Upper bound on output tiles for a variant (the kernel's own count never exceeds it).
int64_t tiles_bound(const VariantInfo* v, int layout, int64_t rows, int64_t G, int64_t N) {
  const int64_t ntn = ceil_div(N, v->w_rows);
  // ragged N: every group's slab rows over its own columns, from the 8-column grid below
  // its first one (a partial tile per group at most); ragged K: a whole slab per group
  if (layout == 2) return ceil_div(rows, v->act_rows) * (ceil_div(N + 7 * G, v->w_rows) + G);
  if (layout == 3) return G * ceil_div(rows, v->act_rows) * ntn;
  if (layout == 0) {
    const int64_t nz = G < rows ? G : rows;  // non-empty groups
    const int64_t mt = (rows + nz * (v->act_rows - 1)) / v->act_rows;
    return mt * ntn;
  }
  return G * ceil_div(rows, v->act_rows) * ntn;  // rows = expected_m here
}

mslkb_status plan(int layout, int64_t rows, int64_t G, int64_t N, int64_t K, int num_sms,
                  int64_t a_align, int64_t b_align, mslkb_plan_info* info) {
  if (layout < 0 || layout > 5) return MSLKB_ERR_SHAPE;
  if (num_sms <= 0 || rows < 0 || G < 0 || N < 0 || K < 0) return MSLKB_ERR_SHAPE;
  const bool dynamic = layout == 1 || layout == 5;
  const int ragged = (layout == 2 || layout == 3) ? layout - 1 : 0;
  // block-scaled stacked (4) or slab (5) layouts
  const int block_scale = (layout == 4 || layout == 5) ? 1 : 0;
  if (block_scale) {  // whole scale blocks along K and N
    if (K % 128 != 0 || N % 128 != 0) return MSLKB_ERR_SHAPE;
    layout = dynamic ? 1 : 0;
  }
  const bool tma = (K % 16 == 0) && (a_align % 16 == 0) && (b_align % 16 == 0);
  if ((ragged || block_scale) && !tma) return MSLKB_ERR_ALIGN;  // TMA-only kernels
  // rows of one group: the slab height (dynamic) or the mean over the groups that can
  // be non-empty (stacked; the counts themselves stay on the device)
  int64_t per_group = rows;
  if (layout == 0 && G > 0 && rows > 0) per_group = rows / (G < rows ? G : rows);
  bool swap;
  int tile_n;
  int cluster = 1;
  if (block_scale) {  // swap-AB up to 32 rows per group; else 128 x 256 / 128 x 128
    swap = per_group <= 32;
    tile_n = per_group <= 16 ? 16 : (swap ? 32 : 128);
    if (!swap) {
      const int wide = find_variant(dynamic, true, false, 256, 1, 0, 1);
      if (wide >= 0 && tiles_bound(variant(wide), layout, rows, G, N) >= num_sms) tile_n = 256;
    }
  } else if (ragged) {  // TMA variants: swap-AB 32, 128 x 256, 128 x 128
    swap = per_group <= 32;
    tile_n = swap ? 32 : 128;
    if (!swap) {
      const int wide = find_variant(false, true, false, 256, 1, ragged);
      if (wide >= 0 && tiles_bound(variant(wide), layout, rows, G, N) >= num_sms) tile_n = 256;
    }
  } else if (per_group <= 16) {
    swap = true;
    tile_n = 16;
  } else if (per_group <= 32 && tma) {
    swap = true;
    tile_n = 32;
  } else {
    swap = false;
    tile_n = 128;
    if (tma) {
      const int wide = find_variant(dynamic, true, false, 256);
      if (wide >= 0 && tiles_bound(variant(wide), layout, rows, G, N) >= num_sms) tile_n = 256;
      // CTA pairs (256 x 256 tiles, a third fewer operand bytes per SM and K block, six
      // stages): measured on GB300 4-5 % ahead of 128 x 256 tiles on full slabs of >= 512
      // rows, 3.5 % ahead on stacked groups of ~1024 rows (16 x 1024 x 16384^2: 3103-3110
      // against 3211-3235 us per call) and ~1.5 % ahead on stacked groups of ~512 rows
      // (16 x 512 x 8192^2, tiles claimed in order: 455-459 against 462-467 us, five
      // alternating rounds); 2.5 % behind on the Zipf-sized groups of the DS-V3 shapes
      // (256 rows on average), where a group's last, half-used pair tile weighs more.
      const int pair = find_variant(dynamic, true, false, 256, 2);
      if (tile_n == 256 && pair >= 0 && per_group >= 512 &&
          tiles_bound(variant(pair), layout, rows, G, N) >= 4 * (num_sms / 2))
        cluster = 2;
    }
  }
  int vi = g_forced_variant.load();
  if (vi < 0) {
    vi = find_variant(dynamic, tma, swap, tile_n, cluster, ragged, block_scale);
    if (vi < 0 && !tma) vi = find_variant(dynamic, false, false, 128);
  }
  const VariantInfo* v = variant(vi);
  if (v == nullptr || v->dynamic != dynamic || v->ragged != ragged ||
      v->block_scale != block_scale || (v->tma && !tma))
    return MSLKB_ERR_SHAPE;
  const int64_t bound = tiles_bound(v, layout, rows, G, N);
  if (bound > INT32_MAX) return MSLKB_ERR_SHAPE;
  const int64_t nkb = ceil_div(K, mslkb::kBK);
  // Measured on GB300: splitting speeds up the swap-AB plans at small M (more SMs stream
  // weights) but slows the 128-row-tile plans by 4-9% (128 KB of partial sums per piece).
  const int policy = g_split_k.load();
  // CTA pairs run whole tiles only (one pair per tile)
  const bool split = nkb > 0 && v->cluster == 1 && !ragged &&
                     (policy == 2 || (policy == 1 && v->swap));
  // with splitting every CTA gets K work as long as there are units to share
  const int64_t work = (split ? bound * nkb : bound) * v->cluster;
  const int64_t max_ctas = (num_sms / v->cluster) * v->cluster;
  int64_t grid = work < max_ctas ? work : max_ctas;
  if (dynamic) {  // padding rows are zeroed by every CTA's epilogue warps
    const int64_t zero_ctas = ceil_div(G * rows, 32);
    if (grid < zero_ctas) grid = zero_ctas < num_sms ? zero_ctas : num_sms;
  }
  if (v->cluster > 1) grid = (grid / v->cluster) * v->cluster;
  if (grid < v->cluster) grid = v->cluster;
  std::memset(info, 0, sizeof(*info));
  info->variant = vi;
  info->swap_ab = v->swap;
  info->tile_m = v->act_rows;
  info->tile_n = v->w_rows;
  info->stages = v->stages;
  info->tma = v->tma;
  info->copy_width = v->tma ? 16 : copy_width_for(K, a_align, b_align);
  info->grid = static_cast<int32_t>(grid);
  info->threads = v->threads;
  info->smem_bytes = v->smem;
  info->tiles_bound = bound;
  info->split_k = split ? 1 : 0;
  return MSLKB_OK;
}

int64_t addr_align(const void* p) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  if (a == 0) return 256;
  return static_cast<int64_t>(a & (~a + 1));  // lowest set bit
}

// ---------------------------------------------------------------------------------
// tensor maps
// ---------------------------------------------------------------------------------
mslkb_status encode_out_map(LaunchArgs* la, const VariantInfo* v, void* out, int64_t rows,
                            int64_t N) {
  std::memset(&la->tmC, 0, sizeof(la->tmC));
  if (v->swap) return MSLKB_OK;  // swap-AB tiles store directly
  if (g_encode == nullptr) return cuda_fail(cudaErrorNotSupported);
  const cuuint32_t elem_strides[2] = {1, 1};
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * 2};
  const cuuint32_t box[2] = {32, 32};  // 32 bf16 (64 bytes) x 32 rows per warp block
  CUresult r = g_encode(&la->tmC, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, out, dims, strides, box,
                        elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    t_last_cuda_error = static_cast<int>(r);
    return MSLKB_ERR_CUDA;
  }
  return MSLKB_OK;
}

mslkb_status encode_maps(LaunchArgs* la, const VariantInfo* v, const void* A, const void* B,
                         int64_t rows, int64_t G, int64_t N, int64_t K) {
  std::memset(&la->tmA, 0, sizeof(la->tmA));
  std::memset(&la->tmB, 0, sizeof(la->tmB));
  std::memset(&la->tmB2, 0, sizeof(la->tmB2));
  if (!v->tma || K == 0) return MSLKB_OK;
  if (g_encode == nullptr) return cuda_fail(cudaErrorNotSupported);
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(mslkb::kBK),
                               static_cast<cuuint32_t>(v->box_act)};
    CUresult r = g_encode(&la->tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(A), dims,
                          strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      t_last_cuda_error = static_cast<int>(r);
      return MSLKB_ERR_CUDA;
    }
  }
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(G)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N * K)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(mslkb::kBK),
                               static_cast<cuuint32_t>(v->box_w), 1};
    CUresult r = g_encode(&la->tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(B), dims,
                          strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      t_last_cuda_error = static_cast<int>(r);
      return MSLKB_ERR_CUDA;
    }
  }
  // swap-AB plans: the weights also as (128 bytes of a K block, N rows, K / 128 blocks, G),
  // so that one box of two K blocks lands as two consecutive stages' [rows][128 B] tiles.
  // Whole K blocks only: with K % 128 != 0 the last block's row would run into the next row.
  la->params.w_pair = 0;
  if (v->swap && v->ragged == 0 && K % 128 == 0) {
    const cuuint64_t dims[4] = {128, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K / 128),
                                static_cast<cuuint64_t>(G)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(K), 128,
                                   static_cast<cuuint64_t>(N * K)};
    const cuuint32_t box[4] = {128, static_cast<cuuint32_t>(v->box_w), 2, 1};
    const cuuint32_t es4[4] = {1, 1, 1, 1};
    CUresult r = g_encode(&la->tmB2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(B),
                          dims, strides, box, es4, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS) la->params.w_pair = 1;  // else the kernel loads one block per box
  }
  return MSLKB_OK;
}

// Two K blocks per weight box (tmB2) for the swap-AB plans that stream long K ranges per
// CTA.  Measured on GB300 against one block per box (three alternating rounds): llama3-70b
// decode with 16 rows 129.2 -> 126.7 us, 128 rows 159.7 -> 155.4; with one row (27 K blocks
// per CTA, where a CTA's first MMA waits for both blocks of its first box) 15.8 -> 16.0, and
// on the block-scaled swap-AB tiles (whose epilogue frees the stages) 130.5 -> 134.4 at 16
// rows: those keep one block per box.
void gate_weight_pairs(LaunchArgs* la, const VariantInfo* v, const mslkb_plan_info& info,
                       int64_t K) {
  const int64_t nkb = ceil_div(K, mslkb::kBK);
  const int64_t per_cta = info.grid > 0 ? info.tiles_bound * nkb / info.grid : 0;
  if (v->block_scale || per_cta < 64) la->params.w_pair = 0;
}

// ---------------------------------------------------------------------------------
// the two entry points share everything but the layout
// ---------------------------------------------------------------------------------
mslkb_status check_sizes(int64_t rows, int64_t G, int64_t N, int64_t K) {
  if (rows < 0 || G < 0 || N < 0 || K < 0) return MSLKB_ERR_SHAPE;
  if (G > MSLKB_MAX_GROUPS) return MSLKB_ERR_SHAPE;
  if (N % 8 != 0) return MSLKB_ERR_SHAPE;
  if (rows > MSLKB_MAX_DIM || N > MSLKB_MAX_DIM || K > MSLKB_MAX_DIM) return MSLKB_ERR_SHAPE;
  return MSLKB_OK;
}

// meta_kind: stacked 0 (int64 m_sizes) / 1 (int32 inclusive offsets); dynamic 0 (int64
// zero_start_index_M) / 2 (no metadata: every slab full)
mslkb_status run(int layout, const void* A, const void* B, const float* scale_a,
                 const float* scale_b, const void* meta, void* out, int64_t rows, int64_t G,
                 int64_t E, int64_t N, int64_t K, void* stream, int meta_kind = 0,
                 bool block_scale = false) {
  // rows: total_M (stacked) or G * E (dynamic)
  if (rows == 0 || N == 0 || G == 0) return MSLKB_OK;  // nothing is owned or written
  // (block scaling over K = 0 has empty scale arrays: nothing reads them)
  const bool scales_needed = !(block_scale && K == 0);
  if (out == nullptr || (meta == nullptr && meta_kind != 2) ||
      (scales_needed && (scale_a == nullptr || scale_b == nullptr)))
    return MSLKB_ERR_NULL;
  if (K > 0 && (A == nullptr || B == nullptr)) return MSLKB_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(out) % 16 != 0) return MSLKB_ERR_ALIGN;
  if (G * N > MSLKB_MAX_DIM || N * K >= (1ll << 40)) return MSLKB_ERR_SHAPE;

  DeviceState* st = nullptr;
  mslkb_status s = device_state(&st);
  if (s != MSLKB_OK) return s;

  mslkb_plan_info info;
  s = plan(block_scale ? (layout == 0 ? 4 : 5) : layout, layout == 0 ? rows : E, G, N, K,
           st->sm_count,
           addr_align(A), addr_align(B), &info);
  if (s != MSLKB_OK) return s;
  const VariantInfo* v = variant(info.variant);
  if ((s = ensure_attr(st, info.variant)) != MSLKB_OK) return s;

  LaunchArgs la{};  // every parameter zero unless set below
  GemmParams& p = la.params;
  p.A = static_cast<const uint8_t*>(A);
  p.B = static_cast<const uint8_t*>(B);
  p.scale_a = scale_a;
  p.scale_b = scale_b;
  p.meta = static_cast<const int64_t*>(meta);
  p.meta_kind = meta_kind;
  p.out = static_cast<uint16_t*>(out);
  p.status = st->status_ptr;
  p.rows = static_cast<int32_t>(rows);
  p.G = static_cast<int32_t>(G);
  p.N = static_cast<int32_t>(N);
  p.K = static_cast<int32_t>(K);
  p.E = static_cast<int32_t>(E);
  p.num_kb = static_cast<int32_t>(ceil_div(K, mslkb::kBK));
  p.copy_width = info.copy_width;
  {
    const int kpc = g_kb_per_chunk.load();
    p.kb_per_chunk = (kpc <= 0 || kpc > p.num_kb) ? (p.num_kb > 0 ? p.num_kb : 1) : kpc;
    if (block_scale) p.kb_per_chunk = 1;  // every K block scaled on its own
  }
  p.timeout_ns = g_wait_timeout_ns.load();
  p.test_stall = g_test_stall.exchange(0);
  p.prefetch_kb = prefetch_kb_for(v);
  {
    const void* spec = g_test_spec_meta.exchange(nullptr);
    p.spec_meta = static_cast<const int64_t*>(spec != nullptr ? spec : p.meta);
  }
  p.split_k = 0;
  if (info.split_k) {
    Workspace ws;
    if ((s = stream_workspace(st, static_cast<cudaStream_t>(stream), &ws)) != MSLKB_OK) return s;
    if (ws.partials != nullptr) {
      p.split_k = 1;
      p.sk_ws = ws.partials;
      p.sk_cnt = ws.counters;
    }
  }
  // Stacked CTA-pair plans claim their tiles from the stream's counter: groups end at any
  // row, and a group's half-used last tile would otherwise put the pairs that share a
  // weight tile out of step (measured on the llama3-405b shape: 5.3 GB of DRAM reads per
  // call instead of up to 9.6, same time in the back-to-back loop).  Slab layouts keep the
  // fixed stride (full slabs have no half tiles; the claims cost ~2 % there).  In a stream
  // capture that has no workspace yet, tiles go in the fixed stride too: same results.
  p.tile_ctr = nullptr;
  if (v->cluster > 1 && !v->dynamic && p.num_kb > 0) {
    Workspace ws;
    if ((s = stream_workspace(st, static_cast<cudaStream_t>(stream), &ws)) != MSLKB_OK) return s;
    if (ws.counters != nullptr) p.tile_ctr = ws.counters + pair_counter_offset(st);
  }
  if ((s = encode_maps(&la, v, A, B, rows, G, N, K)) != MSLKB_OK) return s;
  gate_weight_pairs(&la, v, info, K);
  if ((s = encode_out_map(&la, v, out, rows, N)) != MSLKB_OK) return s;
  la.grid = dim3(launch_grid(st, info.variant, info.grid), 1, 1);
  la.stream = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_traced(info.variant, la, rows);
  if (e != cudaSuccess) return cuda_fail(e);
  return MSLKB_OK;
}


// Ragged layouts: layout 2 (groups partition N: A [G, M, K], B [total_N, K], out [M, total_N])
// or 3 (groups slice K: A [M, total_K], B [N, total_K], out [G, M, N]).  `n_cols` is the
// output width (total_N or N) and `k_row` the row length of A and B (K or total_K).
mslkb_status run_ragged(int layout, const void* A, const void* B, const float* scale_a,
                        const float* scale_b, const int32_t* offsets, void* out, int64_t G,
                        int64_t M, int64_t n_cols, int64_t k_row, void* stream) {
  if (G < 0 || M < 0 || n_cols < 0 || k_row < 0) return MSLKB_ERR_SHAPE;
  if (G > MSLKB_MAX_GROUPS || n_cols % 8 != 0) return MSLKB_ERR_SHAPE;
  if (n_cols > MSLKB_MAX_DIM || k_row > MSLKB_MAX_DIM || M > MSLKB_MAX_DIM) return MSLKB_ERR_SHAPE;
  const int64_t a_rows = layout == 2 ? G * M : M;
  const int64_t out_rows = layout == 2 ? M : G * M;
  const int64_t b_rows = n_cols;  // total_N (ragged N) or N (ragged K) rows of B
  if (a_rows > MSLKB_MAX_DIM || out_rows > MSLKB_MAX_DIM || out_rows * n_cols >= (1ll << 40) ||
      a_rows * k_row >= (1ll << 40) || b_rows * k_row >= (1ll << 40) || G * M > MSLKB_MAX_DIM ||
      G * n_cols > MSLKB_MAX_DIM)
    return MSLKB_ERR_SHAPE;
  if (M == 0 || G == 0 || n_cols == 0) return MSLKB_OK;  // nothing is owned or written
  if (out == nullptr || offsets == nullptr || scale_a == nullptr || scale_b == nullptr)
    return MSLKB_ERR_NULL;
  if (k_row > 0 && (A == nullptr || B == nullptr)) return MSLKB_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(out) % 16 != 0) return MSLKB_ERR_ALIGN;
  if (k_row % 16 != 0 || addr_align(A) % 16 != 0 || addr_align(B) % 16 != 0)
    return MSLKB_ERR_ALIGN;

  DeviceState* st = nullptr;
  mslkb_status s = device_state(&st);
  if (s != MSLKB_OK) return s;
  mslkb_plan_info info;
  s = plan(layout, M, G, n_cols, k_row, st->sm_count, addr_align(A), addr_align(B), &info);
  if (s != MSLKB_OK) return s;
  const VariantInfo* v = variant(info.variant);
  if ((s = ensure_attr(st, info.variant)) != MSLKB_OK) return s;

  LaunchArgs la{};  // every parameter zero unless set below
  GemmParams& p = la.params;
  p.A = static_cast<const uint8_t*>(A);
  p.B = static_cast<const uint8_t*>(B);
  p.scale_a = scale_a;
  p.scale_b = scale_b;
  p.meta = reinterpret_cast<const int64_t*>(offsets);
  p.meta_kind = 1;  // int32 inclusive offsets
  p.out = static_cast<uint16_t*>(out);
  p.status = st->status_ptr;
  p.rows = static_cast<int32_t>(a_rows);
  p.G = static_cast<int32_t>(G);
  p.N = static_cast<int32_t>(n_cols);
  p.K = static_cast<int32_t>(k_row);
  p.E = static_cast<int32_t>(M);
  p.num_kb = static_cast<int32_t>(ceil_div(k_row, mslkb::kBK));
  p.copy_width = 16;
  {
    const int kpc = g_kb_per_chunk.load();
    p.kb_per_chunk = (kpc <= 0 || kpc > p.num_kb) ? (p.num_kb > 0 ? p.num_kb : 1) : kpc;
  }
  p.timeout_ns = g_wait_timeout_ns.load();
  p.test_stall = g_test_stall.exchange(0);
  g_test_spec_meta.store(nullptr);  // no weight prefetch here: the hook is used up
  p.split_k = 0;
  // A [a_rows, k_row]; B as a one-group [1, b_rows, k_row] map; out [out_rows, n_cols]
  if ((s = encode_maps(&la, v, A, B, a_rows, 1, b_rows, k_row)) != MSLKB_OK) return s;
  if ((s = encode_out_map(&la, v, out, out_rows, n_cols)) != MSLKB_OK) return s;
  la.grid = dim3(launch_grid(st, info.variant, info.grid), 1, 1);
  la.stream = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_traced(info.variant, la, a_rows);
  if (e != cudaSuccess) return cuda_fail(e);
  return MSLKB_OK;
}

}  // namespace

namespace mslkb {

// The checks the stacked entry point makes before any CUDA call (0 = go ahead, else the
// status to return; *nothing_to_do set when the call owns no rows).  Used by the
// allocation-free entry point in mslkb_noalloc.cu.
mslkb_status stacked_precheck(const void* A, const void* B, const float* scale_a,
                              const float* scale_b, const int64_t* m_sizes, void* out,
                              int64_t total_M, int64_t G, int64_t N, int64_t K,
                              bool* nothing_to_do) {
  *nothing_to_do = false;
  mslkb_status s = check_sizes(total_M, G, N, K);
  if (s != MSLKB_OK) return s;
  if (total_M == 0 || N == 0 || G == 0) {
    *nothing_to_do = true;
    return MSLKB_OK;
  }
  if (out == nullptr || m_sizes == nullptr || scale_a == nullptr || scale_b == nullptr)
    return MSLKB_ERR_NULL;
  if (K > 0 && (A == nullptr || B == nullptr)) return MSLKB_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(out) % 16 != 0) return MSLKB_ERR_ALIGN;
  if (G * N > MSLKB_MAX_DIM || N * K >= (1ll << 40)) return MSLKB_ERR_SHAPE;
  return MSLKB_OK;
}

// The stacked call with split-tile scratch supplied by the caller (partial sums and
// arrival counters) instead of the per-stream workspace; allocates nothing.  Returns
// MSLKB_ERR_TOO_LARGE when the plan's split tiles need more scratch than supplied.
// The counters the launch uses are cleared on `stream` before the kernel.
mslkb_status run_stacked_with_scratch(const void* A, const void* B, const float* scale_a,
                                      const float* scale_b, const int64_t* m_sizes, void* out,
                                      int64_t total_M, int64_t G, int64_t N, int64_t K,
                                      void* stream, float* partials, size_t partial_bytes,
                                      uint32_t* counters, size_t counter_count) {
  DeviceState* st = nullptr;
  mslkb_status s = device_state(&st);
  if (s != MSLKB_OK) return s;
  mslkb_plan_info info;
  s = plan(0, total_M, G, N, K, st->sm_count, addr_align(A), addr_align(B), &info);
  if (s != MSLKB_OK) return s;
  const VariantInfo* v = variant(info.variant);
  const size_t need_partials = 2 * static_cast<size_t>(info.grid) * v->partial_bytes;
  const size_t need_counters = 2 * static_cast<size_t>(info.grid) * 8;
  if (info.split_k && (need_partials > partial_bytes || need_counters > counter_count))
    return MSLKB_ERR_TOO_LARGE;
  if ((s = ensure_attr(st, info.variant)) != MSLKB_OK) return s;

  LaunchArgs la{};  // every parameter zero unless set below
  GemmParams& p = la.params;
  p.A = static_cast<const uint8_t*>(A);
  p.B = static_cast<const uint8_t*>(B);
  p.scale_a = scale_a;
  p.scale_b = scale_b;
  p.meta = m_sizes;
  p.out = static_cast<uint16_t*>(out);
  p.status = st->status_ptr;
  p.rows = static_cast<int32_t>(total_M);
  p.G = static_cast<int32_t>(G);
  p.N = static_cast<int32_t>(N);
  p.K = static_cast<int32_t>(K);
  p.E = 0;
  p.num_kb = static_cast<int32_t>(ceil_div(K, mslkb::kBK));
  p.copy_width = info.copy_width;
  {
    const int kpc = g_kb_per_chunk.load();
    p.kb_per_chunk = (kpc <= 0 || kpc > p.num_kb) ? (p.num_kb > 0 ? p.num_kb : 1) : kpc;
  }
  p.timeout_ns = g_wait_timeout_ns.load();
  p.test_stall = g_test_stall.exchange(0);
  p.prefetch_kb = prefetch_kb_for(v);
  {
    const void* spec = g_test_spec_meta.exchange(nullptr);
    p.spec_meta = static_cast<const int64_t*>(spec != nullptr ? spec : p.meta);
  }
  p.split_k = info.split_k;
  p.sk_ws = partials;
  p.sk_cnt = counters;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (info.split_k) {
    cudaError_t e = cudaMemsetAsync(counters, 0, need_counters * sizeof(uint32_t), cs);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if ((s = encode_maps(&la, v, A, B, total_M, G, N, K)) != MSLKB_OK) return s;
  gate_weight_pairs(&la, v, info, K);
  if ((s = encode_out_map(&la, v, out, total_M, N)) != MSLKB_OK) return s;
  la.grid = dim3(launch_grid(st, info.variant, info.grid), 1, 1);
  la.stream = cs;
  cudaError_t e = launch_traced(info.variant, la, total_M);
  if (e != cudaSuccess) return cuda_fail(e);
  return MSLKB_OK;
}

void record_cuda_error(cudaError_t e) { t_last_cuda_error = static_cast<int>(e); }

}  // namespace mslkb

extern "C" {

mslkb_status mslkb_f8f8bf16_rowwise_grouped_stacked(const void* A, const void* B,
                                                    const float* scale_a, const float* scale_b,
                                                    const int64_t* m_sizes, void* out,
                                                    int64_t total_M, int64_t G, int64_t N,
                                                    int64_t K, void* stream) {
  mslkb_status s = check_sizes(total_M, G, N, K);
  if (s != MSLKB_OK) return s;
  return run(0, A, B, scale_a, scale_b, m_sizes, out, total_M, G, 0, N, K, stream);
}

mslkb_status mslkb_f8f8bf16_rowwise_grouped_dynamic(const void* A, const void* B,
                                                    const float* scale_a, const float* scale_b,
                                                    const int64_t* zero_start_index_M, void* out,
                                                    int64_t G, int64_t expected_m, int64_t N,
                                                    int64_t K, void* stream) {
  if (expected_m < 0) return MSLKB_ERR_SHAPE;
  mslkb_status s = check_sizes(0, G, N, K);
  if (s != MSLKB_OK) return s;
  if (expected_m > 0 && G > MSLKB_MAX_DIM / expected_m) return MSLKB_ERR_SHAPE;
  return run(1, A, B, scale_a, scale_b, zero_start_index_M, out, G * expected_m, G, expected_m, N,
             K, stream);
}

mslkb_status mslkb_f8f8bf16_rowwise_grouped_offsets(const void* A, const void* B,
                                                    const float* scale_a, const float* scale_b,
                                                    const int32_t* offsets, void* out,
                                                    int64_t total_M, int64_t G, int64_t N,
                                                    int64_t K, void* stream) {
  mslkb_status s = check_sizes(total_M, G, N, K);
  if (s != MSLKB_OK) return s;
  return run(0, A, B, scale_a, scale_b, offsets, out, total_M, G, 0, N, K, stream, 1);
}

mslkb_status mslkb_f8f8bf16_rowwise_grouped_batched(const void* A, const void* B,
                                                    const float* scale_a, const float* scale_b,
                                                    void* out, int64_t G, int64_t M, int64_t N,
                                                    int64_t K, void* stream) {
  if (M < 0) return MSLKB_ERR_SHAPE;
  mslkb_status s = check_sizes(0, G, N, K);
  if (s != MSLKB_OK) return s;
  if (M > 0 && G > MSLKB_MAX_DIM / M) return MSLKB_ERR_SHAPE;
  return run(1, A, B, scale_a, scale_b, nullptr, out, G * M, G, M, N, K, stream, 2);
}

mslkb_status mslkb_f8f8bf16_groupwise_grouped_stacked(const void* A, const void* B,
                                                      const float* scale_a,
                                                      const float* scale_b,
                                                      const int64_t* m_sizes, void* out,
                                                      int64_t total_M, int64_t G, int64_t N,
                                                      int64_t K, void* stream) {
  mslkb_status s = check_sizes(total_M, G, N, K);
  if (s != MSLKB_OK) return s;
  if (K % 128 != 0 || N % 128 != 0) return MSLKB_ERR_SHAPE;  // whole scale blocks
  if (G * (N / 128) * (K / 128) > MSLKB_MAX_DIM) return MSLKB_ERR_SHAPE;
  return run(0, A, B, scale_a, scale_b, m_sizes, out, total_M, G, 0, N, K, stream, 0, true);
}

mslkb_status mslkb_f8f8bf16_groupwise_grouped_dynamic(const void* A, const void* B,
                                                      const float* scale_a,
                                                      const float* scale_b,
                                                      const int64_t* zero_start_index_M,
                                                      void* out, int64_t G, int64_t expected_m,
                                                      int64_t N, int64_t K, void* stream) {
  if (expected_m < 0) return MSLKB_ERR_SHAPE;
  mslkb_status s = check_sizes(0, G, N, K);
  if (s != MSLKB_OK) return s;
  if (expected_m > 0 && G > MSLKB_MAX_DIM / expected_m) return MSLKB_ERR_SHAPE;
  if (K % 128 != 0 || N % 128 != 0) return MSLKB_ERR_SHAPE;  // whole scale blocks
  if (G * (N / 128) * (K / 128) > MSLKB_MAX_DIM || G * expected_m * (K / 128) > MSLKB_MAX_DIM)
    return MSLKB_ERR_SHAPE;
  return run(1, A, B, scale_a, scale_b, zero_start_index_M, out, G * expected_m, G, expected_m,
             N, K, stream, 0, true);
}

mslkb_status mslkb_f8f8bf16_groupwise_grouped_batched(const void* A, const void* B,
                                                      const float* scale_a,
                                                      const float* scale_b, void* out,
                                                      int64_t G, int64_t M, int64_t N,
                                                      int64_t K, void* stream) {
  if (M < 0) return MSLKB_ERR_SHAPE;
  mslkb_status s = check_sizes(0, G, N, K);
  if (s != MSLKB_OK) return s;
  if (M > 0 && G > MSLKB_MAX_DIM / M) return MSLKB_ERR_SHAPE;
  if (K % 128 != 0 || N % 128 != 0) return MSLKB_ERR_SHAPE;  // whole scale blocks
  if (G * (N / 128) * (K / 128) > MSLKB_MAX_DIM || G * M * (K / 128) > MSLKB_MAX_DIM)
    return MSLKB_ERR_SHAPE;
  return run(1, A, B, scale_a, scale_b, nullptr, out, G * M, G, M, N, K, stream, 2, true);
}

mslkb_status mslkb_f8f8bf16_rowwise_grouped_n_offsets(const void* A, const void* B,
                                                      const float* scale_a,
                                                      const float* scale_b,
                                                      const int32_t* offsets, void* out,
                                                      int64_t G, int64_t M, int64_t total_N,
                                                      int64_t K, void* stream) {
  return run_ragged(2, A, B, scale_a, scale_b, offsets, out, G, M, total_N, K, stream);
}

mslkb_status mslkb_f8f8bf16_rowwise_grouped_k_offsets(const void* A, const void* B,
                                                      const float* scale_a,
                                                      const float* scale_b,
                                                      const int32_t* offsets, void* out,
                                                      int64_t G, int64_t M, int64_t N,
                                                      int64_t total_K, void* stream) {
  return run_ragged(3, A, B, scale_a, scale_b, offsets, out, G, M, N, total_K, stream);
}

const char* mslkb_status_string(mslkb_status status) {
  switch (status) {
    case MSLKB_OK: return "ok";
    case MSLKB_ERR_NULL: return "a required pointer is NULL";
    case MSLKB_ERR_SHAPE: return "unsupported or negative size (N must be a multiple of 8)";
    case MSLKB_ERR_ALIGN:
      return "out must be 16-byte aligned (ragged layouts: A and B too, rows a multiple of 16)";
    case MSLKB_ERR_DEVICE: return "the current device is not sm_103 (GB300)";
    case MSLKB_ERR_CUDA: return "a CUDA call failed (see mslkb_last_cuda_error)";
    case MSLKB_ERR_TOO_LARGE:
      return "the problem needs more split-tile scratch than the allocation-free entry "
             "point holds (MSLKB_NOALLOC_SCRATCH_BYTES)";
  }
  return "unknown status";
}

int mslkb_last_cuda_error(void) { return t_last_cuda_error; }

mslkb_status mslkb_get_device_status(void* stream, uint32_t* flags) {
  if (flags == nullptr) return MSLKB_ERR_NULL;
  DeviceState* st = nullptr;
  mslkb_status s = device_state(&st);
  if (s != MSLKB_OK) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  uint32_t value = 0;
  cudaError_t e = cudaMemcpyAsync(&value, st->status_ptr, sizeof(uint32_t),
                                  cudaMemcpyDeviceToHost, cs);
  if (e == cudaSuccess) e = cudaMemsetAsync(st->status_ptr, 0, sizeof(uint32_t), cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) return cuda_fail(e);
  if (value & mslkb::kStatusTimeout) {
    // a kernel that gave up may have left split-tile arrival counters short: clear the
    // counters of every stream workspace of this device (on `stream`), the CTA pairs' tile
    // claim counter with them (its own reset at teardown also runs on the abort path)
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e);
    const size_t ncnt = pair_counter_offset(st) + 2;
    std::lock_guard<std::mutex> lock(g_mutex);
    for (auto& kv : g_workspaces) {
      if (kv.first.first != dev || kv.second.counters == nullptr) continue;
      e = cudaMemsetAsync(kv.second.counters, 0, ncnt * sizeof(uint32_t), cs);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    if ((e = cudaStreamSynchronize(cs)) != cudaSuccess) return cuda_fail(e);
  }
  *flags = value;
  return MSLKB_OK;
}

mslkb_status mslkb_release_workspace(void* stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const auto key = std::make_pair(dev, reinterpret_cast<uintptr_t>(stream));
  Workspace w;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    auto it = g_workspaces.find(key);
    if (it == g_workspaces.end()) return MSLKB_OK;
    w = it->second;
    g_workspaces.erase(it);
  }
  // the stream's enqueued calls may still use it
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if ((e = cudaStreamSynchronize(cs)) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaFree(w.partials)) != cudaSuccess) return cuda_fail(e);
  if ((e = cudaFree(w.counters)) != cudaSuccess) return cuda_fail(e);
  return MSLKB_OK;
}

int32_t mslkb_workspace_count(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(g_mutex);
  int32_t n = 0;
  for (const auto& kv : g_workspaces)
    if (kv.first.first == dev) ++n;
  return n;
}

mslkb_status mslkb_plan(int32_t layout, int64_t rows, int64_t G, int64_t N, int64_t K,
                        int32_t num_sms, int64_t a_align, int64_t b_align,
                        mslkb_plan_info* info) {
  if (info == nullptr) return MSLKB_ERR_NULL;
  mslkb_status s = check_sizes(layout == 0 ? rows : 0, G, N, K);
  if (s != MSLKB_OK) return s;
  if (a_align <= 0 || b_align <= 0) return MSLKB_ERR_SHAPE;
  return plan(layout, rows, G, N, K, num_sms, a_align, b_align, info);
}

int32_t mslkb_num_variants(void) { return num_variants(); }

const char* mslkb_variant_name(int32_t i) {
  const VariantInfo* v = variant(i);
  return v ? v->name : nullptr;
}

mslkb_status mslkb_force_variant(int32_t i) {
  if (i < -1 || i >= num_variants()) return MSLKB_ERR_SHAPE;
  g_forced_variant.store(i);
  return MSLKB_OK;
}

mslkb_status mslkb_variant_resources(int32_t i, int32_t* blocks_per_sm, int32_t* regs_per_thread) {
  if (blocks_per_sm == nullptr || regs_per_thread == nullptr) return MSLKB_ERR_NULL;
  const VariantInfo* v = variant(i);
  if (v == nullptr) return MSLKB_ERR_SHAPE;
  DeviceState* st = nullptr;
  mslkb_status s = device_state(&st);
  if (s != MSLKB_OK) return s;
  cudaError_t e = v->set_attr();
  if (e != cudaSuccess) return cuda_fail(e);
  int blocks = 0, regs = 0, cluster_ctas = 0;
  e = v->occupancy(&blocks, &regs, &cluster_ctas);
  if (e != cudaSuccess) return cuda_fail(e);
  *blocks_per_sm = blocks;
  *regs_per_thread = regs;
  return MSLKB_OK;
}

mslkb_status mslkb_set_split_k(int32_t enable) {
  if (enable < 0 || enable > 2) return MSLKB_ERR_SHAPE;
  g_split_k.store(enable);
  return MSLKB_OK;
}

mslkb_status mslkb_set_accumulation_chunk(int32_t kblocks) {
  // longer chunks (or the whole K) let the tensor core's round-toward-zero adds run past
  // the tolerance on cancelling sums
  if (kblocks < 1 || kblocks > kMaxKbPerChunk) return MSLKB_ERR_SHAPE;
  g_kb_per_chunk.store(kblocks);
  return MSLKB_OK;
}

int32_t mslkb_accumulation_chunk(void) { return g_kb_per_chunk.load(); }

mslkb_status mslkb_set_weight_prefetch(int32_t kblocks) {
  if (kblocks < -1) return MSLKB_ERR_SHAPE;
  g_prefetch_kb.store(kblocks);
  return MSLKB_OK;
}

mslkb_status mslkb_set_wait_timeout_us(int64_t us) {
  if (us < 0) return MSLKB_ERR_SHAPE;
  if (us > 0 && us < 1000) return MSLKB_ERR_SHAPE;  // at least 1 ms
  g_wait_timeout_ns.store(us == 0 ? kWaitTimeoutNs : static_cast<uint64_t>(us) * 1000ull);
  return MSLKB_OK;
}

mslkb_status mslkb_test_speculate_from_next_launch(const void* meta) {
  g_test_spec_meta.store(meta);
  return MSLKB_OK;
}

mslkb_status mslkb_test_stall_next_launch(void) {
  g_test_stall.store(1);
  return MSLKB_OK;
}

int32_t mslkb_version(void) { return kVersion; }

}  // extern "C"
