// mslkb_noalloc.cu -- the allocation-free stacked entry point.
//
// Some callers cannot allocate device memory when they call this library: plug-ins whose
// host framework owns all device memory, and serving loops that cannot take the
// device-wide synchronisation a cudaMalloc can bring.  This entry point runs the same
// stacked kernels, but the split tiles' scratch lives in one static device array instead
// of a workspace the library allocates per stream; nothing here allocates.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "launch.h"
#include "mslkb.h"

namespace {

constexpr size_t kScratchBytes = MSLKB_NOALLOC_SCRATCH_BYTES;
// arrival counters first (up to 256 CTAs x 2 slots x 8 epilogue warps), then partial sums
constexpr size_t kCounterCount = 256 * 2 * 8;
constexpr size_t kCounterBytes = kCounterCount * sizeof(uint32_t);
static_assert(kCounterBytes % 256 == 0, "partial sums stay 256-byte aligned");

// Every GPU that loads the library holds this array until the process exits.  In host
// code its name is only a stand-in for the device copy: the address a kernel needs comes
// from cudaGetSymbolAddress below, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned char* g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device (looked up on the first call there).
mslkb_status scratch_on_current_device(unsigned char** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    mslkb::record_cuda_error(e);
    return MSLKB_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return MSLKB_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      mslkb::record_cuda_error(e);
      return MSLKB_ERR_CUDA;
    }
    g_scratch_addr[dev] = static_cast<unsigned char*>(p);
  }
  *addr = g_scratch_addr[dev];
  return MSLKB_OK;
}

}  // namespace

extern "C" mslkb_status mslkb_f8f8bf16_rowwise_grouped_stacked_noalloc(
    const void* A, const void* B, const float* scale_a, const float* scale_b,
    const int64_t* m_sizes, void* out, int64_t total_M, int64_t G, int64_t N, int64_t K,
    void* stream) {
  bool nothing = false;
  mslkb_status s = mslkb::stacked_precheck(A, B, scale_a, scale_b, m_sizes, out, total_M, G,
                                           N, K, &nothing);
  if (s != MSLKB_OK || nothing) return s;
  unsigned char* base = nullptr;
  if ((s = scratch_on_current_device(&base)) != MSLKB_OK) return s;
  uint32_t* counters = reinterpret_cast<uint32_t*>(base);
  float* partials = reinterpret_cast<float*>(base + kCounterBytes);
  return mslkb::run_stacked_with_scratch(A, B, scale_a, scale_b, m_sizes, out, total_M, G, N,
                                         K, stream, partials, kScratchBytes - kCounterBytes,
                                         counters, kCounterCount);
}
