// Split-TOPK path backed by a fixed, library-owned scratch array.
//
// The split path needs room for its partial results (per split, token and
// head: 512 fp32 of normalised O and one fp32 lse).  The regular entry point
// allocates that room stream-ordered on every call.  This file instead holds
// it in one file-scope device array, so the allocation-free entry point can
// run the same two kernels (small-head kernel in split mode, then combine)
// without any allocation call.
//
// Facts a caller needs:
//   * the array is kNoAllocScratchRows partial rows (8192 x 2052 bytes,
//     16 MiB); every GPU that loads the library holds it until the process
//     exits;
//   * the first call on a device looks up the array's device address (one
//     cudaGetSymbolAddress per device); make that first call before any
//     stream capture;
//   * all calls share the array; two calls whose kernels overlap on the GPU
//     (different streams, or different host threads) race on it;
//   * nothing in the array has to start at zero: every call writes every
//     partial row it later reads.
#include <cuda_runtime.h>

#include <mutex>

#include "smla_internal.h"

namespace smla {
namespace {

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchRows * (kHeadDim + 1)];

struct ScratchAddr {
  bool ready = false;
  float* ptr = nullptr;
};

constexpr int kMaxDevices = 64;

// Device address of the scratch array on the current device (set up once per device).
cudaError_t scratch_address(float** out) {
  static ScratchAddr addrs[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addrs[dev].ready) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addrs[dev].ptr = static_cast<float*>(p);
    addrs[dev].ready = true;
  }
  *out = addrs[dev].ptr;
  return cudaSuccess;
}

}  // namespace

int launch_split_static_scratch(FwdParams p, void* stream) {
  const int64_t rows = int64_t(p.splits) * p.T * p.H;
  if (p.splits < 2 || rows > kNoAllocScratchRows) return static_cast<int>(cudaErrorInvalidValue);
  float* base = nullptr;
  const cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess) return static_cast<int>(e);
  p.part_o = base;                                // [splits, T, H, 512] fp32
  p.part_lse = base + rows * kHeadDim;            // [splits, T, H] fp32
  int r = launch_smallh(p, stream);
  if (r == 0) r = launch_combine(p, stream);
  return r;
}

}  // namespace smla
