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
//     16,809,984 bytes); every GPU that loads the library holds it until the
//     process exits;
//   * the first call on a device looks up the array's device address (one
//     cudaGetSymbolAddress; under lazy module loading that lookup loads the
//     device code and maps the array), so make that first call outside any
//     window in which no allocation may happen;
//   * the address is cached per device together with the id of the context it
//     was taken in; after a device reset the context id changes and the next
//     call looks the address up again instead of using a stale one;
//   * all calls share the array; two calls whose kernels overlap on the GPU
//     (different streams, or different host threads) race on it;
//   * nothing in the array has to start at zero: every call writes every
//     partial row it later reads.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "smla_internal.h"

namespace smla {
namespace {

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchRows * (kHeadDim + 1)];

struct ScratchAddr {
  bool ready = false;
  unsigned long long ctx_id = 0;   // the context the address belongs to
  float* ptr = nullptr;
};

constexpr int kMaxDevices = 64;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the current context (driver entry points looked up once);
// 0 when it cannot be read.
unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array on the current device: looked up on the
// first call and again whenever the device's context has changed (a reset).
cudaError_t scratch_address(float** out) {
  static ScratchAddr addrs[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  ScratchAddr& a = addrs[dev];
  // 0 before the runtime has made the device's context current (the lookup below does)
  const unsigned long long id = current_ctx_id();
  if (!a.ready || id == 0 || a.ctx_id != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    a.ptr = static_cast<float*>(p);
    a.ctx_id = current_ctx_id();   // the context the address was taken in
    a.ready = true;
  }
  *out = a.ptr;
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
