// Combine kernel of the split-TOPK path.
//
// Split s of a token covers a contiguous slot range and left, per head, a
// sink-free partial: O_s normalised by its own softmax sum and lse_s over its
// own slots (-inf when the range had no valid slot).  The merge is the
// log-sum-exp identity over disjoint slot sets, with the sink entering the
// denominator once ("Sparse MLA training backward", section "Contract"; the
// sink-inclusive lse of the same page):
//
//   M   = max(max_s lse_s, sink)
//   den = sum_s exp(lse_s - M) + exp(sink - M)
//   O   = sum_s exp(lse_s - M) O_s / den,   lse = M + ln(den)
//
// A row whose M is -inf (no valid slot anywhere, no finite sink) gives O = 0,
// lse = -inf; an empty split has weight exp(-inf) = 0, never NaN.
//
// One warp per (token, head): 32 lanes x d_v/32 columns (16 at d_v = 512: fp32
// partials read as float4, bf16 output written as 2 x 16 bytes per lane).
#include <cuda_runtime.h>

#include <cmath>

#include "smla_device.cuh"
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kRowsPerBlock = 8;

// kDv output columns per row: each lane owns kC = kDv / 32 consecutive columns.
template <int kDv>
__global__ void __launch_bounds__(kRowsPerBlock * 32) combine_kernel(const FwdParams p) {
  // launched as a programmatic dependent of the split kernel: wait until that
  // grid has completed and its partials are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int kC = kDv / 32;
  static_assert(kC % 2 == 0, "pairs of columns per lane");
  const int lane = threadIdx.x & 31;
  const int64_t TH = p.T * p.H;
  const int64_t row = int64_t(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
  if (row >= TH) return;
  const int h = static_cast<int>(row % p.H);

  float M = -INFINITY;
  for (int s = 0; s < p.splits; ++s) M = fmaxf(M, p.part_lse[int64_t(s) * TH + row] * kLog2e);
  float sk = -INFINITY;
  if (p.sink != nullptr) {
    sk = p.sink[h] * kLog2e;
    M = fmaxf(M, sk);
  }
  uint32_t* out = reinterpret_cast<uint32_t*>(static_cast<char*>(p.out) + row * int64_t(kDv * 2)) +
                  lane * (kC / 2);
  float acc[kC];
#pragma unroll
  for (int i = 0; i < kC; ++i) acc[i] = 0.f;
  float den = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < p.splits; ++s) {
      const int64_t prow = int64_t(s) * TH + row;
      const float w = ex2(p.part_lse[prow] * kLog2e - M);
      den += w;
      if (w == 0.f) continue;   // empty split (or negligible): skip its partial
      const float* po = p.part_o + prow * kDv + lane * kC;
      if constexpr (kC % 4 == 0) {
#pragma unroll
        for (int i = 0; i < kC / 4; ++i) {
          const float4 v = reinterpret_cast<const float4*>(po)[i];
          acc[4 * i + 0] += w * v.x; acc[4 * i + 1] += w * v.y;
          acc[4 * i + 2] += w * v.z; acc[4 * i + 3] += w * v.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < kC / 2; ++i) {
          const float2 v = reinterpret_cast<const float2*>(po)[i];
          acc[2 * i] += w * v.x; acc[2 * i + 1] += w * v.y;
        }
      }
    }
    if (p.sink != nullptr) den += ex2(sk - M);
  }
  // a row whose M is -inf (nothing valid, no finite sink): O = 0, lse = -inf
  const float f = (M == -INFINITY) ? 0.f : 1.f / den;
  uint32_t w[kC / 2];
#pragma unroll
  for (int i = 0; i < kC / 2; ++i) w[i] = pack_bf16x2(acc[2 * i] * f, acc[2 * i + 1] * f);
  if constexpr (kC % 8 == 0) {
#pragma unroll
    for (int i = 0; i < kC / 8; ++i)
      reinterpret_cast<uint4*>(out)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  } else if constexpr (kC % 4 == 0) {
#pragma unroll
    for (int i = 0; i < kC / 4; ++i) reinterpret_cast<uint2*>(out)[i] = make_uint2(w[2 * i], w[2 * i + 1]);
  } else {
#pragma unroll
    for (int i = 0; i < kC / 2; ++i) out[i] = w[i];
  }
  if (lane == 0) p.lse[row] = (M == -INFINITY) ? -INFINITY : (M + log2f(den)) * kLn2;
}

template <int kDv>
cudaError_t launch_dv(const FwdParams& p, cudaStream_t stream) {
  const int64_t rows = p.T * p.H;
  const int64_t blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(kRowsPerBlock * 32, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, combine_kernel<kDv>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

// Launched with programmatic stream serialization: its CTAs may be scheduled
// while the split kernel still runs (that kernel signals it at its start) and
// wait in griddepcontrol.wait, so a decode-sized call does not pay a second
// launch latency.
int launch_combine(const FwdParams& p, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (p.d_v) {
    case 512: return static_cast<int>(launch_dv<512>(p, s));
    case 128: return static_cast<int>(launch_dv<128>(p, s));
    case 576: return static_cast<int>(launch_dv<576>(p, s));
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

}  // namespace smla
