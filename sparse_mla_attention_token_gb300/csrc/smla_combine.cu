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
// One warp per (token, head): 32 lanes x 16 columns, fp32 partials read as
// float4, bf16 output written as 2 x 16 bytes per lane.
#include <cuda_runtime.h>

#include <cmath>

#include "smla_device.cuh"
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kRowsPerBlock = 8;

__global__ void __launch_bounds__(kRowsPerBlock * 32) combine_kernel(const FwdParams p) {
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
  uint4* out = reinterpret_cast<uint4*>(static_cast<char*>(p.out) + row * int64_t(kHeadDim * 2));
  if (M == -INFINITY) {
    out[2 * lane] = make_uint4(0u, 0u, 0u, 0u);
    out[2 * lane + 1] = make_uint4(0u, 0u, 0u, 0u);
    if (lane == 0) p.lse[row] = -INFINITY;
    return;
  }
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  float den = 0.f;
  for (int s = 0; s < p.splits; ++s) {
    const int64_t prow = int64_t(s) * TH + row;
    const float w = ex2(p.part_lse[prow] * kLog2e - M);
    den += w;
    if (w == 0.f) continue;   // empty split (or negligible): skip its partial
    const float4* po = reinterpret_cast<const float4*>(p.part_o + prow * kHeadDim) + lane * 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 v = po[i];
      acc[4 * i + 0] += w * v.x; acc[4 * i + 1] += w * v.y;
      acc[4 * i + 2] += w * v.z; acc[4 * i + 3] += w * v.w;
    }
  }
  if (p.sink != nullptr) den += ex2(sk - M);
  const float f = 1.f / den;
  uint4 o0, o1;
  o0.x = pack_bf16x2(acc[0] * f, acc[1] * f);   o0.y = pack_bf16x2(acc[2] * f, acc[3] * f);
  o0.z = pack_bf16x2(acc[4] * f, acc[5] * f);   o0.w = pack_bf16x2(acc[6] * f, acc[7] * f);
  o1.x = pack_bf16x2(acc[8] * f, acc[9] * f);   o1.y = pack_bf16x2(acc[10] * f, acc[11] * f);
  o1.z = pack_bf16x2(acc[12] * f, acc[13] * f); o1.w = pack_bf16x2(acc[14] * f, acc[15] * f);
  out[2 * lane] = o0;
  out[2 * lane + 1] = o1;
  if (lane == 0) p.lse[row] = (M + log2f(den)) * kLn2;
}

}  // namespace

int launch_combine(const FwdParams& p, void* stream) {
  const int64_t rows = p.T * p.H;
  const int64_t blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  combine_kernel<<<static_cast<unsigned>(blocks), kRowsPerBlock * 32, 0,
                   static_cast<cudaStream_t>(stream)>>>(p);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace smla
