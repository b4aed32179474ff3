// Training backward of the sparse MLA attention ("Sparse MLA training
// backward", aiter PR #4766, sections "Contract" and "Structure").
//
// Given the forward's inputs, its bf16 output O, its sink-inclusive lse and
// the output gradient dO, the backward produces dq, dkv and the sink gradient
// in the page's five steps plus the sink reduction:
//
//   1. delta[t,h] = <O[t,h,:], dO[t,h,:]>                     (bwd_delta_kernel)
//   2. per token and 16-head group, over 32-slot tiles of the gathered rows:
//      S = Q.K^T and dP = dO.V^T from one gathered tile (K == V), the exact
//      probabilities P = exp(scale S - lse) from the saved lse, the scaled
//      score gradient dS' = scale P (dP - delta), dq += dS'.K; P and dS' are
//      written out per compacted slot for step 3              (bwd_dq_kernel;
//      at H = 128, dq = dS'.K is the tcgen05 GEMM of smla_bwd_tc.cu)
//   3. the per-(token, slot) row "interm" = P^T dO + dS'^T Q, a contraction
//      over the heads (bwd_interm_kernel; at H = 128 the tcgen05 kernel of
//      smla_bwd_tc.cu)
//   4. an inverted index: the (token, slot) entries of every kv row
//      (histogram, exclusive scan, fill)                       (bwd_csr_*)
//   5. dkv[r] = sum of the interm rows of r's entries: a gather, no atomics
//      on the data                                             (bwd_gather_kernel)
//   6. dsink[h] = -sum_t exp(sink[h] - lse[t,h]) delta[t,h]    (bwd_dsink_kernel)
//
// Every contraction uses warp-level mma.sync m16n8k16 (bf16 in, fp32 out).
// dq, dkv and dsink are fp32; the per-slot interm rows are bf16 (as the page's
// T * topk * 512 bf16 intermediate) and are summed in fp32 by the gather.  The order in which a row's entries are summed
// in step 5 follows the fill order of step 4 (atomic), so dkv can differ in
// its last bits between calls; everything else is deterministic.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "smla_device.cuh"
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kHG = 16;            // heads per CTA of the dq kernel (mma M)
constexpr int kBN = 32;            // gathered rows per tile
constexpr int kRowBytes = kHeadDim * 2;

__device__ __forceinline__ uint32_t kv_chunk_addr(uint32_t base, int r, int c) {
  return base + r * kRowBytes + ((c ^ (r & 7)) << 4);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ------------------------------------------------------------------ 1. delta
// One warp per (token, head) row: 32 lanes x 16 elements of O and dO.
__global__ void __launch_bounds__(256) bwd_delta_kernel(const BwdParams p) {
  const int64_t row = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= p.T * p.H) return;
  const uint4* o = reinterpret_cast<const uint4*>(static_cast<const char*>(p.out) + row * kRowBytes);
  const uint4* g = reinterpret_cast<const uint4*>(static_cast<const char*>(p.dout) + row * kRowBytes);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 a = o[2 * lane + i], b = g[2 * lane + i];
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
      acc += bf16_lo(aw[k]) * bf16_lo(bw[k]) + bf16_hi(aw[k]) * bf16_hi(bw[k]);
  }
#pragma unroll
  for (int o2 = 16; o2 >= 1; o2 >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o2);
  if (lane == 0) p.delta[row] = acc;
}

// ------------------------------------------------------------------ compaction (H = 128)
// One CTA per token: the valid slots' rows in slot order (full-width check),
// for the tcgen05 kernels that follow.
template <typename IdxT>
__global__ void __launch_bounds__(kThreads) bwd_compact_kernel(const BwdParams p) {
  __shared__ int warp_cnt[kWarps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t t = blockIdx.x;
  const IdxT* idx = static_cast<const IdxT*>(p.idx) + t * p.topk;
  int* out = p.crow + t * p.topk;
  int nv = 0;
  for (int base = 0; base < p.topk; base += kThreads) {
    const int j = base + tid;
    bool v = false;
    int row = -1;
    if (j < p.topk) {
      const IdxT x = idx[j];
      v = slot_valid<IdxT>(x, p.num_kv);
      if (v) row = static_cast<int>(x);   // exact: num_kv < 2^31
    }
    const unsigned ball = __ballot_sync(0xffffffffu, v);
    if (lane == 0) warp_cnt[warp] = __popc(ball);
    __syncthreads();
    int off = nv, total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int c = warp_cnt[w];
      off += (w < warp) ? c : 0;
      total += c;
    }
    if (v) out[off + __popc(ball & ((1u << lane) - 1u))] = row;
    nv += total;
    __syncthreads();
  }
  if (tid == 0) p.ncnt[t] = nv;
}

// ------------------------------------------------------------------ 2. dq, P, dS'
struct __align__(128) DqSmem {
  static constexpr int kRedStride = kBN + 8;   // floats per row of a warp's partials
  static constexpr int kDsStride = kBN + 8;    // bf16 per row of dS' (bank spread for ldmatrix)
  __nv_bfloat16 kv[2][kBN * kHeadDim];         // 2 stages; 16 B chunk c of row r at c ^ (r & 7)
  float red[kWarps][kHG * kRedStride];         // per-warp partials: S, then dP
  __nv_bfloat16 ds[kHG * kDsStride];           // dS' of the tile: A operand of dq += dS'.K
  __nv_bfloat16 pt[kHG * kDsStride];           // P of the tile (staged for its global store)
  float lse2[kHG];                             // lse * log2(e) per head (+inf for pad rows)
  float delta[kHG];
  int rows[kSmallHMaxSlots];                   // compacted valid kv rows, slot order
  int warp_cnt[kWarps];
};

// Two CTAs per SM (at most 128 registers, ~97 KB of shared memory each), so
// that one CTA's barriers overlap the other's contractions.  kDq = false (H =
// 128): only S, dP, P and dS' -- dq then comes from the tcgen05 GEMM of
// smla_bwd_tc.cu.
template <typename IdxT, bool kDq>
__global__ void __launch_bounds__(kThreads, 2) bwd_dq_kernel(const BwdParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  DqSmem& sm = *reinterpret_cast<DqSmem*>(smem_raw);
  constexpr int kRS = DqSmem::kRedStride, kDS = DqSmem::kDsStride;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tig = lane & 3;
  const int64_t t = blockIdx.x;
  const int hg = blockIdx.y;
  const int H = p.H, h0 = hg * kHG, hvalid = min(kHG, H - h0);

  // Q and dO fragments of this warp's 64 columns (rows = the group's heads)
  uint32_t qa[4][4], da[4][4];
  {
    const uint32_t* q32 = static_cast<const uint32_t*>(p.q);
    const uint32_t* d32 = static_cast<const uint32_t*>(p.dout);
    const int64_t rbase = (t * H + h0) * kHeadDim;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const int d = warp * 64 + kk * 16 + 2 * tig;
      const bool lo = g < hvalid, hi = (g + 8) < hvalid;
      const int64_t i0 = (rbase + int64_t(g) * kHeadDim + d) >> 1;
      const int64_t i1 = (rbase + int64_t(g + 8) * kHeadDim + d) >> 1;
      qa[kk][0] = lo ? q32[i0] : 0u;
      qa[kk][1] = hi ? q32[i1] : 0u;
      qa[kk][2] = lo ? q32[i0 + 4] : 0u;
      qa[kk][3] = hi ? q32[i1 + 4] : 0u;
      da[kk][0] = lo ? d32[i0] : 0u;
      da[kk][1] = hi ? d32[i1] : 0u;
      da[kk][2] = lo ? d32[i0 + 4] : 0u;
      da[kk][3] = hi ? d32[i1 + 4] : 0u;
    }
  }
  if (tid < kHG) {
    const bool live = tid < hvalid;
    sm.lse2[tid] = live ? p.lse[t * H + h0 + tid] * kLog2e : INFINITY;   // pad rows: P = 0
    sm.delta[tid] = live ? p.delta[t * H + h0 + tid] : 0.f;
  }

  // classify the token's slots at full width and compact the valid rows (slot order)
  const IdxT* idx = static_cast<const IdxT*>(p.idx) + t * p.topk;
  int nv = 0;
  for (int base = 0; base < p.topk; base += kThreads) {
    const int j = base + tid;
    bool v = false;
    int row = -1;
    if (j < p.topk) {
      const IdxT x = idx[j];
      v = slot_valid<IdxT>(x, p.num_kv);
      if (v) row = static_cast<int>(x);   // exact: num_kv < 2^31
    }
    const unsigned ball = __ballot_sync(0xffffffffu, v);
    if (lane == 0) sm.warp_cnt[warp] = __popc(ball);
    __syncthreads();
    int off = nv, total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int c = sm.warp_cnt[w];
      off += (w < warp) ? c : 0;
      total += c;
    }
    if (v) sm.rows[off + __popc(ball & ((1u << lane) - 1u))] = row;
    nv += total;
    __syncthreads();
  }
  if (hg == 0) {   // the compacted list, for the inverted index
    for (int k = tid; k < nv; k += kThreads) p.crow[t * p.topk + k] = sm.rows[k];
    if (tid == 0) p.ncnt[t] = nv;
  }

  const char* kvb = static_cast<const char*>(p.kv);
  auto issue_tile = [&](int tile, int stage) {
    const uint32_t dst0 = smem_u32(sm.kv[stage]);
#pragma unroll 4
    for (int i = tid; i < kBN * 64; i += kThreads) {
      const int r = i >> 6, c = i & 63;
      const int slot = tile * kBN + r;
      const bool ok = slot < nv;
      const char* src = ok ? kvb + int64_t(sm.rows[slot]) * kRowBytes + c * 16 : kvb;
      cp_async_16(kv_chunk_addr(dst0, r, c), src, ok ? 16u : 0u);   // tail zero-filled
    }
    cp_async_commit();
  };

  const float sl2 = p.scale * kLog2e;
  const int srow = 2 * warp + (lane >> 4);   // row of the reduction owned by this half-warp
  const int sc0 = (lane & 15) * 2;           // its 2 columns
  const int two_h = 2 * H;
  __nv_bfloat16* pds = static_cast<__nv_bfloat16*>(p.pds);
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  const int ntiles = (nv + kBN - 1) / kBN;
  if (ntiles > 0) issue_tile(0, 0);
  for (int it = 0; it < ntiles; ++it) {
    const int stage = it & 1;
    cp_async_wait<0>();
    __syncthreads();   // tile it landed; every warp is done with the other stage
    if (it + 1 < ntiles) issue_tile(it + 1, stage ^ 1);
    const uint32_t kvs = smem_u32(sm.kv[stage]);
    // partial S and dP over this warp's 64 columns
    float s[4][4], dp[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      s[i][0] = s[i][1] = s[i][2] = s[i][3] = dp[i][0] = dp[i][1] = dp[i][2] = dp[i][3] = 0.f;
#pragma unroll
    for (int kp = 0; kp < 2; ++kp) {
      const int c = warp * 8 + kp * 4 + (lane >> 3);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int r = nt * 8 + (lane & 7);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(kv_chunk_addr(kvs, r, c), b0, b1, b2, b3);
        mma_16816(s[nt], qa[2 * kp], b0, b1);
        mma_16816(s[nt], qa[2 * kp + 1], b2, b3);
        mma_16816(dp[nt], da[2 * kp], b0, b1);
        mma_16816(dp[nt], da[2 * kp + 1], b2, b3);
      }
    }
    // the 8 partials of S, then of dP, through one reduction buffer
    float a[2], b[2];
    {
      float* rw = sm.red[warp];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int c0 = nt * 8 + 2 * tig;
        *reinterpret_cast<float2*>(&rw[g * kRS + c0]) = make_float2(s[nt][0], s[nt][1]);
        *reinterpret_cast<float2*>(&rw[(g + 8) * kRS + c0]) = make_float2(s[nt][2], s[nt][3]);
      }
      __syncthreads();
      a[0] = a[1] = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float2 u = *reinterpret_cast<const float2*>(&sm.red[w][srow * kRS + sc0]);
        a[0] += u.x; a[1] += u.y;
      }
      __syncthreads();
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int c0 = nt * 8 + 2 * tig;
        *reinterpret_cast<float2*>(&rw[g * kRS + c0]) = make_float2(dp[nt][0], dp[nt][1]);
        *reinterpret_cast<float2*>(&rw[(g + 8) * kRS + c0]) = make_float2(dp[nt][2], dp[nt][3]);
      }
      __syncthreads();
      b[0] = b[1] = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float2 v = *reinterpret_cast<const float2*>(&sm.red[w][srow * kRS + sc0]);
        b[0] += v.x; b[1] += v.y;
      }
    }
    // P = 2^(S sl2 - lse2), dS' = scale P (dP - delta)
    {
      const float l2 = sm.lse2[srow], dl = sm.delta[srow];
      float pr[2], dsv[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int col = it * kBN + sc0 + k;
        pr[k] = (col < nv) ? ex2(a[k] * sl2 - l2) : 0.f;
        dsv[k] = p.scale * pr[k] * (b[k] - dl);
      }
      *reinterpret_cast<uint32_t*>(&sm.ds[srow * kDS + sc0]) = pack_bf16x2(dsv[0], dsv[1]);
      *reinterpret_cast<uint32_t*>(&sm.pt[srow * kDS + sc0]) = pack_bf16x2(pr[0], pr[1]);
    }
    __syncthreads();
    // P and dS' of the tile's valid slots to [t, slot, P heads | dS' heads]: one
    // 16-byte store per (slot, P or dS', 8 heads)
    if (tid < kBN * 4) {
      const int col = tid >> 2, kind = (tid >> 1) & 1, half = tid & 1;
      const int slot = it * kBN + col;
      if (slot < nv && half * 8 < hvalid) {
        const __nv_bfloat16* src = (kind ? sm.ds : sm.pt) + half * 8 * kDS + col;
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          w[i] = uint32_t(__bfloat16_as_ushort(src[(2 * i) * kDS])) |
                 (uint32_t(__bfloat16_as_ushort(src[(2 * i + 1) * kDS])) << 16);
        __nv_bfloat16* e = pds + (t * p.topk + slot) * int64_t(two_h) + kind * H + h0 + half * 8;
        *reinterpret_cast<uint4*>(e) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    // dq += dS'.K over this warp's 64 columns
    if constexpr (kDq) {
      const uint32_t ds_base = smem_u32(sm.ds);
#pragma unroll
      for (int ks = 0; ks < kBN / 16; ++ks) {
        uint32_t pa[4];
        const int pr_ = ((lane >> 3) & 1) * 8 + (lane & 7);
        const int pc = ks * 16 + (lane >> 4) * 8;
        ldmatrix_x4(ds_base + (pr_ * kDS + pc) * 2, pa[0], pa[1], pa[2], pa[3]);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          const int j = lane >> 3;
          const int r = ks * 16 + (j & 1) * 8 + (lane & 7);
          const int c = warp * 8 + np * 2 + (j >> 1);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4_trans(kv_chunk_addr(kvs, r, c), b0, b1, b2, b3);
          mma_16816(acc[2 * np], pa, b0, b1);
          mma_16816(acc[2 * np + 1], pa, b2, b3);
        }
      }
    }
  }
  cp_async_wait<0>();
  if constexpr (!kDq) return;
  // dq rows of the group (fp32)
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = g + half * 8;
    if (r >= hvalid) continue;
    float* dq = p.dq + (t * H + h0 + r) * int64_t(kHeadDim) + warp * 64 + 2 * tig;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
      *reinterpret_cast<float2*>(dq + nt * 8) = make_float2(acc[nt][2 * half], acc[nt][2 * half + 1]);
  }
}

// ------------------------------------------------------------------ 3. interm
// interm[t, k, :] = [P | dS'](t, k, :) . [dO; Q](t)  (K = 2H, contracted over heads).
// CTA = (token, 128-column chunk); 8 warps each own 16 of the chunk's columns
// and walk the token's compacted slots in 64-slot M tiles.
constexpr int kIChunk = 128;    // output columns per CTA
constexpr int kIM = 64;         // slots per M tile

template <int kH>
struct IntermSmem {
  static constexpr int kK = 2 * kH;               // contraction length
  static constexpr int kBStride = kIChunk + 8;     // bf16 per B row (bank spread)
  static constexpr int kAStride = kK + 8;          // bf16 per A row (bank spread)
  __nv_bfloat16 b[kK * kBStride];                  // [dO; Q] rows, this CTA's columns
  __nv_bfloat16 a[kIM * kAStride];                 // [P | dS'] of 64 slots
};

template <int kH>
__global__ void __launch_bounds__(kThreads, 2) bwd_interm_kernel(const BwdParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  using Sm = IntermSmem<kH>;
  Sm& sm = *reinterpret_cast<Sm*>(smem_raw);
  constexpr int kK = Sm::kK, kBS = Sm::kBStride, kAS = Sm::kAStride;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tig = lane & 3;
  // blockIdx.x = token * 4 + chunk: a token's four column chunks run together,
  // so its [P | dS'] rows are read from L2 by three of them
  const int64_t t = blockIdx.x / (kHeadDim / kIChunk);
  const int col0 = static_cast<int>(blockIdx.x % (kHeadDim / kIChunk)) * kIChunk;
  const int nv = p.ncnt[t];
  if (nv == 0) return;

  // B = [dO; Q] restricted to the chunk's columns: 2H rows x 128 bf16 (256 B, 16 chunks)
  {
    const char* dob = static_cast<const char*>(p.dout) + t * kH * int64_t(kRowBytes) + col0 * 2;
    const char* qb = static_cast<const char*>(p.q) + t * kH * int64_t(kRowBytes) + col0 * 2;
    for (int i = tid; i < kK * 16; i += kThreads) {
      const int r = i >> 4, c = i & 15;
      const char* src = (r < kH ? dob + int64_t(r) * kRowBytes : qb + int64_t(r - kH) * kRowBytes) +
                        c * 16;
      cp_async_16(smem_u32(&sm.b[r * kBS + c * 8]), src, 16u);
    }
    cp_async_commit();
  }
  const __nv_bfloat16* pds = static_cast<const __nv_bfloat16*>(p.pds) + t * p.topk * int64_t(kK);
  __nv_bfloat16* interm =
      static_cast<__nv_bfloat16*>(p.interm) + t * p.topk * int64_t(kHeadDim) + col0 + warp * 16;
  constexpr int kAChunks = kK / 8;   // 16-byte chunks per A row
  for (int m0 = 0; m0 < nv; m0 += kIM) {
    __syncthreads();   // the previous tile's A is no longer read
    for (int i = tid; i < kIM * kAChunks; i += kThreads) {
      const int r = i / kAChunks, c = i % kAChunks;
      const bool ok = m0 + r < nv;
      const __nv_bfloat16* src = ok ? pds + int64_t(m0 + r) * kK + c * 8 : pds;
      cp_async_16(smem_u32(&sm.a[r * kAS + c * 8]), src, ok ? 16u : 0u);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    float acc[4][2][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int n = 0; n < 2; ++n) acc[i][n][0] = acc[i][n][1] = acc[i][n][2] = acc[i][n][3] = 0.f;
#pragma unroll 4
    for (int ks = 0; ks < kK / 16; ++ks) {
      uint32_t b0, b1, b2, b3;   // B fragments: k rows ks*16.., columns warp*16 .. +15
      {
        const int j = lane >> 3;
        const int r = ks * 16 + (j & 1) * 8 + (lane & 7);
        const int c = warp * 16 + (j >> 1) * 8;
        ldmatrix_x4_trans(smem_u32(&sm.b[r * kBS + c]), b0, b1, b2, b3);
      }
#pragma unroll
      for (int mi = 0; mi < 4; ++mi) {
        uint32_t a[4];
        const int r = mi * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
        const int c = ks * 16 + (lane >> 4) * 8;
        ldmatrix_x4(smem_u32(&sm.a[r * kAS + c]), a[0], a[1], a[2], a[3]);
        mma_16816(acc[mi][0], a, b0, b1);
        mma_16816(acc[mi][1], a, b2, b3);
      }
    }
#pragma unroll
    for (int mi = 0; mi < 4; ++mi) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int k = m0 + mi * 16 + g + half * 8;
        if (k >= nv) continue;
        __nv_bfloat16* dst = interm + int64_t(k) * kHeadDim + 2 * tig;
#pragma unroll
        for (int n = 0; n < 2; ++n)
          *reinterpret_cast<uint32_t*>(dst + n * 8) =
              pack_bf16x2(acc[mi][n][2 * half], acc[mi][n][2 * half + 1]);
      }
    }
  }
}

// ------------------------------------------------------------------ 4. inverted index
__global__ void bwd_csr_count_kernel(const BwdParams p) {
  const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= p.T * p.topk) return;
  const int64_t t = e / p.topk;
  const int k = static_cast<int>(e - t * p.topk);
  if (k < p.ncnt[t]) atomicAdd(&p.row_cnt[p.crow[e]], 1);
}

constexpr int kScanBlock = 1024;

// Exclusive scan of row_cnt[0..n) into row_cnt itself, in blocks of 1024;
// each block's total goes to blk[b].
__global__ void __launch_bounds__(kScanBlock) bwd_scan_blocks_kernel(int* v, int64_t n, int* blk) {
  __shared__ int warp_sum[32];
  const int64_t i = int64_t(blockIdx.x) * kScanBlock + threadIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int x = i < n ? v[i] : 0;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sum[lane] = w;   // inclusive over warps
  }
  __syncthreads();
  const int before = warp == 0 ? 0 : warp_sum[warp - 1];
  if (i < n) v[i] = before + incl - x;
  if (threadIdx.x == kScanBlock - 1) blk[blockIdx.x] = before + incl;
}

// Exclusive scan of the block totals (one CTA, serial over chunks of 1024).
__global__ void __launch_bounds__(kScanBlock) bwd_scan_totals_kernel(int* blk, int nblk) {
  __shared__ int warp_sum[32];
  __shared__ int carry;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < nblk; base += kScanBlock) {
    const int i = base + threadIdx.x;
    const int x = i < nblk ? blk[i] : 0;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = warp_sum[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_sum[lane] = w;
    }
    __syncthreads();
    const int before = (warp == 0 ? 0 : warp_sum[warp - 1]) + carry;
    if (i < nblk) blk[i] = before + incl - x;
    __syncthreads();
    if (threadIdx.x == kScanBlock - 1) carry = before + incl;
    __syncthreads();
  }
}

__global__ void bwd_scan_add_kernel(int* v, int64_t n, const int* blk) {
  const int64_t i = int64_t(blockIdx.x) * kScanBlock + threadIdx.x;
  if (i < n) v[i] += blk[blockIdx.x];
}

__global__ void bwd_csr_fill_kernel(const BwdParams p) {
  const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= p.T * p.topk) return;
  const int64_t t = e / p.topk;
  const int k = static_cast<int>(e - t * p.topk);
  if (k >= p.ncnt[t]) return;
  const int r = p.crow[e];
  const int pos = atomicAdd(&p.row_cur[r], 1);
  p.list[p.row_cnt[r] + pos] = static_cast<int>(e);
}

// ------------------------------------------------------------------ 5. dkv gather
// One CTA of 128 threads per kv row: 4 columns each (one 8-byte load of bf16
// per entry), fp32 sums of the row's interm entries in list order.  Entries go
// 16 at a time, and the next 16 list entries are loaded while the current rows
// are summed, so a long row (a pool row named by many tokens) keeps 16 rows and
// the next index chunk in flight instead of paying two latencies per chunk.
__global__ void __launch_bounds__(128) bwd_gather_kernel(const BwdParams p) {
  constexpr int kU = 16;
  const int64_t r = blockIdx.x;
  const int b = p.row_cnt[r], e_end = p.row_cnt[r + 1];
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const uint2* src = reinterpret_cast<const uint2*>(p.interm) + threadIdx.x;
  auto add = [&](uint2 v) {
    acc.x += bf16_lo(v.x); acc.y += bf16_hi(v.x); acc.z += bf16_lo(v.y); acc.w += bf16_hi(v.y);
  };
  int i = b;
  int nx[kU];
  if (i + kU <= e_end) {
#pragma unroll
    for (int u = 0; u < kU; ++u) nx[u] = p.list[i + u];
  }
  for (; i + kU <= e_end; i += kU) {
    uint2 v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) v[u] = src[int64_t(nx[u]) * (kHeadDim / 4)];
    if (i + 2 * kU <= e_end) {
#pragma unroll
      for (int u = 0; u < kU; ++u) nx[u] = p.list[i + kU + u];
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) add(v[u]);
  }
  for (; i < e_end; ++i) add(src[int64_t(p.list[i]) * (kHeadDim / 4)]);
  reinterpret_cast<float4*>(p.dkv + r * kHeadDim)[threadIdx.x] = acc;
}

// ------------------------------------------------------------------ 6. dsink
// One CTA per head: dsink[h] = -sum_t exp(sink[h] - lse[t,h]) delta[t,h].
__global__ void __launch_bounds__(256) bwd_dsink_kernel(const BwdParams p) {
  __shared__ float part[8];
  const int h = blockIdx.x;
  const float sk = p.sink[h] * kLog2e;
  float acc = 0.f;
  for (int64_t t = threadIdx.x; t < p.T; t += 256) {
    const float l = p.lse[t * p.H + h];
    if (l != -INFINITY) acc += ex2(sk - l * kLog2e) * p.delta[t * p.H + h];
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < 8; ++w) s += part[w];
    p.dsink[h] = (sk == -INFINITY) ? 0.f : -s;
  }
}

template <typename IdxT, bool kDq>
cudaError_t launch_dq(const BwdParams& p, cudaStream_t s) {
  auto kern = bwd_dq_kernel<IdxT, kDq>;
  const int smem = static_cast<int>(sizeof(DqSmem)) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(p.T), static_cast<unsigned>((p.H + kHG - 1) / kHG));
  kern<<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <int kH>
cudaError_t launch_interm(const BwdParams& p, cudaStream_t s) {
  auto kern = bwd_interm_kernel<kH>;
  const int smem = static_cast<int>(sizeof(IntermSmem<kH>)) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(p.T * (kHeadDim / kIChunk)));
  kern<<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

BwdWorkspace bwd_workspace_layout(int64_t T, int32_t H, int32_t topk, int64_t num_kv) {
  auto up = [](uint64_t x) { return (x + 255) & ~uint64_t(255); };
  BwdWorkspace w{};
  uint64_t o = 0;
  const uint64_t e = uint64_t(T) * uint64_t(topk);
  w.delta = o;   o += up(uint64_t(T) * H * 4);
  w.pds = o;     o += up(e * 2 * H * 2);
  w.crow = o;    o += up(e * 4);
  w.ncnt = o;    o += up(uint64_t(T) * 4);
  w.interm = o;  o += up(e * kHeadDim * 2);
  w.row_cnt = o; o += up((uint64_t(num_kv) + 1) * 4);
  w.row_cur = o; o += up(uint64_t(num_kv) * 4);
  w.blk = o;     o += up((uint64_t(num_kv) + 1 + kScanBlock) / kScanBlock * 4 + 4);
  w.list = o;    o += up(e * 4);
  w.total = o;
  return w;
}

int launch_bwd(BwdParams p, void* workspace, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const BwdWorkspace w = bwd_workspace_layout(p.T, p.H, p.topk, p.num_kv);
  char* ws = static_cast<char*>(workspace);
  p.delta = reinterpret_cast<float*>(ws + w.delta);
  p.pds = ws + w.pds;
  p.crow = reinterpret_cast<int*>(ws + w.crow);
  p.ncnt = reinterpret_cast<int*>(ws + w.ncnt);
  p.interm = ws + w.interm;
  p.row_cnt = reinterpret_cast<int*>(ws + w.row_cnt);
  p.row_cur = reinterpret_cast<int*>(ws + w.row_cur);
  p.blk = reinterpret_cast<int*>(ws + w.blk);
  p.list = reinterpret_cast<int*>(ws + w.list);
  cudaError_t e;
  const int64_t rows = p.T * p.H;
  bwd_delta_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, s>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // at H = 128: compaction, then S / dP / P / dS' and dq = dS'.K as tcgen05 kernels
  if (p.H == 128) {
    if (p.idx64)
      bwd_compact_kernel<int64_t><<<static_cast<unsigned>(p.T), kThreads, 0, s>>>(p);
    else
      bwd_compact_kernel<int32_t><<<static_cast<unsigned>(p.T), kThreads, 0, s>>>(p);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = static_cast<cudaError_t>(launch_bwd_sdp_tc(p, s));
    if (e == cudaSuccess) e = static_cast<cudaError_t>(launch_bwd_dq_tc(p, s));
  } else {
    e = p.idx64 ? launch_dq<int64_t, true>(p, s) : launch_dq<int32_t, true>(p, s);
  }
  if (e != cudaSuccess) return e;
  switch (p.H) {
    case 128: e = static_cast<cudaError_t>(launch_bwd_interm_tc(p, s)); break;   // tcgen05
    case 8: e = launch_interm<8>(p, s); break;
    case 16: e = launch_interm<16>(p, s); break;
    case 32: e = launch_interm<32>(p, s); break;
    case 64: e = launch_interm<64>(p, s); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  // inverted index: counts, exclusive scan (n + 1 entries: the last is the total), fill
  const int64_t n = p.num_kv + 1;
  if (p.num_kv > 0) {
    if ((e = cudaMemsetAsync(p.row_cnt, 0, n * 4, s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(p.row_cur, 0, p.num_kv * 4, s)) != cudaSuccess) return e;
    const int64_t ents = p.T * p.topk;
    const unsigned eb = static_cast<unsigned>((ents + 255) / 256);
    if (ents > 0) {
      bwd_csr_count_kernel<<<eb, 256, 0, s>>>(p);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const int nblk = static_cast<int>((n + kScanBlock - 1) / kScanBlock);
    bwd_scan_blocks_kernel<<<nblk, kScanBlock, 0, s>>>(p.row_cnt, n, p.blk);
    bwd_scan_totals_kernel<<<1, kScanBlock, 0, s>>>(p.blk, nblk);
    bwd_scan_add_kernel<<<nblk, kScanBlock, 0, s>>>(p.row_cnt, n, p.blk);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (ents > 0) {
      bwd_csr_fill_kernel<<<eb, 256, 0, s>>>(p);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    bwd_gather_kernel<<<static_cast<unsigned>(p.num_kv), 128, 0, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (p.dsink != nullptr) {
    if (p.sink != nullptr) {
      bwd_dsink_kernel<<<p.H, 256, 0, s>>>(p);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    } else if ((e = cudaMemsetAsync(p.dsink, 0, p.H * 4, s)) != cudaSuccess) {
      return e;
    }
  }
  return cudaSuccess;
}

}  // namespace smla
