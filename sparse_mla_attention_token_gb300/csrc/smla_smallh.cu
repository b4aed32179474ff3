// Small-head sparse MLA prefill forward (H = 8/16 per rank, head groups of 16).
//
// One CTA computes one (token, group of 16 heads, slot range).  The op
// ("Sparse MLA training backward", section "Contract"; the forward's
// has_pe=False path) is gather-bound at these head counts: every gathered
// 1 KB kv row feeds only H <= 16 query rows ("Tuned sparse MLA prefill for
// DSv4.1-Flash TP4", description "Perf": the 32-row head tile of the
// autotuned launch is half masked at 16 heads).  So the design spends its
// effort on the gather:
//
//   * the token's index list is classified on the index's full width
//     (0 <= idx < num_kv; int64 never narrowed before the check) and the valid
//     rows are compacted, in slot order, into a shared-memory row list;
//     invalid slots are never read (PR #6002 "Invalid KV rows");
//   * rows are gathered 32 per tile with 16-byte cp.async into a two-stage
//     ring (the next tile lands while this one is computed); the ragged tail
//     of the last tile is zero-filled, so no pad row can inject NaN;
//   * M = 16 heads is below tcgen05's smallest tile (M = 64), so the two
//     contractions use warp-level mma.sync m16n8k16 (bf16 in, fp32 out):
//     the 8 warps split the 512-wide head dim, each owning 64 columns of
//     both S = Q.K^T (partial over its columns, summed across warps in
//     shared memory) and O += P.V;
//   * online softmax in base 2 (exp2 of scale*log2e-scaled scores), the sink
//     folded once in the epilogue: m' = max(m, sink), l' = l 2^(m-m') +
//     2^(sink-m'), lse = ln2 (m' + log2 l') (PR #4766 "Contract" and the
//     sink-inclusive lse note).
//
// Split mode (splits > 1): each slot range writes its sink-free partial
// (O normalised by its own sum, lse of its own slots) for the combine kernel.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "smla_device.cuh"
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kHG = 16;           // heads per CTA (mma M)
constexpr int kOStride = 520;     // bf16 per row of the staged output tile (bank spread)
constexpr int kRowBytes = kHeadDim * 2;

// 32 gathered rows per tile: ~95 KB of shared memory and at most 128
// registers, so two CTAs share an SM and hide each other's gather latency
// (measured faster than 64-row tiles at one CTA per SM for every slot count).
constexpr int kBN = 32;
struct __align__(128) Smem {
  static constexpr int kSredStride = kBN + 8;   // floats per row of a warp's partial scores
  static constexpr int kPStride = kBN + 8;      // bf16 per row of P (bank spread for ldmatrix)
  __nv_bfloat16 kv[2][kBN * kHeadDim];     // 2 stages; 16 B chunk c of row r at c ^ (r & 7)
  float sred[kWarps][kHG * kSredStride];   // per-warp partial scores
  __nv_bfloat16 p[kHG * kPStride];         // probabilities, A operand of P.V
  float alpha[kHG];                        // per-row rescale of O for the current tile
  float row_m[kHG];                        // final running max (log2 units)
  float row_l[kHG];                        // final running sum
  int rows[2][kSmallHMaxSlots];            // compacted valid kv rows, slot order (this token, next)
  int warp_cnt[kWarps];
};
static_assert(sizeof(Smem::kv[0]) >= kHG * kOStride * 2, "output staging fits one stage");

__device__ __forceinline__ uint32_t kv_chunk_addr(uint32_t base, int r, int c) {
  return base + r * kRowBytes + ((c ^ (r & 7)) << 4);
}

template <typename IdxT, bool kSplit>
__global__ void __launch_bounds__(kThreads, 2) smallh_fwd_kernel(const FwdParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  using SmemT = Smem;
  constexpr int kSredStride = SmemT::kSredStride, kPStride = SmemT::kPStride;
  constexpr int kNT = kBN / 8;     // 8-slot n-tiles of S
  constexpr int kCols = kBN / 16;  // softmax columns per lane (16 lanes per row)
  SmemT& sm = *reinterpret_cast<SmemT*>(smem_raw);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = lane >> 2;    // mma groupID
  const int tig = lane & 3;   // mma thread-in-group
  const int hg = blockIdx.y;
  const int split = blockIdx.z;
  const int H = p.H;
  const int h0 = hg * kHG;
  const int hvalid = min(kHG, H - h0);

  const int chunk = (p.topk + p.splits - 1) / p.splits;
  const int j0 = min(p.topk, split * chunk);
  const int j1 = min(p.topk, j0 + chunk);
  const int64_t t0 = blockIdx.x, tstride = gridDim.x;   // tokens t0, t0 + tstride, ...
  if (t0 >= p.T) return;

  // this warp's Q fragments of token t: rows = heads of the group, k = its 64 columns
  uint32_t qa[4][4];
  auto load_q = [&](int64_t t) {
    const uint32_t* q32 = static_cast<const uint32_t*>(p.q);
    const int64_t rbase = (t * H + h0) * kHeadDim;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const int d = warp * 64 + kk * 16 + 2 * tig;
      const bool lo = g < hvalid, hi = (g + 8) < hvalid;
      qa[kk][0] = lo ? q32[(rbase + int64_t(g) * kHeadDim + d) >> 1] : 0u;
      qa[kk][1] = hi ? q32[(rbase + int64_t(g + 8) * kHeadDim + d) >> 1] : 0u;
      qa[kk][2] = lo ? q32[(rbase + int64_t(g) * kHeadDim + d + 8) >> 1] : 0u;
      qa[kk][3] = hi ? q32[(rbase + int64_t(g + 8) * kHeadDim + d + 8) >> 1] : 0u;
    }
  };

  // classify token t's slots at full width and compact the valid rows (slot
  // order) into list `buf`; block-wide (every thread calls it); returns the count
  auto compact = [&](int64_t t, int buf) -> int {
    const IdxT* idx = static_cast<const IdxT*>(p.idx) + t * p.topk;
    int* rows = sm.rows[buf];
    int nvalid = 0;
    for (int base = j0; base < j1; base += kThreads) {
      const int j = base + tid;
      bool v = false;
      int row = -1;
      if (j < j1) {
        const IdxT x = idx[j];
        v = slot_valid<IdxT>(x, p.num_kv);
        if (v) row = static_cast<int>(x);   // exact: num_kv < 2^31
      }
      const unsigned ball = __ballot_sync(0xffffffffu, v);
      if (lane == 0) sm.warp_cnt[warp] = __popc(ball);
      __syncthreads();
      int off = nvalid, total = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const int c = sm.warp_cnt[w];
        off += (w < warp) ? c : 0;
        total += c;
      }
      if (v) rows[off + __popc(ball & ((1u << lane) - 1u))] = row;
      nvalid += total;
      __syncthreads();
    }
    // read trace: the range's entries past its valid count are never read (-1);
    // the gather writes the others
    if (p.trace != nullptr && hg == 0)
      for (int k = j0 + nvalid + tid; k < j1; k += kThreads) p.trace[t * p.topk + k] = -1;
    return nvalid;
  };

  const char* kvb = static_cast<const char*>(p.kv);
  // gather tile `tile` of token t's rows in list `buf` (count nvalid) into `stage`
  auto issue_tile = [&](int64_t t, int buf, int nvalid, int tile, int stage) {
    const uint32_t dst0 = smem_u32(sm.kv[stage]);
    const int* rows = sm.rows[buf];
#pragma unroll 4
    for (int i = tid; i < kBN * 64; i += kThreads) {
      const int r = i >> 6, c = i & 63;
      const int slot = tile * kBN + r;
      const bool ok = slot < nvalid;
      const char* src = ok ? kvb + int64_t(rows[slot]) * kRowBytes + c * 16 : kvb;
      cp_async_16(kv_chunk_addr(dst0, r, c), src, ok ? 16u : 0u);
      // read trace: the row this copy reads, recovered from its source address
      if (p.trace != nullptr && hg == 0 && c == 0 && ok)
        p.trace[t * p.topk + j0 + slot] = (src - kvb) / kRowBytes;
    }
    cp_async_commit();
  };

  const float sl2 = p.scale * kLog2e;
  const int srow = 2 * warp + (lane >> 4);   // softmax row owned by this half-warp
  const int sc0 = (lane & 15) * kCols;       // its kCols columns

  // The CTA's tokens run as one stream of tiles through the two-stage ring:
  // the next token's list is compacted and its first tile gathered while the
  // current token's last tile is computed, so a token's gather latency hides
  // behind the previous token's work.
  load_q(t0);
  int cur = 0;                    // row list of the current token
  int nv_cur = compact(t0, cur);
  uint32_t gt = 0;                // tiles issued before the current one (stage = gt & 1)
  if (nv_cur > 0) issue_tile(t0, cur, nv_cur, 0, 0);

  for (int64_t t = t0; t < p.T; t += tstride) {
    const int64_t tn = t + tstride;
    const int ntiles = (nv_cur + kBN - 1) / kBN;
    int nv_next = 0;
    bool next_done = false;       // the next token's list compacted (and its tile issued)
    float m_run = -INFINITY, l_run = 0.f;
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

    for (int it = 0; it < ntiles; ++it, ++gt) {
      const int stage = gt & 1;
      cp_async_wait<0>();
      __syncthreads();  // tile `it` landed; every warp is done with the other stage
      if (it + 1 < ntiles) {
        issue_tile(t, cur, nv_cur, it + 1, stage ^ 1);
      } else if (tn < p.T) {
        nv_next = compact(tn, cur ^ 1);
        next_done = true;
        if (nv_next > 0) issue_tile(tn, cur ^ 1, nv_next, 0, stage ^ 1);
      }
      const uint32_t kvs = smem_u32(sm.kv[stage]);
      // ---- 3. partial S over this warp's 64 columns
      float s[kNT][4];
  #pragma unroll
      for (int i = 0; i < kNT; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
  #pragma unroll
      for (int kp = 0; kp < 2; ++kp) {
        const int c = warp * 8 + kp * 4 + (lane >> 3);
  #pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          const int r = nt * 8 + (lane & 7);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(kv_chunk_addr(kvs, r, c), b0, b1, b2, b3);
          mma_16816(s[nt], qa[2 * kp], b0, b1);
          mma_16816(s[nt], qa[2 * kp + 1], b2, b3);
        }
      }
      float* sw = sm.sred[warp];
  #pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        *reinterpret_cast<float2*>(&sw[g * kSredStride + nt * 8 + 2 * tig]) =
            make_float2(s[nt][0], s[nt][1]);
        *reinterpret_cast<float2*>(&sw[(g + 8) * kSredStride + nt * 8 + 2 * tig]) =
            make_float2(s[nt][2], s[nt][3]);
      }
      __syncthreads();

      // ---- 4. reduce the 8 partials, online softmax (base 2)
      {
        float a[kCols];
  #pragma unroll
        for (int k = 0; k < kCols; ++k) a[k] = 0.f;
  #pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float* src = &sm.sred[w][srow * kSredStride + sc0];
          if constexpr (kCols == 4) {
            const float4 v = *reinterpret_cast<const float4*>(src);
            a[0] += v.x; a[1] += v.y; a[2] += v.z; a[3] += v.w;
          } else {
            const float2 v = *reinterpret_cast<const float2*>(src);
            a[0] += v.x; a[1] += v.y;
          }
        }
        const int col = it * kBN + sc0;
        float x[kCols];
        float mx = -INFINITY;
  #pragma unroll
        for (int k = 0; k < kCols; ++k) {
          x[k] = (col + k < nv_cur) ? a[k] * sl2 : -INFINITY;
          mx = fmaxf(mx, x[k]);
        }
  #pragma unroll
        for (int o = 8; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m_new = fmaxf(m_run, mx);  // finite: the tile holds >= 1 valid row
        const float alpha = ex2(m_run - m_new);
        float ps = 0.f;
  #pragma unroll
        for (int k = 0; k < kCols; ++k) {
          x[k] = ex2(x[k] - m_new);
          ps += x[k];
        }
  #pragma unroll
        for (int o = 8; o >= 1; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        l_run = l_run * alpha + ps;
        m_run = m_new;
  #pragma unroll
        for (int k = 0; k < kCols; k += 2)
          *reinterpret_cast<uint32_t*>(&sm.p[srow * kPStride + sc0 + k]) = pack_bf16x2(x[k], x[k + 1]);
        if ((lane & 15) == 0) sm.alpha[srow] = alpha;
      }
      __syncthreads();

      // ---- 5. O = alpha * O + P . V over this warp's 64 columns
      {
        const float a_lo = sm.alpha[g], a_hi = sm.alpha[g + 8];
  #pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          acc[nt][0] *= a_lo; acc[nt][1] *= a_lo;
          acc[nt][2] *= a_hi; acc[nt][3] *= a_hi;
        }
        const uint32_t ps = smem_u32(sm.p);
  #pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks) {
          uint32_t pa[4];
          const int pr = ((lane >> 3) & 1) * 8 + (lane & 7);
          const int pc = ks * 16 + (lane >> 4) * 8;
          ldmatrix_x4(ps + (pr * kPStride + pc) * 2, pa[0], pa[1], pa[2], pa[3]);
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

    // ---- epilogue of token t
    if ((lane & 15) == 0) {
      sm.row_m[srow] = m_run;
      sm.row_l[srow] = l_run;
    }
    __syncthreads();

    if constexpr (kSplit) {
      // sink-free partial: O normalised by its own sum; lse of this range alone
      const int64_t TH = p.T * H;
  #pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int r = g + half * 8;
        if (r >= hvalid) continue;
        const float m = sm.row_m[r], l = sm.row_l[r];
        const float f = (l > 0.f) ? 1.f / l : 0.f;
        const int64_t rowid = int64_t(split) * TH + t * H + h0 + r;
        float* po = p.part_o + rowid * kHeadDim + warp * 64 + 2 * tig;
  #pragma unroll
        for (int nt = 0; nt < 8; ++nt)
          *reinterpret_cast<float2*>(po + nt * 8) =
              make_float2(acc[nt][2 * half] * f, acc[nt][2 * half + 1] * f);
        if (warp == 0 && tig == 0) p.part_lse[rowid] = (l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
      }
    } else {
      // fold the sink once, normalise, round to bf16, stage, store 16 B per thread
      // staged in the stage of the token's last tile: every warp has finished
      // reading it (barrier above); the next token's first tile is in the other one
      __nv_bfloat16* ost = sm.kv[(gt - 1) & 1];
  #pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int r = g + half * 8;
        const float m = sm.row_m[r], l = sm.row_l[r];
        float m2 = m, l2 = l;
        if (p.sink != nullptr && r < hvalid) {
          const float sk = p.sink[h0 + r] * kLog2e;
          m2 = fmaxf(m, sk);
          if (m2 != -INFINITY) l2 = l * ex2(m - m2) + ex2(sk - m2);
        }
        const bool live = (m2 != -INFINITY) && (l2 > 0.f);
        const float f = live ? ex2(m - m2) / l2 : 0.f;
  #pragma unroll
        for (int nt = 0; nt < 8; ++nt)
          *reinterpret_cast<uint32_t*>(&ost[r * kOStride + warp * 64 + nt * 8 + 2 * tig]) =
              pack_bf16x2(acc[nt][2 * half] * f, acc[nt][2 * half + 1] * f);
        if (warp == 0 && tig == 0 && r < hvalid)
          p.lse[t * H + h0 + r] = live ? (m2 + log2f(l2)) * kLn2 : -INFINITY;
      }
      __syncthreads();
      uint4* outp = reinterpret_cast<uint4*>(static_cast<char*>(p.out) +
                                             (t * H + h0) * int64_t(kRowBytes));
      for (int i = tid; i < hvalid * 64; i += kThreads) {
        const int r = i >> 6, c = i & 63;
        outp[i] = *reinterpret_cast<const uint4*>(&ost[r * kOStride + c * 8]);
      }
    }

    // the next token: its list (unless compacted already with the last tile) and Q
    if (tn < p.T) {
      if (!next_done) {
        nv_next = compact(tn, cur ^ 1);
        if (nv_next > 0) issue_tile(tn, cur ^ 1, nv_next, 0, gt & 1);
      }
      load_q(tn);
    }
    cur ^= 1;
    nv_cur = nv_next;
  }
  cp_async_wait<0>();   // nothing of ours may land after the CTA exits
}

// CTAs that fit on the current device at once (2 per SM), looked up once per device.
cudaError_t resident_ctas(int* out) {
  static int per_dev[64] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (per_dev[dev] == 0) {
    const int smem = static_cast<int>(sizeof(Smem)) + 1024;
    auto kern = smallh_fwd_kernel<int32_t, false>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
        cudaSuccess)
      return e;
    int per_sm = 0, sms = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem)) !=
        cudaSuccess)
      return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    per_dev[dev] = std::max(1, per_sm * sms);
  }
  *out = per_dev[dev];
  return cudaSuccess;
}

// Grid: (token CTAs, head groups, splits).  Without splits the CTAs are
// persistent, each walking tokens blockIdx.x, +gridDim.x, ...; with splits
// (small T) one CTA per (token, group, split).
cudaError_t grid_of(int64_t T, int32_t H, int32_t splits, dim3* grid) {
  const int groups = (H + kHG - 1) / kHG;
  int64_t x = T;
  if (splits == 1) {
    int resident = 0;
    const cudaError_t e = resident_ctas(&resident);
    if (e != cudaSuccess) return e;
    x = std::min<int64_t>(T, std::max(1, resident / groups));
  }
  *grid = dim3(static_cast<unsigned>(std::max<int64_t>(x, 1)), static_cast<unsigned>(groups),
               static_cast<unsigned>(splits));
  return cudaSuccess;
}

template <typename IdxT, bool kSplit>
cudaError_t launch_typed(const FwdParams& p, cudaStream_t stream) {
  auto kern = smallh_fwd_kernel<IdxT, kSplit>;
  const int smem = static_cast<int>(sizeof(Smem)) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid;
  if ((e = grid_of(p.T, p.H, p.splits, &grid)) != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int smallh_geometry(int64_t T, int32_t H, int32_t splits, LaunchGeom* g) {
  dim3 grid;
  const cudaError_t e = grid_of(T, H, splits, &grid);
  if (e != cudaSuccess) return static_cast<int>(e);
  g->grid_ctas = static_cast<int>(grid.x * grid.y * grid.z);
  g->threads = kThreads;
  g->cluster = 1;
  g->smem = static_cast<int>(sizeof(Smem)) + 1024;
  return 0;
}

int launch_smallh(const FwdParams& p, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool split = p.splits > 1;
  cudaError_t e;
  if (p.idx64)
    e = split ? launch_typed<int64_t, true>(p, s) : launch_typed<int64_t, false>(p, s);
  else
    e = split ? launch_typed<int32_t, true>(p, s) : launch_typed<int32_t, false>(p, s);
  return static_cast<int>(e);
}

}  // namespace smla
