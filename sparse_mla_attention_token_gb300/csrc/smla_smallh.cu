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
//     ring (the next tile lands while this one is computed), each warp the
//     64 columns it reads, so that (bf16) a warp waits for its own copies
//     only; the ragged tail of the last tile is zero-filled, so no pad row
//     can inject NaN;
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
//
// Head dims: the kernel is instantiated for score width kDqk in {128, 512,
// 576} (kDqk / 64 warps, one 64-column slice each) and value width kDv <= kDqk
// (the first kDv columns of each gathered row; kDv = 512 with kDqk = 576 is the
// MLA layout whose last 64 columns are a positional part used in the scores
// only: "Add DSv4 sparse MLA prefill Triton and unified with MLA Gluon kernel
// on GFX950", the has_pe flag; head dims 128 and 576: "Tuned sparse MLA
// prefill for DSv4.1-Flash TP4", its tests).
//
// fp8 cache (kFp8, 512 columns): each kv row is 512 e4m3 bytes and 4 fp32
// scales, one per 128-column block (value = code * scale).  The gather moves
// the 512 + 16 bytes with cp.async into an fp8 ring (16-byte chunk c of row r
// at chunk c ^ 4 (r & 7), so that a warp's reads of 8 rows x 64 bytes spread
// over the banks); at the start of each tile every warp decodes the codes of
// its own 64 columns exactly into the bf16 stage (e4m3 is a subset of bf16)
// behind a warp-level sync; the scales are applied in fp32: to each warp's partial scores (a warp's
// 64 columns lie in one block) and to the probabilities, one bf16 copy of P per
// block, so that P.V and the scores see code * scale without a second rounding
// of the values.
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "smla_device.cuh"
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kHG = 16;           // heads per CTA (mma M)
// 32 gathered rows per tile: ~95 KB of shared memory at 512 columns and at
// most 128 registers, so two CTAs share an SM and hide each other's gather
// latency (measured faster than 64-row tiles at one CTA per SM for every slot
// count).
constexpr int kBN = 32;

// Shape constants of one (score width, value width) instantiation.
template <int kDqk, int kDv>
struct Dims {
  static_assert(kDqk % 64 == 0 && kDv % 64 == 0 && kDv <= kDqk, "64-column slices");
  static constexpr int kWarps = kDqk / 64;          // one 64-column slice of the scores each
  static constexpr int kVWarps = kDv / 64;          // warps that also own value columns
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kRowBytes = kDqk * 2;        // one gathered row
  static constexpr int kOStride = kDv + 8;          // bf16 per row of the staged output tile
  static constexpr int kHW = 2 * kWarps;            // half-warps; one owns a softmax row at a time
  static constexpr int kRowsPerHW = (kHG + kHW - 1) / kHW;
  static constexpr int kMinBlocks = kDqk <= 512 ? 2 : 1;
};

// Shared memory of the bf16 instantiations: two bf16 stages of the gather ring.
template <int kDqk, int kDv, bool kFp8 = false>
struct __align__(128) Smem {
  using Dm = Dims<kDqk, kDv>;
  static constexpr int kSredStride = kBN + 8;   // floats per row of a warp's partial scores
  static constexpr int kPStride = kBN + 8;      // bf16 per row of P (bank spread for ldmatrix)
  __nv_bfloat16 kv[2][kBN * kDqk];         // 2 stages; 16 B chunk c of row r at c ^ (r & 7)
  float sred[Dm::kWarps][kHG * kSredStride];   // per-warp partial scores
  __nv_bfloat16 p[1][kHG * kPStride];      // probabilities, A operand of P.V
  float alpha[kHG];                        // per-row rescale of O for the current tile
  float row_m[kHG];                        // final running max (log2 units)
  float row_l[kHG];                        // final running sum
  int rows[2][kSmallHMaxSlots];            // compacted valid kv rows, slot order (this token, next)
  int warp_cnt[Dm::kWarps];
  static_assert(sizeof(kv[0]) >= kHG * Dm::kOStride * 2, "output staging fits one stage");
};

// The fp8-cache instantiation: a two-stage ring of raw e4m3 rows and their
// scales, decoded tile by tile into one bf16 stage.
template <>
struct __align__(128) Smem<512, 512, true> {
  using Dm = Dims<512, 512>;
  static constexpr int kSredStride = kBN + 8;
  static constexpr int kPStride = kBN + 8;
  __nv_bfloat16 kv[1][kBN * 512];          // the decoded tile (same layout as a bf16 stage)
  float sred[Dm::kWarps][kHG * kSredStride];
  __nv_bfloat16 p[4][kHG * kPStride];      // P times each 128-column block's scale
  float alpha[kHG];
  float row_m[kHG];
  float row_l[kHG];
  int rows[2][kSmallHMaxSlots];
  int warp_cnt[Dm::kWarps];
  uint8_t f8[2][kBN * 512];                // fp8 ring: raw e4m3 rows
  float scl[2][Dm::kWarps][kBN];           // per warp: its 128-column block's scale of each row
  static_assert(sizeof(kv[0]) >= kHG * Dm::kOStride * 2, "output staging fits one stage");
};

// 4-byte async copy global -> shared; src_bytes = 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}

template <int kRowBytes>
__device__ __forceinline__ uint32_t kv_chunk_addr(uint32_t base, int r, int c) {
  return base + r * kRowBytes + ((c ^ (r & 7)) << 4);
}

// kTrace: the instantiation that writes the read trace (p.trace); the others
// carry no trace code in their gather loop.  kFp8: kv is the fp8 cache.
template <typename IdxT, bool kSplit, int kDqk, int kDv, bool kTrace, bool kFp8 = false>
__global__ void __launch_bounds__(Dims<kDqk, kDv>::kThreads, Dims<kDqk, kDv>::kMinBlocks)
    smallh_fwd_kernel(const FwdParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  using Dm = Dims<kDqk, kDv>;
  using SmemT = Smem<kDqk, kDv, kFp8>;
  constexpr int kWarps = Dm::kWarps, kThreads = Dm::kThreads, kRowBytes = Dm::kRowBytes;
  constexpr int kOStride = Dm::kOStride, kHW = Dm::kHW, kRPH = Dm::kRowsPerHW;
  constexpr int kSredStride = SmemT::kSredStride, kPStride = SmemT::kPStride;
  constexpr int kNT = kBN / 8;     // 8-slot n-tiles of S
  constexpr int kCols = kBN / 16;  // softmax columns per lane (16 lanes per row)
  SmemT& sm = *reinterpret_cast<SmemT*>(smem_raw);
  const auto kv_chunk = [](uint32_t base, int r, int c) { return kv_chunk_addr<kRowBytes>(base, r, c); };

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
  // the combine kernel that follows a split launch may be scheduled now: it
  // waits for this whole grid to finish before it reads a partial
  if constexpr (kSplit) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (t0 >= p.T) return;

  // this warp's Q fragments of token t: rows = heads of the group, k = its 64 columns
  uint32_t qa[4][4];
  auto load_q = [&](int64_t t) {
    const uint32_t* q32 = static_cast<const uint32_t*>(p.q);
    const int64_t rbase = (t * H + h0) * kDqk;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const int d = warp * 64 + kk * 16 + 2 * tig;
      const bool lo = g < hvalid, hi = (g + 8) < hvalid;
      qa[kk][0] = lo ? q32[(rbase + int64_t(g) * kDqk + d) >> 1] : 0u;
      qa[kk][1] = hi ? q32[(rbase + int64_t(g + 8) * kDqk + d) >> 1] : 0u;
      qa[kk][2] = lo ? q32[(rbase + int64_t(g) * kDqk + d + 8) >> 1] : 0u;
      qa[kk][3] = hi ? q32[(rbase + int64_t(g + 8) * kDqk + d + 8) >> 1] : 0u;
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
    if constexpr (kTrace)
      if (hg == 0)
        for (int k = j0 + nvalid + tid; k < j1; k += kThreads) p.trace[t * p.topk + k] = -1;
    return nvalid;
  };

  const char* kvb = static_cast<const char*>(p.kv);
  // gather tile `tile` of token t's rows in list `buf` (count nvalid) into `stage`
  auto issue_tile = [&](int64_t t, int buf, int nvalid, int tile, int stage) {
    const int* rows = sm.rows[buf];
    if constexpr (kFp8) {
      // each warp copies the codes of its own 64 columns (4 chunks of each row; chunk
      // c at c ^ 4(r & 7), so that its decode reads of 8 rows x 64 B spread over the
      // banks) and its 128-column block's scale of each row: all a warp reads before
      // the next block barrier.  The tail is zero-filled.
      static_assert(kBN == 32, "one row per lane for the scales");
      const uint32_t f0 = smem_u32(sm.f8[stage]), s0 = smem_u32(&sm.scl[stage][warp][0]);
      const uint8_t* cb = static_cast<const uint8_t*>(p.kv);
      const char* sb = reinterpret_cast<const char*>(p.kv_scale);
#pragma unroll
      for (int k = 0; k < kBN / 8; ++k) {
        const int r = (lane >> 2) + 8 * k, c = warp * 4 + (lane & 3);
        const int slot = tile * kBN + r;
        const bool ok = slot < nvalid;
        const int64_t row = ok ? rows[slot] : 0;
        cp_async_16(f0 + r * 512 + ((c ^ ((r & 7) << 2)) << 4), cb + row * 512 + c * 16, ok ? 16u : 0u);
      }
      {
        const int slot = tile * kBN + lane;
        const bool ok = slot < nvalid;
        const int64_t row = ok ? rows[slot] : 0;
        cp_async_4(s0 + lane * 4, sb + row * 16 + (warp >> 1) * 4, ok ? 4u : 0u);
      }
      cp_async_commit();
      return;
    }
    const uint32_t dst0 = smem_u32(sm.kv[stage]);
    // each warp copies its own 64 columns of the tile's rows (the only ones it
    // reads: its score slice and its value columns), 8 lanes per 128-byte row
    // piece, so a warp waits for its own copies alone
#pragma unroll
    for (int k = 0; k < kBN / 4; ++k) {
      const int r = (lane >> 3) + 4 * k, c = warp * 8 + (lane & 7);
      const int slot = tile * kBN + r;
      const bool ok = slot < nvalid;
      const char* src = ok ? kvb + int64_t(rows[slot]) * kRowBytes + c * 16 : kvb;
      cp_async_16(kv_chunk(dst0, r, c), src, ok ? 16u : 0u);
      // read trace: the row this copy reads, recovered from its source address
      if constexpr (kTrace)
        if (hg == 0 && c == 0 && ok) p.trace[t * p.topk + j0 + slot] = (src - kvb) / kRowBytes;
    }
    cp_async_commit();
  };

  const float sl2 = p.scale * kLog2e;
  const int hw = 2 * warp + (lane >> 4);     // half-warp: owns softmax rows hw, hw + kHW, ...
  const int sc0 = (lane & 15) * kCols;       // its kCols columns

  // The CTA's tokens run as one stream of tiles through the two-stage ring:
  // the next token's list is compacted and its first tile gathered while the
  // current token's last tile is computed, so a token's gather latency hides
  // behind the previous token's work.
  // this thread's epilogue rows g and g + 8: their sinks (base-2 logits), read
  // once for all of the CTA's tokens (the head group is fixed), not in every
  // token's epilogue between its two barriers
  float sk2[2] = {-INFINITY, -INFINITY};
  if constexpr (!kSplit) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = g + half * 8;
      if (p.sink != nullptr && r < hvalid) sk2[half] = p.sink[h0 + r] * kLog2e;
    }
  }
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
    float m_run[kRPH], l_run[kRPH];
#pragma unroll
    for (int i = 0; i < kRPH; ++i) {
      m_run[i] = -INFINITY;
      l_run[i] = 0.f;
    }
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

    for (int it = 0; it < ntiles; ++it, ++gt) {
      const int stage = gt & 1;
      cp_async_wait<0>();
      // tile `it` landed: a warp gathered, and reads before the next block barrier,
      // its own columns (and, fp8, its own block's scales) only, so its own copies
      // and a warp-level sync suffice; it is also done with its part of the other
      // stage.  fp8: the decode stage also holds the previous token's staged
      // output, which every warp must have copied out before a token's first decode.
      if constexpr (kFp8) {
        if (it == 0) __syncthreads(); else __syncwarp();
      } else {
        __syncwarp();
      }
      if (it + 1 < ntiles) {
        // bf16: tile 1 goes into the stage the previous token's epilogue staged its
        // output in; every warp must have copied that out first (other gathers into
        // it follow a compaction, whose block barriers order them)
        if constexpr (!kFp8)
          if (it == 0) __syncthreads();
        issue_tile(t, cur, nv_cur, it + 1, stage ^ 1);
      } else if (tn < p.T) {
        nv_next = compact(tn, cur ^ 1);
        next_done = true;
        if (nv_next > 0) issue_tile(tn, cur ^ 1, nv_next, 0, stage ^ 1);
      }
      if constexpr (kFp8) {
        // decode the tile's e4m3 codes exactly into the bf16 stage: each warp only
        // its own 64 columns (the only ones it reads, for its score slice and for
        // its value columns), so a warp-level sync is enough; the barrier above
        // ordered the stage's previous readers (the output copy included)
        static_assert(kDqk == 512 && kDv == 512 && Dm::kVWarps == kWarps, "fp8: 64 columns per warp");
        const uint32_t kv0 = smem_u32(sm.kv[0]);
#pragma unroll
        for (int k = 0; k < kBN * 4 / 32; ++k) {
          const int i = lane + k * 32, r = i >> 2, c = warp * 4 + (i & 3);
          const uint4 raw = *reinterpret_cast<const uint4*>(&sm.f8[stage][r * 512 + ((c ^ ((r & 7) << 2)) << 4)]);
          const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t o[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const __nv_fp8x2_storage_t two =
                static_cast<__nv_fp8x2_storage_t>((w4[j >> 1] >> (16 * (j & 1))) & 0xffffu);
            const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(two, __NV_E4M3);
            o[j] = pack_bf16x2(__half2float(__half(__half_raw{h.x})),
                               __half2float(__half(__half_raw{h.y})));
          }
          sts_u4(kv_chunk(kv0, r, 2 * c), make_uint4(o[0], o[1], o[2], o[3]));
          sts_u4(kv_chunk(kv0, r, 2 * c + 1), make_uint4(o[4], o[5], o[6], o[7]));
        }
        __syncwarp();
      }
      const uint32_t kvs = smem_u32(sm.kv[kFp8 ? 0 : stage]);
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
          ldmatrix_x4(kv_chunk(kvs, r, c), b0, b1, b2, b3);
          mma_16816(s[nt], qa[2 * kp], b0, b1);
          mma_16816(s[nt], qa[2 * kp + 1], b2, b3);
        }
      }
      if constexpr (kFp8) {
        // this warp's 64 columns lie in scale block warp / 2: scale each slot's partial
  #pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          const float c0 = sm.scl[stage][warp][nt * 8 + 2 * tig];
          const float c1 = sm.scl[stage][warp][nt * 8 + 2 * tig + 1];
          s[nt][0] *= c0; s[nt][1] *= c1; s[nt][2] *= c0; s[nt][3] *= c1;
        }
      }
      float* sw = sm.sred[warp];
      const bool hi_row = g + 8 < hvalid;   // rows past the group's heads are never reduced
  #pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        *reinterpret_cast<float2*>(&sw[g * kSredStride + nt * 8 + 2 * tig]) =
            make_float2(s[nt][0], s[nt][1]);
        if (hi_row)
          *reinterpret_cast<float2*>(&sw[(g + 8) * kSredStride + nt * 8 + 2 * tig]) =
              make_float2(s[nt][2], s[nt][3]);
      }
      __syncthreads();

      // ---- 4. reduce the kWarps partials, online softmax (base 2)
#pragma unroll
      for (int ri = 0; ri < kRPH; ++ri) {
        const int srow = hw + ri * kHW;
        if (srow >= kHG) break;   // warp-uniform: kHW divides 16, or whole warps have no row
        // a warp whose two rows are both past the group's heads (H = 8: warps 4-7)
        // skips them (warp-uniform test): an MMA row of O depends only on the same
        // row of P and alpha, and those rows' outputs are never stored
        if (2 * warp + ri * kHW >= hvalid) continue;
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
        const float m_new = fmaxf(m_run[ri], mx);  // finite: the tile holds >= 1 valid row
        const float alpha = ex2(m_run[ri] - m_new);
        float ps = 0.f;
  #pragma unroll
        for (int k = 0; k < kCols; ++k) {
          x[k] = ex2(x[k] - m_new);
          ps += x[k];
        }
  #pragma unroll
        for (int o = 8; o >= 1; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        l_run[ri] = l_run[ri] * alpha + ps;
        m_run[ri] = m_new;
        if constexpr (kFp8) {
          // P times each block's scale of the slot: the A operand of that block's warps
  #pragma unroll
          for (int b = 0; b < 4; ++b)
  #pragma unroll
            for (int k = 0; k < kCols; k += 2)
              *reinterpret_cast<uint32_t*>(&sm.p[b][srow * kPStride + sc0 + k]) =
                  pack_bf16x2(x[k] * sm.scl[stage][2 * b][sc0 + k], x[k + 1] * sm.scl[stage][2 * b][sc0 + k + 1]);
        } else {
  #pragma unroll
          for (int k = 0; k < kCols; k += 2)
            *reinterpret_cast<uint32_t*>(&sm.p[0][srow * kPStride + sc0 + k]) = pack_bf16x2(x[k], x[k + 1]);
        }
        if ((lane & 15) == 0) sm.alpha[srow] = alpha;
      }
      __syncthreads();

      // ---- 5. O = alpha * O + P . V over this warp's 64 columns (value warps)
      if (warp < Dm::kVWarps) {
        const float a_lo = sm.alpha[g], a_hi = sm.alpha[g + 8];
  #pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          acc[nt][0] *= a_lo; acc[nt][1] *= a_lo;
          acc[nt][2] *= a_hi; acc[nt][3] *= a_hi;
        }
        const uint32_t ps = smem_u32(sm.p[kFp8 ? warp >> 1 : 0]);
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
            ldmatrix_x4_trans(kv_chunk(kvs, r, c), b0, b1, b2, b3);
            mma_16816(acc[2 * np], pa, b0, b1);
            mma_16816(acc[2 * np + 1], pa, b2, b3);
          }
        }
      }
    }

    // ---- epilogue of token t
#pragma unroll
    for (int ri = 0; ri < kRPH; ++ri) {
      const int srow = hw + ri * kHW;
      if ((lane & 15) == 0 && srow < kHG) {
        sm.row_m[srow] = m_run[ri];
        sm.row_l[srow] = l_run[ri];
      }
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
        if (warp < Dm::kVWarps) {
          float* po = p.part_o + rowid * kDv + warp * 64 + 2 * tig;
  #pragma unroll
          for (int nt = 0; nt < 8; ++nt)
            *reinterpret_cast<float2*>(po + nt * 8) =
                make_float2(acc[nt][2 * half] * f, acc[nt][2 * half + 1] * f);
        }
        if (warp == 0 && tig == 0) p.part_lse[rowid] = (l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
      }
    } else {
      // fold the sink once, normalise, round to bf16, stage, store 16 B per thread
      // staged in the stage of the token's last tile: every warp has finished
      // reading it (barrier above); the next token's first tile is in the other one
      __nv_bfloat16* ost = sm.kv[kFp8 ? 0 : (gt - 1) & 1];
  #pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int r = g + half * 8;
        if (r >= hvalid) continue;   // never stored (the copy below takes hvalid rows)
        const float m = sm.row_m[r], l = sm.row_l[r];
        float m2 = m, l2 = l;
        if (sk2[half] != -INFINITY) {
          const float sk = sk2[half];
          m2 = fmaxf(m, sk);
          l2 = l * ex2(m - m2) + ex2(sk - m2);
        }
        const bool live = (m2 != -INFINITY) && (l2 > 0.f);
        const float f = live ? ex2(m - m2) / l2 : 0.f;
        if (warp < Dm::kVWarps) {
  #pragma unroll
          for (int nt = 0; nt < 8; ++nt)
            *reinterpret_cast<uint32_t*>(&ost[r * kOStride + warp * 64 + nt * 8 + 2 * tig]) =
                pack_bf16x2(acc[nt][2 * half] * f, acc[nt][2 * half + 1] * f);
        }
        if (warp == 0 && tig == 0)
          p.lse[t * H + h0 + r] = live ? (m2 + log2f(l2)) * kLn2 : -INFINITY;
      }
      __syncthreads();
      constexpr int kOChunks = kDv / 8;   // 16-byte chunks per output row
      uint4* outp = reinterpret_cast<uint4*>(static_cast<char*>(p.out) +
                                             (t * H + h0) * int64_t(kDv * 2));
      for (int i = tid; i < hvalid * kOChunks; i += kThreads) {
        const int r = static_cast<int>(unsigned(i) / kOChunks), c = static_cast<int>(unsigned(i) % kOChunks);
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

template <int kDqk, int kDv, bool kFp8 = false>
constexpr int smem_bytes() {
  return static_cast<int>(sizeof(Smem<kDqk, kDv, kFp8>)) + 1024;
}

// CTAs of one instantiation that fit on the current device at once, looked up
// once per device (index `slot` per (kDqk, kDv, fp8) variant).
template <int kDqk, int kDv, bool kFp8 = false>
cudaError_t resident_ctas(int slot, int* out) {
  static int per_dev[5][64] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (per_dev[slot][dev] == 0) {
    const int smem = smem_bytes<kDqk, kDv, kFp8>();
    auto kern = smallh_fwd_kernel<int32_t, false, kDqk, kDv, false, kFp8>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
        cudaSuccess)
      return e;
    int per_sm = 0, sms = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Dims<kDqk, kDv>::kThreads,
                                                           smem)) != cudaSuccess)
      return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    per_dev[slot][dev] = std::max(1, per_sm * sms);
  }
  *out = per_dev[slot][dev];
  return cudaSuccess;
}

// Grid: (token CTAs, head groups, splits).  Without splits the CTAs are
// persistent, each walking tokens blockIdx.x, +gridDim.x, ...; with splits
// (small T) one CTA per (token, group, split).
template <int kDqk, int kDv, bool kFp8 = false>
cudaError_t grid_of(int slot, int64_t T, int32_t H, int32_t splits, dim3* grid) {
  const int groups = (H + kHG - 1) / kHG;
  int64_t x = T;
  if (splits == 1) {
    int resident = 0;
    const cudaError_t e = resident_ctas<kDqk, kDv, kFp8>(slot, &resident);
    if (e != cudaSuccess) return e;
    x = std::min<int64_t>(T, std::max(1, resident / groups));
  }
  *grid = dim3(static_cast<unsigned>(std::max<int64_t>(x, 1)), static_cast<unsigned>(groups),
               static_cast<unsigned>(splits));
  return cudaSuccess;
}

template <typename IdxT, bool kSplit, int kDqk, int kDv, bool kTrace, bool kFp8 = false>
cudaError_t launch_typed(int slot, const FwdParams& p, cudaStream_t stream) {
  auto kern = smallh_fwd_kernel<IdxT, kSplit, kDqk, kDv, kTrace, kFp8>;
  const int smem = smem_bytes<kDqk, kDv, kFp8>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid;
  if ((e = grid_of<kDqk, kDv, kFp8>(slot, p.T, p.H, p.splits, &grid)) != cudaSuccess) return e;
  kern<<<grid, Dims<kDqk, kDv>::kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int kDqk, int kDv, bool kTrace>
cudaError_t launch_dims(int slot, const FwdParams& p, cudaStream_t s) {
  const bool split = p.splits > 1;
  if (p.idx64)
    return split ? launch_typed<int64_t, true, kDqk, kDv, kTrace>(slot, p, s)
                 : launch_typed<int64_t, false, kDqk, kDv, kTrace>(slot, p, s);
  return split ? launch_typed<int32_t, true, kDqk, kDv, kTrace>(slot, p, s)
               : launch_typed<int32_t, false, kDqk, kDv, kTrace>(slot, p, s);
}

template <int kDqk, int kDv, bool kFp8 = false>
cudaError_t geometry_dims(int slot, int64_t T, int32_t H, int32_t splits, LaunchGeom* g) {
  dim3 grid;
  const cudaError_t e = grid_of<kDqk, kDv, kFp8>(slot, T, H, splits, &grid);
  if (e != cudaSuccess) return e;
  g->grid_ctas = static_cast<int>(grid.x * grid.y * grid.z);
  g->threads = Dims<kDqk, kDv>::kThreads;
  g->cluster = 1;
  g->smem = smem_bytes<kDqk, kDv, kFp8>();
  return cudaSuccess;
}

}  // namespace

bool smallh_dims_supported(int32_t d_qk, int32_t d_v) {
  return (d_qk == 512 && d_v == 512) || (d_qk == 128 && d_v == 128) ||
         (d_qk == 576 && d_v == 576) || (d_qk == 576 && d_v == 512);
}

int smallh_geometry(int64_t T, int32_t H, int32_t splits, int32_t d_qk, int32_t d_v,
                    LaunchGeom* g, bool fp8) {
  cudaError_t e;
  if (fp8) return static_cast<int>(geometry_dims<512, 512, true>(4, T, H, splits, g));
  if (d_qk == 512 && d_v == 512) e = geometry_dims<512, 512>(0, T, H, splits, g);
  else if (d_qk == 128 && d_v == 128) e = geometry_dims<128, 128>(1, T, H, splits, g);
  else if (d_qk == 576 && d_v == 576) e = geometry_dims<576, 576>(2, T, H, splits, g);
  else if (d_qk == 576 && d_v == 512) e = geometry_dims<576, 512>(3, T, H, splits, g);
  else e = cudaErrorInvalidValue;
  return static_cast<int>(e);
}

int launch_smallh(const FwdParams& p, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (p.kv_fp8) {   // the fp8 cache: 512-wide rows, no read trace
    if (p.d_qk != 512 || p.d_v != 512 || p.trace != nullptr) return cudaErrorInvalidValue;
    const bool split = p.splits > 1;
    if (p.idx64)
      e = split ? launch_typed<int64_t, true, 512, 512, false, true>(4, p, s)
                : launch_typed<int64_t, false, 512, 512, false, true>(4, p, s);
    else
      e = split ? launch_typed<int32_t, true, 512, 512, false, true>(4, p, s)
                : launch_typed<int32_t, false, 512, 512, false, true>(4, p, s);
    return static_cast<int>(e);
  }
  // the read trace is built for the 512-wide op only (sparse_mla_fwd_ex)
  if (p.d_qk == 512 && p.d_v == 512)
    e = p.trace != nullptr ? launch_dims<512, 512, true>(0, p, s) : launch_dims<512, 512, false>(0, p, s);
  else if (p.trace != nullptr) e = cudaErrorInvalidValue;
  else if (p.d_qk == 128 && p.d_v == 128) e = launch_dims<128, 128, false>(1, p, s);
  else if (p.d_qk == 576 && p.d_v == 576) e = launch_dims<576, 576, false>(2, p, s);
  else if (p.d_qk == 576 && p.d_v == 512) e = launch_dims<576, 512, false>(3, p, s);
  else e = cudaErrorInvalidValue;
  return static_cast<int>(e);
}

}  // namespace smla
