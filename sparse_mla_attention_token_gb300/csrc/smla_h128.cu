// tcgen05 sparse MLA prefill forward for H = 128 (one token per 2-CTA cluster).
//
// The op is the has_pe=False forward of "Sparse MLA training backward"
// (aiter PR #4766, section "Contract"): all 128 heads of a token share the
// token's gathered kv rows, so heads are the MMA M dimension (M = 128).
//
// Why a CTA pair.  O[128 x 512] in fp32 is 256 KB, the whole tensor memory
// of one SM, and S needs a 512-deep contraction.  Each CTA of the pair owns
// one 256-wide half of the head dim (rank r: columns 256r..256r+255):
//   * S_r = Q[:, half r] . K[:, half r]^T, its partial scores over that half;
//   * the pair swaps partials: each CTA scales its partial to base-2 logits,
//     takes each row's maximum o_r off it, rounds the remainder to fp16 and
//     sends remainder and o_r with st.async (the bytes are counted on the
//     peer's mbarrier, so no fence per thread is needed); CTA r forms
//     S = (S_r - o_r) + f16(S_peer - o_peer) relative to o_0 + o_1 in fp32,
//     its own remainder unrounded.  Taking the row maximum off first makes the
//     rounding error depend on how far a score lies below its row's top (as
//     softmax does), not on the size of the logits;
//   * each CTA runs the online softmax on its S (the two differ only by the
//     rounding of one half's remainder; P, l and the O half of a CTA all come
//     from the same S, and rank 0 writes lse);
//   * O[:, half r] += P . V[:, half r] into its own TMEM.
//   TMEM per CTA: O half 256 columns, one 64-column S buffer (read out early
//   by its warpgroup), four 32-column P buffers (bf16 pairs, the A operand of
//   P.V: each warpgroup's P waits for the P.V two of its tiles back) and the first 128 of the
//   half's Q columns (64 columns of bf16 pairs, the A operand of the first 8
//   of S's 16 MMAs; the other 128 Q columns stay in shared memory).  Holding
//   part of Q in TMEM frees the shared memory for a fourth KV stage: a stage
//   is busy from its gather through S, the score exchange and softmax to its
//   P.V, so the ring's depth sets how many tiles are in flight.
//
// Data movement.  Producer warp 0 compacts the token's valid slots
// (0 <= idx < num_kv at the index's full width; PR #6002 "Invalid KV rows",
// "int64 indices") into a row list one token ahead and loads Q columns 0-127
// of the token's half with 2-D TMA into a 32 KB buffer; the MMA thread copies
// them into TMEM (tcgen05.cp) and then loads columns 128-255 into the same
// buffer.  Producer warps 0-6 gather each tile's 64 half rows
// (512 B each) with 16-byte cp.async straight into the 128-byte-swizzled
// layout of a 4-stage ring; each fences its landed copies into the async
// proxy before it arrives on the stage's barrier.  One tile serves as the
// K-major B operand of Q.K^T and the MN-major B operand of P.V.  The ragged
// tail of a token's last tile is zero-filled and its scores are masked: no
// invalid slot is read.
//
// Pipeline.  The MMA thread issues S and P.V as their inputs arrive, across
// token boundaries too.  Two score warpgroups take alternate tiles end to end
// (exchange, combine, softmax, P), handing the running max to each other.
// Softmax is base 2 with the sink folded once in the epilogue (m' = max(m,
// sink), l' = l 2^(m-m') + 2^(sink-m'), lse = ln2 (m' + log2 l')); the running
// max is only raised when it grows by more than 2^8, which keeps O rescales
// rare and is exact because O and l use the same stale max.  Producer warps
// 0-3 run each token's epilogue while the score warps start the next token.
//
// Warps (512 threads): 0-6 producers, 7 TMEM owner + single-thread MMA issuer,
// 8-15 two score warpgroups (thread = TMEM lane = head).  Every mbarrier wait
// is bounded: on expiry the kernel sets an error word, every role leaves its
// loop, in-flight copies and MMAs are drained, TMEM is freed and the kernel
// returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "smla_device.cuh"
#include "smla_internal.h"
#include "smla_sm100.cuh"

namespace smla {
namespace {

using namespace sm100;

constexpr int kThreads = 512;
constexpr int kProducerWarps = 7;     // warps 0-6
constexpr int kProducerThreads = kProducerWarps * 32;
constexpr int kMmaWarp = 7;
constexpr int kScoreWarp0 = 8;        // warps 8-15: two score warpgroups
constexpr int kWgThreads = 128;       // one thread per head row
constexpr int kTileN = 64;            // slots per tile
constexpr int kStages = 4;
constexpr int kMaxTopk = 1024;        // row-list capacity (two lists)
constexpr uint32_t kTmemCols = 512;
constexpr int kSBufs = 2;
constexpr int kPBufs = 2;
constexpr uint32_t kTmemS = 256;      // S buffers (64 columns each); O at 0
constexpr uint32_t kTmemP = kTmemS + kSBufs * 64;   // P buffers (32 columns of bf16 pairs each)
constexpr uint32_t kTmemQ = kTmemP + kPBufs * 32;   // Q columns 0-127 of this CTA's half (64 columns)
static_assert(kTmemQ + 64 <= kTmemCols, "TMEM columns");

// shared memory layout (offsets from a 1024-byte aligned base)
constexpr uint32_t kQOff = 0;                         // [2 col blocks][128 rows][128 B]
constexpr uint32_t kQBytes = 128 * 128 * 2;           // 32 KB: Q columns 0-127 (staged for TMEM), then 128-255
constexpr uint32_t kKVOff = kQOff + kQBytes;          // [stage][4 col blocks][64 rows][128 B]
constexpr uint32_t kStageBytes = kTileN * 256 * 2;    // 32 KB
// peer partials: [2 buffers][8 chunks][128 rows][16 B] (chunk c of row r at c * 2 KB + r * 16,
// so that a warp's 16-byte stores of one chunk for its 32 rows are 512 contiguous bytes)
constexpr uint32_t kXOff = kKVOff + kStages * kStageBytes;
constexpr int kXBufs = 2;
constexpr uint32_t kXBufBytes = 128 * kTileN * 2;     // 16 KB per buffer
constexpr uint32_t kStgOff = kXOff + kXBufs * kXBufBytes;    // O store staging: [4 warps][2][32][32 bf16]
constexpr uint32_t kStgBytes = 32 * 32 * 2;                  // 2 KB per block
constexpr uint32_t kRowsOff = kStgOff + 8 * kStgBytes;       // int32 row lists
constexpr uint32_t kMaxOff = kRowsOff + 2 * kMaxTopk * 4;    // running max handoff [2][128]
constexpr uint32_t kSumOff = kMaxOff + 2 * 128 * 4;          // epilogue sums [2][2][2][128]
constexpr uint32_t kXMaxOff = kSumOff + 2 * 512 * 4;         // peer row maxima: [2][128] fp32
constexpr uint32_t kXMaxBytes = 128 * 4;
constexpr uint32_t kXTxBytes = kXBufBytes + kXMaxBytes;      // bytes a peer sends per tile
constexpr uint32_t kBarOff = kXMaxOff + kXBufs * kXMaxBytes;
constexpr uint32_t kSmemBytes = kBarOff + 512 + 1024;  // + barriers + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

constexpr long long kTimeoutCycles = 4000000000LL;    // ~2 s at 2 GHz

struct Bars {
  uint64_t q_lo_full, q_hi_full;   // Q columns 0-127 / 128-255 of the half landed (TMA)
  uint64_t qcp_done;               // Q columns 0-127 copied into TMEM (MMA commit)
  uint64_t q_empty;                // the token's last S has completed
  uint64_t kv_full[kStages], kv_empty[kStages];
  // per tile parity (= score warpgroup), so that each barrier completes once per
  // tile of its warpgroup, in order, although the tiles share one S buffer
  uint64_t s_full[2];   // partial S(g) in TMEM (MMA commit)
  uint64_t s_free[2];   // the score warpgroup has read S(g)
  uint64_t m_ready[2][4];    // running max of tile g published (per tile parity, per quadrant)
  uint64_t epi[2];           // both score warpgroups have published their sums (per token
                             // parity: a warpgroup with no tile in a token may already
                             // be done with the next one)
  uint64_t p_full[kPBufs], pv_done[kPBufs];   // per P buffer
  uint64_t x_full[kXBufs], x_free[kXBufs];
  uint64_t o_free;
  uint64_t meta_full[2], meta_empty[2];
  uint64_t drain;
  int nvalid[2];
  int prod_nv[2];
  int prod_stop;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

struct H128Params {
  const void* idx;
  const __nv_bfloat16* kv;
  const float* sink;
  __nv_bfloat16* out;
  float* lse;
  int64_t* trace;
  unsigned int* err;
  int64_t T;
  int64_t num_kv;
  int32_t topk;
  int32_t idx64;
  float scale;
};

__device__ unsigned int g_h128_error;

// Optional per-role timeline of cluster 0 (clock64 per event, 64 tiles from
// tile SMLA_TL_START), compiled only with -DSMLA_TIMELINE for performance
// investigations.
#ifdef SMLA_TIMELINE
#ifndef SMLA_TL_START
#define SMLA_TL_START 0
#endif
__device__ long long g_timeline[2][4][64][8];
#define SMLA_TL(role, g, ev)                                                        \
  do {                                                                              \
    const uint32_t tl_g_ = static_cast<uint32_t>(g) - SMLA_TL_START;                \
    if (cluster_id_x() == 0 && tl_g_ < 64u)                                         \
      g_timeline[cluster_ctarank()][role][tl_g_][ev] = clock64();                   \
  } while (0)
#else
#define SMLA_TL(role, g, ev) \
  do {                       \
  } while (0)
#endif

// Bounded mbarrier wait; false on timeout or (unless kDrain) when another role
// gave up.  Drain waits ignore the abort flag: they wait for work already in
// flight (copies, MMAs), bounded by time alone.
template <bool kClusterScope, bool kDrain = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, Bars* b, unsigned* err,
                                         unsigned code) {
  if (kClusterScope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t n = 1;; ++n) {
    if (kClusterScope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity))
      return true;
    if ((n & 15) == 0) {
      if (!kDrain && *reinterpret_cast<volatile int*>(&b->abort_flag)) return false;
      if (clock64() - t0 > kTimeoutCycles) {
        *reinterpret_cast<volatile int*>(&b->abort_flag) = 1;
        atomicOr(err, code);
        return false;
      }
    }
  }
}

__device__ __forceinline__ uint32_t bar_addr(const uint64_t& b) { return smem_u32(&b); }

// Compact one token's valid slots (slot order) into `rows`; returns the count.
// Warp-collective (warp 0).  Loads are issued kUnroll deep before use, so a
// list of 32 * kUnroll slots costs one round trip to L2; the compaction sits
// between a token's last gather and the next token's first.  int64 lists load
// 32 deep (one round for 1024 slots: 3.7% faster than 16 deep on 1024-slot
// int64 lists), int32 lists 16 deep (32 deep measured 2.3% slower on 512-slot
// lists).  With a read trace, the entries past the token's valid count are set
// to -1 here (no copy ever reads for them); the gather writes the others.
template <typename IdxT>
__device__ __forceinline__ int compact_token(const H128Params& p, int64_t tok, int* rows,
                                             bool write_trace, int lane) {
  constexpr int kUnroll = sizeof(IdxT) == 8 ? 32 : 16;
  const IdxT* ip = static_cast<const IdxT*>(p.idx) + tok * p.topk;
  int nv = 0;
  for (int base = 0; base < p.topk; base += 32 * kUnroll) {
    IdxT v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int j = base + u * 32 + lane;
      v[u] = (j < p.topk) ? ip[j] : IdxT(-1);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int j = base + u * 32 + lane;
      const bool ok = (j < p.topk) && slot_valid<IdxT>(v[u], p.num_kv);
      const unsigned ball = __ballot_sync(0xffffffffu, ok);
      if (ok) rows[nv + __popc(ball & ((1u << lane) - 1u))] = static_cast<int>(v[u]);  // exact: num_kv < 2^31
      nv += __popc(ball);
    }
  }
  if (write_trace)
    for (int k = nv + lane; k < p.topk; k += 32) p.trace[tok * p.topk + k] = -1;
  __syncwarp();
  return nv;
}

// One arrive per warp on a barrier that counts warps: the warp-level sync orders
// every lane's prior accesses (each lane fences its own first where a proxy or
// tcgen05 ordering needs it) before lane 0's release arrive.  Warp-collective.
// Per-thread arrives (224 a tile from the producers, 128 from a score warpgroup)
// all update one barrier word; one per warp measured 1% faster on the kernel.
__device__ __forceinline__ void warp_arrive(uint32_t bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// This warp's cp.async copies of a tile have landed (wait_group in every lane):
// each lane makes its own visible to the tensor core's async proxy, then the warp
// counts them on the barrier.
__device__ __forceinline__ void land_and_arrive(uint32_t bar, int lane) {
  fence_proxy_async_smem();
  warp_arrive(bar, lane);
}

// Warps 0-6 gather every tile together: warp w copies rows w, w+7, ... (lane c
// copies 16-byte chunk c of each 512-byte half row, one contiguous half row
// per instruction).  Each warp counts its copies on the stage's barrier as soon
// as they have landed and been fenced into the async proxy.  Warp 0 also
// compacts the index lists one token ahead into a double-buffered row list,
// publishes each token's valid count, loads Q columns 0-127 of the token's half
// with 2-D TMA once the previous token's last S has completed (the MMA thread
// copies them into TMEM and loads columns 128-255) and prefetches the next
// token's Q into L2.
template <typename IdxT, bool kTrace>
__device__ void producer_role(const H128Params& p, const CUtensorMap* tm_q, const CUtensorMap* tm_o,
                              uint8_t* base, Bars* b, uint32_t tmem, uint32_t rank, int warp,
                              int lane) {
  const uint32_t sbase = smem_u32(base);
  int* rows_buf = reinterpret_cast<int*>(base + kRowsOff);   // [2][kMaxTopk]
  const int64_t cid = cluster_id_x(), ncl = nclusters_x();
  const char* kvb = reinterpret_cast<const char*>(p.kv) + 512 * rank;   // this CTA's half
  const int c = lane;                                  // 16-byte chunk of the half row
  const uint32_t chunk_off = (c >> 3) * 8192;          // its 64-column block
  // the read trace exists only in the instantiation built for it, so that the
  // production gather loop carries no trace code
  const bool trace = kTrace && rank == 0;
  uint32_t gt = 0, qn = 0, q_loads = 0;
  int it = 0;

  // epilogue state (warps 0-3, warp = TMEM lane quadrant)
  const bool epi_warp = warp < 4;
  const int qd = warp & 3;
  const int row = 32 * qd + lane;
  const uint32_t tl = tmem + (static_cast<uint32_t>(32 * qd) << 16);
  const float sk = (epi_warp && p.sink != nullptr) ? p.sink[row] * kLog2e : -INFINITY;
  const float* l_sh = reinterpret_cast<const float*>(base + kSumOff);
  const uint32_t stg = sbase + kStgOff + qd * 2 * kStgBytes;   // two 2 KB blocks per warp
  bool ep_pend = false;   // a token whose epilogue has not run yet
  int64_t ep_tok = 0;
  uint32_t ep_gl = 0, et = 0;
  auto epilogue = [&]() -> bool {
    ep_pend = false;
    const uint32_t e = et++;
    // both score warpgroups have published their sums
    if (!__all_sync(0xffffffffu, wait_bar<false>(bar_addr(b->epi[e & 1]), (e >> 1) & 1, b, p.err,
                                                 1u)))
      return false;
    const float* lsh = l_sh + (e & 1) * 512;
    const float l0 = lsh[row], m0 = lsh[128 + row], l1 = lsh[256 + row], m1 = lsh[384 + row];
    const float m_run = fmaxf(m0, m1);   // the max of the token's last tile
    const float l_run = l0 * ex2(m0 - m_run) + l1 * ex2(m1 - m_run);
    // the token's last P.V has completed
    if (!__all_sync(0xffffffffu, wait_bar<false>(bar_addr(b->pv_done[ep_gl % kPBufs]),
                                                 (ep_gl / kPBufs) & 1, b, p.err, 1u)))
      return false;
    if (lane == 0) SMLA_TL(3, ep_gl, 5);
    tc_fence_after();
    float m2 = m_run, l2 = l_run;
    if (sk != -INFINITY) {
      m2 = fmaxf(m_run, sk);
      l2 = l_run * ex2(m_run - m2) + ex2(sk - m2);
    }
    const float f = ex2(m_run - m2) / l2;
    // 32 x 32 bf16 blocks through a double-buffered staging block (64-byte
    // rows, 64-byte swizzle: 16-byte chunk q of row r at q ^ ((r >> 1) & 3)),
    // written to global memory by TMA.  O is released as soon as all of it has
    // been read from TMEM: the first kHeld blocks wait in registers (packed
    // bf16) while the others go through the staging blocks.
    constexpr int kHeld = 3;
    uint32_t held[kHeld][16];
    auto put = [&](int cc, const uint32_t* w16, int slot) {   // one block: staging -> TMA
      const uint32_t sb = stg + (slot & 1) * kStgBytes;
      if (lane == 0) bulk_wait_read<1>();   // the block stored two slots ago has left sb
      __syncwarp();
#pragma unroll
      for (int q = 0; q < 4; ++q)
        st_shared_v4(sb + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4),
                     make_uint4(w16[4 * q], w16[4 * q + 1], w16[4 * q + 2], w16[4 * q + 3]));
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(tm_o, sb, 256 * int(rank) + 32 * cc, static_cast<int>(ep_tok * 128 + 32 * qd));
        bulk_commit();
      }
    };
    auto load = [&](int cc, uint32_t* w16) {   // one block: TMEM -> normalised bf16 pairs
      uint32_t o[32];
      tmem_ld32(tl + 32 * cc, o);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i)
        w16[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * f, __uint_as_float(o[2 * i + 1]) * f);
    };
#pragma unroll
    for (int cc = 0; cc < kHeld; ++cc) load(cc, held[cc]);
#pragma unroll 1
    for (int cc = kHeld; cc < 8; ++cc) {
      uint32_t w16[16];
      load(cc, w16);
      put(cc, w16, cc - kHeld);
    }
    tc_fence_before();
    warp_arrive(bar_addr(b->o_free), lane);   // all of O has been read
#pragma unroll
    for (int cc = 0; cc < kHeld; ++cc) put(cc, held[cc], 8 - kHeld + cc);
    if (lane == 0) SMLA_TL(3, ep_gl, 6);
    if (rank == 0) p.lse[ep_tok * 128 + row] = (m2 + log2f(l2)) * kLn2;
    return true;
  };
  bool run = true;

  if (warp == 0 && cid < p.T) {
    const int nv = compact_token<IdxT>(p, cid, rows_buf, trace, lane);
    if (lane == 0) b->prod_nv[0] = nv;
  }
  for (int64_t tok = cid; tok < p.T; tok += ncl, ++it) {
    const int buf = it & 1;
    if (warp == 0 && lane == 0) b->prod_stop = *reinterpret_cast<volatile int*>(&b->abort_flag);
    named_bar_sync(1, kProducerThreads);   // this token's list is complete; token it-1 is done
    if (b->prod_stop) break;
    const int nv = b->prod_nv[buf];
    const int* rows = rows_buf + buf * kMaxTopk;
    if (warp == 0 && tok + ncl < p.T) {
      // the next token's index row into L2: warp 0 compacts it at the end of
      // this token, on the way to the next token's first gather
      const int64_t bytes = int64_t(p.topk) * int64_t(sizeof(IdxT));
      const char* ip = static_cast<const char*>(p.idx) + (tok + ncl) * bytes;
      for (int64_t o = int64_t(lane) * 128; o < bytes; o += 32 * 128) prefetch_l2(ip + o);
    }
    if (warp == 0) {
      const int slot = it & 1;
      bool ok = __all_sync(0xffffffffu, wait_bar<false>(bar_addr(b->meta_empty[slot]),
                                                        ((it >> 1) & 1) ^ 1, b, p.err, 1u));
      if (ok && lane == 0) {
        b->nvalid[slot] = nv;
        mbar_arrive(bar_addr(b->meta_full[slot]));
      }
      if (ok && nv > 0) {
        if (lane == 0) SMLA_TL(0, gt, 4);
        ok = __all_sync(0xffffffffu,
                        wait_bar<false>(bar_addr(b->q_empty), (qn & 1) ^ 1, b, p.err, 1u));
        if (ok && lane == 0) {
          SMLA_TL(0, gt, 3);
          // columns 0-127 of the half; the MMA thread copies them into TMEM and
          // then loads columns 128-255 into the same buffer
          mbar_arrive_expect_tx(bar_addr(b->q_lo_full), kQBytes);
#pragma unroll
          for (int cb = 0; cb < 2; ++cb)
            tma_load_2d(sbase + kQOff + cb * 16384, tm_q, 256 * int(rank) + 64 * cb,
                        static_cast<int>(tok * 128), bar_addr(b->q_lo_full));
          ++q_loads;
          // the next token's Q half into L2 now, so its load at the token switch is short
          if (tok + ncl < p.T) {
#pragma unroll
            for (int cb = 0; cb < 4; ++cb)
              tma_prefetch_2d(tm_q, 256 * int(rank) + 64 * cb, static_cast<int>((tok + ncl) * 128));
          }
        }
      }
    }
    if (nv == 0 && epi_warp) {   // nothing valid: O = 0; lse = sink (finite) or -inf
      uint4* orow = reinterpret_cast<uint4*>(p.out + (tok * 128 + row) * int64_t(kHeadDim) +
                                             256 * rank);
#pragma unroll
      for (int cc = 0; cc < 32; ++cc) orow[cc] = make_uint4(0u, 0u, 0u, 0u);
      if (rank == 0) p.lse[tok * 128 + row] = (sk != -INFINITY) ? sk * kLn2 : -INFINITY;
    }
    const int64_t next = tok + ncl;
    bool compacted = (warp != 0) || (next >= p.T);
    auto compact_next = [&]() {
      const int nn = compact_token<IdxT>(p, next, rows_buf + (buf ^ 1) * kMaxTopk, trace, lane);
      if (lane == 0) b->prod_nv[buf ^ 1] = nn;
      compacted = true;
    };
    if (nv > 0) {
      ++qn;
      const int ntiles = (nv + kTileN - 1) / kTileN;
      for (int j = 0; j < ntiles; ++j) {
        const uint32_t g = gt + j;
        const uint32_t s = g % kStages, ph = (g / kStages) & 1;
        // this stage is freed by P.V(g - kStages): once that is the pending
        // token's last P.V (or a later one), run the token's epilogue before
        // waiting for the stage
        if (epi_warp && ep_pend && g >= ep_gl + kStages) {
          if (!(run = epilogue())) break;
        }
        const bool ok = __all_sync(0xffffffffu, wait_bar<false>(bar_addr(b->kv_empty[s]),
                                                                ph ^ 1, b, p.err, 1u));
        if (!ok) break;
        if (lane == 0) SMLA_TL(0, g, 0);
        const uint32_t dst = sbase + kKVOff + s * kStageBytes + chunk_off;
        // this warp copies rows r = warp + 7k; lane k holds row k's index
        const int rk = warp + kProducerWarps * lane, sl = j * kTileN + rk;
        const int my_row = (rk < kTileN && sl < nv) ? rows[sl] : -1;
#pragma unroll
        for (int k = 0; k < (kTileN + kProducerWarps - 1) / kProducerWarps; ++k) {
          const int r = warp + kProducerWarps * k;
          const int rr = __shfl_sync(0xffffffffu, my_row, k);
          if (r < kTileN) {
            const bool valid = rr >= 0;                // the ragged tail is zero-filled
            const char* src = valid ? kvb + int64_t(rr) * 1024 + c * 16 : kvb;
            cp_async_16(dst + r * 128 + (((c & 7) ^ (r & 7)) << 4), src, valid ? 16u : 0u);
            // read trace: the row this copy reads, recovered from its source address
            if constexpr (kTrace)
              if (trace && c == 0 && valid) p.trace[tok * p.topk + j * kTileN + r] = (src - kvb) >> 10;
          }
        }
        cp_async_commit();
        if (lane == 0) SMLA_TL(0, g, 1);
        // count this tile as soon as its copies have landed: the MMA waits for the
        // slowest warp, so counting it after the next tile's issue (overlapping
        // the two) made every tile ready later (2% slower overall)
        cp_async_wait<0>();
        land_and_arrive(bar_addr(b->kv_full[s]), lane);
        if (lane == 0) SMLA_TL(0, g, 2);
        if (!compacted && j == ntiles - 1) compact_next();   // after counting the tile
      }
      gt += ntiles;
      if (epi_warp && run) {   // epilogues run in token order
        if (ep_pend) run = epilogue();
        ep_pend = true;
        ep_tok = tok;
        ep_gl = gt - 1;
      }
    }
    if (!compacted) compact_next();
    // after a failed epilogue (the abort flag is set) every producer warp leaves
    // together at the next token's start, never from here
  }
  if (epi_warp && run && ep_pend) epilogue();
  if (epi_warp && lane == 0) bulk_wait<0>();   // every O block stored before the CTA exits
  cp_async_wait<0>();   // drain: no copy of ours may land after the CTA exits
  if (warp == 0 && lane == 0 && q_loads > 0)
    wait_bar<false, true>(bar_addr(b->q_lo_full), (q_loads - 1) & 1, b, p.err, 1u);
}

// Warp 7, lane 0: issues every tcgen05.mma and tcgen05.cp of the CTA.
//   S(g)  = Q_half . K_half(g)^T -> the S buffer (M=128, N=64, K=256: 16 MMAs,
//           the first 8 with Q columns 0-127 from TMEM, the last 8 with
//           columns 128-255 from shared memory)
//   PV(g) : O_half += P(g) . V_half(g)       (M=128, N=256, K=64: 4 MMAs,
//           P(g) read from TMEM buffer g%4, V from the shared-memory stage)
// Per token it also copies Q columns 0-127 into TMEM once they have landed and
// then loads columns 128-255 into the freed buffer.
// Event-driven: each pass polls (without blocking) whether the next P.V or the
// next S has its inputs and issues whichever is ready, P.V first because it
// releases a KV stage.  No operation waits behind another one's inputs.  A
// pass without progress for ~2 s (or another role giving up) ends the loop.
__device__ void mma_role(const H128Params& p, uint8_t* base, Bars* b, uint32_t tmem,
                         const CUtensorMap* tm_q, uint32_t rank) {
  const uint32_t sbase = smem_u32(base);
  const int64_t cid = cluster_id_x(), ncl = nclusters_x();
  constexpr uint32_t kIdescS = idesc_bf16_f32(128, kTileN, false, false);
  constexpr uint32_t kIdescO = idesc_bf16_f32(128, 256, false, true);
  constexpr int kRing = 8;   // issued-S tiles awaiting their P.V (at most kSBufs + 2; < 32 bits)
  // Operand descriptors are built once and advanced by adding (byte offset / 16)
  // to their start-address field (shared addresses < 256 KB: no carry out of it):
  // a thread issuing tcgen05.mma back to back is bound by its own issue path.
  const uint64_t d_k0 = sdesc_sw128(sbase + kKVOff, 16, 1024);     // stage 0, K-major
  const uint64_t d_v0 = sdesc_sw128(sbase + kKVOff, 8192, 1024);   // stage 0, MN-major
  const uint64_t d_q0 = sdesc_sw128(sbase + kQOff, 16, 1024);

  // S side: token walk
  int64_t tok = cid;
  int it = 0;                 // token iteration (meta slot / parity)
  int nt = 0, j = 0;          // tiles of the current token, next tile index in it
  bool have_meta = false;
  int q_state = 0;            // 0: wait Q low half, 1: copy done?, 2: wait Q high half, 3: Q ready
  uint32_t hi_loads = 0;      // Q high-half loads issued
  uint32_t qn = 0, tokn = 0;  // tokens with tiles: Q loads consumed, token index
  uint32_t sg = 0;            // next S tile (global)
  // P.V side
  uint32_t pg = 0;            // next P.V tile (global)
  // per issued S awaiting its P.V, bit (g mod 32): the tile is its token's first /
  // its token's index is odd (registers, not a dynamically indexed local array)
  uint32_t first_bits = 0, todd_bits = 0;

  // inputs already seen ready for the next P.V / the next S: none of them can
  // complete another phase before that operation issues, so they are polled
  // until seen once (every poll is a shared-memory access behind the
  // producers' and score warps' traffic)
  bool p_ok = false, kv_ok = false, sf_ok = false;
  uint32_t idle = 0;          // passes since the last progress
  long long last = 0;
  while (true) {
    bool progress = false;
    // ---- the next token's Q (gates its first S): ahead of a ready P.V
    if (have_meta && q_state < 3) {
      if (q_state == 0) {
        // Q columns 0-127 landed (loaded once the previous token's last S completed):
        // into TMEM, 16 K elements (8 columns) per copy
        if (mbar_test_wait(bar_addr(b->q_lo_full), qn & 1)) {
          SMLA_TL(1, sg, 6);
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tmem_cp_128x256b(tmem + kTmemQ + 8 * kk, d_q0 + (kk >> 2) * 1024 + (kk & 3) * 2);
          mma_commit(bar_addr(b->qcp_done));
          q_state = 1;
          progress = true;
        }
      } else if (q_state == 1) {
        // the copies have read the buffer: columns 128-255 into it
        if (mbar_test_wait(bar_addr(b->qcp_done), qn & 1)) {
          SMLA_TL(1, sg, 7);
          mbar_arrive_expect_tx(bar_addr(b->q_hi_full), kQBytes);
#pragma unroll
          for (int cb = 0; cb < 2; ++cb)
            tma_load_2d(sbase + kQOff + cb * 16384, tm_q, 256 * int(rank) + 128 + 64 * cb,
                        static_cast<int>(tok * 128), bar_addr(b->q_hi_full));
          ++hi_loads;
          q_state = 2;
          progress = true;
        }
      } else if (q_state == 2) {
        if (mbar_test_wait(bar_addr(b->q_hi_full), qn & 1)) {
          SMLA_TL(1, sg, 5);
          tc_fence_after();
          q_state = 3;
          progress = true;
        }
      }
    }
    // ---- next P.V
    if (pg < sg) {
      const uint32_t bit = 1u << (pg & 31u);
      const bool first = (first_bits & bit) != 0;
      if (!p_ok) p_ok = mbar_test_wait(bar_addr(b->p_full[pg % kPBufs]), (pg / kPBufs) & 1);
      if (p_ok && (!first || mbar_test_wait(bar_addr(b->o_free), ((todd_bits & bit) ? 1u : 0u) ^ 1u))) {
        SMLA_TL(1, pg, 3);
        tc_fence_after();
        const uint32_t s = pg % kStages;
        const uint32_t ptm = tmem + kTmemP + (pg % kPBufs) * 32;   // P: 64 bf16 = 32 columns
        // V as MN-major B: 64-column blocks 8 KB apart, 8-slot groups 1 KB apart; a K
        // step is 16 slot rows (2 KB = 128 in the descriptor's start-address field)
        const uint64_t vd = d_v0 + s * (kStageBytes >> 4);
        mma_bf16_ts(tmem, ptm, vd, kIdescO, first ? 0u : 1u);
#pragma unroll
        for (int kk = 1; kk < kTileN / 16; ++kk) mma_bf16_ts(tmem, ptm + kk * 8, vd + kk * 128, kIdescO, 1u);
        mma_commit(bar_addr(b->kv_empty[s]));
        mma_commit(bar_addr(b->pv_done[pg % kPBufs]));
        SMLA_TL(1, pg, 4);
        ++pg;
        p_ok = false;
        progress = true;
      }
    }
    // ---- next S (walking tokens; tokens without valid slots have no tiles), in
    // the same pass as a P.V issued above (P.V still goes first)
    if (tok < p.T && sg - pg < kRing) {
      if (!have_meta) {
        const int slot = it & 1;
        if (mbar_test_wait(bar_addr(b->meta_full[slot]), (it >> 1) & 1)) {
          const int nv = b->nvalid[slot];
          mbar_arrive(bar_addr(b->meta_empty[slot]));
          nt = (nv + kTileN - 1) / kTileN;
          j = 0;
          have_meta = true;
          q_state = 0;
          progress = true;
          if (nt == 0) {   // nothing to compute for this token
            have_meta = false;
            tok += ncl;
            ++it;
          }
        }
      } else if (q_state < 3) {
        // the Q chain advances above
      } else {
        const uint32_t s = sg % kStages, ph = (sg / kStages) & 1;
        const uint32_t sb = sg % kSBufs;
        // the tile has landed and the S buffer's previous tile, S(sg - kSBufs), has been read
        if (!kv_ok) kv_ok = mbar_test_wait(bar_addr(b->kv_full[s]), ph);
        if (kv_ok && !sf_ok)
          sf_ok = sg < kSBufs ||
                  mbar_test_wait(bar_addr(b->s_free[(sg - kSBufs) & 1]), ((sg - kSBufs) >> 1) & 1);
        if (kv_ok && sf_ok) {
          kv_ok = sf_ok = false;
          SMLA_TL(1, sg, 1);
          tc_fence_after();
          // K rows as K-major B (64-column blocks 8 KB apart); a K step of 16 elements is
          // 32 B inside a 128 B row (2 in the descriptor's start-address field)
          const uint64_t kd = d_k0 + s * (kStageBytes >> 4);
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) {
            const uint64_t bd = kd + (kk >> 2) * 512 + (kk & 3) * 2;
            if (kk < 8) {   // Q columns 0-127 from TMEM
              mma_bf16_ts(tmem + kTmemS + sb * kTileN, tmem + kTmemQ + 8 * kk, bd, kIdescS,
                          kk > 0 ? 1u : 0u);
            } else {        // Q columns 128-255 from shared memory (16 KB per 64 columns)
              const uint64_t a = d_q0 + ((kk - 8) >> 2) * 1024 + (kk & 3) * 2;
              mma_bf16_ss(tmem + kTmemS + sb * kTileN, a, bd, kIdescS, 1u);
            }
          }
          mma_commit(bar_addr(b->s_full[sg & 1]));
          SMLA_TL(1, sg, 0);
          {
            const uint32_t bit = 1u << (sg & 31u);
            first_bits = j == 0 ? (first_bits | bit) : (first_bits & ~bit);
            todd_bits = (tokn & 1u) ? (todd_bits | bit) : (todd_bits & ~bit);
          }
          ++sg;
          progress = true;
          if (++j == nt) {   // the token's last S: its Q may be replaced
            mma_commit(bar_addr(b->q_empty));
            ++qn;
            ++tokn;
            have_meta = false;
            tok += ncl;
            ++it;
          }
        }
      }
    }
    if (tok >= p.T && pg == sg) break;   // every S and every P.V issued
    // keep polling without a sleep: the next MMA issues as soon as its inputs are
    // ready (a 32 ns sleep here cost 1-2%); the abort flag and the no-progress
    // timer are looked at every 16th idle pass
    if (progress) {
      idle = 0;
    } else if ((++idle & 15u) == 0) {
      if (idle == 16) last = clock64();   // the idle stretch's first look
      if (*reinterpret_cast<volatile int*>(&b->abort_flag)) break;
      if (clock64() - last > kTimeoutCycles) {
        *reinterpret_cast<volatile int*>(&b->abort_flag) = 1;
        atomicOr(p.err, 2u);
        break;
      }
    }
  }
  // drain: every MMA and copy issued must complete before TMEM is freed, and
  // no Q load of ours may land after the CTA exits
  mma_commit(bar_addr(b->drain));
  wait_bar<false, true>(bar_addr(b->drain), 0, b, p.err, 2u);
  if (hi_loads > 0) wait_bar<false, true>(bar_addr(b->q_hi_full), (hi_loads - 1) & 1, b, p.err, 2u);
}

// Largest / smallest of a row's 64 raw fp32 partial scores (bit patterns).
__device__ __forceinline__ float row_max64(const uint32_t* v) {
  float t[22];
#pragma unroll
  for (int k = 0; k < 21; ++k)
    t[k] = max3f(__uint_as_float(v[3 * k]), __uint_as_float(v[3 * k + 1]), __uint_as_float(v[3 * k + 2]));
  t[21] = __uint_as_float(v[63]);
  float u[8];
#pragma unroll
  for (int k = 0; k < 7; ++k) u[k] = max3f(t[3 * k], t[3 * k + 1], t[3 * k + 2]);
  u[7] = t[21];
  return max3f(max3f(u[0], u[1], u[2]), max3f(u[3], u[4], u[5]), fmaxf(u[6], u[7]));
}
__device__ __forceinline__ float row_min64(const uint32_t* v) {
  float t[22];
#pragma unroll
  for (int k = 0; k < 21; ++k)
    t[k] = min3f(__uint_as_float(v[3 * k]), __uint_as_float(v[3 * k + 1]), __uint_as_float(v[3 * k + 2]));
  t[21] = __uint_as_float(v[63]);
  float u[8];
#pragma unroll
  for (int k = 0; k < 7; ++k) u[k] = min3f(t[3 * k], t[3 * k + 1], t[3 * k + 2]);
  u[7] = t[21];
  return min3f(min3f(u[0], u[1], u[2]), min3f(u[3], u[4], u[5]), fminf(u[6], u[7]));
}

// Warps 8-15: two score warpgroups.  Warpgroup w handles the tiles g with
// g % 2 == w (tile numbers count every tile of this CTA); thread = TMEM lane =
// head `row`.  For its tile g a warpgroup
//   1. reads this CTA's partial scores S_r(g) (64 fp32) from the S buffer and
//      frees the buffer; scales them to base-2 logits, takes the row's largest
//      o_r off and rounds the remainder to fp16;
//   2. st.asyncs remainder and o_r into the peer's receive buffer g%2 (the
//      bytes are counted on the peer's mbarrier);
//   3. once the peer's are in, forms S - off = (S_r - o_r) + f16(S_peer - o_peer)
//      in fp32 with off = o_0 + o_1 (its own remainder unrounded);
//   4. takes the running max: it waits for the max the other warpgroup
//      settled for tile g-1 (per row, through shared memory), raises it only
//      when the tile's max exceeds it by more than 2^8, and publishes it for
//      tile g+1;
//   5. writes P = 2^(S - m) (bf16) into TMEM P buffer g%4 and, when the max
//      was raised, first rescales O (after P.V(g-1) has completed).
// Each warpgroup keeps the sum l of its own tiles (relative to the max it last
// saw); at the end of a token the two sums are merged through shared memory
// and the warpgroups normalise and store one half each of this CTA's O half.
__device__ void score_role(const H128Params& p, uint8_t* base, Bars* b, uint32_t tmem,
                           uint32_t rank, int warp, int lane) {
  const uint32_t sbase = smem_u32(base);
  const int wg = (warp - kScoreWarp0) >> 2;   // 0 or 1
  const int qd = warp & 3;                    // TMEM lane quadrant
  const int row = 32 * qd + lane;
  const uint32_t tl = tmem + (static_cast<uint32_t>(32 * qd) << 16);
  const int64_t cid = cluster_id_x(), ncl = nclusters_x();
  const uint32_t peer = rank ^ 1u;
  const float sl2 = p.scale * kLog2e;
  float* m_sh = reinterpret_cast<float*>(base + kMaxOff);   // [2 tile parities][128]
  float* l_sh = reinterpret_cast<float*>(base + kSumOff);   // [2 tokens][2 wg][2 (l, m)][128]
  const float* xmax_sh = reinterpret_cast<const float*>(base + kXMaxOff);   // [2][128]
  uint32_t recv_local[kXBufs], recv_peer[kXBufs], xfull_peer[kXBufs], xfree_peer[kXBufs];
  uint32_t xmax_peer[kXBufs];
#pragma unroll
  for (int i = 0; i < kXBufs; ++i) {
    recv_local[i] = sbase + kXOff + i * kXBufBytes + row * 16;   // chunk c at + c * 2 KB
    recv_peer[i] = map_peer(recv_local[i], peer);
    xmax_peer[i] = map_peer(sbase + kXMaxOff + (i * 128 + row) * 4, peer);
    xfull_peer[i] = map_peer(bar_addr(b->x_full[i]), peer);
    xfree_peer[i] = map_peer(bar_addr(b->x_free[i]), peer);
  }

  uint32_t gt = 0, et = 0;   // tiles before this token; tokens with tiles so far
  int it = 0;
  bool ok = true;
  for (int64_t tok = cid; tok < p.T && ok; tok += ncl, ++it) {
    const int slot = it & 1;
    ok = __all_sync(0xffffffffu, wait_bar<false>(bar_addr(b->meta_full[slot]), (it >> 1) & 1,
                                                 b, p.err, 4u));
    if (!ok) break;
    const int nv = b->nvalid[slot];
    warp_arrive(bar_addr(b->meta_empty[slot]), lane);
    if (nv == 0) continue;   // written by the producer warps
    const int ntiles = (nv + kTileN - 1) / kTileN;
    float l_w = 0.f, m_lw = -INFINITY;   // this warpgroup's sum and the max it is relative to
    for (int j = 0; j < ntiles; ++j) {
      const uint32_t g = gt + j;
      if (static_cast<int>(g & 1u) != wg) continue;
      const uint32_t sb = g % kSBufs, xb = g % kXBufs, pb = g % kPBufs;
      // 1. my partial scores, rounded to fp16; the S buffer is free again
      if (!(ok = __all_sync(0xffffffffu, wait_bar<false>(bar_addr(b->s_full[g & 1]),
                                                         (g >> 1) & 1, b, p.err, 8u))))
        break;
      if (row == 0) SMLA_TL(2, g, 0);
      tc_fence_after();
      const int nvt = min(kTileN, nv - j * kTileN);   // valid columns of this tile
      float2 ownf[32];   // this CTA's remainders, kept in fp32
      uint32_t own[32];
      float o_own;   // this row's largest scaled partial: o_own - (what was sent) is the partial
      {
        uint32_t sv[64];
        tmem_ld32(tl + kTmemS + sb * kTileN, sv);
        tmem_ld32(tl + kTmemS + sb * kTileN + 32, sv + 32);
        tmem_wait_ld();
        tc_fence_before();
        warp_arrive(bar_addr(b->s_free[g & 1]), lane);
        // the row's top partial in base-2 logits over the valid columns (rounding
        // is monotone, so the extreme raw value scales to the largest scaled one;
        // a negative scale turns the smallest raw value into it).  The zero-filled
        // tail of a ragged tile takes column 0's value, which changes neither.
        if (nvt < kTileN) {
#pragma unroll
          for (int i = 1; i < 64; ++i) sv[i] = (i < nvt) ? sv[i] : sv[0];
        }
        o_own = sl2 * (sl2 >= 0.f ? row_max64(sv) : row_min64(sv));
        // S sl2 - o_own in one rounding, then fp16
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float2 t = fma2(make_float2(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])),
                                make_float2(sl2, sl2), make_float2(-o_own, -o_own));
          ownf[i] = t;
          own[i] = pack_f16x2(t.x, t.y);
        }
      }
      if (row == 0) SMLA_TL(3, g, 0);
      // 2. to the peer, once it has consumed what it got in buffer xb two tiles ago
      if (!(ok = __all_sync(0xffffffffu, wait_bar<true>(bar_addr(b->x_free[xb]),
                                                        ((g / kXBufs) & 1) ^ 1, b, p.err, 8u))))
        break;
      if (row == 0) SMLA_TL(3, g, 1);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_async_v4(recv_peer[xb] + c * 2048,
                    make_uint4(own[4 * c], own[4 * c + 1], own[4 * c + 2], own[4 * c + 3]),
                    xfull_peer[xb]);
      st_async_b32(xmax_peer[xb], __float_as_uint(o_own), xfull_peer[xb]);
      if (row == 0) mbar_arrive_expect_tx(bar_addr(b->x_full[xb]), kXTxBytes);
      if (row == 0) SMLA_TL(2, g, 1);
      // 3. the peer's partial scores; full base-2 scores, tail masked
      if (!(ok = __all_sync(0xffffffffu, wait_bar<true>(bar_addr(b->x_full[xb]),
                                                        (g / kXBufs) & 1, b, p.err, 8u))))
        break;
      if (row == 0) SMLA_TL(2, g, 2);
      // scores relative to off = o_0 + o_1
      const float off = o_own + xmax_sh[xb * 128 + row];
      float s[64];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(base + (recv_local[xb] - sbase) + c * 2048);
        const uint32_t pv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 t = add_f32_f16x2(ownf[4 * c + q], pv[q]);   // own + f16(peer)
          s[8 * c + 2 * q] = t.x;
          s[8 * c + 2 * q + 1] = t.y;
        }
      }
      if (nvt < kTileN) {   // the token's ragged last tile
#pragma unroll
        for (int i = 0; i < 64; ++i) s[i] = (i < nvt) ? s[i] : -INFINITY;
      }
      if (row == 0) SMLA_TL(3, g, 2);
      // 4. running max: the one settled for tile g-1 (also across tokens, so that
      //    its slot is read before it is written again), raised by more than 2^8 only
      float mx;
      {
        float t[22];
#pragma unroll
        for (int k = 0; k < 21; ++k) t[k] = max3f(s[3 * k], s[3 * k + 1], s[3 * k + 2]);
        t[21] = s[63];
        float u[8];
#pragma unroll
        for (int k = 0; k < 7; ++k) u[k] = max3f(t[3 * k], t[3 * k + 1], t[3 * k + 2]);
        u[7] = t[21];
        mx = max3f(max3f(u[0], u[1], u[2]), max3f(u[3], u[4], u[5]), fmaxf(u[6], u[7])) + off;
      }
      float m_prev = -INFINITY;
      if (g >= 1) {
        if (!(ok = __all_sync(0xffffffffu,
                              wait_bar<false>(bar_addr(b->m_ready[(g - 1) & 1][qd]),
                                              ((g - 1) >> 1) & 1, b, p.err, 4u))))
          break;
        if (j > 0) m_prev = m_sh[((g - 1) & 1) * 128 + row];
      }
      if (row == 0) SMLA_TL(3, g, 3);
      const bool need = mx > m_prev + 8.f;
      const float m_new = need ? mx : m_prev;
      m_sh[(g & 1) * 128 + row] = m_new;
      warp_arrive(bar_addr(b->m_ready[g & 1][qd]), lane);
      if (row == 0) SMLA_TL(2, g, 3);
      // 5. P = 2^(S - m), this warpgroup's sum (s holds S - off)
      const float m_rel = m_new - off;
      float2 sum4[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) sum4[k] = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float2 t = add2(make_float2(s[2 * i], s[2 * i + 1]), make_float2(-m_rel, -m_rel));
        t.x = ex2(t.x);
        t.y = ex2(t.y);
        s[2 * i] = t.x;
        s[2 * i + 1] = t.y;
        sum4[i & 3] = add2(sum4[i & 3], t);
      }
      const float2 sa = add2(add2(sum4[0], sum4[1]), add2(sum4[2], sum4[3]));
      l_w = l_w * ex2(m_lw - m_new) + (sa.x + sa.y);
      m_lw = m_new;
      // P buffer pb was last read by P.V(g-4); O may only be rescaled after P.V(g-1)
      if (g >= kPBufs) {
        if (!(ok = __all_sync(0xffffffffu, wait_bar<false>(bar_addr(b->pv_done[pb]),
                                                           ((g / kPBufs) & 1) ^ 1, b, p.err, 4u))))
          break;
        tc_fence_after();
      }
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        if (!(ok = __all_sync(0xffffffffu,
                              wait_bar<false>(bar_addr(b->pv_done[(g - 1) % kPBufs]),
                                              ((g - 1) / kPBufs) & 1, b, p.err, 4u))))
          break;
        tc_fence_after();
        const float alpha = ex2(m_prev - m_new);   // 1 for rows whose max stayed
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t o[32];
          tmem_ld32(tl + 32 * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tl + 32 * c, o);
        }
      }
      if (row == 0) SMLA_TL(3, g, 4);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(s[32 * h + 2 * i], s[32 * h + 2 * i + 1]);
        tmem_st16(tl + kTmemP + pb * 32 + 16 * h, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(bar_addr(b->p_full[pb]), lane);
      // receive buffer xb may be refilled: every lane's reads of it were consumed above
      __syncwarp();
      if (lane == 0) mbar_arrive_remote_relaxed(xfree_peer[xb]);
      if (row == 0) SMLA_TL(2, g, 4);
    }
    if (!ok) break;
    gt += ntiles;
    // publish this warpgroup's sum for the token's epilogue (run by producer warps 0-3)
    float* lsh = l_sh + (et & 1) * 512;
    lsh[wg * 256 + row] = l_w;
    lsh[wg * 256 + 128 + row] = m_lw;
    warp_arrive(bar_addr(b->epi[et & 1]), lane);
    ++et;
  }
}

template <typename IdxT, bool kTrace>
__global__ void __launch_bounds__(kThreads, 1)
    h128_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
                    const H128Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* b = reinterpret_cast<Bars*>(base + kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();

  if (threadIdx.x == 0) {
    mbar_init(bar_addr(b->q_lo_full), 1);
    mbar_init(bar_addr(b->q_hi_full), 1);
    mbar_init(bar_addr(b->qcp_done), 1);
    mbar_init(bar_addr(b->q_empty), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_addr(b->kv_full[s]), kProducerWarps);
      mbar_init(bar_addr(b->kv_empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_addr(b->s_full[i]), 1);
      mbar_init(bar_addr(b->s_free[i]), kWgThreads / 32);
    }
    for (int i = 0; i < 2; ++i)
      for (int q = 0; q < 4; ++q) mbar_init(bar_addr(b->m_ready[i][q]), 1);
    for (int i = 0; i < 2; ++i) mbar_init(bar_addr(b->epi[i]), 2 * kWgThreads / 32);
    for (int i = 0; i < kPBufs; ++i) {
      mbar_init(bar_addr(b->p_full[i]), kWgThreads / 32);
      mbar_init(bar_addr(b->pv_done[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_addr(b->meta_full[i]), 1);
      mbar_init(bar_addr(b->meta_empty[i]), 1 + 2 * kWgThreads / 32);
    }
    for (int i = 0; i < kXBufs; ++i) {
      mbar_init(bar_addr(b->x_full[i]), 1);     // local expect_tx + the peer's st.async bytes
      mbar_init(bar_addr(b->x_free[i]), 4);     // one arrive per peer swap warp
    }
    mbar_init(bar_addr(b->o_free), 4);     // producer warps 0-3 after the epilogue
    mbar_init(bar_addr(b->drain), 1);
    b->abort_flag = 0;
    b->prod_stop = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) prefetch_tmap(&tm_q);
  if (warp == 1 && lane == 0) prefetch_tmap(&tm_o);
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&b->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();   // the peer's barriers are initialised before any remote arrive
  const uint32_t tmem = b->tmem_base;

  if (warp < kMmaWarp) {
    producer_role<IdxT, kTrace>(p, &tm_q, &tm_o, base, b, tmem, rank, warp, lane);
  } else if (warp == kMmaWarp) {
    if (lane == 0) mma_role(p, base, b, tmem, &tm_q, rank);
    __syncwarp();
  } else {
    score_role(p, base, b, tmem, rank, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();   // no remote store or arrive may target an exited CTA
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D bf16 tensor map over a [rows, 512] row-major matrix.
bool make_map(CUtensorMap* map, const void* ptr, uint64_t rows, uint32_t box_cols,
              uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim * 2)};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct DeviceState {
  bool ready = false;
  int max_clusters = 0;
};

cudaLaunchConfig_t launch_config(unsigned ctas, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <typename IdxT, bool kTrace>
cudaError_t prepare(DeviceState& st) {
  auto kern = h128_fwd_kernel<IdxT, kTrace>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = launch_config(2, nullptr, attr);
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (n <= 0) return cudaErrorInvalidConfiguration;
  st.max_clusters = n;
  st.ready = true;
  return cudaSuccess;
}

constexpr int kMaxDev = 64;

// Per-device, per-instantiation launch state (shared-memory attribute set,
// co-resident cluster count), prepared on first use.
template <typename IdxT, bool kTrace>
cudaError_t device_state(DeviceState** out) {
  static DeviceState states[kMaxDev];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!states[dev].ready && (e = prepare<IdxT, kTrace>(states[dev])) != cudaSuccess) return e;
  *out = &states[dev];
  return cudaSuccess;
}

template <typename IdxT, bool kTrace>
cudaError_t launch_typed(const FwdParams& fp, cudaStream_t stream) {
  DeviceState* st = nullptr;
  cudaError_t e = device_state<IdxT, kTrace>(&st);
  if (e != cudaSuccess) return e;
  CUtensorMap tq, to;
  if (!make_map(&tq, fp.q, static_cast<uint64_t>(fp.T) * 128, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&to, fp.out, static_cast<uint64_t>(fp.T) * 128, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  unsigned int* err = nullptr;
  if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&err), g_h128_error)) != cudaSuccess)
    return e;
  H128Params p;
  p.idx = fp.idx;
  p.kv = static_cast<const __nv_bfloat16*>(fp.kv);
  p.sink = fp.sink;
  p.out = static_cast<__nv_bfloat16*>(fp.out);
  p.lse = fp.lse;
  p.trace = fp.trace;
  p.err = err;
  p.T = fp.T;
  p.num_kv = fp.num_kv;
  p.topk = fp.topk;
  p.idx64 = fp.idx64;
  p.scale = fp.scale;
  const int64_t clusters = fp.T < st->max_clusters ? fp.T : st->max_clusters;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = launch_config(static_cast<unsigned>(2 * clusters), stream, attr);
  e = cudaLaunchKernelEx(&cfg, h128_fwd_kernel<IdxT, kTrace>, tq, to, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Self-test of the bounded-wait path: one thread waits on an mbarrier that
// nothing ever arrives at, gives up after `limit` cycles, records the expiry
// in the same error word the H=128 kernel uses and returns.
__global__ void wait_timeout_selftest_kernel(unsigned int* err, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t a = smem_u32(&bar);
  mbar_init(a, 1);
  const long long t0 = clock64();
  while (!mbar_try_wait(a, 0)) {
    if (clock64() - t0 > limit) {
      atomicOr(err, 16u);
      return;
    }
  }
}

}  // namespace

int selftest_wait_timeout(void* stream) {
  unsigned int* err = nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&err), g_h128_error);
  if (e != cudaSuccess) return static_cast<int>(e);
  wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, 2000000LL);
  return static_cast<int>(cudaGetLastError());
}

bool h128_supported(int64_t T, int32_t H, int32_t topk, int64_t num_kv) {
  return H == 128 && topk >= 1 && topk <= kMaxTopk && num_kv >= 1 && T >= 1 &&
         T < (int64_t(1) << 24);
}

int launch_h128(const FwdParams& p, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool tr = p.trace != nullptr;
  const cudaError_t e = p.idx64 ? (tr ? launch_typed<int64_t, true>(p, s) : launch_typed<int64_t, false>(p, s))
                                : (tr ? launch_typed<int32_t, true>(p, s) : launch_typed<int32_t, false>(p, s));
  return static_cast<int>(e);
}

int h128_geometry(int64_t T, LaunchGeom* g) {
  DeviceState* st = nullptr;
  const cudaError_t e = device_state<int32_t, false>(&st);
  if (e != cudaSuccess) return static_cast<int>(e);
  const int64_t clusters = T < st->max_clusters ? T : st->max_clusters;
  g->grid_ctas = static_cast<int>(2 * clusters);
  g->threads = kThreads;
  g->cluster = 2;
  g->smem = static_cast<int>(kSmemBytes);
  return 0;
}

#ifdef SMLA_TIMELINE
int h128_timeline(long long* host) {
  return static_cast<int>(cudaMemcpyFromSymbol(host, g_timeline, sizeof(g_timeline)));
}
#endif

int h128_error_word(unsigned int** addr) {
  return static_cast<int>(cudaGetSymbolAddress(reinterpret_cast<void**>(addr), g_h128_error));
}

}  // namespace smla
