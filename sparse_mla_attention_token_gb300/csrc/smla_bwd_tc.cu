// tcgen05 form of the backward's per-slot dkv contraction, H = 128 ("Sparse
// MLA training backward", aiter PR #4766, section "Structure": the dKV-interm
// step, a contraction over all heads of the gathered slots' P and dS).
//
//   interm[t, k, d] = sum_c A[t, k, c] * B[t, c, d],   c < 2H = 256
//   A[t, k, :] = [P(t, :, k) | scale * dS(t, :, k)]    (the workspace rows the
//                                                       dq kernel writes, bf16)
//   B[t, c, :] = dO[t, c, :] for c < H, q[t, c - H, :] for c >= H
//
// One CTA per (token, 128-slot tile, 256-column half of D): M = 128 slots,
// N = 256, K = 256 in four 64-wide chunks.  Warp 0 lane 0 loads each chunk with
// 2-D TMA (A: one 128 x 64 box of the [T * topk, 256] workspace; B: four 64 x
// 64 boxes of dO or q, the MN-major operand) into a two-stage ring; warp 1
// lane 0 owns the 256 TMEM columns and issues four M128 N256 K16 MMAs per
// chunk; all four warps then read the accumulator (thread = TMEM lane = slot)
// and store the tile's valid rows as bf16.  96 KB of shared memory and 256
// TMEM columns: two CTAs per SM, one's epilogue under the other's MMAs.
//
// Every wait is bounded (~2 s): on expiry the CTA records an error in the
// backward's error word (read by sparse_mla_device_status), waits for what it
// issued, frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "smla_device.cuh"
#include "smla_internal.h"
#include "smla_sm100.cuh"

namespace smla {

__device__ unsigned int g_bwd_error;

namespace {

using namespace sm100;

constexpr int kThreadsTc = 128;
constexpr int kM = 128;                          // slots per tile
constexpr int kNh = 256;                         // output columns per CTA
constexpr int kKc = 64;                          // contraction chunk
constexpr int kH = 128;
constexpr int kChunks = 2 * kH / kKc;            // 4
constexpr int kStagesTc = 2;
constexpr uint32_t kABytes = kM * kKc * 2;       // 16 KB: [128 rows][128 B]
constexpr uint32_t kBBytes = kKc * kNh * 2;      // 32 KB: [4 column blocks][64 K rows][128 B]
constexpr uint32_t kStageBytesTc = kABytes + kBBytes;
constexpr uint32_t kBarOffTc = kStagesTc * kStageBytesTc;
constexpr uint32_t kSmemTc = kBarOffTc + 128 + 1024;   // barriers + alignment slack
constexpr long long kTimeoutTc = 4000000000LL;         // ~2 s at 2 GHz

__device__ __forceinline__ uint32_t bar_addr_tc(const uint64_t& b) { return smem_u32(&b); }

struct TcBars {
  uint64_t full[kStagesTc], empty[kStagesTc], done, drain;
  uint32_t tmem_base;
  int abort_flag;
};

template <typename BarsT>
__device__ __forceinline__ bool wait_tc(uint32_t bar, uint32_t parity, BarsT* b, bool drain) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 15) == 0) {
      if (!drain && *reinterpret_cast<volatile int*>(&b->abort_flag)) return false;
      if (clock64() - t0 > kTimeoutTc) {
        *reinterpret_cast<volatile int*>(&b->abort_flag) = 1;
        atomicOr(&g_bwd_error, 1u);
        return false;
      }
    }
  }
}

__global__ void __launch_bounds__(kThreadsTc, 2)
    bwd_interm_tc_kernel(const __grid_constant__ CUtensorMap tm_a,
                         const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_out, const BwdParams p, int ntile) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  TcBars* b = reinterpret_cast<TcBars*>(base + kBarOffTc);
  const uint32_t sbase = smem_u32(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int dh = blockIdx.x & 1;
  const int64_t unit = blockIdx.x >> 1;
  const int64_t t = unit / ntile;
  const int tile = static_cast<int>(unit % ntile);
  const int nv = p.ncnt[t];
  if (tile * kM >= nv) return;   // uniform: this tile holds no valid slot

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesTc; ++s) {
      mbar_init(bar_addr_tc(b->full[s]), 1);
      mbar_init(bar_addr_tc(b->empty[s]), 1);
    }
    mbar_init(bar_addr_tc(b->done), 1);
    mbar_init(bar_addr_tc(b->drain), 1);
    b->abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_do);
    prefetch_tmap(&tm_q);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&b->tmem_base), kNh);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = b->tmem_base;
  const int row0 = static_cast<int>(t * p.topk + int64_t(tile) * kM);   // < 2^31 (host check)
  const int qrow0 = static_cast<int>(t * kH);

  if (warp == 0 && lane == 0) {
    // producer: chunk c = heads 64c..64c+63 of [P | dS'] against rows of dO (c < 2) or q
    uint32_t loaded = 0;
    for (int c = 0; c < kChunks; ++c) {
      const int s = c % kStagesTc;
      if (c >= kStagesTc && !wait_tc(bar_addr_tc(b->empty[s]), ((c / kStagesTc) - 1) & 1, b, false))
        break;
      const uint32_t st = sbase + s * kStageBytesTc;
      mbar_arrive_expect_tx(bar_addr_tc(b->full[s]), kStageBytesTc);
      tma_load_2d(st, &tm_a, kKc * c, row0, bar_addr_tc(b->full[s]));
      const CUtensorMap* mb = c < 2 ? &tm_do : &tm_q;
      const int brow = qrow0 + kKc * (c & 1);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        tma_load_2d(st + kABytes + j * 8192, mb, kNh * dh + 64 * j, brow, bar_addr_tc(b->full[s]));
      ++loaded;
    }
    // drain: every load issued has landed before the CTA may exit
    for (uint32_t c = loaded >= kStagesTc ? loaded - kStagesTc : 0; c < loaded; ++c)
      wait_tc(bar_addr_tc(b->full[c % kStagesTc]), (c / kStagesTc) & 1, b, true);
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t kIdesc = idesc_bf16_f32(kM, kNh, false, true);
    // descriptors advanced from two built before the loop (byte offset / 16 added to
    // the start-address field; shared addresses < 256 KB, so nothing carries out)
    const uint64_t d_a0 = sdesc_sw128(sbase, 16, 1024);               // K-major A
    const uint64_t d_b0 = sdesc_sw128(sbase + kABytes, 8192, 1024);   // MN-major B
    bool ok = true;
    for (int c = 0; c < kChunks && ok; ++c) {
      const int s = c % kStagesTc;
      if (!(ok = wait_tc(bar_addr_tc(b->full[s]), (c / kStagesTc) & 1, b, false))) break;
      tc_fence_after();
      const uint64_t so = s * (kStageBytesTc >> 4);
#pragma unroll
      for (int kk = 0; kk < kKc / 16; ++kk) {
        const uint64_t ad = d_a0 + so + kk * 2;            // + kk * 32 bytes
        const uint64_t bd = d_b0 + so + kk * (16 * 128 >> 4);   // + kk * 16 rows of 128 bytes
        mma_bf16_ss(tmem, ad, bd, kIdesc, (c > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit(bar_addr_tc(b->empty[s]));
    }
    mma_commit(bar_addr_tc(ok ? b->done : b->drain));
    if (!ok) wait_tc(bar_addr_tc(b->drain), 0, b, true);   // MMAs issued so far completed
  }
  __syncwarp();
  // epilogue: thread = TMEM lane = slot of the tile; bf16 rows to the workspace.
  // When the tile's 128 rows lie inside the token's topk rows (rows past the
  // valid count are never read), the tile is staged in the finished ring
  // (four 64-column blocks, 128-byte swizzle) and stored by four 2-D TMA
  // boxes: a warp's row-per-lane stores would touch 32 lines per instruction.
  const bool done = __all_sync(0xffffffffu, wait_tc(bar_addr_tc(b->done), 0, b, false));
  const bool boxed = (tile + 1) * kM <= p.topk;
  if (done && boxed) {
    tc_fence_after();
    const int r = 32 * warp + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * warp) << 16);
#pragma unroll 1
    for (int cc = 0; cc < kNh / 32; ++cc) {
      uint32_t v[32];
      tmem_ld32(tl + 32 * cc, v);
      tmem_wait_ld();
      // columns 32 cc .. +31: block cc / 2, 16-byte chunks 4 (cc & 1) .. +3 of row r
      const uint32_t rowa = sbase + (cc >> 1) * (kM * 128) + r * 128;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        st_shared_v4(rowa + ((((cc & 1) * 4 + q) ^ (r & 7)) << 4),
                     make_uint4(pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                                pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                                pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                                pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]))));
    }
    fence_proxy_async_smem();   // the staged tile is read by the TMA (async proxy)
  }
  if (boxed) {
    __syncthreads();
    if (done && threadIdx.x == 0) {
#pragma unroll
      for (int j = 0; j < kNh / 64; ++j) tma_store_2d(&tm_out, sbase + j * (kM * 128), kNh * dh + 64 * j, row0);
      bulk_commit();
      bulk_wait<0>();   // the boxes are written before the CTA exits
    }
  } else if (done) {
    tc_fence_after();
    const int r = 32 * warp + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * warp) << 16);
    const bool live = tile * kM + r < nv;
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.interm) +
                         (int64_t(row0) + r) * kHeadDim + kNh * dh;
#pragma unroll 1
    for (int cc = 0; cc < kNh / 32; ++cc) {
      uint32_t v[32];
      tmem_ld32(tl + 32 * cc, v);
      tmem_wait_ld();
      if (live) {
        uint4* o = reinterpret_cast<uint4*>(dst + 32 * cc);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          o[q] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                            pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                            pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                            pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kNh);
  }
}

// dq = scale * dS . K for H = 128: M = 128 heads, N = 256 (a D half), K = the
// token's valid slots in 32-slot chunks.  A = (scale dS)^T, MN-major: each
// slot's 128 dS' values (256 bytes of the workspace row) as two 128-byte rows of
// two 64-head blocks; B = the gathered kv half rows, MN-major (the forward's
// stage layout).  Warps 0-3 gather both with 16-byte cp.async into a four-stage
// ring, up to three chunks in flight per thread (slots past the valid count
// zero-filled, so the uninitialised workspace past them never enters a sum),
// and then run the epilogue; warp 4 lane 0 owns TMEM and issues two M128 N256
// K16 MMAs per chunk.
constexpr int kDqThreads = 160;
constexpr int kDqChunk = 32;                         // slots per chunk
constexpr int kDqStages = 4;
constexpr uint32_t kDqBlk = kDqChunk * 128;          // 4 KB: one 64-element block of 32 slots
constexpr uint32_t kDqA = kDqChunk * kH * 2;         // 8 KB: [2 head blocks][32 slots][128 B]
constexpr uint32_t kDqB = kDqChunk * kNh * 2;        // 16 KB: [4 column blocks][32 slots][128 B]
constexpr uint32_t kDqStage = kDqA + kDqB;
constexpr uint32_t kDqBarOff = kDqStages * kDqStage;   // 96 KB (also the epilogue's staging)
constexpr uint32_t kDqSmem = kDqBarOff + 128 + 1024;

struct DqBars {
  uint64_t full[kDqStages], empty[kDqStages], done, drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(DqBars) <= 128, "barriers fit their slot");

__global__ void __launch_bounds__(kDqThreads, 2)
    bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  DqBars* b = reinterpret_cast<DqBars*>(base + kDqBarOff);
  const uint32_t sbase = smem_u32(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int dh = blockIdx.x & 1;
  const int64_t t = blockIdx.x >> 1;
  const int nv = p.ncnt[t];
  float* dq = p.dq + (t * kH) * int64_t(kHeadDim) + kNh * dh;
  if (nv == 0) {   // no valid slot: dq = 0 (uniform)
    if (tid < kH) {
      float4* o = reinterpret_cast<float4*>(dq + int64_t(tid) * kHeadDim);
      for (int i = 0; i < kNh / 4; ++i) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }
  if (tid == 0) {
    for (int s = 0; s < kDqStages; ++s) {
      mbar_init(bar_addr_tc(b->full[s]), 128);     // the four gather warps
      mbar_init(bar_addr_tc(b->empty[s]), 1);
    }
    mbar_init(bar_addr_tc(b->done), 1);
    mbar_init(bar_addr_tc(b->drain), 1);
    b->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(smem_u32(&b->tmem_base), kNh);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = b->tmem_base;
  const int nchunks = (nv + kDqChunk - 1) / kDqChunk;

  if (warp < 4) {
    const char* pds = static_cast<const char*>(p.pds) + t * p.topk * int64_t(2 * kH * 2);
    const int* crow = p.crow + t * p.topk;
    const char* kvb = static_cast<const char*>(p.kv) + kNh * 2 * dh;   // this CTA's D half
    // copies of a chunk: A k = 0..3 is piece qa = tid % 16 of slot 8 k + tid / 16 (16
    // lanes read one slot's 256 dS' bytes); B k = 0..7 is piece qb = tid % 32 of slot
    // 4 k + tid / 32 (a warp reads one kv half row)
    const int qa = tid & 15, ra = tid >> 4, qb = lane, rb = warp;
    const uint32_t a_off = (qa >> 3) * kDqBlk + ra * 128 + (((qa & 7) ^ (ra & 7)) << 4);
    const uint32_t b_off = kDqA + (qb >> 3) * kDqBlk + rb * 128;   // + row 4 k, swizzled below
    // A chunk's copies are counted on its barrier once kDepth - 1 later chunks are
    // issued; before any wait that may block, the pending chunks are counted first
    // (the slot waited for is freed by MMAs that need them).  Pending chunks are
    // consecutive, from `first`.
    constexpr int kDepth = 3;
    int first = 0, npend = 0;
    auto count_oldest = [&]() {
      mbar_arrive(bar_addr_tc(b->full[first % kDqStages]));
      ++first;
      --npend;
    };
    auto flush = [&]() {
      if (npend > 0) {
        cp_async_wait<0>();
        fence_proxy_async_smem();   // visible to the tensor core's async proxy
        while (npend > 0) count_oldest();
      }
    };
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % kDqStages;
      if (c >= kDqStages) {
        const uint32_t eb = bar_addr_tc(b->empty[s]), ep = ((c / kDqStages) - 1) & 1;
        if (!mbar_test_wait(eb, ep)) {
          flush();
          if (!(ok = wait_tc(eb, ep, b, false))) break;
        }
      }
      const uint32_t st = sbase + s * kDqStage;
      const int s0 = c * kDqChunk;
      int rowb[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int slot = s0 + 4 * k + rb;
        rowb[k] = slot < nv ? crow[slot] : -1;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int slot = s0 + 8 * k + ra;
        const bool v = slot < nv;
        const char* src = v ? pds + int64_t(slot) * (2 * kH * 2) + kH * 2 + qa * 16 : pds;
        cp_async_16(st + a_off + k * 8 * 128, src, v ? 16u : 0u);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const bool v = rowb[k] >= 0;
        const char* src = v ? kvb + int64_t(rowb[k]) * 1024 + qb * 16 : kvb;
        // row 4 k + rb: its low three bits are rb + 4 (k & 1)
        cp_async_16(st + b_off + k * 4 * 128 + (((qb & 7) ^ ((rb + 4 * k) & 7)) << 4), src, v ? 16u : 0u);
      }
      cp_async_commit();
      if (npend == 0) first = c;
      if (++npend == kDepth) {
        cp_async_wait<kDepth - 1>();   // the oldest pending chunk has landed
        fence_proxy_async_smem();
        count_oldest();
      }
    }
    flush();
    cp_async_wait<0>();
  } else if (lane == 0) {
    constexpr uint32_t kIdesc = idesc_bf16_f32(kH, kNh, true, true);
    // MN-major A and B: 64-element blocks kDqBlk apart, 8-slot groups 1 KB apart; a K
    // step is 16 slots (2 KB, 128 in the descriptor's start-address field)
    const uint64_t d0 = sdesc_sw128(sbase, kDqBlk, 1024);
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      const int s = c % kDqStages;
      if (!(ok = wait_tc(bar_addr_tc(b->full[s]), (c / kDqStages) & 1, b, false))) break;
      tc_fence_after();
      const uint64_t ad = d0 + s * (kDqStage >> 4), bd = ad + (kDqA >> 4);
#pragma unroll
      for (int kk = 0; kk < kDqChunk / 16; ++kk)
        mma_bf16_ss(tmem, ad + kk * 128, bd + kk * 128, kIdesc, (c > 0 || kk > 0) ? 1u : 0u);
      mma_commit(bar_addr_tc(b->empty[s]));
    }
    mma_commit(bar_addr_tc(ok ? b->done : b->drain));
    if (!ok) wait_tc(bar_addr_tc(b->drain), 0, b, true);
  }
  __syncwarp();
  if (warp < 4) {
    // epilogue: thread = TMEM lane = head; its 256 dq columns in fp32
    const bool done = __all_sync(0xffffffffu, wait_tc(bar_addr_tc(b->done), 0, b, false));
    // the 128 x 256 fp32 tile goes out through the finished ring in two 128-column
    // passes, each four 32-column boxes (128-byte swizzle) stored by 2-D TMA: a
    // warp's row-per-lane stores would touch 32 lines per instruction
    tc_fence_after();
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * warp) << 16);
    const int r = tid;
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
      if (done) {
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t v[32];
          tmem_ld32(tl + 128 * pass + 32 * cc, v);
          tmem_wait_ld();
          const uint32_t rowa = sbase + cc * (kH * 128) + r * 128;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            st_shared_v4(rowa + ((q ^ (r & 7)) << 4),
                         make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
        }
        fence_proxy_async_smem();   // the staged boxes are read by the TMA (async proxy)
      }
      named_bar_sync(1, 128);
      if (done && tid == 0) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          tma_store_2d(&tm_dq, sbase + j * (kH * 128), kNh * dh + 128 * pass + 32 * j,
                       static_cast<int>(t * kH));
        bulk_commit();
        bulk_wait_read<0>();   // the boxes have left shared memory
      }
      named_bar_sync(1, 128);
    }
    if (done && tid == 0) bulk_wait<0>();   // written before the CTA exits
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kNh);
  }
}

// S and dP for H = 128, transposed so that the slots are the MMA's M: per
// (token, 128-slot tile), S^T = K . Q^T and dP^T = K . dO^T (M = 128 slots,
// N = 128 heads, K = 512 in eight 64-column chunks; both operands K-major).
// Warps 0-3 gather the tile's kv rows chunk by chunk (16-byte cp.async, 128 B a
// row, slots past the valid count zero-filled); warp 4 lane 0 loads the Q and
// dO chunks with 2-D TMA, owns 256 TMEM columns (S^T, then dP^T) and issues
// eight M128 N128 K16 MMAs a chunk.  The epilogue (thread = TMEM lane = slot)
// forms P = 2^(S scale log2e - lse log2e) from the saved lse and
// dS' = scale P (dP - delta), and writes the slot's workspace row [P | dS'].
constexpr int kSdThreads = 160;
constexpr int kSdM = 128;                            // slots per tile
constexpr int kSdChunks = kHeadDim / 64;             // 8
constexpr uint32_t kSdA = kSdM * 128;                // 16 KB: [128 slots][128 B]
constexpr uint32_t kSdB = kH * 128;                  // 16 KB: [128 heads][128 B]
constexpr uint32_t kSdStage = kSdA + 2 * kSdB;       // 48 KB
constexpr uint32_t kSdBarOff = 2 * kSdStage;
constexpr uint32_t kSdSmem = kSdBarOff + 128 + 2 * kH * 4 + 1024;

struct SdBars {
  uint64_t full[2], tma[2], empty[2], done, drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ bool wait_sd(uint32_t bar, uint32_t parity, SdBars* b, bool drain) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 15) == 0) {
      if (!drain && *reinterpret_cast<volatile int*>(&b->abort_flag)) return false;
      if (clock64() - t0 > kTimeoutTc) {
        *reinterpret_cast<volatile int*>(&b->abort_flag) = 1;
        atomicOr(&g_bwd_error, 2u);
        return false;
      }
    }
  }
}

__global__ void __launch_bounds__(kSdThreads, 2)
    bwd_sdp_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_do,
                      const __grid_constant__ CUtensorMap tm_pds, const BwdParams p, int ntile) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  SdBars* b = reinterpret_cast<SdBars*>(base + kSdBarOff);
  float* lse2 = reinterpret_cast<float*>(base + kSdBarOff + 128);   // [128] lse * log2 e
  float* dlt = lse2 + kH;                                           // [128] delta
  const uint32_t sbase = smem_u32(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int64_t t = blockIdx.x / ntile;
  const int tile = static_cast<int>(blockIdx.x % ntile);
  const int nv = p.ncnt[t];
  if (tile * kSdM >= nv) return;   // uniform

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_addr_tc(b->full[s]), 128);   // the four gather warps
      mbar_init(bar_addr_tc(b->tma[s]), 1);      // Q and dO chunks (TMA bytes)
      mbar_init(bar_addr_tc(b->empty[s]), 1);
    }
    mbar_init(bar_addr_tc(b->done), 1);
    mbar_init(bar_addr_tc(b->drain), 1);
    b->abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_do);
  }
  if (tid < kH) {
    lse2[tid] = p.lse[t * kH + tid] * kLog2e;
    dlt[tid] = p.delta[t * kH + tid];
  }
  if (warp == 4) {
    tmem_alloc(smem_u32(&b->tmem_base), 2 * kH);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = b->tmem_base;
  const int slot0 = tile * kSdM;
  const int* crow = p.crow + t * p.topk;

  if (warp < 4) {
    // gather: a 64-column chunk is 128 rows x 8 pieces of 16 B; copy j of this thread
    // is piece q = tid % 8 of row 16 j + tid / 8, so 8 lanes read one row's 128
    // contiguous bytes and a warp instruction four whole lines
    const int q = tid & 7, r0 = tid >> 3;
    const char* src_row[8];
    bool vr[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = 16 * j + r0;
      vr[j] = slot0 + r < nv;
      src_row[j] = static_cast<const char*>(p.kv) + (vr[j] ? int64_t(crow[slot0 + r]) * 1024 : 0) + q * 16;
    }
    const uint32_t dst_off = r0 * 128 + ((q ^ (r0 & 7)) << 4);   // row 16 j + r0 adds 2 KB j
    // a chunk's copies are counted once the next chunk is issued (two in flight per
    // thread); before a wait that may block, the pending chunk is counted first
    int pend = -1;
    auto flush = [&]() {
      if (pend >= 0) {
        cp_async_wait<0>();
        fence_proxy_async_smem();
        mbar_arrive(bar_addr_tc(b->full[pend & 1]));
        pend = -1;
      }
    };
    bool ok = true;
    for (int c = 0; c < kSdChunks && ok; ++c) {
      const int s = c & 1;
      if (c >= 2) {
        const uint32_t eb = bar_addr_tc(b->empty[s]), ep = ((c >> 1) - 1) & 1;
        if (!mbar_test_wait(eb, ep)) {
          flush();
          if (!(ok = wait_sd(eb, ep, b, false))) break;
        }
      }
      const uint32_t dst = sbase + s * kSdStage + dst_off;
#pragma unroll
      for (int j = 0; j < 8; ++j) cp_async_16(dst + j * 2048, src_row[j] + c * 128, vr[j] ? 16u : 0u);
      cp_async_commit();
      if (pend >= 0) {
        cp_async_wait<1>();   // the previous chunk has landed
        fence_proxy_async_smem();
        mbar_arrive(bar_addr_tc(b->full[pend & 1]));
      }
      pend = c;
    }
    flush();
    cp_async_wait<0>();
  } else if (lane == 0) {
    constexpr uint32_t kIdesc = idesc_bf16_f32(kSdM, kH, false, false);
    const uint64_t d_sd0 = sdesc_sw128(sbase, 16, 1024);   // stage 0, K-major, 128-byte rows
    const int qrow = static_cast<int>(t * kH);
    bool ok = true;
    uint32_t loaded = 0;
    auto load = [&](int c) {
      const int s = c & 1;
      const uint32_t st = sbase + s * kSdStage;
      mbar_arrive_expect_tx(bar_addr_tc(b->tma[s]), 2 * kSdB);
      tma_load_2d(st + kSdA, &tm_q, 64 * c, qrow, bar_addr_tc(b->tma[s]));
      tma_load_2d(st + kSdA + kSdB, &tm_do, 64 * c, qrow, bar_addr_tc(b->tma[s]));
      ++loaded;
    };
    load(0);
    load(1);
    for (int c = 0; c < kSdChunks && ok; ++c) {
      const int s = c & 1;
      if (!(ok = wait_sd(bar_addr_tc(b->full[s]), (c >> 1) & 1, b, false))) break;
      if (!(ok = wait_sd(bar_addr_tc(b->tma[s]), (c >> 1) & 1, b, false))) break;
      tc_fence_after();
      // descriptors advanced from one built before the loop (byte offset / 16 added to
      // the start-address field; shared addresses < 256 KB, so nothing carries out)
      const uint64_t da = d_sd0 + s * (kSdStage >> 4);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = da + kk * 2;
        const uint64_t bq = da + (kSdA >> 4) + kk * 2;
        const uint64_t bd = da + ((kSdA + kSdB) >> 4) + kk * 2;
        const uint32_t acc = (c > 0 || kk > 0) ? 1u : 0u;
        mma_bf16_ss(tmem, ad, bq, kIdesc, acc);            // S^T
        mma_bf16_ss(tmem + kH, ad, bd, kIdesc, acc);       // dP^T
      }
      mma_commit(bar_addr_tc(b->empty[s]));
      if (c + 2 < kSdChunks) {
        // the stage's Q / dO may be replaced once these MMAs have read it
        if (!(ok = wait_sd(bar_addr_tc(b->empty[s]), (c >> 1) & 1, b, false))) break;
        load(c + 2);
      }
    }
    mma_commit(bar_addr_tc(ok ? b->done : b->drain));
    if (!ok) wait_sd(bar_addr_tc(b->drain), 0, b, true);
    // every TMA load issued has landed
    for (uint32_t c = loaded >= 2 ? loaded - 2 : 0; c < loaded; ++c)
      wait_sd(bar_addr_tc(b->tma[c & 1]), (c >> 1) & 1, b, true);
  }
  __syncwarp();
  // When the tile's 128 rows lie inside the token's topk rows (rows past the
  // valid count are never read), the [P | dS'] tile is staged in the finished
  // ring (four 64-column blocks, 128-byte swizzle) and stored by four 2-D TMA
  // boxes: a warp's row-per-lane stores would touch 32 lines per instruction.
  const bool boxed = (tile + 1) * kSdM <= p.topk;
  bool done = true;
  if (warp < 4) {
    done = __all_sync(0xffffffffu, wait_sd(bar_addr_tc(b->done), 0, b, false));
    if (done && boxed) {
      tc_fence_after();
      const int r = tid;
      const uint32_t tl = tmem + (static_cast<uint32_t>(32 * warp) << 16);
      const float sl2 = p.scale * kLog2e;
#pragma unroll 1
      for (int hc = 0; hc < kH / 32; ++hc) {
        uint32_t sv[32], dv[32];
        tmem_ld32(tl + 32 * hc, sv);
        tmem_ld32(tl + kH + 32 * hc, dv);
        tmem_wait_ld();
        uint32_t pw[16], dw[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int h = 32 * hc + 2 * i;
          const float p0 = ex2(__uint_as_float(sv[2 * i]) * sl2 - lse2[h]);
          const float p1 = ex2(__uint_as_float(sv[2 * i + 1]) * sl2 - lse2[h + 1]);
          pw[i] = pack_bf16x2(p0, p1);
          dw[i] = pack_bf16x2(p.scale * p0 * (__uint_as_float(dv[2 * i]) - dlt[h]),
                              p.scale * p1 * (__uint_as_float(dv[2 * i + 1]) - dlt[h + 1]));
        }
        // P columns 32 hc .. +31: block hc / 2; dS' the same two blocks further
        const uint32_t rp = sbase + (hc >> 1) * (kSdM * 128) + r * 128;
        const uint32_t rd = rp + 2 * (kSdM * 128);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t ch = ((((hc & 1) * 4 + q) ^ (r & 7)) << 4);
          st_shared_v4(rp + ch, make_uint4(pw[4 * q], pw[4 * q + 1], pw[4 * q + 2], pw[4 * q + 3]));
          st_shared_v4(rd + ch, make_uint4(dw[4 * q], dw[4 * q + 1], dw[4 * q + 2], dw[4 * q + 3]));
        }
      }
      fence_proxy_async_smem();   // the staged tile is read by the TMA (async proxy)
    }
  }
  if (boxed) {
    __syncthreads();
    if (done && tid == 0) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        tma_store_2d(&tm_pds, sbase + j * (kSdM * 128), 64 * j, static_cast<int>(t * p.topk + slot0));
      bulk_commit();
      bulk_wait<0>();   // the boxes are written before the CTA exits
    }
  } else if (warp < 4) {
    if (done) {
      tc_fence_after();
      const int r = tid;
      const bool v = slot0 + r < nv;
      const uint32_t tl = tmem + (static_cast<uint32_t>(32 * warp) << 16);
      const float sl2 = p.scale * kLog2e;
      uint4* row = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.pds) +
                                            (t * p.topk + slot0 + r) * int64_t(2 * kH));
#pragma unroll 1
      for (int hc = 0; hc < kH / 32; ++hc) {
        uint32_t sv[32], dv[32];
        tmem_ld32(tl + 32 * hc, sv);
        tmem_ld32(tl + kH + 32 * hc, dv);
        tmem_wait_ld();
        uint32_t pw[16], dw[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int h = 32 * hc + 2 * i;
          const float p0 = ex2(__uint_as_float(sv[2 * i]) * sl2 - lse2[h]);
          const float p1 = ex2(__uint_as_float(sv[2 * i + 1]) * sl2 - lse2[h + 1]);
          pw[i] = pack_bf16x2(p0, p1);
          dw[i] = pack_bf16x2(p.scale * p0 * (__uint_as_float(dv[2 * i]) - dlt[h]),
                              p.scale * p1 * (__uint_as_float(dv[2 * i + 1]) - dlt[h + 1]));
        }
        if (v) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            row[4 * hc + q] = make_uint4(pw[4 * q], pw[4 * q + 1], pw[4 * q + 2], pw[4 * q + 3]);
            row[16 + 4 * hc + q] = make_uint4(dw[4 * q], dw[4 * q + 1], dw[4 * q + 2], dw[4 * q + 3]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kH);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_tc() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D tensor map over a [rows, cols] row-major bf16 (or fp32) matrix, 128-byte swizzle.
bool make_map_2d(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols,
                 uint32_t box_cols, uint32_t box_rows, bool fp32 = false) {
  auto fn = encode_tc();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * (fp32 ? 4 : 2))};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int launch_bwd_interm_tc(const BwdParams& p, void* stream) {
  if (p.H != kH || p.T <= 0 || p.topk <= 0) return static_cast<int>(cudaErrorInvalidValue);
  auto kern = bwd_interm_tc_kernel;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemTc));
  if (e != cudaSuccess) return static_cast<int>(e);
  CUtensorMap ta, tdo, tq, to;
  if (!make_map_2d(&ta, p.pds, uint64_t(p.T) * p.topk, 2 * kH, 64, kM) ||
      !make_map_2d(&tdo, p.dout, uint64_t(p.T) * kH, kHeadDim, 64, 64) ||
      !make_map_2d(&tq, p.q, uint64_t(p.T) * kH, kHeadDim, 64, 64) ||
      !make_map_2d(&to, p.interm, uint64_t(p.T) * p.topk, kHeadDim, 64, kM))
    return static_cast<int>(cudaErrorInvalidValue);
  const int ntile = (p.topk + kM - 1) / kM;
  const int64_t blocks = p.T * ntile * 2;
  kern<<<static_cast<unsigned>(blocks), kThreadsTc, kSmemTc, static_cast<cudaStream_t>(stream)>>>(
      ta, tdo, tq, to, p, ntile);
  return static_cast<int>(cudaGetLastError());
}

int launch_bwd_dq_tc(const BwdParams& p, void* stream) {
  if (p.H != kH || p.T <= 0) return static_cast<int>(cudaErrorInvalidValue);
  auto kern = bwd_dq_tc_kernel;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kDqSmem));
  if (e != cudaSuccess) return static_cast<int>(e);
  CUtensorMap tdq;
  if (!make_map_2d(&tdq, p.dq, uint64_t(p.T) * kH, kHeadDim, 32, kH, /*fp32=*/true))
    return static_cast<int>(cudaErrorInvalidValue);
  kern<<<static_cast<unsigned>(p.T * 2), kDqThreads, kDqSmem, static_cast<cudaStream_t>(stream)>>>(tdq, p);
  return static_cast<int>(cudaGetLastError());
}

int launch_bwd_sdp_tc(const BwdParams& p, void* stream) {
  if (p.H != kH || p.T <= 0 || p.topk <= 0) return static_cast<int>(cudaErrorInvalidValue);
  auto kern = bwd_sdp_tc_kernel;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSdSmem));
  if (e != cudaSuccess) return static_cast<int>(e);
  CUtensorMap tq, tdo, tp;
  if (!make_map_2d(&tq, p.q, uint64_t(p.T) * kH, kHeadDim, 64, kH) ||
      !make_map_2d(&tdo, p.dout, uint64_t(p.T) * kH, kHeadDim, 64, kH) ||
      !make_map_2d(&tp, p.pds, uint64_t(p.T) * p.topk, 2 * kH, 64, kSdM))
    return static_cast<int>(cudaErrorInvalidValue);
  const int ntile = (p.topk + kSdM - 1) / kSdM;
  kern<<<static_cast<unsigned>(p.T * ntile), kSdThreads, kSdSmem,
         static_cast<cudaStream_t>(stream)>>>(tq, tdo, tp, p, ntile);
  return static_cast<int>(cudaGetLastError());
}

int bwd_error_word(unsigned int** addr) {
  return static_cast<int>(cudaGetSymbolAddress(reinterpret_cast<void**>(addr), g_bwd_error));
}

}  // namespace smla
