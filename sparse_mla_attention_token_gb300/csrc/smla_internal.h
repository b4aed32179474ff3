// Internal interface between the host planner (api.cpp) and the kernel
// translation units.  Plain C++ types only; no CUDA headers needed here.
#pragma once

#include <cstddef>
#include <cstdint>

namespace smla {

constexpr int kHeadDim = 512;

// Everything one forward launch needs.  Pointers are device pointers.
struct FwdParams {
  const void* q;          // [T, H, 512] bf16
  const void* kv;         // [num_kv, 512] bf16
  const void* idx;        // [T, topk] int32 | int64
  const float* sink;      // [H] fp32 or nullptr
  void* out;              // [T, H, 512] bf16
  float* lse;             // [T, H] fp32
  int64_t* trace;         // [T, topk] int64 or nullptr (row read per slot, -1 = none)
  float* part_o;          // split path: [splits, T, H, d_v] fp32 (sink-free, normalised)
  float* part_lse;        // split path: [splits, T, H] fp32 (sink-free)
  int64_t T;
  int64_t num_kv;
  int32_t H;
  int32_t topk;
  int32_t splits;         // >= 1
  int32_t idx64;          // 1: int64 indices
  int32_t d_qk;           // score width: q and kv rows (512 unless stated)
  int32_t d_v;            // value width: the first d_v columns of a kv row; out rows
  int32_t kv_fp8;         // 1: kv holds e4m3 codes [num_kv, 512] (the fp8 cache)
  const float* kv_scale;  // fp8 cache: [num_kv, 4] fp32 block scales, else unused
  float scale;
};

// Largest slot range one CTA of the small-head kernel compacts in shared memory.
constexpr int kSmallHMaxSlots = 2048;

// Small-head kernel (mma.sync, head groups of 16); any H in {8,...,128}.
// Returns a cudaError_t value (0 = success).
int launch_smallh(const FwdParams& p, void* stream);
// (d_qk, d_v) pairs the small-head kernel is built for: (512, 512), (128, 128),
// (576, 576) and (576, 512) (a 64-wide positional part used in the scores only).
bool smallh_dims_supported(int32_t d_qk, int32_t d_v);

// tcgen05 kernel for H == 128, splits == 1.
int launch_h128(const FwdParams& p, void* stream);
// Whether launch_h128 supports this problem (H == 128, 1 <= topk <= 1024,
// num_kv >= 1, T < 2^24).
bool h128_supported(int64_t T, int32_t H, int32_t topk, int64_t num_kv);
#ifdef SMLA_TIMELINE
int h128_timeline(long long* host);
#endif
// Launch the bounded-wait self-test kernel (its wait always expires).
int selftest_wait_timeout(void* stream);
// Device address of the h128 kernel's error word (bounded waits), or nullptr.
int h128_error_word(unsigned int** addr);

// Launch geometry of each kernel family: grid CTAs, threads, cluster size, smem.
struct LaunchGeom {
  int grid_ctas;
  int threads;
  int cluster;
  int smem;
};
int smallh_geometry(int64_t T, int32_t H, int32_t splits, int32_t d_qk, int32_t d_v,
                    LaunchGeom* g, bool fp8 = false);
int h128_geometry(int64_t T, LaunchGeom* g);

// Partial rows (splits * T * H) the static scratch of the allocation-free
// split path holds: 8192 rows of 512 + 1 fp32 = 16 MiB.
constexpr int64_t kNoAllocScratchRows = 8192;
// Split path (splits >= 2) with its partials in the library's static scratch;
// fills p.part_o / p.part_lse itself.  Returns a cudaError_t value.
int launch_split_static_scratch(FwdParams p, void* stream);

// Merge split partials into out / lse, folding the sink once.
int launch_combine(const FwdParams& p, void* stream);

// ---------------------------------------------------------------- backward
// Everything one backward call needs.  Pointers are device pointers; the
// workspace pointers are filled in by launch_bwd from the caller's workspace.
struct BwdParams {
  const void* q;          // [T, H, 512] bf16
  const void* kv;         // [num_kv, 512] bf16
  const void* idx;        // [T, topk] int32 | int64
  const float* sink;      // [H] fp32 or nullptr
  const void* out;        // [T, H, 512] bf16 (the forward's output)
  const float* lse;       // [T, H] fp32 (the forward's sink-inclusive lse)
  const void* dout;       // [T, H, 512] bf16
  float* dq;              // [T, H, 512] fp32
  float* dkv;             // [num_kv, 512] fp32
  float* dsink;           // [H] fp32 or nullptr
  // workspace
  float* delta;           // [T, H]
  void* pds;              // [T, topk, 2H] bf16: P, then scale * dS, per compacted slot
  int* crow;              // [T, topk] kv row of each compacted slot
  int* ncnt;              // [T] valid slots per token
  void* interm;           // [T, topk, 512] bf16: each compacted slot's dkv contribution
  int* row_cnt;           // [num_kv + 1] counts, then exclusive starts (last = total)
  int* row_cur;           // [num_kv] fill cursors
  int* blk;               // scan block totals
  int* list;              // [T * topk] entry ids (t * topk + slot) grouped by kv row
  int64_t T;
  int64_t num_kv;
  int32_t H;
  int32_t topk;
  int32_t idx64;
  float scale;
};

// Byte offsets of the backward's workspace regions (each 256-byte aligned).
struct BwdWorkspace {
  uint64_t delta, pds, crow, ncnt, interm, row_cnt, row_cur, blk, list, total;
};
BwdWorkspace bwd_workspace_layout(int64_t T, int32_t H, int32_t topk, int64_t num_kv);
// All backward kernels on `stream`; returns a cudaError_t value.
int launch_bwd(BwdParams p, void* workspace, void* stream);
// tcgen05 forms of the per-slot dkv contraction and of dq = dS'.K (H = 128);
// workspace pointers set, P / dS' and the compacted rows written.
int launch_bwd_interm_tc(const BwdParams& p, void* stream);
int launch_bwd_dq_tc(const BwdParams& p, void* stream);
int launch_bwd_sdp_tc(const BwdParams& p, void* stream);
// Device address of the backward's error word (bounded waits of its tcgen05 kernel).
int bwd_error_word(unsigned int** addr);

}  // namespace smla
