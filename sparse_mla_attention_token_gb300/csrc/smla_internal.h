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
  float* part_o;          // split path: [splits, T, H, 512] fp32 (sink-free, normalised)
  float* part_lse;        // split path: [splits, T, H] fp32 (sink-free)
  int64_t T;
  int64_t num_kv;
  int32_t H;
  int32_t topk;
  int32_t splits;         // >= 1
  int32_t idx64;          // 1: int64 indices
  float scale;
};

// Largest slot range one CTA of the small-head kernel compacts in shared memory.
constexpr int kSmallHMaxSlots = 2048;

// Small-head kernel (mma.sync, head groups of 16); any H in {8,...,128}.
// Returns a cudaError_t value (0 = success).
int launch_smallh(const FwdParams& p, void* stream);

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
int smallh_geometry(int64_t T, int32_t H, int32_t splits, LaunchGeom* g);
int h128_geometry(int64_t T, LaunchGeom* g);

// Partial rows (splits * T * H) the static scratch of the allocation-free
// split path holds: 8192 rows of 512 + 1 fp32 = 16 MiB.
constexpr int64_t kNoAllocScratchRows = 8192;
// Split path (splits >= 2) with its partials in the library's static scratch;
// fills p.part_o / p.part_lse itself.  Returns a cudaError_t value.
int launch_split_static_scratch(FwdParams p, void* stream);

// Merge split partials into out / lse, folding the sink once.
int launch_combine(const FwdParams& p, void* stream);

}  // namespace smla
