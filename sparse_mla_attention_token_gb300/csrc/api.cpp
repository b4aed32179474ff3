// C ABI of the sparse MLA prefill forward: argument validation, planning
// (kernel family and split count), launches and status reporting.
//
// Validation mirrors the checks of the pages' public entry ("Tuned sparse MLA
// prefill for DSv4.1-Flash TP4; fix attn_sink in Triton fallback": clear
// errors for a bad q, a kv mismatch and an unusable out=, out= on q's device
// with a unit-stride last dim) in C terms: null pointers, shapes, alignment,
// aliasing and a finite scale, all decided on the host before any CUDA call.
// Index values are never errors: any value outside [0, num_kv) is an invalid
// slot, resolved on the device.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "smla_internal.h"
#include "sparse_mla.h"

namespace {

constexpr int32_t kAbiVersion = 1;
constexpr int kMaxSplits = 64;
constexpr int kDefaultSMs = 152;  // planning without a device (host-only checks)

thread_local char g_last_cuda_error[256] = "";

smla_status_t cuda_fail(cudaError_t e, const char* where) {
  std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s (%d)", where,
                cudaGetErrorString(e), static_cast<int>(e));
  return SMLA_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlap(const void* a, uint64_t na, const void* b, uint64_t nb) {
  if (a == nullptr || b == nullptr || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

struct Plan {
  int family;    // 0 small-head, 1 tcgen05 H=128
  int splits;
  int launches;
};

// Streaming multiprocessors of the current device (looked up once per device),
// or kDefaultSMs when no device can be queried.
int device_sms() {
  static int per_dev[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();   // no device here: clear the error and plan for the default
    return kDefaultSMs;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (per_dev[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return kDefaultSMs;
    }
    per_dev[dev] = n;
  }
  return per_dev[dev];
}

// kernel family and split count; `dims512` false for other head dims (the
// tcgen05 kernel is built for 512-wide rows only)
smla_status_t make_plan(int64_t T, int32_t H, int32_t topk, int64_t num_kv, int32_t num_splits,
                        int num_sms, Plan* pl, bool dims512 = true) {
  if (num_splits < 0 || num_splits > kMaxSplits) return SMLA_ERR_BAD_SPLITS;
  const int min_splits =
      std::max(1, (topk + smla::kSmallHMaxSlots - 1) / smla::kSmallHMaxSlots);
  int splits;
  const int64_t ctas = T * ((H + 15) / 16);          // small-head CTAs without splits
  const int decode_splits = (topk + 127) / 128;      // about 128 slots per split
  if (num_splits > 0) {
    splits = num_splits;
  } else if (decode_splits >= 2 && ctas > 0 && ctas * decode_splits <= 2 * num_sms) {
    // a decode-sized call (a few tokens): the split path with ~128 slots per
    // split, while its grid fits the GPU twice (measured faster than the
    // persistent kernels and than more, shorter splits for 1-16 tokens)
    splits = std::min(decode_splits, 16);
  } else if (dims512 && smla::h128_supported(T, H, topk, num_kv)) {
    splits = 1;
  } else {
    // enough CTAs to cover the GPU twice; each split keeps >= 64 slots
    splits = 1;
    if (ctas > 0 && ctas < 2 * num_sms) {
      const int64_t want = (2 * num_sms + ctas - 1) / ctas;
      splits = static_cast<int>(std::min<int64_t>(want, std::max(1, topk / 64)));
      splits = std::min(splits, 16);
    }
  }
  splits = std::max(splits, min_splits);
  if (num_splits > 0 && splits != num_splits) return SMLA_ERR_BAD_SPLITS;  // too few for topk
  if (splits > kMaxSplits) return SMLA_ERR_BAD_SPLITS;
  const bool tc = dims512 && (splits == 1) && smla::h128_supported(T, H, topk, num_kv);
  pl->family = tc ? 1 : 0;
  pl->splits = splits;
  pl->launches = (T == 0) ? 0 : (splits > 1 ? 2 : 1);
  return SMLA_OK;
}

smla_status_t validate(const void* q, const void* kv, const void* idx, int32_t index_dtype,
                       const float* sink, float scale, void* out, float* lse, int64_t T,
                       int32_t H, int64_t num_kv, int32_t topk, const int64_t* trace,
                       int32_t d_qk = smla::kHeadDim, int32_t d_v = smla::kHeadDim,
                       uint64_t kv_row_bytes = 0) {
  if (T < 0 || num_kv < 0 || num_kv >= (int64_t(1) << 31) || topk < 0) return SMLA_ERR_BAD_SHAPE;
  if (T > (int64_t(1) << 31) - 1) return SMLA_ERR_BAD_SHAPE;
  if (!(H == 8 || H == 16 || H == 32 || H == 64 || H == 128)) return SMLA_ERR_UNSUPPORTED_H;
  if (index_dtype != SMLA_IDX_INT32 && index_dtype != SMLA_IDX_INT64)
    return SMLA_ERR_BAD_INDEX_DTYPE;
  if (!std::isfinite(scale)) return SMLA_ERR_BAD_SCALE;
  if (T == 0) return SMLA_OK;
  if (q == nullptr || out == nullptr || lse == nullptr) return SMLA_ERR_NULL_PTR;
  if (num_kv > 0 && kv == nullptr) return SMLA_ERR_NULL_PTR;
  if (topk > 0 && idx == nullptr) return SMLA_ERR_NULL_PTR;
  const uintptr_t isz = index_dtype == SMLA_IDX_INT64 ? 8 : 4;
  if (!aligned(q, 16) || !aligned(out, 16) || (kv && !aligned(kv, 16)) || !aligned(lse, 4) ||
      (idx && !aligned(idx, isz)) || (sink && !aligned(sink, 4)) || (trace && !aligned(trace, 8)))
    return SMLA_ERR_MISALIGNED;
  const uint64_t qb = uint64_t(T) * H * d_qk * 2;
  const uint64_t ob = uint64_t(T) * H * d_v * 2;
  const uint64_t kvb = uint64_t(num_kv) * (kv_row_bytes ? kv_row_bytes : uint64_t(d_qk) * 2);
  const uint64_t ib = uint64_t(T) * topk * isz;
  const uint64_t lb = uint64_t(T) * H * 4;
  const uint64_t sb = sink ? uint64_t(H) * 4 : 0;
  const uint64_t tb = trace ? uint64_t(T) * topk * 8 : 0;
  const void* ins[4] = {q, kv, idx, sink};
  const uint64_t inb[4] = {qb, kvb, ib, sb};
  for (int i = 0; i < 4; ++i) {
    if (overlap(out, ob, ins[i], inb[i]) || overlap(lse, lb, ins[i], inb[i]) ||
        overlap(trace, tb, ins[i], inb[i]))
      return SMLA_ERR_ALIASING;
  }
  if (overlap(out, ob, lse, lb) || overlap(out, ob, trace, tb) || overlap(lse, lb, trace, tb))
    return SMLA_ERR_ALIASING;
  return SMLA_OK;
}

smla_status_t run(const void* q, const void* kv, const void* idx, int32_t index_dtype,
                  const float* sink, float scale, void* out, float* lse, int64_t T, int32_t H,
                  int64_t num_kv, int32_t topk, void* stream, int32_t num_splits,
                  int64_t* trace, int32_t d_qk = smla::kHeadDim, int32_t d_v = smla::kHeadDim,
                  bool fp8 = false, const float* kv_scale = nullptr) {
  smla_status_t st = validate(q, kv, idx, index_dtype, sink, scale, out, lse, T, H, num_kv, topk,
                              trace, d_qk, d_v, fp8 ? uint64_t(d_qk) : 0);
  if (st != SMLA_OK) return st;
  // the tcgen05 kernel serves 512-wide bf16 rows only
  const bool dims512 = d_qk == smla::kHeadDim && d_v == smla::kHeadDim && !fp8;
  Plan pl;
  st = make_plan(T, H, topk, num_kv, num_splits, T > 0 ? device_sms() : kDefaultSMs, &pl,
                 dims512);
  if (st != SMLA_OK) return st;
  if (T == 0) return SMLA_OK;

  smla::FwdParams p{};
  p.q = q;
  p.kv = kv;
  p.idx = idx;
  p.sink = sink;
  p.out = out;
  p.lse = lse;
  p.trace = trace;
  p.T = T;
  p.num_kv = num_kv;
  p.H = H;
  p.topk = topk;
  p.splits = pl.splits;
  p.idx64 = index_dtype == SMLA_IDX_INT64 ? 1 : 0;
  p.d_qk = d_qk;
  p.d_v = d_v;
  p.kv_fp8 = fp8 ? 1 : 0;
  p.kv_scale = kv_scale;
  p.scale = scale;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (pl.family == 1) {
    const int e = smla::launch_h128(p, stream);
    if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "h128 kernel launch");
    return SMLA_OK;
  }
  if (pl.splits == 1) {
    const int e = smla::launch_smallh(p, stream);
    if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "small-head kernel launch");
    return SMLA_OK;
  }
  // split path: stream-ordered workspace for the partials
  const uint64_t rows = uint64_t(pl.splits) * uint64_t(T) * uint64_t(H);
  const size_t bytes = rows * d_v * 4 + rows * 4;
  void* ws = nullptr;
  cudaError_t ce = cudaMallocAsync(&ws, bytes, s);
  if (ce != cudaSuccess) return cuda_fail(ce, "cudaMallocAsync(split workspace)");
  p.part_o = static_cast<float*>(ws);
  p.part_lse = reinterpret_cast<float*>(static_cast<char*>(ws) + rows * d_v * 4);
  int e = smla::launch_smallh(p, stream);
  if (e == 0) e = smla::launch_combine(p, stream);
  ce = cudaFreeAsync(ws, s);
  if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "split path launch");
  if (ce != cudaSuccess) return cuda_fail(ce, "cudaFreeAsync(split workspace)");
  return SMLA_OK;
}

// Device workspace of the host-buffer call: kv | q | idx | sink | out | lse,
// each region 256-byte aligned.
struct HostWs {
  uint64_t kv, q, idx, sink, out, lse, total;
};

HostWs host_ws_layout(int64_t T, int32_t H, int32_t topk, int64_t num_kv, int32_t index_dtype,
                      bool has_sink) {
  auto up = [](uint64_t x) { return (x + 255) & ~uint64_t(255); };
  const uint64_t isz = index_dtype == SMLA_IDX_INT64 ? 8 : 4;
  HostWs w{};
  uint64_t o = 0;
  w.kv = o;
  o += up(uint64_t(num_kv) * smla::kHeadDim * 2);
  w.q = o;
  o += up(uint64_t(T) * H * smla::kHeadDim * 2);
  w.idx = o;
  o += up(uint64_t(T) * topk * isz);
  w.sink = o;
  o += up(has_sink ? uint64_t(H) * 4 : 0);
  w.out = o;
  o += up(uint64_t(T) * H * smla::kHeadDim * 2);
  w.lse = o;
  o += up(uint64_t(T) * H * 4);
  w.total = o;
  return w;
}

// Copy streams and events of the host-buffer call, per device, made on first
// use and reused (calls enqueue under the lock, so they serialise on them).
constexpr int kMaxHostChunks = 16;
struct HostStreams {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t in_ev[kMaxHostChunks] = {}, k_ev[kMaxHostChunks] = {};
};

cudaError_t host_streams(HostStreams** out, std::unique_lock<std::mutex>* lock) {
  static HostStreams per_dev[64];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  *lock = std::unique_lock<std::mutex>(mu);
  HostStreams& h = per_dev[dev];
  if (!h.ready) {
    const unsigned f = cudaEventDisableTiming;
    e = cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.start, f);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.done, f);
    for (int i = 0; i < kMaxHostChunks && e == cudaSuccess; ++i) {
      e = cudaEventCreateWithFlags(&h.in_ev[i], f);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.k_ev[i], f);
    }
    if (e != cudaSuccess) {   // release what was made, so that a later call starts afresh
      if (h.in) cudaStreamDestroy(h.in);
      if (h.out) cudaStreamDestroy(h.out);
      if (h.start) cudaEventDestroy(h.start);
      if (h.done) cudaEventDestroy(h.done);
      for (int i = 0; i < kMaxHostChunks; ++i) {
        if (h.in_ev[i]) cudaEventDestroy(h.in_ev[i]);
        if (h.k_ev[i]) cudaEventDestroy(h.k_ev[i]);
      }
      h = HostStreams{};
      return e;
    }
    h.ready = true;
  }
  *out = &h;
  return cudaSuccess;
}

}  // namespace

extern "C" {

smla_status_t sparse_mla_fwd_host_workspace(int64_t T, int32_t H, int32_t topk, int64_t num_kv,
                                            int32_t index_dtype, int32_t has_sink,
                                            uint64_t* bytes) {
  if (T < 0 || topk < 0 || num_kv < 0 || num_kv >= (int64_t(1) << 31)) return SMLA_ERR_BAD_SHAPE;
  if (!(H == 8 || H == 16 || H == 32 || H == 64 || H == 128)) return SMLA_ERR_UNSUPPORTED_H;
  if (index_dtype != SMLA_IDX_INT32 && index_dtype != SMLA_IDX_INT64)
    return SMLA_ERR_BAD_INDEX_DTYPE;
  if (bytes == nullptr) return SMLA_ERR_NULL_PTR;
  *bytes = host_ws_layout(T, H, topk, num_kv, index_dtype, has_sink != 0).total;
  return SMLA_OK;
}

smla_status_t sparse_mla_fwd_host(const void* q_host, const void* kv_host,
                                  const void* topk_indices_host, int32_t index_dtype,
                                  const float* attn_sink_host, float scale, void* out_host,
                                  float* lse_host, int64_t T, int32_t H, int64_t num_kv,
                                  int32_t topk, void* workspace, uint64_t workspace_bytes,
                                  void* stream) {
  smla_status_t st = validate(q_host, kv_host, topk_indices_host, index_dtype, attn_sink_host,
                              scale, out_host, lse_host, T, H, num_kv, topk, nullptr);
  if (st != SMLA_OK) return st;
  Plan pl;
  st = make_plan(T, H, topk, num_kv, 0, T > 0 ? device_sms() : kDefaultSMs, &pl);
  if (st != SMLA_OK) return st;
  if (T == 0) return SMLA_OK;
  const HostWs w = host_ws_layout(T, H, topk, num_kv, index_dtype, attn_sink_host != nullptr);
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < w.total)
    return SMLA_ERR_WORKSPACE;

  char* ws = static_cast<char*>(workspace);
  const uint64_t isz = index_dtype == SMLA_IDX_INT64 ? 8 : 4;
  const uint64_t q_tok = uint64_t(H) * smla::kHeadDim * 2, i_tok = uint64_t(topk) * isz,
                 l_tok = uint64_t(H) * 4;
  // chunks of at least 256 tokens (a full-GPU grid each), at most kMaxHostChunks
  const int64_t nch = std::max<int64_t>(1, std::min<int64_t>(kMaxHostChunks, T / 256));
  const int64_t per = (T + nch - 1) / nch;

  HostStreams* hs = nullptr;
  std::unique_lock<std::mutex> lock;
  cudaError_t e = host_streams(&hs, &lock);
  if (e != cudaSuccess) return cuda_fail(e, "host-call streams");
  cudaStream_t s0 = static_cast<cudaStream_t>(stream);
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
  // the copies start after the caller's earlier work on `stream`
  if ((e = cudaEventRecord(hs->start, s0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(hs->in, hs->start, 0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(hs->out, hs->start, 0)) != cudaSuccess)
    return cuda_fail(e, "host-call ordering");
  if (num_kv > 0 &&
      (e = cudaMemcpyAsync(ws + w.kv, kv_host, uint64_t(num_kv) * smla::kHeadDim * 2, h2d,
                           hs->in)) != cudaSuccess)
    return cuda_fail(e, "copy in kv");
  if (attn_sink_host != nullptr &&
      (e = cudaMemcpyAsync(ws + w.sink, attn_sink_host, uint64_t(H) * 4, h2d, hs->in)) !=
          cudaSuccess)
    return cuda_fail(e, "copy in sink");
  for (int64_t c = 0; c < nch; ++c) {
    const int64_t t0 = c * per, tc = std::min<int64_t>(per, T - t0);
    if (tc <= 0) break;
    if ((e = cudaMemcpyAsync(ws + w.q + t0 * q_tok, static_cast<const char*>(q_host) + t0 * q_tok,
                             tc * q_tok, h2d, hs->in)) != cudaSuccess ||
        (topk > 0 && (e = cudaMemcpyAsync(ws + w.idx + t0 * i_tok,
                                          static_cast<const char*>(topk_indices_host) + t0 * i_tok,
                                          tc * i_tok, h2d, hs->in)) != cudaSuccess) ||
        (e = cudaEventRecord(hs->in_ev[c], hs->in)) != cudaSuccess)
      return cuda_fail(e, "copy in chunk");
  }
  for (int64_t c = 0; c < nch; ++c) {
    const int64_t t0 = c * per, tc = std::min<int64_t>(per, T - t0);
    if (tc <= 0) break;
    if ((e = cudaStreamWaitEvent(s0, hs->in_ev[c], 0)) != cudaSuccess)
      return cuda_fail(e, "chunk ordering");
    st = run(ws + w.q + t0 * q_tok, num_kv > 0 ? ws + w.kv : nullptr,
             topk > 0 ? ws + w.idx + t0 * i_tok : nullptr, index_dtype,
             attn_sink_host != nullptr ? reinterpret_cast<const float*>(ws + w.sink) : nullptr,
             scale, ws + w.out + t0 * q_tok, reinterpret_cast<float*>(ws + w.lse + t0 * l_tok), tc,
             H, num_kv, topk, stream, pl.splits, nullptr);   // the whole call's plan
    if (st != SMLA_OK) return st;
    if ((e = cudaEventRecord(hs->k_ev[c], s0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(hs->out, hs->k_ev[c], 0)) != cudaSuccess ||
        (e = cudaMemcpyAsync(static_cast<char*>(out_host) + t0 * q_tok, ws + w.out + t0 * q_tok,
                             tc * q_tok, d2h, hs->out)) != cudaSuccess ||
        (e = cudaMemcpyAsync(reinterpret_cast<char*>(lse_host) + t0 * l_tok,
                             ws + w.lse + t0 * l_tok, tc * l_tok, d2h, hs->out)) != cudaSuccess)
      return cuda_fail(e, "copy out chunk");
  }
  // the caller's stream passes this call once the last result is in host memory
  if ((e = cudaEventRecord(hs->done, hs->out)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(s0, hs->done, 0)) != cudaSuccess)
    return cuda_fail(e, "host-call completion");
  return SMLA_OK;
}

smla_status_t sparse_mla_fwd(const void* q, const void* kv, const void* topk_indices,
                             int32_t index_dtype, const float* attn_sink, float scale,
                             void* out, float* lse, int64_t T, int32_t H, int64_t num_kv,
                             int32_t topk, void* stream) {
  return run(q, kv, topk_indices, index_dtype, attn_sink, scale, out, lse, T, H, num_kv, topk,
             stream, 0, nullptr);
}

smla_status_t sparse_mla_fwd_fp8kv(const void* q, const void* kv_fp8, const float* kv_scale,
                                   const void* topk_indices, int32_t index_dtype,
                                   const float* attn_sink, float scale, void* out, float* lse,
                                   int64_t T, int32_t H, int64_t num_kv, int32_t topk,
                                   void* stream) {
  if (T < 0 || num_kv < 0 || num_kv >= (int64_t(1) << 31) || topk < 0) return SMLA_ERR_BAD_SHAPE;
  if (T > 0 && num_kv > 0 && (kv_fp8 == nullptr || kv_scale == nullptr)) return SMLA_ERR_NULL_PTR;
  if ((kv_fp8 && !aligned(kv_fp8, 16)) || (kv_scale && !aligned(kv_scale, 16)))
    return SMLA_ERR_MISALIGNED;
  // the scales are one more input that the outputs may not overlap
  const uint64_t sb = uint64_t(num_kv) * 16;
  const uint64_t ob = uint64_t(T) * H * smla::kHeadDim * 2, lb = uint64_t(T) * H * 4;
  if (overlap(out, ob, kv_scale, sb) || overlap(lse, lb, kv_scale, sb)) return SMLA_ERR_ALIASING;
  return run(q, kv_fp8, topk_indices, index_dtype, attn_sink, scale, out, lse, T, H, num_kv, topk,
             stream, 0, nullptr, smla::kHeadDim, smla::kHeadDim, true, kv_scale);
}

smla_status_t sparse_mla_fwd_dims(const void* q, const void* kv, const void* topk_indices,
                                  int32_t index_dtype, const float* attn_sink, float scale,
                                  void* out, float* lse, int64_t T, int32_t H, int64_t num_kv,
                                  int32_t topk, int32_t d_qk, int32_t d_v, void* stream) {
  if (!smla::smallh_dims_supported(d_qk, d_v)) return SMLA_ERR_BAD_SHAPE;
  return run(q, kv, topk_indices, index_dtype, attn_sink, scale, out, lse, T, H, num_kv, topk,
             stream, 0, nullptr, d_qk, d_v);
}

smla_status_t sparse_mla_fwd_ex(const void* q, const void* kv, const void* topk_indices,
                                int32_t index_dtype, const float* attn_sink, float scale,
                                void* out, float* lse, int64_t T, int32_t H, int64_t num_kv,
                                int32_t topk, void* stream, int32_t num_splits,
                                int64_t* read_trace) {
  return run(q, kv, topk_indices, index_dtype, attn_sink, scale, out, lse, T, H, num_kv, topk,
             stream, num_splits, read_trace);
}

smla_status_t sparse_mla_fwd_static_scratch(const void* q, const void* kv,
                                            const void* topk_indices, int32_t index_dtype,
                                            const float* attn_sink, float scale, void* out,
                                            float* lse, int64_t T, int32_t H, int64_t num_kv,
                                            int32_t topk, void* stream, int32_t num_splits) {
  smla_status_t st = validate(q, kv, topk_indices, index_dtype, attn_sink, scale, out, lse, T, H,
                              num_kv, topk, nullptr);
  if (st != SMLA_OK) return st;
  if (num_splits == 1) return SMLA_ERR_BAD_SPLITS;   // this path always splits
  Plan pl;
  st = make_plan(T, H, topk, num_kv, num_splits, T > 0 ? device_sms() : kDefaultSMs, &pl);
  if (st != SMLA_OK) return st;
  const int splits = std::max(2, pl.splits);
  if (T == 0) return SMLA_OK;
  if (int64_t(splits) * T * H > smla::kNoAllocScratchRows) return SMLA_ERR_SCRATCH_LIMIT;
  smla::FwdParams p{};
  p.q = q;
  p.kv = kv;
  p.idx = topk_indices;
  p.sink = attn_sink;
  p.out = out;
  p.lse = lse;
  p.trace = nullptr;
  p.T = T;
  p.num_kv = num_kv;
  p.H = H;
  p.topk = topk;
  p.splits = splits;
  p.idx64 = index_dtype == SMLA_IDX_INT64 ? 1 : 0;
  p.d_qk = smla::kHeadDim;
  p.d_v = smla::kHeadDim;
  p.scale = scale;
  const int e = smla::launch_split_static_scratch(p, stream);
  if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "static-scratch split path launch");
  return SMLA_OK;
}

smla_status_t sparse_mla_bwd_workspace(int64_t T, int32_t H, int32_t topk, int64_t num_kv,
                                       uint64_t* bytes) {
  if (T < 0 || topk < 0 || topk > smla::kSmallHMaxSlots || num_kv < 0 ||
      num_kv >= (int64_t(1) << 31) || T * int64_t(topk) >= (int64_t(1) << 31))
    return SMLA_ERR_BAD_SHAPE;
  if (!(H == 8 || H == 16 || H == 32 || H == 64 || H == 128)) return SMLA_ERR_UNSUPPORTED_H;
  if (bytes == nullptr) return SMLA_ERR_NULL_PTR;
  *bytes = smla::bwd_workspace_layout(T, H, topk, num_kv).total;
  return SMLA_OK;
}

smla_status_t sparse_mla_bwd(const void* q, const void* kv, const void* topk_indices,
                             int32_t index_dtype, const float* attn_sink, float scale,
                             const void* out, const float* lse, const void* dout, float* dq,
                             float* dkv, float* dsink, int64_t T, int32_t H, int64_t num_kv,
                             int32_t topk, void* workspace, uint64_t workspace_bytes,
                             void* stream) {
  uint64_t need = 0;
  smla_status_t st = sparse_mla_bwd_workspace(T, H, topk, num_kv, &need);
  if (st != SMLA_OK) return st;
  if (index_dtype != SMLA_IDX_INT32 && index_dtype != SMLA_IDX_INT64)
    return SMLA_ERR_BAD_INDEX_DTYPE;
  if (!std::isfinite(scale)) return SMLA_ERR_BAD_SCALE;
  if (num_kv > 0 && (kv == nullptr || dkv == nullptr)) return SMLA_ERR_NULL_PTR;
  if (T > 0 && (q == nullptr || out == nullptr || lse == nullptr || dout == nullptr ||
                dq == nullptr || (topk > 0 && topk_indices == nullptr)))
    return SMLA_ERR_NULL_PTR;
  const uintptr_t isz = index_dtype == SMLA_IDX_INT64 ? 8 : 4;
  if ((q && !aligned(q, 16)) || (kv && !aligned(kv, 16)) || (out && !aligned(out, 16)) ||
      (dout && !aligned(dout, 16)) || (dq && !aligned(dq, 16)) || (dkv && !aligned(dkv, 16)) ||
      (lse && !aligned(lse, 4)) || (dsink && !aligned(dsink, 4)) ||
      (attn_sink && !aligned(attn_sink, 4)) || (topk_indices && !aligned(topk_indices, isz)))
    return SMLA_ERR_MISALIGNED;
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < need)
    return SMLA_ERR_WORKSPACE;
  const uint64_t qb = uint64_t(T) * H * smla::kHeadDim * 2;
  const uint64_t kvb = uint64_t(num_kv) * smla::kHeadDim * 2;
  const uint64_t ib = uint64_t(T) * topk * isz;
  const uint64_t lb = uint64_t(T) * H * 4;
  const uint64_t sb = attn_sink ? uint64_t(H) * 4 : 0;
  const void* ins[6] = {q, kv, topk_indices, attn_sink, out, dout};
  const uint64_t inb[6] = {qb, kvb, ib, sb, qb, qb};
  void* outs[4] = {dq, dkv, dsink, workspace};
  const uint64_t outb[4] = {qb * 2, kvb * 2, dsink ? uint64_t(H) * 4 : 0, need};
  for (int o = 0; o < 4; ++o) {
    for (int i = 0; i < 6; ++i)
      if (overlap(outs[o], outb[o], ins[i], inb[i])) return SMLA_ERR_ALIASING;
    if (overlap(outs[o], outb[o], lse, lb)) return SMLA_ERR_ALIASING;
    for (int o2 = o + 1; o2 < 4; ++o2)
      if (overlap(outs[o], outb[o], outs[o2], outb[o2])) return SMLA_ERR_ALIASING;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (T == 0) {   // no token: every gradient is zero
    if (num_kv > 0 && (e = cudaMemsetAsync(dkv, 0, kvb * 2, s)) != cudaSuccess)
      return cuda_fail(e, "zero dkv");
    if (dsink && (e = cudaMemsetAsync(dsink, 0, uint64_t(H) * 4, s)) != cudaSuccess)
      return cuda_fail(e, "zero dsink");
    return SMLA_OK;
  }
  smla::BwdParams p{};
  p.q = q;
  p.kv = kv;
  p.idx = topk_indices;
  p.sink = attn_sink;
  p.out = out;
  p.lse = lse;
  p.dout = dout;
  p.dq = dq;
  p.dkv = dkv;
  p.dsink = dsink;
  p.T = T;
  p.num_kv = num_kv;
  p.H = H;
  p.topk = topk;
  p.idx64 = index_dtype == SMLA_IDX_INT64 ? 1 : 0;
  p.scale = scale;
  const int r = smla::launch_bwd(p, workspace, stream);
  if (r != 0) return cuda_fail(static_cast<cudaError_t>(r), "backward launch");
  return SMLA_OK;
}

smla_status_t sparse_mla_plan(int64_t T, int32_t H, int32_t topk, int32_t num_splits,
                              int32_t* kernel_family, int32_t* splits_out,
                              int32_t* launches_out) {
  if (T < 0 || topk < 0) return SMLA_ERR_BAD_SHAPE;
  if (!(H == 8 || H == 16 || H == 32 || H == 64 || H == 128)) return SMLA_ERR_UNSUPPORTED_H;
  Plan pl;
  const smla_status_t st = make_plan(T, H, topk, 1, num_splits, device_sms(), &pl);
  if (st != SMLA_OK) return st;
  if (kernel_family) *kernel_family = pl.family;
  if (splits_out) *splits_out = pl.splits;
  if (launches_out) *launches_out = pl.launches;
  return SMLA_OK;
}

smla_status_t sparse_mla_launch_config(int64_t T, int32_t H, int32_t topk, int64_t num_kv,
                                       int32_t num_splits, int32_t* grid_ctas,
                                       int32_t* cta_threads, int32_t* cluster_size,
                                       int32_t* smem_bytes) {
  if (T < 0 || topk < 0 || num_kv < 0) return SMLA_ERR_BAD_SHAPE;
  if (!(H == 8 || H == 16 || H == 32 || H == 64 || H == 128)) return SMLA_ERR_UNSUPPORTED_H;
  Plan pl;
  smla_status_t st = make_plan(T, H, topk, num_kv, num_splits, device_sms(), &pl);
  if (st != SMLA_OK) return st;
  smla::LaunchGeom g{0, 0, 0, 0};
  const int e = pl.family == 1 ? smla::h128_geometry(T, &g)
                               : smla::smallh_geometry(T, H, pl.splits, smla::kHeadDim,
                                                       smla::kHeadDim, &g);
  if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "launch geometry");
  if (grid_ctas) *grid_ctas = g.grid_ctas;
  if (cta_threads) *cta_threads = g.threads;
  if (cluster_size) *cluster_size = g.cluster;
  if (smem_bytes) *smem_bytes = g.smem;
  return SMLA_OK;
}

smla_status_t sparse_mla_selftest_wait_timeout(void* stream) {
  const int e = smla::selftest_wait_timeout(stream);
  if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "self-test launch");
  return SMLA_OK;
}

smla_status_t sparse_mla_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  // the forward's and the backward's error words (bounded waits of their tcgen05 kernels)
  bool expired = false;
  for (int w = 0; w < 2; ++w) {
    unsigned int* word = nullptr;
    const int ge = w == 0 ? smla::h128_error_word(&word) : smla::bwd_error_word(&word);
    if (ge != 0) return cuda_fail(static_cast<cudaError_t>(ge), "cudaGetSymbolAddress(error word)");
    if (word == nullptr) continue;
    unsigned int v = 0;
    e = cudaMemcpy(&v, word, sizeof(v), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read device error word");
    if (v != 0) {
      const unsigned int zero = 0;
      e = cudaMemcpy(word, &zero, sizeof(zero), cudaMemcpyHostToDevice);
      if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
      expired = true;
    }
  }
  return expired ? SMLA_ERR_DEVICE_TIMEOUT : SMLA_OK;
}

const char* sparse_mla_strerror(int32_t status) {
  switch (status) {
    case SMLA_OK: return "ok";
    case SMLA_ERR_NULL_PTR: return "a required pointer is NULL";
    case SMLA_ERR_BAD_SHAPE: return "bad shape (T, num_kv or topk out of range)";
    case SMLA_ERR_UNSUPPORTED_H: return "unsupported head count (H must be 8, 16, 32, 64 or 128)";
    case SMLA_ERR_BAD_INDEX_DTYPE: return "index dtype must be int32 or int64";
    case SMLA_ERR_MISALIGNED: return "misaligned buffer (q, kv, out need 16 bytes)";
    case SMLA_ERR_BAD_SCALE: return "scale must be finite";
    case SMLA_ERR_ALIASING: return "an output buffer overlaps another buffer";
    case SMLA_ERR_CUDA: return "CUDA runtime error";
    case SMLA_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait (outputs unspecified)";
    case SMLA_ERR_BAD_SPLITS: return "split count out of range for this topk";
    case SMLA_ERR_SCRATCH_LIMIT:
      return "splits*T*H exceeds the 8192 partial rows of the static scratch "
             "(use sparse_mla_fwd for calls this large)";
    case SMLA_ERR_WORKSPACE:
      return "workspace is NULL, smaller than sparse_mla_fwd_host_workspace() or not "
             "256-byte aligned";
    default: return "unknown status";
  }
}

const char* sparse_mla_last_cuda_error(void) { return g_last_cuda_error; }

#ifdef SMLA_TIMELINE
// Debug builds only (-DSMLA_TIMELINE): copy the H=128 kernel's cluster-0 role
// timeline (2 ranks x 4 roles x 64 tiles x 8 events of clock64) to host memory.
int sparse_mla_debug_timeline(long long* host) { return smla::h128_timeline(host); }
#endif

int32_t sparse_mla_abi_version(void) { return kAbiVersion; }

}  // extern "C"
