/*
 * sparse_mla.h -- C ABI of the GB300 (sm_103a) sparse MLA prefill forward.
 *
 * The operation (DeepSeek-V4 sparse MLA, "has_pe = False" path) is the one
 * defined in "Sparse MLA training backward" (aiter PR #4766), section
 * "Contract", and in "Tuned sparse MLA prefill for DSv4.1-Flash TP4; fix
 * attn_sink in Triton fallback" (aiter PR #6002), description items
 * "attn_sink", "int64 indices" and "Invalid KV rows":
 *
 *   for every token t and head h, over the slots j whose row r = idx[t, j]
 *   lies in [0, num_kv) (any other value is an invalid slot, never read):
 *     s_j = scale * <q[t,h,:], kv[r,:]>            (K == V == kv, 512 wide)
 *     m   = max(max_j s_j, sink[h])
 *     den = sum_j exp(s_j - m) + exp(sink[h] - m)  (sink: denominator only)
 *     out[t,h,:] = bf16( sum_j exp(s_j - m) * kv[r,:] / den )
 *     lse[t,h]   = m + ln(den)                     (sink-inclusive, natural log)
 *   A row with no valid slot gives out = 0 and lse = -inf without a sink
 *   (or with sink = -inf), lse = sink[h] with a finite sink.
 *   A duplicated row counts once per slot that names it.
 *
 * Numerics: S and the softmax run in fp32 (base 2, scale folded into one
 * multiply); the probabilities P are rounded to bf16 before P.V (a choice
 * the definition above leaves open); O is accumulated in fp32 and rounded to
 * bf16 once.  The H = 128 kernel splits the 512-wide contraction between the two
 * CTAs of a cluster: each takes its row's largest partial score off, rounds
 * the remainder it sends to the other CTA to fp16 and adds the received one to
 * its own in fp32, so a score's error is at most 2^-11 of how far its partial
 * lies below the row's largest partial (shared score components cost nothing).
 * Results are deterministic for given inputs and launch configuration.
 *
 * Ownership: the caller owns every buffer passed in; all pointers except the
 * stream are device pointers unless stated.  Calls are asynchronous on
 * `stream` (a cudaStream_t; NULL = the legacy default stream) and return once
 * the work is queued.  Argument errors are detected on the host before any
 * CUDA call and leave every buffer untouched.  The library itself allocates
 * only the split path's partial-result workspace, stream-ordered on `stream`
 * (cudaMallocAsync / cudaFreeAsync).
 */
#ifndef SPARSE_MLA_H
#define SPARSE_MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of topk_indices. */
typedef enum {
  SMLA_IDX_INT32 = 0,
  SMLA_IDX_INT64 = 1
} smla_index_dtype_t;

/* Return codes.  Every entry point returns one of these. */
typedef enum {
  SMLA_OK = 0,
  SMLA_ERR_NULL_PTR = 1,         /* a required pointer is NULL                      */
  SMLA_ERR_BAD_SHAPE = 2,        /* T < 0, num_kv < 0 or >= 2^31, topk < 0, ...      */
  SMLA_ERR_UNSUPPORTED_H = 3,    /* H not in {8, 16, 32, 64, 128}                    */
  SMLA_ERR_BAD_INDEX_DTYPE = 4,  /* index_dtype not a smla_index_dtype_t value       */
  SMLA_ERR_MISALIGNED = 5,       /* q, kv or out not 16-byte aligned, lse not 4     */
  SMLA_ERR_BAD_SCALE = 6,        /* scale is NaN or infinite                         */
  SMLA_ERR_ALIASING = 7,         /* out or lse overlaps an input                     */
  SMLA_ERR_CUDA = 8,             /* a CUDA runtime call failed (see _last_cuda_error)*/
  SMLA_ERR_DEVICE_TIMEOUT = 9,   /* a kernel's bounded wait expired (device status)  */
  SMLA_ERR_BAD_SPLITS = 10,      /* forced split count out of range                  */
  SMLA_ERR_SCRATCH_LIMIT = 11,   /* splits*T*H beyond the library's static scratch   */
  SMLA_ERR_WORKSPACE = 12        /* host-buffer call: workspace NULL, short or       */
                                 /* not 256-byte aligned                             */
} smla_status_t;

/*
 * sparse_mla_fwd -- the op.
 *
 *   q            [T, H, 512] bf16, contiguous, 16-byte aligned.
 *   kv           [num_kv, 512] bf16, contiguous, 16-byte aligned; may sit at
 *                any 16-byte aligned offset inside a larger allocation
 *                (offsets beyond 2 GiB are fine: all address math is 64-bit).
 *   topk_indices [T, topk] int32 or int64 (index_dtype), contiguous.  Values
 *                are compared at their full width: anything outside
 *                [0, num_kv) is an invalid slot (never an error, never read).
 *   attn_sink    [H] fp32, or NULL for no sink.  -inf behaves as no sink.
 *   scale        finite; 1/sqrt(512) for DeepSeek-V4.  Negative is allowed.
 *   out          [T, H, 512] bf16, contiguous, 16-byte aligned, caller-allocated;
 *                must not overlap q, kv or topk_indices.
 *   lse          [T, H] fp32, contiguous, caller-allocated.
 *   T >= 0 (T == 0: nothing is launched), H in {8,16,32,64,128},
 *   0 <= num_kv < 2^31, topk >= 0 (num_kv == 0 or topk == 0: every row is
 *   fully masked).
 *   stream       cudaStream_t.
 *
 * The split count over the topk slots is chosen by the library.
 */
smla_status_t sparse_mla_fwd(const void* q, const void* kv, const void* topk_indices,
                             int32_t index_dtype, const float* attn_sink, float scale,
                             void* out, float* lse, int64_t T, int32_t H, int64_t num_kv,
                             int32_t topk, void* stream);

/*
 * sparse_mla_fwd_ex -- sparse_mla_fwd with two test/benchmark controls.
 *
 *   num_splits   0 = library choice; otherwise 1..64: the topk slots of each
 *                token are cut into num_splits contiguous ranges of
 *                ceil(topk / num_splits) slots, computed independently and
 *                merged by a combine kernel (the split-TOPK path;
 *                lse-weighted merge, the sink folded once).
 *   read_trace   NULL, or a device int64 [T, topk] buffer that records which
 *                kv rows the kernel's copies read.  Per token and per slot
 *                range (one range when the call does not split), the entries
 *                hold, in order, the row each gather reads for the range's
 *                valid slots (slot order; a duplicated row appears once per
 *                slot), then -1 for the rest of the range.  Each row entry is
 *                recovered from the source address of the copy that reads it,
 *                where that address is formed; the -1 entries are written
 *                where the slots are classified (nothing is read for them).
 */
smla_status_t sparse_mla_fwd_ex(const void* q, const void* kv, const void* topk_indices,
                                int32_t index_dtype, const float* attn_sink, float scale,
                                void* out, float* lse, int64_t T, int32_t H, int64_t num_kv,
                                int32_t topk, void* stream, int32_t num_splits,
                                int64_t* read_trace);

/*
 * sparse_mla_fwd_dims -- the op at other head dims, and with a positional part.
 *
 *   d_qk         score width: q is [T, H, d_qk], kv is [num_kv, d_qk] (bf16).
 *   d_v          value width: the values are the first d_v columns of each kv
 *                row; out is [T, H, d_v] bf16.
 *   Supported (d_qk, d_v): (512, 512) -- exactly sparse_mla_fwd; (128, 128)
 *   and (576, 576), K == V at the head dims "Tuned sparse MLA prefill for
 *   DSv4.1-Flash TP4" tests; (576, 512), the MLA layout of "Add DSv4 sparse
 *   MLA prefill Triton and unified with MLA Gluon kernel on GFX950" with
 *   has_pe = True: each row is [512 no-pe | 64 pe] (q the same), the scores
 *   use all 576 columns and only the no-pe part is a value.  Other pairs
 *   return SMLA_ERR_BAD_SHAPE.  scale is the caller's (1/sqrt(d_qk) is the
 *   usual choice).  Other arguments, layouts, errors and the allocation of
 *   the split path's workspace: as sparse_mla_fwd.  Pairs other than
 *   (512, 512) run on the small-head kernel family for every H.
 */
smla_status_t sparse_mla_fwd_dims(const void* q, const void* kv, const void* topk_indices,
                                  int32_t index_dtype, const float* attn_sink, float scale,
                                  void* out, float* lse, int64_t T, int32_t H, int64_t num_kv,
                                  int32_t topk, int32_t d_qk, int32_t d_v, void* stream);

/*
 * sparse_mla_fwd_fp8kv -- the op on an fp8 KV cache.
 *
 * The pages leave the fp8 cache out ("Add DSv4 sparse MLA prefill Triton and
 * unified with MLA Gluon kernel on GFX950": the fp8 paged decode cache is not
 * part of that change) and make the bf16 entry reject an fp8 pool with a dtype
 * error ("Tuned sparse MLA prefill for DSv4.1-Flash TP4", which the Python
 * binding's sparse_mla_fwd follows).  This entry point serves such a cache in
 * the layout this library reads it in:
 *
 *   kv_fp8       [num_kv, 512] bytes, OCP FP8 E4M3 (e4m3fn) codes, 16-byte
 *                aligned.
 *   kv_scale     [num_kv, 4] fp32, 16-byte aligned: one scale per 128-column
 *                block; the row's value in column c is
 *                decode(kv_fp8[r, c]) * kv_scale[r, c / 128].
 *   Everything else as sparse_mla_fwd: q, out bf16 [T, H, 512], the same
 *   checks, the split path's stream-ordered workspace.  Every H runs on the
 *   small-head kernel family.  Only the rows valid slots name are read.
 * Numerics: the codes are decoded exactly into bf16; the scales are applied in
 * fp32 to the partial scores and, per block, to P before its bf16 rounding.
 */
smla_status_t sparse_mla_fwd_fp8kv(const void* q, const void* kv_fp8, const float* kv_scale,
                                   const void* topk_indices, int32_t index_dtype,
                                   const float* attn_sink, float scale, void* out, float* lse,
                                   int64_t T, int32_t H, int64_t num_kv, int32_t topk,
                                   void* stream);

/*
 * sparse_mla_fwd_static_scratch -- the split-TOPK path without any allocation.
 *
 * The pages have no counterpart to this entry point.  It exists for callers
 * that must not allocate device memory while they run: serving loops with a
 * fixed memory budget, code running inside a window in which no allocation may
 * happen, and hosts whose allocator is owned by another runtime.
 * sparse_mla_fwd_ex allocates the split path's partial results on every call;
 * this entry point keeps them in one fixed array inside the library instead
 * (8192 x 2052 bytes = 16,809,984 bytes of device memory, held by every GPU
 * that loads the library until the process exits) and calls no cudaMalloc /
 * cudaFree or any allocating routine.
 *
 *   Arguments and results: as sparse_mla_fwd (same layouts, same validation).
 *   num_splits   0 = the library's split count (at least 2); otherwise 2..64.
 *   Limit        num_splits * T * H <= 8192 partial rows, else
 *                SMLA_ERR_SCRATCH_LIMIT before any CUDA call.  This suits
 *                decode-sized calls (a few tokens); larger calls belong on
 *                sparse_mla_fwd.
 *   First call   on each device (and again after that device's context has
 *                been reset) looks up the array's device address.  With CUDA's
 *                lazy module loading that lookup is what loads the library's
 *                device code and maps the array, an allocation made by the
 *                driver: make the first call outside any window in which no
 *                allocation may happen.
 *   Sharing      every call uses the same array: calls whose kernels overlap
 *                on the GPU (other streams, other host threads) race and give
 *                wrong results.  Serialise them on one stream.  No state
 *                carries over between calls: every partial row a call reads,
 *                it wrote first.
 */
smla_status_t sparse_mla_fwd_static_scratch(const void* q, const void* kv,
                                            const void* topk_indices, int32_t index_dtype,
                                            const float* attn_sink, float scale, void* out,
                                            float* lse, int64_t T, int32_t H, int64_t num_kv,
                                            int32_t topk, void* stream, int32_t num_splits);

/*
 * sparse_mla_fwd_host -- the forward on HOST buffers: copies the inputs in,
 * runs sparse_mla_fwd and copies O and lse out, overlapping the copies with
 * the computation.
 *
 * The pages have no counterpart to this entry point; it is the call for a
 * caller whose tensors live in host memory (the end-to-end path).  Tokens are
 * independent, so the call splits them into chunks and pipelines them on two
 * copy streams of its own: while chunk c is computed, chunk c+1's q and index
 * rows are copied in and chunk c-1's O and lse copied out.  kv (and the sink)
 * go in first, whole: any token may read any kv row.  Every chunk runs with
 * the kernel and split count sparse_mla_fwd would pick for the whole call, so
 * the results are bit-identical to sparse_mla_fwd's on the same inputs.
 *
 *   q_host, kv_host, topk_indices_host, attn_sink_host (or NULL), out_host,
 *   lse_host     HOST pointers, the layouts of sparse_mla_fwd.  For the copies
 *                to overlap they must be page-locked (cudaHostAlloc or
 *                cudaHostRegister); pageable memory works but serialises.
 *   workspace    DEVICE memory of at least sparse_mla_fwd_host_workspace()
 *                bytes, 256-byte aligned, owned by the caller and not touched
 *                by other work until `stream` has passed this call; the call
 *                allocates nothing.
 *   stream       the call is ordered on it: its copies start after the
 *                stream's earlier work, and the stream waits for the last
 *                copy out, so out_host / lse_host hold the results once
 *                `stream` has passed the call.
 *   Errors       as sparse_mla_fwd (same host checks on the host pointers),
 *                plus SMLA_ERR_WORKSPACE; all before any CUDA call.
 */
smla_status_t sparse_mla_fwd_host(const void* q_host, const void* kv_host,
                                  const void* topk_indices_host, int32_t index_dtype,
                                  const float* attn_sink_host, float scale, void* out_host,
                                  float* lse_host, int64_t T, int32_t H, int64_t num_kv,
                                  int32_t topk, void* workspace, uint64_t workspace_bytes,
                                  void* stream);

/*
 * sparse_mla_fwd_host_workspace -- device workspace bytes sparse_mla_fwd_host
 * needs for these sizes (host only, no CUDA call): room for kv, q, the index
 * rows, the sink, O and lse, each 256-byte aligned.  has_sink: 0 or 1.
 */
smla_status_t sparse_mla_fwd_host_workspace(int64_t T, int32_t H, int32_t topk, int64_t num_kv,
                                            int32_t index_dtype, int32_t has_sink,
                                            uint64_t* bytes);

/*
 * sparse_mla_bwd -- the training backward ("Sparse MLA training backward",
 * aiter PR #4766, sections "Contract" and "Structure").
 *
 * For the forward above, with its output O and sink-inclusive lse saved, and
 * the output gradient dO, over the valid slots of each token and head:
 *   P_j = exp(scale <q, kv[r_j]> - lse)        (lse from the forward)
 *   delta = <O, dO>,  dS_j = P_j (<dO, kv[r_j]> - delta)
 *   dq         = scale sum_j dS_j kv[r_j]
 *   dkv[r_j]  += scale dS_j q + P_j dO          (K == V: both terms on the row;
 *                                               summed over heads and slots)
 *   dsink[h]   = -sum_t exp(sink[h] - lse[t,h]) delta[t,h]
 *
 *   q, kv, topk_indices, index_dtype, attn_sink, scale, T, H, num_kv: as
 *                sparse_mla_fwd (same layouts and checks).
 *   out          [T, H, 512] bf16: the forward's output O.
 *   lse          [T, H] fp32: the forward's lse (sink-inclusive).
 *   dout         [T, H, 512] bf16: dO, 16-byte aligned.
 *   dq           [T, H, 512] fp32, 16-byte aligned (written whole).
 *   dkv          [num_kv, 512] fp32, 16-byte aligned (written whole: rows no
 *                valid slot names get 0).
 *   dsink        [H] fp32 or NULL (not computed); 0 when attn_sink is NULL.
 *   topk         0..2048; T * topk < 2^31.
 *   workspace    DEVICE memory of at least sparse_mla_bwd_workspace() bytes,
 *                256-byte aligned, owned by the caller and not touched by
 *                other work until `stream` has passed the call; the call
 *                allocates nothing.
 *   Errors       as sparse_mla_fwd, plus SMLA_ERR_WORKSPACE; all before any
 *                CUDA call.  Outputs and the workspace may not overlap inputs
 *                or each other.
 * Numerics: the contractions run in bf16 with fp32 accumulation; P and
 * scale * dS are rounded to bf16 before the two contractions over them (the
 * dq and the per-slot dkv terms).  The summation order of a kv row's terms
 * follows an atomic fill, so dkv can differ between calls in its last bits.
 */
smla_status_t sparse_mla_bwd(const void* q, const void* kv, const void* topk_indices,
                             int32_t index_dtype, const float* attn_sink, float scale,
                             const void* out, const float* lse, const void* dout, float* dq,
                             float* dkv, float* dsink, int64_t T, int32_t H, int64_t num_kv,
                             int32_t topk, void* workspace, uint64_t workspace_bytes,
                             void* stream);

/*
 * sparse_mla_bwd_workspace -- device workspace bytes sparse_mla_bwd needs for
 * these sizes (host only, no CUDA call): per-row delta, P and scale * dS per
 * valid slot and head (bf16), the compacted rows, each slot's dkv term
 * (fp32, T * topk * 2 KB) and the inverted index.
 */
smla_status_t sparse_mla_bwd_workspace(int64_t T, int32_t H, int32_t topk, int64_t num_kv,
                                       uint64_t* bytes);

/*
 * sparse_mla_plan -- what sparse_mla_fwd_ex would launch, without launching.
 * Launches nothing and touches no memory; its one CUDA query is the current
 * device's SM count (looked up once per device), which the split count
 * depends on (152 SMs are assumed when no device can be queried).  Writes the
 * kernel family (0 = small-head kernel, 1 = tcgen05 H=128 kernel), the split
 * count and the number of kernel launches per call.  num_splits as in
 * sparse_mla_fwd_ex.
 */
smla_status_t sparse_mla_plan(int64_t T, int32_t H, int32_t topk, int32_t num_splits,
                              int32_t* kernel_family, int32_t* splits_out,
                              int32_t* launches_out);

/*
 * sparse_mla_launch_config -- the launch geometry sparse_mla_fwd_ex would use on
 * the current device for these sizes (queries the device's occupancy, so it
 * makes CUDA runtime calls but launches nothing).  Writes the CTAs of the
 * main kernel's grid, threads per CTA, CTAs per cluster and dynamic shared
 * memory bytes per CTA.  Any output pointer may be NULL.
 */
smla_status_t sparse_mla_launch_config(int64_t T, int32_t H, int32_t topk, int64_t num_kv,
                                       int32_t num_splits, int32_t* grid_ctas,
                                       int32_t* cta_threads, int32_t* cluster_size,
                                       int32_t* smem_bytes);

/*
 * sparse_mla_device_status -- synchronises `stream`, then reads and clears
 * the library's device error word on the current device.  Returns
 * SMLA_ERR_DEVICE_TIMEOUT if a kernel gave up a bounded wait since the last
 * call (its outputs are then unspecified), SMLA_OK otherwise.
 */
smla_status_t sparse_mla_device_status(void* stream);

/*
 * sparse_mla_selftest_wait_timeout -- exercise the failure-detection path.
 * Queues on `stream` a one-thread kernel whose bounded mbarrier wait can never
 * be satisfied: after ~1 ms it records the expiry in the library's device
 * error word and returns normally (no fault, no trap; the context stays
 * usable).  The next sparse_mla_device_status on that device then returns
 * SMLA_ERR_DEVICE_TIMEOUT and clears the word.  For tests and health checks.
 */
smla_status_t sparse_mla_selftest_wait_timeout(void* stream);

/* Static description of a status code (never NULL). */
const char* sparse_mla_strerror(int32_t status);

/* Text of the last CUDA error seen by this thread inside the library ("" if none). */
const char* sparse_mla_last_cuda_error(void);

/* ABI version: bumped on any incompatible change of the declarations above. */
int32_t sparse_mla_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_MLA_H */
