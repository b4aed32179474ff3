"""fp64 CPU oracle for the DeepSeek-V4 sparse MLA prefill forward.

TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this module.  It shares no code with the CUDA
path: no kernels, headers, helpers or constants.

What it computes (the plain definition of the op, in float64):

For every token ``t`` and head ``h``, over the slots ``j`` of the token's index
list whose value ``r = idx[t, j]`` lies in ``[0, num_kv)``::

    s_j   = scale * <q[t, h, :], kv[r, :]>          (K == V == kv, one 512-wide row)
    m     = max(max_j s_j, sink[h])                   (sink folded into the max)
    den   = sum_j exp(s_j - m) + exp(sink[h] - m)     (sink in the denominator only)
    O     = sum_j exp(s_j - m) * kv[r, :] / den
    lse   = m + log(den)                              (natural log, sink-inclusive)

Passages followed:

* "Sparse MLA training backward" (aiter PR #4766), section "Contract": shared-KV
  GQA with K == V == kv as one dense 512-wide tensor, scale 1/sqrt(512), the
  sink folded into the softmax denominator only, ``-1`` slots masked out, kv
  ``[num_kv, 512]`` with ``num_kv >= T``.
* same page, the paragraph under the ``mla_gluon`` call: the forward's lse is
  sink-inclusive, the sink folded into the running max and sum before
  ``lse = max + log(sum)``.
* same page, review thread on the fp32 test reference: fold the sink into the
  max, so ``exp(sink - m)`` cannot overflow.
* same page, review reply on the reference's all-invalid row: such a row gives
  O = 0 and lse = -inf (no sink); with a finite sink the formula gives O = 0
  and lse = sink.
* "Tuned sparse MLA prefill for DSv4.1-Flash TP4; fix attn_sink in Triton
  fallback" (aiter PR #6002), description: invalid KV rows are never loaded,
  int64 indices are kept at full width (no wrap of slots >= 2**31); a commit
  note on that page: slots outside ``[0, len(kv))`` are masked, including
  ``num_kv`` itself and values up to the int32 maximum.

Readings where the pages are silent: a duplicated index counts once per slot
(the sum runs over slots); ``sink = -inf`` is the same as no sink; NaN/Inf in a
row that only invalid slots name never reaches the output, because such rows
are never read.  O is returned in float64 and is not rounded to bf16.

Steps that use a library primitive: the row gather (numpy fancy indexing) and
two matrix products per token (numpy ``@``), each a plain sum over the
definition's index, with no blocking or reordering beyond that.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float64 exactly."""
    b = np.ascontiguousarray(bits).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def valid_slots(idx: np.ndarray, num_kv: int) -> np.ndarray:
    """Which slots are read: ``0 <= idx < num_kv`` on the full index width.

    PR #6002 description ("int64 indices", "Invalid KV rows") and its commit
    note on ``-1`` / ``num_kv`` / int32-maximum slots.
    """
    i = np.asarray(idx).astype(np.int64)  # int32 widens exactly; int64 stays full width
    return (i >= 0) & (i < int(num_kv))


def token_forward(q_t: np.ndarray, kv: np.ndarray, idx_t: np.ndarray, num_kv: int,
                  sink, scale: float, d_v=None):
    """One token: returns (O [H, d_v] float64, lse [H] float64).

    ``q_t`` is float64 ``[H, D]``, ``kv`` ``[num_kv, D]`` either float64 or
    bf16 bit patterns (uint16, widened exactly after the gather), ``sink`` a
    float64 ``[H]`` array or None.  Scores use all D columns; the values are
    the first ``d_v`` columns of the same rows (default all D).  d_v < D is
    the MLA layout with a positional part: each row is ``[no-pe | pe]`` and
    only the no-pe part is a value ("Add DSv4 sparse MLA prefill Triton and
    unified with MLA Gluon kernel on GFX950", the ``has_pe`` flag with a
    64-wide positional part).
    """
    H, D = q_t.shape
    dv = D if d_v is None else int(d_v)
    rows = np.asarray(idx_t).astype(np.int64)[valid_slots(idx_t, num_kv)]
    k = kv[rows]                                   # [v, D]; a duplicated row appears twice
    if k.dtype == np.uint16:
        k = bf16_to_f64(k)
    s = scale * (q_t @ k.T)                        # [H, v]
    m = s.max(axis=1) if rows.size else np.full(H, -np.inf)
    if sink is not None:
        m = np.maximum(m, sink)                    # sink folded into the max
    out = np.zeros((H, dv))
    lse = np.full(H, -np.inf)
    live = np.isfinite(m)                          # m = -inf: nothing valid and no finite sink
    if np.any(live):
        ml = m[live]
        e = np.exp(s[live] - ml[:, None])          # [h_live, v]
        den = e.sum(axis=1)
        if sink is not None:
            den = den + np.exp(sink[live] - ml)    # sink in the denominator only
        out[live] = (e @ k[:, :dv]) / den[:, None]
        lse[live] = ml + np.log(den)
    return out, lse


def sparse_mla_fwd(q_bits: np.ndarray, kv_bits: np.ndarray, idx: np.ndarray, sink,
                   scale: float, tokens=None, d_v=None):
    """The whole op (or a subset of tokens) in float64.

    q_bits: uint16 bf16 bits ``[T, H, D]``; kv_bits: uint16 bf16 bits
    ``[num_kv, D]``; idx: int32/int64 ``[T, TOPK]``; sink: float32 ``[H]`` or
    None; tokens: optional iterable of token ids (default all); d_v: value
    width (the first d_v columns of each kv row; default D).
    Returns (O float64 ``[n, H, d_v]``, lse float64 ``[n, H]``) for those tokens.
    """
    num_kv = kv_bits.shape[0]
    kv = np.asarray(kv_bits, dtype=np.uint16)      # rows are widened once gathered
    sk = None if sink is None else np.asarray(sink, dtype=np.float32).astype(np.float64)
    T, H, D = q_bits.shape
    dv = D if d_v is None else int(d_v)
    toks = range(T) if tokens is None else list(tokens)
    n = len(toks)
    O = np.zeros((n, H, dv))
    L = np.full((n, H), -np.inf)
    for i, t in enumerate(toks):
        O[i], L[i] = token_forward(bf16_to_f64(q_bits[t]), kv, idx[t], num_kv, sk, scale,
                                   d_v=dv)
    return O, L
