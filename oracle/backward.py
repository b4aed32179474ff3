"""fp64 CPU oracle for the training backward of the sparse MLA attention.

TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this module.  It shares no code with the CUDA
path: no kernels, headers, helpers or constants.

What it computes: the exact gradient, in float64, of the forward of
``oracle.oracle`` with respect to q, kv and the sink, given the output
gradient dO ("Sparse MLA training backward", aiter PR #4766, sections
"Contract" and "Structure").  For every token ``t`` and head ``h``, over the
valid slots ``j`` (row ``r_j = idx[t, j]`` in ``[0, num_kv)``)::

    s_j     = scale * <q, kv[r_j]>
    m       = max(max_j s_j, sink)
    den     = sum_j exp(s_j - m) + exp(sink - m)
    P_j     = exp(s_j - m) / den            P_sink = exp(sink - m) / den
    O       = sum_j P_j kv[r_j]             (the sink's value is zero)
    dP_j    = <dO, kv[r_j]>                 (K == V: the same row)
    delta   = <dO, O>  = sum_j P_j dP_j     (the "delta" kernel: rowsum(O * dO))
    dS_j    = P_j (dP_j - delta)
    dq      = scale * sum_j dS_j kv[r_j]
    dkv[r_j] += scale * dS_j q + P_j dO     (K and V are one tensor: both terms
                                             land on the row; a duplicated row
                                             collects once per slot)
    dsink  += -P_sink * delta               (summed over tokens, per head)

The page splits the work into the same quantities: delta as rowsum(O * dO);
dQ from S and dP of one gathered tile; a per-(token, slot) "interm" row
``scale * dS^T q + P^T dO`` contracted over the heads; an inverted index so
that each kv row gathers its contributors; and the sink gradient.  This
oracle follows that order per token with dense numpy products.

Readings where the page is silent: the backward takes dO only (lse and O are
outputs the forward saved, not inputs with gradients of their own); a row
with no valid slot has O = 0, so delta = 0 and it contributes nothing; sink =
-inf (or no sink) gives a zero sink gradient.
"""
from __future__ import annotations

import numpy as np

from .oracle import bf16_to_f64, valid_slots


def token_backward(q_t, kv, idx_t, num_kv: int, sink, scale: float, do_t):
    """One token.

    ``q_t`` and ``do_t`` float64 ``[H, D]``; ``kv`` ``[num_kv, D]`` float64 or
    bf16 bits (uint16); ``sink`` float64 ``[H]`` or None.  Returns
    ``(dq [H, D], rows [v], dk [v, D], dsink [H])``: the rows this token's
    valid slots name (duplicates kept) and each slot's contribution to
    ``dkv[row]``.
    """
    H, D = q_t.shape
    rows = np.asarray(idx_t).astype(np.int64)[valid_slots(idx_t, num_kv)]
    k = kv[rows]
    if k.dtype == np.uint16:
        k = bf16_to_f64(k)
    dq = np.zeros((H, D))
    dsink = np.zeros(H)
    dk = np.zeros((rows.size, D))
    s = scale * (q_t @ k.T)                                    # [H, v]
    m = s.max(axis=1) if rows.size else np.full(H, -np.inf)
    if sink is not None:
        m = np.maximum(m, sink)
    live = np.isfinite(m)
    if not np.any(live) or rows.size == 0:
        return dq, rows, dk, dsink                             # O = 0: nothing flows back
    ml = m[live]
    e = np.exp(s[live] - ml[:, None])
    den = e.sum(axis=1)
    if sink is not None:
        den = den + np.exp(sink[live] - ml)
    P = e / den[:, None]                                       # [h_live, v]
    O = P @ k                                                  # [h_live, D]
    dP = do_t[live] @ k.T                                      # [h_live, v]
    delta = (do_t[live] * O).sum(axis=1)                       # rowsum(O * dO)
    dS = P * (dP - delta[:, None])
    dq[live] = scale * (dS @ k)
    dk = scale * (dS.T @ q_t[live]) + P.T @ do_t[live]         # [v, D], summed over heads
    if sink is not None:
        p_sink = np.exp(sink[live] - ml) / den
        dsink[live] = -p_sink * delta
    return dq, rows, dk, dsink


def accumulate_rows(dkv, rows, dk):
    """dkv[rows[i]] += dk[i] for every i; a row named several times collects each."""
    np.add.at(dkv, rows, dk)


def sparse_mla_bwd(q_bits, kv_bits, idx, sink, scale: float, do_bits, tokens=None):
    """The whole backward (or the contributions of a subset of tokens).

    q_bits, do_bits: uint16 bf16 bits ``[T, H, D]``; kv_bits: uint16 bf16 bits
    ``[num_kv, D]``; idx ``[T, TOPK]`` int32/int64; sink float32 ``[H]`` or
    None.  Returns (dq float64 ``[n, H, D]`` for the tokens, dkv float64
    ``[num_kv, D]`` from those tokens, dsink float64 ``[H]`` from those tokens).
    """
    num_kv = kv_bits.shape[0]
    kv = np.asarray(kv_bits, dtype=np.uint16)
    sk = None if sink is None else np.asarray(sink, dtype=np.float32).astype(np.float64)
    T, H, D = q_bits.shape
    toks = range(T) if tokens is None else list(tokens)
    dq = np.zeros((len(toks), H, D))
    dkv = np.zeros((num_kv, D))
    dsink = np.zeros(H)
    for i, t in enumerate(toks):
        g, rows, dk, ds = token_backward(bf16_to_f64(q_bits[t]), kv, idx[t], num_kv, sk, scale,
                                         bf16_to_f64(do_bits[t]))
        dq[i] = g
        accumulate_rows(dkv, rows, dk)
        dsink += ds
    return dq, dkv, dsink
