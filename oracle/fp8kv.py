"""fp64 CPU oracle for the forward on an fp8 KV cache.

TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this module.  It shares no code with the CUDA
path.

The pages name an fp8 KV cache ("Add DSv4 sparse MLA prefill Triton and
unified with MLA Gluon kernel on GFX950": the fp8 paged decode cache is left
out of that change; "Tuned sparse MLA prefill for DSv4.1-Flash TP4": an fp8
pool must be rejected with a clear dtype error by the bf16 entry point) but do
not define its layout.  The reading taken here: each kv row is 512 OCP FP8
E4M3 (e4m3fn) bytes and 4 fp32 scales, one per 128-column block; the row's
value in column c is ``decode(byte[c]) * scale[c // 128]``.  The op is then the
bf16 op's definition (``oracle.oracle``) applied to those values, exactly.

e4m3fn: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is
subnormal (m / 8 * 2^-6); exponent 15 with mantissa 7 is NaN (no infinities).
"""
from __future__ import annotations

import numpy as np

from .oracle import token_forward

BLOCK = 128   # columns per scale


def e4m3_to_f64(b: np.ndarray) -> np.ndarray:
    """Decode e4m3fn bytes (uint8) to float64 exactly."""
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    s = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return s * val


def dequant_rows(kv8: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Rows ``[n, 512]`` of e4m3 bytes and ``[n, 4]`` fp32 scales -> float64 values."""
    v = e4m3_to_f64(kv8)
    sc = np.asarray(scales, dtype=np.float32).astype(np.float64)
    return v * np.repeat(sc, BLOCK, axis=1)


def sparse_mla_fwd_fp8kv(q_bits, kv8, kv_scale, idx, sink, scale: float, tokens=None):
    """The forward on the fp8 cache (or a subset of tokens), float64.

    q_bits: uint16 bf16 bits ``[T, H, 512]``; kv8: uint8 e4m3 ``[num_kv, 512]``;
    kv_scale: float32 ``[num_kv, 4]``; idx ``[T, TOPK]``; sink float32 ``[H]`` or
    None.  Returns (O ``[n, H, 512]``, lse ``[n, H]``).
    """
    from .oracle import bf16_to_f64
    num_kv = kv8.shape[0]
    T, H, D = q_bits.shape
    sk = None if sink is None else np.asarray(sink, dtype=np.float32).astype(np.float64)
    toks = range(T) if tokens is None else list(tokens)
    O = np.zeros((len(toks), H, D))
    L = np.full((len(toks), H), -np.inf)
    for i, t in enumerate(toks):
        it = np.asarray(idx[t]).astype(np.int64)
        ok = (it >= 0) & (it < num_kv)
        # only the rows this token names are decoded; the others are never read
        rows = np.unique(it[ok])
        kv = _SparseRows(rows, dequant_rows(kv8[rows], kv_scale[rows]), num_kv, D)
        O[i], L[i] = token_forward(bf16_to_f64(q_bits[t]), kv, idx[t], num_kv, sk, scale)
    return O, L


class _SparseRows:
    """The decoded rows of one token, indexable like a ``[num_kv, D]`` array by
    the row numbers the token names."""

    def __init__(self, rows, values, num_kv, D):
        self._pos = {int(r): k for k, r in enumerate(rows)}
        self._values = values
        self.shape = (num_kv, D)
        self.dtype = np.dtype(np.float64)

    def __getitem__(self, rows):
        rows = np.asarray(rows)
        if rows.size == 0:
            return np.zeros((0, self.shape[1]))
        return self._values[[self._pos[int(r)] for r in rows]]
