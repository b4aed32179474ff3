"""Pins for the oracle's other head dims and its positional-part layout (CPU only).

The forward with head dim D in {128, 576} (K == V, D-wide rows) and the MLA
layout with a 64-wide positional part (rows ``[512 no-pe | 64 pe]``: scores
over all 576 columns, values the first 512; "Add DSv4 sparse MLA prefill
Triton and unified with MLA Gluon kernel on GFX950", the ``has_pe`` flag and
its 64-wide positional part; "Tuned sparse MLA prefill for DSv4.1-Flash TP4",
tests at head dims 128 and 576) are pinned by:

* brute force: torch ``scaled_dot_product_attention`` in float64 over the whole
  pool, values being the first d_v columns of the keys, multiplicities as
  ``log(count)`` offsets and the sink as one extra key with a zero value;
* a closed form: one valid slot gives O = v[:d_v] e^s / (e^s + e^sink);
* a reduction: with the positional part of q set to zero the result equals the
  512-wide op on the no-pe columns alone.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from sparse_mla_attention_token_gb300 import synth


def _f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _inputs(D, seed, T=20, H=4, N=48, K=24):
    rng = np.random.default_rng(seed)
    q = synth.bf16_bits(rng.standard_normal((T, H, D)).astype(np.float32))
    kv = synth.bf16_bits(rng.standard_normal((N, D)).astype(np.float32))
    idx = rng.integers(-3, N + 3, size=(T, K)).astype(np.int64)   # some invalid, some repeats
    sink = rng.standard_normal(H).astype(np.float32)
    return q, kv, idx, sink


def _dense(q_bits, kv_bits, idx, sink, scale, d_v):
    T, H, D = q_bits.shape
    N = kv_bits.shape[0]
    count = np.zeros((T, N))
    for t in range(T):
        for r in idx[t].tolist():
            if r in range(N):
                count[t, r] += 1
    q = torch.from_numpy(_f64(q_bits)).permute(1, 0, 2)
    k = torch.cat([torch.from_numpy(_f64(kv_bits)), torch.zeros(1, D, dtype=torch.float64)], 0)
    v = k[:, :d_v].clone()
    with np.errstate(divide="ignore"):
        logc = torch.from_numpy(np.log(count))
    mask = torch.empty(H, T, N + 1, dtype=torch.float64)
    mask[:, :, :N] = logc[None]
    mask[:, :, N] = torch.from_numpy(sink.astype(np.float64))[:, None]
    o = torch.nn.functional.scaled_dot_product_attention(
        q, k[None].expand(H, -1, -1), v[None].expand(H, -1, -1), attn_mask=mask, scale=scale)
    lse = torch.logsumexp(scale * (q @ k.T[None]) + mask, dim=-1)
    return o.permute(1, 0, 2).numpy(), lse.permute(1, 0).numpy()


@pytest.mark.parametrize("D,d_v", [(128, 128), (576, 576), (576, 512)])
def test_dims_match_dense_sdpa(D, d_v):
    q, kv, idx, sink = _inputs(D, seed=D + d_v)
    scale = 1 / math.sqrt(D)
    O, L = orc.sparse_mla_fwd(q, kv, idx, sink, scale, d_v=d_v)
    Od, Ld = _dense(q, kv, idx, sink, scale, d_v)
    assert O.shape == (q.shape[0], q.shape[1], d_v)
    np.testing.assert_allclose(O, Od, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(L, Ld, rtol=1e-12, atol=1e-12)


def test_pe_layout_single_slot_closed_form():
    q, kv, _, sink = _inputs(576, seed=3, T=1, H=2)
    idx = np.array([[-1, 9, 48, -7]], dtype=np.int64)
    scale = 1 / math.sqrt(576)
    O, L = orc.sparse_mla_fwd(q, kv, idx, sink, scale, d_v=512)
    for h in range(2):
        s = scale * math.fsum(_f64(q[0, h]) * _f64(kv[9]))
        w = math.exp(s) / (math.exp(s) + math.exp(float(sink[h])))
        np.testing.assert_allclose(O[0, h], w * _f64(kv[9])[:512], rtol=1e-12, atol=1e-15)
        assert abs(L[0, h] - math.log(math.exp(s) + math.exp(float(sink[h])))) < 1e-12


def test_pe_layout_without_positional_query_is_the_512_op():
    q, kv, idx, sink = _inputs(576, seed=5)
    q0 = q.copy()
    q0[:, :, 512:] = 0                      # q_pe = 0: the pe columns add nothing to a score
    scale = 1 / math.sqrt(512)
    O, L = orc.sparse_mla_fwd(q0, kv, idx, sink, scale, d_v=512)
    O5, L5 = orc.sparse_mla_fwd(np.ascontiguousarray(q[:, :, :512]),
                                np.ascontiguousarray(kv[:, :512]), idx, sink, scale)
    np.testing.assert_allclose(O, O5, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(L, L5, rtol=1e-13, atol=1e-13)
