"""Pins for the fp64 oracle, against things other than itself (CPU only).

* brute force: dense attention over the whole kv pool in float64 with
  torch's ``scaled_dot_product_attention`` (a library routine), the slot
  multiplicities entering as ``log(count)`` logit offsets and the sink as one
  extra key whose logit is ``sink[h]`` and whose value is the zero vector;
  lse from ``torch.logsumexp`` over the same dense logits;
* closed forms evaluated with ``math`` (one slot, one slot repeated, q = 0,
  two slots, a sink far above every score);
* invariants: all-invalid rows, sink = -inf equals no sink, permuting a
  token's list, appending invalid slots, poisoning rows only invalid slots
  name, full-width int64 slots that would wrap onto valid rows.

Semantics pinned: "Sparse MLA training backward" (aiter PR #4766), sections
"Contract" and the review notes on the sink-inclusive lse and the all-invalid
row; "Tuned sparse MLA prefill for DSv4.1-Flash TP4; fix attn_sink in Triton
fallback" (aiter PR #6002), description items "attn_sink", "int64 indices",
"Invalid KV rows".
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from sparse_mla_attention_token_gb300 import synth

D = 512


def _f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _dense_reference(q_bits, kv_bits, idx, sink, scale):
    """Dense masked attention with multiplicities, via torch SDPA in float64."""
    T, H, _ = q_bits.shape
    N = kv_bits.shape[0]
    count = np.zeros((T, N))
    for t in range(T):                      # per-slot loop, independent of the oracle's mask
        for r in idx[t].tolist():
            if r in range(N):
                count[t, r] += 1
    q = torch.from_numpy(_f64(q_bits)).permute(1, 0, 2)          # [H, T, D]
    kv = torch.from_numpy(_f64(kv_bits))
    keys = torch.cat([kv, torch.zeros(1, D, dtype=torch.float64)], 0)   # sink key = 0
    vals = keys.clone()                                                  # sink value = 0
    with np.errstate(divide="ignore"):
        logc = torch.from_numpy(np.log(count))                         # -inf where count = 0
    mask = torch.empty(H, T, N + 1, dtype=torch.float64)
    mask[:, :, :N] = logc[None]
    if sink is None:
        mask[:, :, N] = -math.inf
    else:
        mask[:, :, N] = torch.from_numpy(sink.astype(np.float64))[:, None]
    K = keys[None].expand(H, -1, -1)
    V = vals[None].expand(H, -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(q, K, V, attn_mask=mask, scale=scale)
    logits = scale * (q @ K.transpose(1, 2)) + mask
    lse = torch.logsumexp(logits, dim=-1)
    return o.permute(1, 0, 2).numpy(), lse.permute(1, 0).numpy()


def _tiny(seed=0, sink=True, T=None, topk=None, window=None):
    cfg = synth.CONFIGS["tiny"].with_(seed=seed, sink=sink)
    if T is not None:
        cfg = cfg.with_(T=T)
    if topk is not None:
        cfg = cfg.with_(topk=topk, window=window)
    return cfg, synth.make_inputs(cfg)


@pytest.mark.parametrize("variant", ["plain", "shuffled", "dups", "oob", "nosink", "int64"])
def test_oracle_matches_dense_sdpa(variant):
    cfg, x = _tiny(seed=11, sink=(variant != "nosink"))
    idx = x["idx"]
    if variant == "shuffled":
        idx = synth.shuffle_rows(idx, 5)
    elif variant == "dups":
        idx = synth.inject_duplicates(idx, cfg.num_kv, 6, frac=0.2)
    elif variant == "oob":
        idx = synth.inject_out_of_range(idx, cfg.num_kv, 7, frac=0.3)
    elif variant == "int64":
        idx = synth.inject_out_of_range(idx.astype(np.int64), cfg.num_kv, 8, frac=0.3)
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], idx, x["sink"], x["scale"])
    Od, Ld = _dense_reference(x["q"], x["kv"], idx, x["sink"], x["scale"])
    live = np.isfinite(Ld)
    assert live.sum() > 0.9 * live.size
    np.testing.assert_allclose(O[live], Od[live], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(L[live], Ld[live], rtol=1e-12, atol=1e-12)
    # rows SDPA cannot score (nothing valid, no sink): O = 0 and lse = -inf
    assert np.all(O[~live] == 0) and np.all(L[~live] == -np.inf)


def _dot(a, b):
    return math.fsum(float(x) * float(y) for x, y in zip(a, b))


def _one_token(rows, sink_h=None, q_zero=False, seed=3, H=4):
    rng = np.random.default_rng(seed)
    kv_bits = synth.bf16_bits(rng.standard_normal((20, D)).astype(np.float32))
    q_bits = synth.bf16_bits(rng.standard_normal((1, H, D)).astype(np.float32))
    if q_zero:
        q_bits[:] = 0
    idx = np.array([rows], dtype=np.int32)
    sink = None if sink_h is None else np.full(H, sink_h, dtype=np.float32)
    return q_bits, kv_bits, idx, sink


@pytest.mark.parametrize("sink_h", [None, 0.75, -2.5])
def test_closed_form_single_slot(sink_h):
    r = 7
    q_bits, kv_bits, idx, sink = _one_token([-1, r, 20, -1, 99], sink_h)
    scale = 1 / math.sqrt(D)
    O, L = orc.sparse_mla_fwd(q_bits, kv_bits, idx, sink, scale)
    kvr = _f64(kv_bits[r])
    for h in range(q_bits.shape[1]):
        s = scale * _dot(_f64(q_bits[0, h]), kvr)
        if sink_h is None:
            w, lse = 1.0, s
        else:
            sk = float(np.float32(sink_h))
            w = math.exp(s) / (math.exp(s) + math.exp(sk))
            lse = math.log(math.exp(s) + math.exp(sk))
        np.testing.assert_allclose(O[0, h], w * kvr, rtol=1e-12, atol=1e-14)
        assert abs(L[0, h] - lse) < 1e-12


@pytest.mark.parametrize("k", [2, 3, 5])
def test_closed_form_repeated_slot(k):
    r = 4
    q_bits, kv_bits, idx, sink = _one_token([r] * k + [-1, 20], 0.3)
    scale = 1 / math.sqrt(D)
    O, L = orc.sparse_mla_fwd(q_bits, kv_bits, idx, sink, scale)
    kvr = _f64(kv_bits[r])
    sk = float(np.float32(0.3))
    for h in range(q_bits.shape[1]):
        s = scale * _dot(_f64(q_bits[0, h]), kvr)
        den = k * math.exp(s) + math.exp(sk)
        np.testing.assert_allclose(O[0, h], kvr * k * math.exp(s) / den, rtol=1e-12, atol=1e-14)
        assert abs(L[0, h] - math.log(den)) < 1e-12


def test_closed_form_q_zero_is_weighted_mean():
    rows = [1, 2, 2, 9, -1, 19]
    q_bits, kv_bits, idx, sink = _one_token(rows, 1.25, q_zero=True)
    O, L = orc.sparse_mla_fwd(q_bits, kv_bits, idx, sink, 1 / math.sqrt(D))
    n = 5
    sk = float(np.float32(1.25))
    tot = sum(_f64(kv_bits[r]) for r in rows if r >= 0)
    for h in range(q_bits.shape[1]):
        np.testing.assert_allclose(O[0, h], tot / (n + math.exp(sk)), rtol=1e-12, atol=1e-14)
        assert abs(L[0, h] - math.log(n + math.exp(sk))) < 1e-12


def test_closed_form_two_slots_and_sign():
    q_bits, kv_bits, idx, sink = _one_token([3, 12], -0.5, seed=9)
    scale = -0.2  # a negative scale is allowed (no positivity check on the pages)
    O, L = orc.sparse_mla_fwd(q_bits, kv_bits, idx, sink, scale)
    k3, k12 = _f64(kv_bits[3]), _f64(kv_bits[12])
    sk = float(np.float32(-0.5))
    for h in range(q_bits.shape[1]):
        qh = _f64(q_bits[0, h])
        s1, s2 = scale * _dot(qh, k3), scale * _dot(qh, k12)
        den = math.exp(s1) + math.exp(s2) + math.exp(sk)
        np.testing.assert_allclose(O[0, h], (math.exp(s1) * k3 + math.exp(s2) * k12) / den,
                                   rtol=1e-11, atol=1e-14)
        assert abs(L[0, h] - math.log(den)) < 1e-12


def test_sink_far_above_scores_does_not_overflow():
    # exp(800) overflows float64: the sink must be folded into the max.
    q_bits, kv_bits, idx, sink = _one_token([1, 2, 3], 800.0)
    scale = 1 / math.sqrt(D)
    O, L = orc.sparse_mla_fwd(q_bits, kv_bits, idx, sink, scale)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
    for h in range(q_bits.shape[1]):
        ss = [scale * _dot(_f64(q_bits[0, h]), _f64(kv_bits[r])) for r in (1, 2, 3)]
        lse = 800.0 + math.log1p(sum(math.exp(s - 800.0) for s in ss))
        assert abs(L[0, h] - lse) < 1e-9
        # every weight exp(s - 800) underflows: O is 0 to double precision
        assert np.all(np.abs(O[0, h]) < 1e-300)


def test_large_scores_stable():
    # scores near 700: exp(s) alone would overflow if the max were not subtracted
    q_bits, kv_bits, idx, sink = _one_token([5, 6], None, seed=2)
    O, L = orc.sparse_mla_fwd(q_bits, kv_bits, idx, sink, 300.0)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))


def test_all_invalid_rows():
    cfg, x = _tiny(seed=1)
    idx = np.full_like(x["idx"], -1)
    idx[:, 3] = cfg.num_kv                       # first row past the pool: invalid too
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], idx, None, x["scale"])
    assert np.all(O == 0) and np.all(L == -np.inf)
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], idx, x["sink"], x["scale"])
    assert np.all(O == 0)
    np.testing.assert_array_equal(L, np.broadcast_to(x["sink"].astype(np.float64), L.shape))
    neg = np.full_like(x["sink"], -np.inf)
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], idx, neg, x["scale"])
    assert np.all(O == 0) and np.all(L == -np.inf) and not np.any(np.isnan(O))


def test_sink_minus_inf_equals_no_sink():
    cfg, x = _tiny(seed=2)
    neg = np.full_like(x["sink"], -np.inf)
    a = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], neg, x["scale"])
    b = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], None, x["scale"])
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_sink_changes_denominator_only():
    # with a sink, O scales by den_nosink/den_sink and the direction is unchanged
    cfg, x = _tiny(seed=4)
    O1, L1 = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], None, x["scale"])
    O2, L2 = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"])
    ratio = np.exp(L1 - L2)                     # den_nosink / den_sink
    np.testing.assert_allclose(O2, O1 * ratio[..., None], rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(np.exp(L2), np.exp(L1) + np.exp(x["sink"].astype(np.float64)),
                               rtol=1e-10)


def test_permutation_invariance():
    cfg, x = _tiny(seed=5)
    a = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"])
    b = orc.sparse_mla_fwd(x["q"], x["kv"], synth.shuffle_rows(x["idx"], 1), x["sink"], x["scale"])
    np.testing.assert_allclose(a[0], b[0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(a[1], b[1], rtol=1e-13, atol=1e-13)


def test_duplicate_counts_twice():
    # duplicating slot j is the same as adding log 2 to that slot's logit
    q_bits, kv_bits, idx, sink = _one_token([2, 5, 5, -1], 0.1)
    scale = 1 / math.sqrt(D)
    O, L = orc.sparse_mla_fwd(q_bits, kv_bits, idx, sink, scale)
    sk = float(np.float32(0.1))
    for h in range(q_bits.shape[1]):
        qh = _f64(q_bits[0, h])
        s2, s5 = scale * _dot(qh, _f64(kv_bits[2])), scale * _dot(qh, _f64(kv_bits[5]))
        den = math.exp(s2) + math.exp(s5 + math.log(2)) + math.exp(sk)
        exp_o = (math.exp(s2) * _f64(kv_bits[2]) + 2 * math.exp(s5) * _f64(kv_bits[5])) / den
        np.testing.assert_allclose(O[0, h], exp_o, rtol=1e-11, atol=1e-14)


@pytest.mark.parametrize("dtype", [np.int32, np.int64])
def test_appending_invalid_slots_changes_nothing(dtype):
    cfg, x = _tiny(seed=6)
    idx = x["idx"].astype(dtype)
    bad = [-1, cfg.num_kv, cfg.num_kv + 1, np.iinfo(np.int32).max, -(2 ** 31)]
    if dtype == np.int64:
        bad += [2 ** 31, 2 ** 32, 2 ** 32 + 5, 2 ** 40 + 1, -(2 ** 33)]
    extra = np.tile(np.array(bad, dtype=dtype), (idx.shape[0], 1))
    a = orc.sparse_mla_fwd(x["q"], x["kv"], idx, x["sink"], x["scale"])
    b = orc.sparse_mla_fwd(x["q"], x["kv"], np.concatenate([extra, idx, extra], 1),
                           x["sink"], x["scale"])
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_int64_slots_do_not_wrap():
    # 2**32 + r narrows to r in int32; at full width it is out of range
    cfg, x = _tiny(seed=7)
    idx = x["idx"].astype(np.int64)
    wrapped = idx.copy()
    sel = idx >= 0
    wrapped[sel] = idx[sel] + (1 << 32)
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], wrapped, None, x["scale"])
    assert np.all(O == 0) and np.all(L == -np.inf)
    assert orc.valid_slots(np.array([2 ** 31, 2 ** 32 + 1, -1, 0, 79, 80]), 80).tolist() == \
        [False, False, False, True, True, False]


def test_poisoned_unreferenced_rows_do_not_reach_output():
    cfg, x = _tiny(seed=8)
    idx = x["idx"].copy()
    idx[idx == 0] = -1                           # nothing valid names row 0 any more
    used = np.unique(idx[(idx >= 0) & (idx < cfg.num_kv)])
    kv = x["kv"].copy()
    poison = np.setdiff1d(np.arange(cfg.num_kv), used)
    assert 0 in poison
    kv[poison] = 0x7FC0                          # bf16 NaN
    kv[0, ::2] = 0x7F80                          # +inf
    a = orc.sparse_mla_fwd(x["q"], x["kv"], idx, x["sink"], x["scale"])
    b = orc.sparse_mla_fwd(x["q"], kv, idx, x["sink"], x["scale"])
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_token_subset_matches_full():
    cfg, x = _tiny(seed=9)
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"])
    toks = [0, 17, 63, 5]
    Os, Ls = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"], tokens=toks)
    np.testing.assert_array_equal(Os, O[toks])
    np.testing.assert_array_equal(Ls, L[toks])
