"""Pins for the fp64 backward oracle, against things other than itself (CPU only).

* torch autograd (float64) through dense masked attention over the whole kv
  pool: slot multiplicities as ``log(count)`` logit offsets, the sink as one
  extra key whose logit is ``sink[h]`` and whose value is zero, K and V the
  same leaf tensor so that autograd sums both uses of a row;
* central finite differences of the forward oracle's ``sum(dO * O)`` along
  random directions in q, kv and the sink;
* closed forms (one valid slot with a sink, evaluated with ``math``);
* invariants: rows no valid slot names get exactly zero gradient, sink = -inf
  equals no sink, permuting a token's list, an all-invalid token;
* planted mistakes in the backward must each fail one of the pins above.

Semantics pinned: "Sparse MLA training backward" (aiter PR #4766), sections
"Contract" (K == V, the sink in the denominator only, scale 1/sqrt(512)) and
"Structure" (delta = rowsum(O * dO), dS from S and dP, the dKV row gathers all
its contributors, the sink gradient).
"""
import math

import numpy as np
import pytest
import torch

from oracle import backward as bwd
from oracle import oracle as orc
from sparse_mla_attention_token_gb300 import synth

D = 512


def _f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _inputs(seed=0, sink=True, T=24, H=4, topk=40, window=16, pool=16):
    cfg = synth.CONFIGS["tiny"].with_(seed=seed, sink=sink, T=T, H=H, topk=topk, window=window,
                                      pool=pool)
    x = synth.make_inputs(cfg)
    rng = np.random.default_rng(seed + 1000)
    x["do"] = synth.bf16_bits(rng.standard_normal((T, H, D)).astype(np.float32))
    return cfg, x


def _autograd_reference(q_bits, kv_bits, idx, sink, scale, do_bits):
    """dq, dkv, dsink by torch autograd through dense masked attention (float64)."""
    T, H, _ = q_bits.shape
    N = kv_bits.shape[0]
    count = np.zeros((T, N))
    for t in range(T):                      # per-slot loop, independent of the oracle's mask
        for r in idx[t].tolist():
            if r in range(N):
                count[t, r] += 1
    q = torch.tensor(_f64(q_bits), requires_grad=True)                 # [T, H, D]
    kv = torch.tensor(_f64(kv_bits), requires_grad=True)               # [N, D]
    sk = torch.tensor(np.zeros(H) if sink is None else sink.astype(np.float64),
                      requires_grad=True)
    with np.errstate(divide="ignore"):
        logc = torch.from_numpy(np.log(count))                         # -inf where count = 0
    logits = scale * torch.einsum("thd,nd->thn", q, kv) + logc[:, None, :]
    sink_col = sk[None, :, None].expand(T, H, 1)
    if sink is None:
        sink_col = torch.full((T, H, 1), -math.inf, dtype=torch.float64)
    full = torch.cat([logits, sink_col], dim=-1)                       # [T, H, N + 1]
    live = torch.isfinite(full.max(dim=-1).values)
    safe = torch.where(live[..., None], full, torch.zeros_like(full))
    p = torch.where(live[..., None], torch.softmax(safe, dim=-1), torch.zeros_like(full))
    o = torch.einsum("thn,nd->thd", p[..., :N], kv)                   # the sink's value is 0
    loss = (o * torch.from_numpy(_f64(do_bits))).sum()
    loss.backward()
    ds = sk.grad.numpy() if sink is not None else np.zeros(H)
    return q.grad.numpy(), kv.grad.numpy(), ds


def _close(a, b, rtol=1e-9):
    scale = max(np.abs(b).max(), 1e-300)
    return np.abs(a - b).max() <= rtol * scale


@pytest.mark.parametrize("variant", ["plain", "dups", "oob", "nosink", "sinkneg", "allbad_rows"])
def test_backward_matches_autograd(variant):
    cfg, x = _inputs(seed=3, sink=(variant != "nosink"))
    idx = x["idx"]
    sink = x["sink"]
    if variant == "dups":
        idx = synth.inject_duplicates(idx, cfg.num_kv, 4, frac=0.25)
    elif variant == "oob":
        idx = synth.inject_out_of_range(idx.astype(np.int64), cfg.num_kv, 5, frac=0.3)
    elif variant == "sinkneg":
        sink = np.full_like(sink, -np.inf)
    elif variant == "allbad_rows":
        idx = idx.copy()
        idx[::3] = -1
    dq, dkv, ds = bwd.sparse_mla_bwd(x["q"], x["kv"], idx, sink, x["scale"], x["do"])
    rq, rkv, rs = _autograd_reference(x["q"], x["kv"], idx,
                                      None if variant == "sinkneg" else sink, x["scale"], x["do"])
    assert _close(dq, rq) and _close(dkv, rkv)
    if variant in ("nosink", "sinkneg"):
        assert np.all(ds == 0)
    else:
        assert _close(ds, rs)


def _loss(q, kv, idx, sink, scale, do, num_kv):
    """sum(dO * O) from the forward oracle's per-token definition (float64 inputs)."""
    tot = 0.0
    for t in range(q.shape[0]):
        o, _ = orc.token_forward(q[t], kv, idx[t], num_kv, sink, scale)
        tot += float((o * do[t]).sum())
    return tot


def test_backward_matches_finite_differences():
    cfg, x = _inputs(seed=7, T=6, H=3, topk=24, window=8, pool=8)
    idx = synth.inject_duplicates(x["idx"], cfg.num_kv, 8, frac=0.2)
    q, kv, do = _f64(x["q"]), _f64(x["kv"]), _f64(x["do"])
    sink = x["sink"].astype(np.float64)
    dq, dkv, ds = bwd.sparse_mla_bwd(x["q"], x["kv"], idx, x["sink"], x["scale"], x["do"])
    rng = np.random.default_rng(9)
    eps = 1e-5
    for _ in range(3):
        uq, ukv, us = (rng.standard_normal(q.shape), rng.standard_normal(kv.shape),
                       rng.standard_normal(sink.shape))
        lp = _loss(q + eps * uq, kv + eps * ukv, idx, sink + eps * us, x["scale"], do, cfg.num_kv)
        lm = _loss(q - eps * uq, kv - eps * ukv, idx, sink - eps * us, x["scale"], do, cfg.num_kv)
        fd = (lp - lm) / (2 * eps)
        an = float((dq * uq).sum() + (dkv * ukv).sum() + (ds * us).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (fd, an)


def test_backward_single_slot_closed_form():
    # one valid slot r with a sink: O = v * sig, sig = e^s / (e^s + e^sink), s = scale <q, v>;
    # L = sig <dO, v>: dL/dsink = -sig (1 - sig) <dO, v>,
    # dL/dq = sig (1 - sig) <dO, v> scale v, dL/dv = sig dO + sig (1 - sig) <dO, v> scale q
    rng = np.random.default_rng(12)
    H = 2
    q_bits = synth.bf16_bits(rng.standard_normal((1, H, D)).astype(np.float32))
    kv_bits = synth.bf16_bits(rng.standard_normal((30, D)).astype(np.float32))
    do_bits = synth.bf16_bits(rng.standard_normal((1, H, D)).astype(np.float32))
    sink = np.array([0.3, -1.2], dtype=np.float32)
    idx = np.array([[-1, 17, 30, -5]], dtype=np.int64)
    scale = 1 / math.sqrt(D)
    dq, dkv, ds = bwd.sparse_mla_bwd(q_bits, kv_bits, idx, sink, scale, do_bits)
    v = _f64(kv_bits[17])
    dv_want = np.zeros(D)
    for h in range(H):
        qh, doh = _f64(q_bits[0, h]), _f64(do_bits[0, h])
        s = scale * math.fsum(qh * v)
        sig = math.exp(s) / (math.exp(s) + math.exp(float(sink[h])))
        dov = math.fsum(doh * v)
        assert abs(ds[h] - (-sig * (1 - sig) * dov)) <= 1e-12 * max(1, abs(dov))
        np.testing.assert_allclose(dq[0, h], sig * (1 - sig) * dov * scale * v, rtol=1e-10,
                                   atol=1e-14)
        dv_want += sig * doh + sig * (1 - sig) * dov * scale * qh
    np.testing.assert_allclose(dkv[17], dv_want, rtol=1e-10, atol=1e-13)
    others = np.delete(np.arange(30), 17)
    assert np.all(dkv[others] == 0)


def test_backward_invariants():
    cfg, x = _inputs(seed=21)
    dq, dkv, ds = bwd.sparse_mla_bwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"], x["do"])
    used = np.unique(x["idx"][(x["idx"] >= 0) & (x["idx"] < cfg.num_kv)])
    unused = np.setdiff1d(np.arange(cfg.num_kv), used)
    assert np.all(dkv[unused] == 0)
    # permuting each token's list changes nothing (up to summation order)
    idx_p = synth.shuffle_rows(x["idx"], 3)
    dq2, dkv2, ds2 = bwd.sparse_mla_bwd(x["q"], x["kv"], idx_p, x["sink"], x["scale"], x["do"])
    assert _close(dq2, dq, 1e-12) and _close(dkv2, dkv, 1e-12) and _close(ds2, ds, 1e-12)
    # sink = -inf is no sink
    dq3, dkv3, ds3 = bwd.sparse_mla_bwd(x["q"], x["kv"], x["idx"],
                                        np.full_like(x["sink"], -np.inf), x["scale"], x["do"])
    dq4, dkv4, ds4 = bwd.sparse_mla_bwd(x["q"], x["kv"], x["idx"], None, x["scale"], x["do"])
    assert np.array_equal(dq3, dq4) and np.array_equal(dkv3, dkv4)
    assert np.all(ds3 == 0) and np.all(ds4 == 0)
    # an all-invalid token contributes nothing
    idx_b = x["idx"].copy()
    idx_b[:] = -1
    dq5, dkv5, ds5 = bwd.sparse_mla_bwd(x["q"], x["kv"], idx_b, x["sink"], x["scale"], x["do"])
    assert np.all(dq5 == 0) and np.all(dkv5 == 0) and np.all(ds5 == 0)


# ------------------------------------------------------------ planted mistakes
_orig = bwd.token_backward


def _mutant(kind):
    def fwd(q_t, kv, idx_t, num_kv, sink, scale, do_t):
        H, Dd = q_t.shape
        rows = np.asarray(idx_t).astype(np.int64)
        v = (rows >= 0) & (rows < num_kv)
        rows = rows[v]
        k = kv[rows]
        if k.dtype == np.uint16:
            k = orc.bf16_to_f64(k)
        dq = np.zeros((H, Dd))
        dsink = np.zeros(H)
        dk = np.zeros((rows.size, Dd))
        s = scale * (q_t @ k.T)
        m = s.max(axis=1) if rows.size else np.full(H, -np.inf)
        if sink is not None:
            m = np.maximum(m, sink)
        live = np.isfinite(m)
        if not np.any(live) or rows.size == 0:
            return dq, rows, dk, dsink
        ml = m[live]
        e = np.exp(s[live] - ml[:, None])
        den = e.sum(axis=1)
        if sink is not None and kind != "sink_not_in_den":
            den = den + np.exp(sink[live] - ml)
        P = e / den[:, None]
        O = P @ k
        dP = do_t[live] @ k.T
        delta = (do_t[live] * O).sum(axis=1)
        if kind == "no_delta":
            delta = 0 * delta
        dS = P * (dP - delta[:, None])
        dq[live] = (1.0 if kind == "dq_no_scale" else scale) * (dS @ k)
        dk = scale * (dS.T @ q_t[live])
        if kind != "dkv_no_value_term":
            dk = dk + P.T @ do_t[live]
        if kind == "dkv_no_key_term":
            dk = P.T @ do_t[live]
        if sink is not None:
            p_sink = np.exp(sink[live] - ml) / den
            dsink[live] = (p_sink if kind == "dsink_sign" else -p_sink) * delta
        return dq, rows, dk, dsink
    return fwd


def _dedupe_add_at(a, rows, vals):
    a[rows] += vals       # buffered: a duplicated row keeps only one slot's contribution


BWD_MUTANTS = ["sink_not_in_den", "no_delta", "dq_no_scale", "dkv_no_value_term",
               "dkv_no_key_term", "dsink_sign", "dup_rows_once"]


def _battery():
    try:
        cfg, x = _inputs(seed=31)
        idx = synth.inject_duplicates(x["idx"], cfg.num_kv, 6, frac=0.3)
        dq, dkv, ds = bwd.sparse_mla_bwd(x["q"], x["kv"], idx, x["sink"], x["scale"], x["do"])
        rq, rkv, rs = _autograd_reference(x["q"], x["kv"], idx, x["sink"], x["scale"], x["do"])
        return _close(dq, rq) and _close(dkv, rkv) and _close(ds, rs)
    except Exception:
        return False


def test_unmutated_backward_passes_battery():
    assert _battery()


def test_mutant_template_is_faithful(monkeypatch):
    monkeypatch.setattr(bwd, "token_backward", _mutant("none"))
    assert _battery()


@pytest.mark.parametrize("kind", BWD_MUTANTS)
def test_backward_mutant_is_caught(kind, monkeypatch):
    if kind == "dup_rows_once":
        monkeypatch.setattr(bwd, "accumulate_rows", _dedupe_add_at)
    else:
        monkeypatch.setattr(bwd, "token_backward", _mutant(kind))
    assert not _battery(), f"backward pins miss the planted mistake {kind!r}"
