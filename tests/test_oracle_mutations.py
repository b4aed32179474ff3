"""Planted mistakes in the oracle must each fail at least one pin (CPU only).

Each mutant replaces one step of the oracle's per-token forward with a
plausible slip (a dropped sink term, a wrong axis, a narrowed index, a lost
duplicate, ...).  The battery below is the pins' own checks: dense SDPA brute
force, the one-slot closed form and the all-invalid row.  A mutant that passes
the whole battery means the pins have a hole.
"""
import math

import numpy as np
import pytest

from oracle import oracle as orc
from sparse_mla_attention_token_gb300 import synth
from tests.test_oracle_pins import _dense_reference, _dot, _f64, _one_token

D = 512
_orig_token_forward = orc.token_forward
_orig_valid = orc.valid_slots


def _battery():
    """True when every pin passes for the current (possibly mutated) oracle."""
    try:
        cfg = synth.CONFIGS["tiny"].with_(seed=21)
        x = synth.make_inputs(cfg)
        idx = synth.inject_duplicates(x["idx"], cfg.num_kv, 3, frac=0.2)
        idx = synth.inject_out_of_range(idx.astype(np.int64), cfg.num_kv, 4, frac=0.2)
        # pull row 0 into many lists so a mutant that drops it is visible
        idx[:, 0] = 0
        O, L = orc.sparse_mla_fwd(x["q"], x["kv"], idx, x["sink"], x["scale"])
        Od, Ld = _dense_reference(x["q"], x["kv"], idx, x["sink"], x["scale"])
        live = np.isfinite(Ld)
        if not (np.allclose(O[live], Od[live], rtol=1e-10, atol=1e-12)
                and np.allclose(L[live], Ld[live], rtol=1e-12, atol=1e-12)):
            return False
        q_bits, kv_bits, idx1, sink = _one_token([-1, 7, 20], 0.75)
        scale = 1 / math.sqrt(D)
        O, L = orc.sparse_mla_fwd(q_bits, kv_bits, idx1, sink, scale)
        s = scale * _dot(_f64(q_bits[0, 0]), _f64(kv_bits[7]))
        sk = float(np.float32(0.75))
        if abs(L[0, 0] - math.log(math.exp(s) + math.exp(sk))) > 1e-12:
            return False
        allbad = np.full_like(x["idx"], -1)
        O, L = orc.sparse_mla_fwd(x["q"], x["kv"], allbad, x["sink"], x["scale"])
        if not (np.all(O == 0) and np.allclose(L, x["sink"].astype(np.float64)[None])):
            return False
        return True
    except Exception:
        return False


def _mutant_token_forward(kind):
    def fwd(q_t, kv, idx_t, num_kv, sink, scale, d_v=None):
        H, Dd = q_t.shape
        i = np.asarray(idx_t).astype(np.int64)
        if kind == "int32_wrap":
            i = np.asarray(idx_t).astype(np.int32).astype(np.int64)
        v = (i >= 0) & (i < num_kv)
        if kind == "drop_row0":
            v = (i > 0) & (i < num_kv)
        rows = i[v]
        if kind == "dedupe":
            rows = np.unique(rows)
        k = kv[rows]
        if k.dtype == np.uint16:
            k = orc.bf16_to_f64(k)
        sc = scale * scale if kind == "scale_squared" else scale
        s = sc * (q_t @ k.T)
        if kind == "neg_score":
            s = -s
        m = s.max(axis=1) if rows.size else np.full(H, -np.inf)
        if sink is not None:
            m = np.maximum(m, sink)
        out = np.zeros((H, Dd))
        lse = np.full(H, -np.inf)
        live = np.isfinite(m)
        if np.any(live):
            ml = m[live]
            e = np.exp(s[live] - ml[:, None])
            den = e.sum(axis=1)
            if sink is not None and kind != "no_sink_den":
                den = den + np.exp(sink[live] - ml)
            num = e @ k
            if kind == "sink_in_numerator" and sink is not None:
                num = num + np.exp(sink[live] - ml)[:, None]
            out[live] = num / den[:, None]
            lse[live] = ml + np.log(den)
            if kind == "lse_no_sink" and sink is not None:
                lse[live] = ml + np.log(e.sum(axis=1))
            if kind == "lse_log2":
                lse[live] = ml + np.log2(den)
            if kind == "softmax_wrong_axis":
                e2 = np.exp(s[live] - s[live].max(axis=0, keepdims=True))
                out[live] = (e2 / e2.sum(axis=0, keepdims=True)) @ k
        if kind == "allinvalid_lse_zero":
            lse[~live] = 0.0
        if kind == "allinvalid_with_sink_wrong" and sink is not None and rows.size == 0:
            lse[:] = -np.inf
        return out, lse

    def quiet(*args, **kw):
        # a planted mistake may divide by zero or take log(0); the pins judge the result
        with np.errstate(divide="ignore", invalid="ignore"):
            return fwd(*args, **kw)
    return quiet


MUTANTS = ["int32_wrap", "drop_row0", "dedupe", "scale_squared", "neg_score", "no_sink_den",
           "sink_in_numerator", "lse_no_sink", "lse_log2", "softmax_wrong_axis",
           "allinvalid_with_sink_wrong"]


def test_unmutated_oracle_passes_battery():
    assert _battery()


@pytest.mark.parametrize("kind", MUTANTS)
def test_mutant_is_caught(kind, monkeypatch):
    monkeypatch.setattr(orc, "token_forward", _mutant_token_forward(kind))
    assert not _battery(), f"pins miss the planted mistake {kind!r}"


def test_mutant_harness_is_faithful(monkeypatch):
    # the mutant template with no mutation must pass, or the test above proves nothing
    monkeypatch.setattr(orc, "token_forward", _mutant_token_forward("none"))
    assert _battery()
