"""Helpers shared by the GPU parity tests: device copies of the seeded inputs
and the comparison against the fp64 oracle.

Bar (tolerances for the floating-point outputs): max|dO| <= 2e-2,
max|dlse| <= 5e-3, cosine(O) >= 0.9999 per tensor.  lse entries that are -inf
on either side must be -inf on both and are left out of the differences and
of the cosine; O rows of such entries must be exactly 0.
"""
from __future__ import annotations

import numpy as np

TOL_O = 2e-2
TOL_LSE = 5e-3
TOL_COS = 0.9999


def to_dev(x, dev, kv_offset_bytes: int = 0, guard_rows: int = 0, guard_value=None):
    """Device tensors for one input dict.

    kv is placed ``kv_offset_bytes`` into one larger allocation, with
    ``guard_rows`` rows after it set to ``guard_value`` (bf16 bits), so reads
    past ``num_kv`` would pick up the guard.
    """
    import torch
    q = torch.from_numpy(x["q"].view(np.int16)).view(torch.bfloat16).to(dev)
    kvh = torch.from_numpy(x["kv"].view(np.int16))
    n, d = x["kv"].shape
    if kv_offset_bytes or guard_rows:
        assert kv_offset_bytes % 1024 == 0 or kv_offset_bytes % 16 == 0
        total = kv_offset_bytes // 2 + (n + guard_rows) * d
        buf = torch.zeros(total, dtype=torch.int16, device=dev)
        start = kv_offset_bytes // 2
        buf[start:start + n * d] = kvh.reshape(-1).to(dev)
        if guard_rows:
            g = int(np.int16(np.uint16(guard_value).view(np.int16)))
            buf[start + n * d:] = g
        kv = buf[start:start + n * d].view(n, d).view(torch.bfloat16)
        keep = buf
    else:
        kv = kvh.to(dev).view(torch.bfloat16)
        keep = None
    idx = torch.from_numpy(x["idx"]).to(dev)
    sink = None if x["sink"] is None else torch.from_numpy(x["sink"]).to(dev)
    return q, kv, idx, sink, keep


def compare(out, lse, O, L, tokens=None, o_tol=TOL_O):
    """Return a dict of parity numbers; raises AssertionError outside the bar.

    ``o_tol`` replaces the max|dO| bar for callers that check O themselves.
    """
    og = out.float().cpu().numpy().astype(np.float64)
    lg = lse.float().cpu().numpy().astype(np.float64)
    if tokens is not None:
        og, lg = og[tokens], lg[tokens]
    assert og.shape == O.shape and lg.shape == L.shape
    assert not np.any(np.isnan(og)), "NaN in O"
    assert not np.any(np.isnan(lg)), "NaN in lse"
    ninf_o, ninf_g = np.isneginf(L), np.isneginf(lg)
    assert np.array_equal(ninf_o, ninf_g), \
        f"-inf lse mismatch at {np.argwhere(ninf_o != ninf_g)[:5].tolist()}"
    assert np.all(og[ninf_g] == 0), "rows with lse = -inf must have O = 0"
    live = ~ninf_g
    d_o = float(np.max(np.abs(og - O))) if og.size else 0.0
    d_l = float(np.max(np.abs(lg[live] - L[live]))) if live.any() else 0.0
    a, b = og[live].ravel(), O[live].ravel()
    nab = np.sqrt((a * a).sum() * (b * b).sum())
    cos = float((a * b).sum() / nab) if nab > 0 else 1.0
    res = {"max_dO": d_o, "max_dlse": d_l, "cos": cos}
    assert d_o <= o_tol, f"max|dO| {d_o} > {o_tol} ({res})"
    assert d_l <= TOL_LSE, f"max|dlse| {d_l} > {TOL_LSE} ({res})"
    assert cos >= TOL_COS, f"cos {cos} < {TOL_COS} ({res})"
    return res
