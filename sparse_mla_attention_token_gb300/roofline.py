"""Algorithmic FLOP and byte counts of one forward call, and the roofline.

Per unit (one valid slot of one token): 4 * H * 512 FLOPs (S = Q.K^T and
O = P.V, 2 FLOPs per multiply-add each) and one gathered 1024-byte kv row.
Per call, fixed bytes: Q and O (T*H*1024 each), lse (T*H*4), the index list
(T*topk*4 or 8) and the sink (H*4).

Two byte counts, as the roofline of this op is defined:
* gathered = fixed + 1024 B per valid slot (the bytes the method moves per
  token; most of them come from L2 when the pool is small);
* unique   = fixed + 1024 B per distinct valid kv row (perfect reuse).
The roofline time is max(FLOPs / bf16 peak, bytes / HBM bandwidth).
"""
from __future__ import annotations

import json
import os
from dataclasses import dataclass

import numpy as np

D = 512
ROW_BYTES = D * 2

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


@dataclass
class Counts:
    T: int
    H: int
    topk: int
    num_kv: int
    valid: int          # sum over tokens of valid slots
    unique_rows: int    # distinct valid kv rows over the whole call
    index_bytes: int
    sink: bool

    @property
    def flops(self) -> float:
        return 4.0 * self.H * D * self.valid

    @property
    def flops_all_slots(self) -> float:
        return 4.0 * self.T * self.H * self.topk * D

    @property
    def fixed_bytes(self) -> float:
        return (2.0 * self.T * self.H * ROW_BYTES + 4.0 * self.T * self.H +
                self.T * self.topk * self.index_bytes + (4.0 * self.H if self.sink else 0.0))

    @property
    def gathered_bytes(self) -> float:
        return self.fixed_bytes + float(self.valid) * ROW_BYTES

    @property
    def unique_bytes(self) -> float:
        return self.fixed_bytes + float(self.unique_rows) * ROW_BYTES


def count(idx: np.ndarray, num_kv: int, H: int, sink: bool) -> Counts:
    """Counts for one call from its index list (validity: 0 <= idx < num_kv)."""
    i = np.asarray(idx)
    ok = (i >= 0) & (i < num_kv)
    rows = np.unique(i[ok]) if ok.any() else np.zeros(0, dtype=np.int64)
    return Counts(T=i.shape[0], H=H, topk=i.shape[1], num_kv=num_kv, valid=int(ok.sum()),
                  unique_rows=int(rows.size), index_bytes=i.dtype.itemsize, sink=sink)


def load_peaks(root: str) -> tuple[dict, str]:
    """Measured peaks (``MEASURED_PEAKS.json``), else the fallback; returns (peaks, source)."""
    p = os.path.join(root, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def terms(c: Counts, seconds: float, peaks: dict, sustained: bool = False) -> dict:
    """Each roofline term's time, the achieved rate and the fraction of its peak."""
    tflops_peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    hbm = peaks["hbm_gbs"]
    t_flop = c.flops / (tflops_peak * 1e12)
    t_gath = c.gathered_bytes / (hbm * 1e9)
    t_uniq = c.unique_bytes / (hbm * 1e9)
    return {
        "flop": {"time_s": t_flop, "achieved": c.flops / seconds / 1e12, "peak": tflops_peak,
                 "unit": "TFLOP/s", "frac": t_flop / seconds},
        "gathered": {"time_s": t_gath, "achieved": c.gathered_bytes / seconds / 1e9, "peak": hbm,
                     "unit": "GB/s", "frac": t_gath / seconds},
        "unique": {"time_s": t_uniq, "achieved": c.unique_bytes / seconds / 1e9, "peak": hbm,
                   "unit": "GB/s", "frac": t_uniq / seconds},
        "roofline_gathered_s": max(t_flop, t_gath),
        "roofline_unique_s": max(t_flop, t_uniq),
        "frac_of_roofline_gathered": max(t_flop, t_gath) / seconds,
        "frac_of_roofline_unique": max(t_flop, t_uniq) / seconds,
    }
