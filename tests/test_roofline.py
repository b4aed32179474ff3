"""Roofline arithmetic against the workload sizes (CPU only).

FLOPs = 4*H*512*valid slots; gathered bytes = Q + O + lse + indices + sink +
1 KB per valid slot; unique bytes count each distinct valid row once.
"""
import numpy as np
import pytest

from sparse_mla_attention_token_gb300 import roofline, synth

# (GFLOP, fixed MB, gathered-row MB) per workload, 1 MB = 1e6 bytes
EXPECTED = {
    "tiny": (0.067, 2.1, 2.1),
    "sweep_k32": (2.14, 67.8, 133.7),
    "sweep_k640": (34.22, 77.7, 2138.6),
    "h128": (470.2, 1084.2, 1836.8),
}


@pytest.mark.parametrize("name", list(EXPECTED))
def test_counts(name):
    cfg = synth.CONFIGS[name]
    idx = synth.make_indices(cfg, np.random.Generator(np.random.PCG64(cfg.seed)))
    c = roofline.count(idx, cfg.num_kv, cfg.H, cfg.sink)
    gf, fixed, gath = EXPECTED[name]
    assert abs(c.flops / 1e9 - gf) <= 0.01 * gf + 0.001
    assert abs(c.fixed_bytes / 1e6 - fixed) <= 0.1
    assert abs((c.gathered_bytes - c.fixed_bytes) / 1e6 - gath) <= 0.1
    assert c.unique_rows <= cfg.num_kv
    assert c.unique_bytes <= c.gathered_bytes


def test_terms_pick_the_slower_term():
    cfg = synth.CONFIGS["h128"]
    idx = synth.make_indices(cfg, np.random.Generator(np.random.PCG64(cfg.seed)))
    c = roofline.count(idx, cfg.num_kv, cfg.H, cfg.sink)
    peaks = {"hbm_gbs": 6801.3, "bf16_tflops": 1891.6, "bf16_tflops_sustained": 1694.3}
    t = roofline.terms(c, 1e-3, peaks)
    assert abs(t["flop"]["time_s"] - 0.2486e-3) < 0.002e-3
    assert abs(t["gathered"]["time_s"] - 0.270e-3 - 0.16e-3) < 0.01e-3
    assert t["roofline_gathered_s"] == max(t["flop"]["time_s"], t["gathered"]["time_s"])
    assert abs(t["frac_of_roofline_gathered"] - t["roofline_gathered_s"] / 1e-3) < 1e-12
