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


def _bench_module():
    import importlib.util
    import os
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(root, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_committed_traffic_only_for_the_profiled_source(tmp_path, monkeypatch):
    # The bench reports an ncu DRAM traffic figure only from a summary taken on
    # the kernel source it runs (same sha256 prefix), and null otherwise.
    b = _bench_module()
    src = tmp_path / "sparse_mla_attention_token_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "smla_h128.cu").write_text("// kernel v1\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    assert b.committed_traffic(1, "h128") == (None, "no ncu summary for this kernel/workload")
    sha = b.kernel_source_sha(1)
    (tmp_path / "profiles" / "k.md").write_text(
        f"traffic_per_launch: kernel=h128_fwd_kernel workload=h128 source_sha={sha} "
        f"dram_bytes=12345\n")
    assert b.committed_traffic(1, "h128") == (12345, "profiles/k.md")
    assert b.committed_traffic(1, "h128_long")[0] is None
    (src / "smla_h128.cu").write_text("// kernel v2\n")
    v, why = b.committed_traffic(1, "h128")
    assert v is None and "another source" in why
