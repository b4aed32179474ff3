"""Structure of the synthetic workloads (CPU only).

The index lists follow the window + causally visible compressed-pool recipe
("Sparse MLA training backward", section "Performance": realistic top-k is a
sliding window plus a causally visible pool, not uniform random).  The valid
slot count of each workload has a closed form that depends only on
visibility; the totals below are the ones the workloads are sized by.
"""
import numpy as np
import pytest
import torch

from sparse_mla_attention_token_gb300 import synth

# Sum over tokens of valid slots for each workload (closed form below).
EXPECTED_VALID = {
    "tiny": 2048,
    "small_head": 9952832,
    "sweep_k32": 130576,
    "sweep_k128": 516160,
    "sweep_k256": 1007552,
    "sweep_k640": 2088512,
    "h128": 1793728,
    "h128_long": 5994368,
    "glm_k2048": 26171584,
    "decode_h8_t1": 640,
    "decode_h16_t16": 10240,
    "decode_h128_t4": 2048,
}


def _closed_form_valid(cfg):
    t = cfg.pos0 + np.arange(cfg.T, dtype=np.int64)
    win = np.minimum(cfg.window, t + 1)
    vis = np.minimum(cfg.pool, (t + 1) // cfg.ratio)
    return int(win.sum() + np.minimum(vis, cfg.topk - cfg.window).sum())


@pytest.mark.parametrize("name", list(EXPECTED_VALID))
def test_valid_count_closed_form(name):
    cfg = synth.CONFIGS[name]
    assert _closed_form_valid(cfg) == EXPECTED_VALID[name]


@pytest.mark.parametrize("name", ["tiny", "sweep_k32", "sweep_k256", "h128", "glm_k2048",
                                  "decode_h8_t1", "decode_h16_t16", "decode_h128_t4"])
def test_index_structure(name):
    cfg = synth.CONFIGS[name]
    idx = synth.make_indices(cfg, np.random.Generator(np.random.PCG64(cfg.seed)))
    assert idx.shape == (cfg.T, cfg.topk)
    assert idx.dtype == (np.int64 if cfg.index_dtype == "int64" else np.int32)
    W = cfg.window
    for t in range(0, cfg.T, max(1, cfg.T // 97)):
        pos = cfg.pos0 + t                              # the token's position in its sequence
        row = idx[t].astype(np.int64)
        exp_win = np.arange(pos - W + 1, pos + 1)
        exp_win = np.where(exp_win < 0, -1, cfg.base_row + exp_win)
        np.testing.assert_array_equal(row[:W], exp_win)
        pool = row[W:]
        got = pool[pool >= 0]
        vis = min(cfg.pool, (pos + 1) // cfg.ratio)
        assert len(got) == min(vis, cfg.topk - W)
        assert np.all(np.diff(got) > 0)                 # sorted, no repeats
        p = got - (cfg.base_row + cfg.ctx)
        assert np.all(p >= 0) and np.all(cfg.ratio * (p + 1) <= pos + 1)
        assert np.all(pool[len(got):] == -1)
    valid = ((idx >= 0) & (idx < cfg.num_kv)).sum()
    assert valid == EXPECTED_VALID[name]
    # rows of other sequences in a shared pool are never named
    assert not np.any((idx >= 0) & (idx < cfg.base_row))


def test_decode_configs_cover_the_sweep():
    for h in synth.DECODE_H:
        for t in synth.DECODE_T:
            cfg = synth.CONFIGS[f"decode_h{h}_t{t}"]
            assert (cfg.T, cfg.H, cfg.ctx) == (t, h, 8192)


def test_shared_pool_rows_hold_nan():
    # a small stand-in of the 2 GiB shared pool: the other sequences' rows are NaN
    cfg = synth.CONFIGS["tiny"].with_(base_row=40)
    x = synth.make_inputs(cfg)
    assert x["kv"].shape == (cfg.num_kv, 512)
    assert np.all(x["kv"][:40] == synth.NAN_BITS)
    base = synth.make_inputs(synth.CONFIGS["tiny"])
    np.testing.assert_array_equal(x["q"], base["q"])
    np.testing.assert_array_equal(x["kv"][40:], base["kv"])
    np.testing.assert_array_equal(np.where(x["idx"] >= 0, x["idx"] - 40, -1), base["idx"])


def test_generator_is_deterministic():
    cfg = synth.CONFIGS["tiny"]
    a, b = synth.make_inputs(cfg), synth.make_inputs(cfg)
    for k in ("q", "kv", "idx", "sink"):
        np.testing.assert_array_equal(a[k], b[k])
    c = synth.make_inputs(cfg.with_(seed=99))
    assert not np.array_equal(a["q"], c["q"])


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32),
                        np.array([1.00390625, 1.01171875, -1.00390625, 3.0e38, 1e-40],
                                 dtype=np.float32)])
    ours = synth.bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_out_of_range_injection_values():
    cfg = synth.CONFIGS["tiny"]
    idx = synth.make_indices(cfg, np.random.Generator(np.random.PCG64(0))).astype(np.int64)
    bad = synth.inject_out_of_range(idx, cfg.num_kv, 1, frac=0.5)
    changed = bad != idx
    assert changed.sum() > 0.3 * idx.size
    assert np.all((bad[changed] < 0) | (bad[changed] >= cfg.num_kv))
    assert (bad >= 2 ** 31).any()
