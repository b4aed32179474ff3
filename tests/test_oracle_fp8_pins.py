"""Pins for the fp8-cache oracle (CPU only).

* the e4m3fn decoder against torch's float8_e4m3fn (a library routine) on all
  256 codes, NaN included;
* closed forms of the format: 1.0 = 0x38, 448 = 0x7E, the smallest subnormal
  0x01 = 2^-9, -2 = 0xC0;
* the cache forward equals the bf16 op's definition on the decoded values
  (dequantised rows written out as float64 and fed to the plain oracle), and
  rows no valid slot names never matter (NaN codes there change nothing).
"""
import math

import numpy as np
import torch

from oracle import fp8kv
from oracle import oracle as orc
from sparse_mla_attention_token_gb300 import synth


def test_e4m3_decoder_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = fp8kv.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])


def test_e4m3_closed_forms():
    d = fp8kv.e4m3_to_f64(np.array([0x38, 0x7E, 0x01, 0xC0, 0x00, 0x80], dtype=np.uint8))
    assert d[0] == 1.0 and d[1] == 448.0 and d[2] == 2.0 ** -9 and d[3] == -2.0
    assert d[4] == 0.0 and d[5] == 0.0 and math.copysign(1, d[5]) == -1


def test_cache_forward_is_the_definition_on_decoded_rows():
    cfg = synth.CONFIGS["tiny"].with_(seed=51)
    x = synth.make_inputs(cfg)
    kv8, sc = synth.fp8_cache(x["kv"])
    # rows no valid slot names hold NaN codes: they must never matter
    idx = synth.inject_out_of_range(x["idx"].astype(np.int64), cfg.num_kv, 7, frac=0.2)
    used = np.unique(idx[(idx >= 0) & (idx < cfg.num_kv)])
    unused = np.setdiff1d(np.arange(cfg.num_kv), used)
    kv8[unused] = 0x7F
    O, L = fp8kv.sparse_mla_fwd_fp8kv(x["q"], kv8, sc, idx, x["sink"], x["scale"])
    dense = fp8kv.dequant_rows(kv8, sc)              # the decoded values, written out
    dense[unused] = 0.0
    ref_O = np.zeros_like(O)
    ref_L = np.zeros_like(L)
    q = orc.bf16_to_f64(x["q"])
    for t in range(cfg.T):
        ref_O[t], ref_L[t] = orc.token_forward(q[t], dense, idx[t], cfg.num_kv,
                                               x["sink"].astype(np.float64), x["scale"])
    np.testing.assert_array_equal(O, ref_O)
    np.testing.assert_array_equal(L, ref_L)
    assert not np.isnan(O).any()


def test_cache_writer_round_trip():
    # the generator's cache holds each bf16 value to e4m3's precision (2^-4 relative
    # of the block's scale step): a coarse check that the inputs are what they claim
    cfg = synth.CONFIGS["tiny"].with_(seed=52)
    x = synth.make_inputs(cfg)
    kv8, sc = synth.fp8_cache(x["kv"])
    v = orc.bf16_to_f64(x["kv"])
    d = fp8kv.dequant_rows(kv8, sc)
    blk_amax = np.repeat(np.abs(v).reshape(v.shape[0], 4, 128).max(axis=2), 128, axis=1)
    assert np.all(np.abs(d - v) <= blk_amax * 2.0 ** -4 + 1e-12)
