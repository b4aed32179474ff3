"""Load the golden fixtures of this folder (written by ``make_golden.py``).

A fixture stores its inputs sparsely (non-zero entries, every value exact in
bf16) and its expected outputs as decimal strings from the closed form the
fixture's ``derivation`` states; entries of O not listed are exactly 0.
"""
from __future__ import annotations

import json
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
NAMES = ("uniform_scores", "two_level_scores", "large_scores")
D = 512


def _bf16_bits(vals) -> np.ndarray:
    f = np.asarray(vals, dtype=np.float64)
    f32 = f.astype(np.float32)
    assert np.array_equal(f32.astype(np.float64), f), "fixture value not exact in fp32"
    u = f32.view(np.uint32)
    assert np.all(u & 0xFFFF == 0), "fixture value not exact in bf16"
    return (u >> 16).astype(np.uint16)


def load(name: str) -> dict:
    """Inputs in the layout of ``synth.make_inputs`` plus ``O`` / ``lse`` (float64)."""
    with open(os.path.join(HERE, name + ".json")) as f:
        fx = json.load(f)
    T, H, N = fx["T"], fx["H"], fx["num_kv"]
    q = np.zeros((T, H, D), np.uint16)
    for t, h, d, v in fx["q"]:
        q[t, h, d] = _bf16_bits([v])[0]
    kv = np.zeros((N, D), np.uint16)
    for r, d, v in fx["kv"]:
        kv[r, d] = _bf16_bits([v])[0]
    idx = np.asarray(fx["idx"], dtype=np.int64 if fx["index_dtype"] == "int64" else np.int32)
    assert idx.shape == (T, fx["topk"])
    sink = None
    if fx["sink"] is not None:
        sink = np.asarray(fx["sink"], np.float32)
        assert np.array_equal(sink.astype(np.float64), np.asarray(fx["sink"], np.float64))
    scale = float(fx["scale"])
    assert float(np.float32(scale)) == scale, "scale must be exact in fp32"
    lse = np.array([[float(v) for v in row] for row in fx["expected"]["lse"]], np.float64)
    O = np.zeros((T, H, D), np.float64)
    for t, h, d, v in fx["expected"]["O"]:
        O[t, h, d] = float(v)
    return dict(name=name, q=q, kv=kv, idx=idx, sink=sink, scale=scale, O=O, lse=lse,
                cite=fx["cite"], derivation=fx["derivation"])
