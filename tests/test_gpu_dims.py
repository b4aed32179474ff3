"""GPU parity of the other head dims and the positional-part layout (needs a GB300).

``sparse_mla_fwd_dims`` through the C ABI against the fp64 oracle at head dims
128 and 576 with K == V ("Tuned sparse MLA prefill for DSv4.1-Flash TP4", its
tests at those dims) and at 576 score / 512 value columns, the MLA layout with
a 64-wide positional part ("Add DSv4 sparse MLA prefill Triton and unified with
MLA Gluon kernel on GFX950", has_pe = True).  Same bar as the 512-wide op.
"""
import math

import numpy as np
import pytest

from oracle import oracle as orc
from sparse_mla_attention_token_gb300 import synth
from tests.parity import compare

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DIMS = [(128, 128), (576, 576), (576, 512)]


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_attention_token_gb300 import binding
    binding.lib()
    return binding


def _inputs(cfg, D):
    """The workload's index lists with D-wide q / kv rows (N(0,1), bf16), seeded."""
    rng = np.random.Generator(np.random.PCG64(cfg.seed + 31 * D))
    x = synth.make_inputs(cfg)
    x["q"] = synth.bf16_bits(rng.standard_normal((cfg.T, cfg.H, D), dtype=np.float32))
    x["kv"] = synth.bf16_bits(rng.standard_normal((cfg.num_kv, D), dtype=np.float32))
    x["scale"] = 1.0 / math.sqrt(D)
    return x


def _dev(x):
    q = torch.from_numpy(x["q"].view(np.int16)).view(torch.bfloat16).to(DEV)
    kv = torch.from_numpy(x["kv"].view(np.int16)).view(torch.bfloat16).to(DEV)
    idx = torch.from_numpy(x["idx"]).to(DEV)
    sink = None if x["sink"] is None else torch.from_numpy(x["sink"]).to(DEV)
    return q, kv, idx, sink


def _check(B, x, d_v, splits_note=""):
    q, kv, idx, sink = _dev(x)
    out, lse = B.sparse_mla_fwd_dims(q, kv, idx, sink, x["scale"], d_v=d_v)
    torch.cuda.synchronize()
    assert B.sparse_mla_device_status() == 0
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"], d_v=d_v)
    return compare(out, lse, O, L)


@pytest.mark.parametrize("d_qk,d_v", DIMS)
@pytest.mark.parametrize("H", [8, 16, 128])
def test_dims_tiny(B, d_qk, d_v, H):
    cfg = synth.CONFIGS["tiny"].with_(H=H, T=96, pool=24, seed=300 + H)
    _check(B, _inputs(cfg, d_qk), d_v)


@pytest.mark.parametrize("d_qk,d_v", DIMS)
def test_dims_many_tokens_per_cta(B, d_qk, d_v):
    # more tokens than resident CTAs: the persistent walk with its one-token-ahead
    # compaction and gather; invalid slots and all-invalid tokens among them
    cfg = synth.CONFIGS["tiny"].with_(T=900, H=16, pool=300, ratio=1, topk=96, window=40, seed=310)
    x = _inputs(cfg, d_qk)
    x["idx"] = synth.inject_out_of_range(x["idx"].astype(np.int64), cfg.num_kv, 3, frac=0.2)
    x["idx"][4::9] = -1
    _check(B, x, d_v)


@pytest.mark.parametrize("d_qk,d_v", DIMS)
@pytest.mark.parametrize("T", [1, 4, 16])
def test_dims_decode_sized(B, d_qk, d_v, T):
    # split-TOPK path and the combine at the other value widths
    cfg = synth.CONFIGS[f"decode_h16_t{T}"]
    _check(B, _inputs(cfg, d_qk), d_v)


@pytest.mark.parametrize("d_qk,d_v", DIMS)
def test_dims_no_sink_and_long_lists(B, d_qk, d_v):
    cfg = synth.CONFIGS["tiny"].with_(T=64, H=16, pool=2400, ratio=1, topk=2048, window=200,
                                      sink=False, seed=320)
    _check(B, _inputs(cfg, d_qk), d_v)


def test_dims_512_is_the_op(B):
    cfg = synth.CONFIGS["tiny"].with_(seed=330)
    x = synth.make_inputs(cfg)
    q, kv, idx, sink = _dev(x)
    o1, l1 = B.sparse_mla_fwd_dims(q, kv, idx, sink, x["scale"])
    o2, l2 = B.sparse_mla_fwd(q, kv, idx, sink, x["scale"])
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


def test_dims_rejects_unsupported(B):
    cfg = synth.CONFIGS["tiny"].with_(seed=340)
    x = _inputs(cfg, 256)
    q, kv, idx, sink = _dev(x)
    with pytest.raises(B.SparseMLAError) as ei:
        B.sparse_mla_fwd_dims(q, kv, idx, sink)
    assert ei.value.status == 2
