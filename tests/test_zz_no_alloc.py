"""The allocation-free entry point against the regular one (needs a GB300).

``sparse_mla_fwd_static_scratch`` serves callers that may not allocate device
memory while they run (a fixed memory budget, a window in which no allocation
may happen, an allocator owned by another runtime): it runs the split-TOPK path
with its partial results in the library's fixed scratch array.  Two calls in a
row, with different shapes and inputs, must each agree with
``sparse_mla_fwd_ex`` (the same split count: the same kernels, so bit for
bit), with the regular ``sparse_mla_fwd`` and with the fp64 oracle within the
parity tolerances.  A repeated call must leave the device's free memory
unchanged.  The file is named to be collected last, so a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest

from oracle import oracle as orc
from sparse_mla_attention_token_gb300 import synth
from tests.parity import compare, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_attention_token_gb300 import binding
    binding.lib()
    return binding


def _as_ref(out, lse):
    return (out.float().cpu().numpy().astype(np.float64),
            lse.float().cpu().numpy().astype(np.float64))


def _one_call(B, x, num_splits, want_splits):
    q, kv, idx, sink, _ = to_dev(x, DEV)
    T, H, _ = q.shape
    out = torch.full_like(q, float("nan"))
    lse = torch.full((T, H), float("nan"), dtype=torch.float32, device=DEV)
    o_s, l_s = B.sparse_mla_fwd_static_scratch(q, kv, idx, out, lse, sink, x["scale"],
                                               num_splits=num_splits)
    torch.cuda.synchronize()
    assert o_s.data_ptr() == out.data_ptr()
    # same split count through the allocating entry point: the same kernels
    o_x, l_x = B.sparse_mla_fwd(q, kv, idx, sink, x["scale"], num_splits=want_splits)
    # the regular call (the library's own kernel choice)
    o_r, l_r = B.sparse_mla_fwd(q, kv, idx, sink, x["scale"])
    torch.cuda.synchronize()
    assert B.sparse_mla_device_status() == 0
    assert torch.equal(o_s.view(torch.int16), o_x.view(torch.int16))
    assert torch.equal(l_s.view(torch.int32), l_x.view(torch.int32))
    compare(o_s, l_s, *_as_ref(o_r, l_r))
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"])
    compare(o_s, l_s, O, L)
    # the same call again allocates nothing: the device's free memory is unchanged
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    B.sparse_mla_fwd_static_scratch(q, kv, idx, out, lse, sink, x["scale"],
                                    num_splits=num_splits)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.equal(out.view(torch.int16), o_x.view(torch.int16))


def test_static_scratch_two_calls_in_a_row(B):
    # first call: 64 tokens, 16 heads, library split count (2)
    cfg1 = synth.CONFIGS["tiny"].with_(seed=71)
    x1 = synth.make_inputs(cfg1)
    _one_call(B, x1, num_splits=0, want_splits=2)
    # second call: a decode-sized H=128 call with int64 indices, some out of range
    cfg2 = synth.CONFIGS["h128"].with_(T=8, pool=64, seed=72, index_dtype="int64")
    x2 = synth.make_inputs(cfg2)
    x2["idx"] = synth.inject_out_of_range(x2["idx"], cfg2.num_kv, 5, frac=0.2)
    _one_call(B, x2, num_splits=4, want_splits=4)


def test_static_scratch_rejects_oversize(B):
    cfg = synth.CONFIGS["tiny"].with_(T=300, seed=73)
    x = synth.make_inputs(cfg)
    q, kv, idx, sink, _ = to_dev(x, DEV)
    out = torch.empty_like(q)
    lse = torch.empty((cfg.T, cfg.H), dtype=torch.float32, device=DEV)
    with pytest.raises(B.SparseMLAError) as ei:
        B.sparse_mla_fwd_static_scratch(q, kv, idx, out, lse, sink, x["scale"], num_splits=2)
    assert ei.value.status == 11
