"""The host-buffer entry point against the device-buffer one (needs a GB300).

``sparse_mla_fwd_host`` copies host inputs in, runs the forward in token
chunks overlapped with the copies and copies O and lse back.  Every chunk
runs the kernel and split count of the whole call, so the results must be
bit-identical to ``sparse_mla_fwd`` on the same inputs; they are also checked
against the oracle.
"""
import numpy as np
import pytest

from sparse_mla_attention_token_gb300 import synth
from tests.parity import compare, to_dev
import oracle.oracle as orc

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


def _host(x):
    q = torch.from_numpy(x["q"].view(np.int16)).view(torch.bfloat16).pin_memory()
    kv = torch.from_numpy(x["kv"].view(np.int16)).view(torch.bfloat16).pin_memory()
    idx = torch.from_numpy(x["idx"]).pin_memory()
    sink = torch.from_numpy(x["sink"]).pin_memory() if x["sink"] is not None else None
    return q, kv, idx, sink


@pytest.mark.parametrize("name,T,seed,i64", [("h128", 600, 81, False), ("h128", 100, 82, False),
                                             ("h128", 300, 85, True), ("small_head", 1100, 83, False),
                                             ("tiny", 64, 84, True)])
def test_host_call_bit_identical(B, name, T, seed, i64):
    cfg = synth.CONFIGS[name].with_(T=T, seed=seed, index_dtype="int64" if i64 else "int32")
    x = synth.make_inputs(cfg)
    q, kv, idx, sink = _host(x)
    out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    lse = torch.full((cfg.T, cfg.H), float("nan"), dtype=torch.float32).pin_memory()
    nb = B.sparse_mla_fwd_host_workspace(cfg.T, cfg.H, cfg.topk, cfg.num_kv,
                                         B.SMLA_IDX_INT64 if i64 else B.SMLA_IDX_INT32,
                                         sink is not None)
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
    B.sparse_mla_fwd_host(q, kv, idx, out, lse, sink, ws, x["scale"])
    torch.cuda.current_stream().synchronize()
    assert B.sparse_mla_device_status() == 0
    dq, dkv, didx, dsink, _ = to_dev(x, DEV)
    o_d, l_d = B.sparse_mla_fwd(dq, dkv, didx, dsink, x["scale"])
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), o_d.cpu().view(torch.int16))
    assert torch.equal(lse.view(torch.int32), l_d.cpu().view(torch.int32))
    toks = list(range(0, cfg.T, max(1, cfg.T // 40)))
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"], tokens=toks)
    compare(out[toks].to(DEV), lse[toks].to(DEV), O, L)
