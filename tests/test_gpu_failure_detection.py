"""Failure detection without a GPU fault (needs a GB300).

Every wait in the H=128 kernel is bounded: on expiry it records an error word
and returns, and the host reads the status with ``sparse_mla_device_status``.
The self-test kernel makes exactly such a wait run out (an mbarrier nothing
arrives at); the test checks the status is reported once, is cleared by the
read, and that the context keeps working for a normal forward call.
"""
import numpy as np
import pytest

from oracle import oracle as orc
from sparse_mla_attention_token_gb300 import synth
from tests.parity import compare, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_attention_token_gb300 import binding
    binding.lib()
    return binding


def test_bounded_wait_expiry_is_reported_and_cleared(B):
    assert B.sparse_mla_device_status() == 0
    B.sparse_mla_selftest_wait_timeout()
    assert B.sparse_mla_device_status() == 9          # SMLA_ERR_DEVICE_TIMEOUT
    assert B.sparse_mla_device_status() == 0          # read clears it
    # the context is healthy: a normal H=128 call still matches the oracle
    cfg = synth.CONFIGS["h128"].with_(T=40, pool=16, seed=91)
    x = synth.make_inputs(cfg)
    q, kv, idx, sink, _ = to_dev(x, "cuda:0")
    out, lse = B.sparse_mla_fwd(q, kv, idx, sink, x["scale"])
    torch.cuda.synchronize()
    assert B.sparse_mla_device_status() == 0
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"])
    compare(out, lse, O, L)
