"""The C ABI library on the host (CPU only, no compute call).

* the library loads and exports every function ``include/*.h`` declares;
* argument validation returns its documented status before any CUDA call
  (fake, never-dereferenced pointer values are enough to reach each check);
* the planner's kernel / split choices.
"""
import ctypes
import glob
import os
import re

import pytest

from sparse_mla_attention_token_gb300 import binding
from sparse_mla_attention_token_gb300 import build as bld

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(binding.LIB_PATH):
        bld.build()
    return binding.lib()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"\b([A-Za-z_][A-Za-z0-9_]*)\s*\(", src):
            n = m.group(1)
            if n.startswith("sparse_mla"):
                names.add(n)
    return names


def test_exports_every_declared_function(L):
    names = _declared_functions()
    assert {"sparse_mla_fwd", "sparse_mla_fwd_ex", "sparse_mla_strerror"} <= names
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"
    assert set(binding.SIGNATURES) >= names


def test_abi_version_and_strerror(L):
    assert binding.abi_version() == 1
    for code in range(0, 12):
        s = binding.strerror(code)
        assert s and s != "unknown status"
    assert binding.strerror(999) == "unknown status"


# fake device addresses: 16-byte aligned, far apart, never dereferenced
Q, KV, IDX, SINK, OUT, LSE = (0x10000000 * k for k in range(1, 7))


def _fwd(L, q=Q, kv=KV, idx=IDX, idt=0, sink=SINK, scale=0.0441941738, out=OUT, lse=LSE,
         T=4, H=16, num_kv=80, topk=64, splits=0, trace=None):
    return L.sparse_mla_fwd_ex(q, kv, idx, idt, sink, scale, out, lse, T, H, num_kv, topk,
                               None, splits, trace)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(out=None), 1), (dict(lse=None), 1), (dict(kv=None), 1),
    (dict(idx=None), 1),
    (dict(T=-1), 2), (dict(num_kv=-1), 2), (dict(num_kv=1 << 31), 2), (dict(topk=-3), 2),
    (dict(H=12), 3), (dict(H=256), 3), (dict(H=0), 3),
    (dict(idt=2), 4), (dict(idt=-1), 4),
    (dict(q=Q + 8), 5), (dict(kv=KV + 4), 5), (dict(out=OUT + 2), 5), (dict(lse=LSE + 2), 5),
    (dict(idx=IDX + 2), 5), (dict(idx=IDX + 4, idt=1), 5),
    (dict(scale=float("nan")), 6), (dict(scale=float("inf")), 6), (dict(scale=float("-inf")), 6),
    (dict(out=Q), 7), (dict(out=KV + 1024), 7), (dict(lse=IDX + 64), 7), (dict(lse=OUT + 16), 7),
    (dict(splits=65), 10), (dict(splits=-1), 10), (dict(topk=5000, splits=1), 10),
])
def test_validation_codes(L, kw, code):
    assert _fwd(L, **kw) == code


def test_empty_problem_is_ok_without_cuda(L):
    # T == 0: validated, nothing launched, no CUDA call
    assert _fwd(L, T=0, q=None, out=None, lse=None) == 0
    assert L.sparse_mla_fwd(None, None, None, 0, None, 1.0, None, None, 0, 8, 0, 0, None) == 0


def test_plan(L):
    # many CTAs: no split; small-head family for H <= 64
    assert binding.sparse_mla_plan(4096, 8, 640) == (0, 1, 1)
    assert binding.sparse_mla_plan(16384, 16, 640) == (0, 1, 1)
    # few tokens: split over topk (about 128 slots per split), plus the combine launch
    assert binding.sparse_mla_plan(4, 16, 640) == (0, 5, 2)
    assert binding.sparse_mla_plan(8, 128, 512) == (0, 4, 2)
    assert binding.sparse_mla_plan(16, 128, 512) == (1, 1, 1)   # the grid would exceed 2 x SMs
    # forced splits are honoured; topk beyond one CTA's list forces splits
    assert binding.sparse_mla_plan(4096, 16, 640, 4) == (0, 4, 2)
    assert binding.sparse_mla_plan(4096, 16, 5000)[1] >= 3
    assert binding.sparse_mla_plan(0, 16, 64)[2] == 0
    with pytest.raises(binding.SparseMLAError):
        binding.sparse_mla_plan(4096, 16, 5000, 1)


def test_static_scratch_entry_validates_before_cuda(L):
    f = L.sparse_mla_fwd_static_scratch
    args = [Q, KV, IDX, 0, SINK, 0.04, OUT, LSE]
    # 8192 partial rows at most: 2 splits x 300 tokens x 16 heads is over
    assert f(*args, 300, 16, 80, 64, None, 2) == 11
    assert f(*args, 64, 128, 80, 64, None, 0) == 11        # 2 x 64 x 128 = 16384
    assert f(*args, 4, 16, 80, 64, None, 1) == 10          # this path always splits
    assert f(*args, 4, 16, 80, 64, None, 65) == 10
    assert f(*args, 4, 12, 80, 64, None, 2) == 3
    assert f(None, KV, IDX, 0, SINK, 0.04, OUT, LSE, 4, 16, 80, 64, None, 2) == 1
    assert f(*args, 0, 16, 80, 64, None, 2) == 0           # T == 0: nothing to do


def test_host_call_workspace_and_validation_before_cuda(L):
    # workspace bytes: kv | q | idx | sink | out | lse, each rounded up to 256 bytes
    up = lambda x: (x + 255) // 256 * 256
    T, H, topk, nkv = 300, 16, 80, 64
    want = up(nkv * 1024) + up(T * H * 1024) + up(T * topk * 4) + up(H * 4) + up(T * H * 1024) + \
        up(T * H * 4)
    assert binding.sparse_mla_fwd_host_workspace(T, H, topk, nkv) == want
    assert binding.sparse_mla_fwd_host_workspace(T, H, topk, nkv, binding.SMLA_IDX_INT64, False) == \
        want - up(T * topk * 4) + up(T * topk * 8) - up(H * 4)
    with pytest.raises(binding.SparseMLAError) as ei:
        binding.sparse_mla_fwd_host_workspace(T, 12, topk, nkv)
    assert ei.value.status == 3
    f = L.sparse_mla_fwd_host
    args = [Q, KV, IDX, 0, SINK, 0.04, OUT, LSE, T, H, nkv, topk]
    WS = 0x7f0000400000
    assert f(*args, None, want, None) == 12                 # no workspace
    assert f(*args, WS, want - 1, None) == 12               # one byte short
    assert f(*args, WS + 16, want, None) == 12              # not 256-byte aligned
    assert f(Q, KV, IDX, 0, SINK, float("nan"), OUT, LSE, T, H, nkv, topk, WS, want, None) == 6
    assert f(Q, KV, IDX, 0, SINK, 0.04, Q, LSE, T, H, nkv, topk, WS, want, None) == 7
    assert f(*args[:8], 0, H, nkv, topk, None, 0, None) == 0   # T == 0: nothing to do
