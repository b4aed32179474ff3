"""GPU parity of the training backward against the fp64 backward oracle (needs a GB300).

Every call goes through the C ABI (``sparse_mla_bwd`` via the ctypes binding).
The forward's O and lse that the backward consumes come from the fp64 oracle
(rounded to bf16 / fp32, as the forward stores them), so that the comparison
isolates the backward; one test also chains the CUDA forward into the CUDA
backward.

Bar (derived in the design notes from the arithmetic): P and scale * dS are
rounded to bf16 (2^-9 relative) before the two contractions over them, all
sums are fp32.  Per tensor: cosine >= 0.9999 and max|delta| <= 1e-2 * max|ref|
for dq and dkv; dsink to 1e-2 of its largest magnitude (plus 1e-6).
"""
import numpy as np
import pytest

from oracle import backward as obwd
from oracle import oracle as orc
from sparse_mla_attention_token_gb300 import synth
from tests.parity import to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"
COS = 0.9999
REL = 1e-2


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_attention_token_gb300 import binding
    binding.lib()
    return binding


def _bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


def _cos(a, b):
    a, b = a.ravel(), b.ravel()
    n = np.sqrt((a * a).sum() * (b * b).sum())
    return float((a * b).sum() / n) if n > 0 else float(np.abs(a).max() == np.abs(b).max() == 0)


def _check(name, got, ref, rel=REL, atol=0.0):
    assert not np.any(np.isnan(got)), f"NaN in {name}"
    scale = np.abs(ref).max()
    err = np.abs(got - ref).max() if ref.size else 0.0
    assert err <= rel * scale + atol, f"{name}: max|d| {err:.3e} > {rel} * {scale:.3e}"
    if scale > 0:
        c = _cos(got, ref)
        assert c >= COS, f"{name}: cos {c}"
    return err, scale


def _run(B, x, dout_bits, out=None, lse=None):
    """CUDA backward with the oracle forward's O / lse unless given."""
    if out is None:
        O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"])
        out = _bf16_dev(synth.bf16_bits(O.astype(np.float32)))
        lse = torch.from_numpy(L.astype(np.float32)).to(DEV)
    q, kv, idx, sink, _ = to_dev(x, DEV)
    dq, dkv, ds = B.sparse_mla_bwd(q, kv, idx, out, lse, _bf16_dev(dout_bits), sink, x["scale"])
    torch.cuda.synchronize()
    return (dq.cpu().numpy().astype(np.float64), dkv.cpu().numpy().astype(np.float64),
            None if ds is None else ds.cpu().numpy().astype(np.float64))


def _compare(B, x, dout):
    dq, dkv, ds = _run(B, x, dout)
    rq, rkv, rs = obwd.sparse_mla_bwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"], dout)
    _check("dq", dq, rq)
    _check("dkv", dkv, rkv)
    if x["sink"] is not None:
        _check("dsink", ds, rs, atol=1e-6)
    return dq, dkv, ds


@pytest.mark.parametrize("H", [8, 16, 32, 64, 128])
def test_bwd_head_counts(B, H):
    cfg = synth.CONFIGS["tiny"].with_(H=H, T=96, pool=24, seed=200 + H)
    x = synth.make_inputs(cfg)
    _compare(B, x, synth.make_dout(cfg))


@pytest.mark.parametrize("variant", ["dups", "oob64", "nosink", "sinkneg", "empty_tokens",
                                     "shuffled"])
def test_bwd_variants(B, variant):
    cfg = synth.CONFIGS["tiny"].with_(seed=210, T=80)
    x = synth.make_inputs(cfg)
    if variant == "dups":
        x["idx"] = synth.inject_duplicates(x["idx"], cfg.num_kv, 3, frac=0.3)
    elif variant == "oob64":
        x["idx"] = synth.inject_out_of_range(x["idx"].astype(np.int64), cfg.num_kv, 4, frac=0.3)
    elif variant == "nosink":
        x["sink"] = None
    elif variant == "sinkneg":
        x["sink"] = np.full(cfg.H, -np.inf, dtype=np.float32)
    elif variant == "empty_tokens":
        x["idx"][::3] = -1
    elif variant == "shuffled":
        x["idx"] = synth.shuffle_rows(x["idx"], 6)
    dq, dkv, ds = _compare(B, x, synth.make_dout(cfg))
    if variant == "sinkneg":
        assert np.all(ds == 0)
    if variant == "empty_tokens":
        assert np.all(dq[::3] == 0)


@pytest.mark.parametrize("topk,window", [(1, 1), (67, 40), (700, 200), (2048, 300)])
def test_bwd_ragged_topk(B, topk, window):
    cfg = synth.CONFIGS["tiny"].with_(T=40, H=16, pool=2400, ratio=1, topk=topk, window=window,
                                      seed=220)
    x = synth.make_inputs(cfg)
    _compare(B, x, synth.make_dout(cfg))


def test_bwd_h128_sampled_rows(B):
    # the backward's page shape at a reduced token count (T=512, H=128, topk 512)
    cfg = synth.CONFIGS["h128"].with_(T=512, pool=128, seed=230)
    x = synth.make_inputs(cfg)
    _compare(B, x, synth.make_dout(cfg))


@pytest.mark.parametrize("topk,window", [(300, 128), (1024, 256)])
def test_bwd_h128_tile_boundaries(B, topk, window):
    # H = 128 on the tcgen05 kernels: topk 300 ends in a partial 128-slot tile (its
    # rows stored lane by lane, the full tiles by TMA boxes); topk 1024 with int64
    # indices is the page's second backward shape at reduced T
    # (2048 earlier context rows: every slot of every token is valid)
    cfg = synth.CONFIGS["h128"].with_(T=192, pos0=2048, pool=1200, ratio=2, topk=topk,
                                      window=window, seed=235 + topk)
    x = synth.make_inputs(cfg)
    if topk == 1024:
        x["idx"] = x["idx"].astype(np.int64)
    _compare(B, x, synth.make_dout(cfg))


def test_bwd_unused_rows_are_zero_and_shared_pool(B):
    # the sequence's rows sit 3000 rows into a shared pool; the NaN rows of the
    # other sequences are never read and their gradient rows are exactly zero
    cfg = synth.CONFIGS["tiny"].with_(seed=240, base_row=3000)
    x = synth.make_inputs(cfg)
    dq, dkv, ds = _compare(B, x, synth.make_dout(cfg))
    used = np.unique(x["idx"][(x["idx"] >= 0) & (x["idx"] < cfg.num_kv)])
    unused = np.setdiff1d(np.arange(cfg.num_kv), used)
    assert np.all(dkv[unused] == 0)


def test_bwd_after_cuda_forward(B):
    # the CUDA forward's own O and lse feed the CUDA backward (both kernels of the
    # forward: the tcgen05 H=128 kernel here)
    cfg = synth.CONFIGS["h128"].with_(T=96, pool=24, seed=250)
    x = synth.make_inputs(cfg)
    q, kv, idx, sink, _ = to_dev(x, DEV)
    out, lse = B.sparse_mla_fwd(q, kv, idx, sink, x["scale"])
    dout = synth.make_dout(cfg)
    dq, dkv, ds = _run(B, x, dout, out=out, lse=lse)
    rq, rkv, rs = obwd.sparse_mla_bwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"], dout)
    _check("dq", dq, rq)
    _check("dkv", dkv, rkv)
    _check("dsink", ds, rs, atol=1e-6)


def test_bwd_zero_tokens_zero_gradients(B):
    cfg = synth.CONFIGS["tiny"].with_(seed=260)
    x = synth.make_inputs(cfg)
    q, kv, idx, sink, _ = to_dev(x, DEV)
    q0, idx0 = q[:0], idx[:0]
    out0 = torch.empty_like(q0)
    lse0 = torch.empty((0, cfg.H), dtype=torch.float32, device=DEV)
    dkv = torch.full(kv.shape, 7.0, dtype=torch.float32, device=DEV)
    dsink = torch.full((cfg.H,), 7.0, dtype=torch.float32, device=DEV)
    B.sparse_mla_bwd(q0, kv, idx0, out0, lse0, out0, sink, x["scale"], dkv=dkv, dsink=dsink)
    torch.cuda.synchronize()
    assert torch.all(dkv == 0) and torch.all(dsink == 0)


def test_bwd_rejections(B):
    cfg = synth.CONFIGS["tiny"].with_(seed=270)
    x = synth.make_inputs(cfg)
    q, kv, idx, sink, _ = to_dev(x, DEV)
    out = torch.empty_like(q)
    lse = torch.zeros((cfg.T, cfg.H), dtype=torch.float32, device=DEV)
    small = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(B.SparseMLAError) as ei:
        B.sparse_mla_bwd(q, kv, idx, out, lse, out, sink, workspace=small)
    assert ei.value.status == 12
    buf = torch.zeros((cfg.T, cfg.H, 512), dtype=torch.float32, device=DEV)
    out_in_dq = buf.view(torch.bfloat16).view(-1)[:q.numel()].view(q.shape)   # O inside dq
    with pytest.raises(B.SparseMLAError) as ei:
        B.sparse_mla_bwd(q, kv, idx, out_in_dq, lse, out, sink, dq=buf)
    assert ei.value.status == 7
    big = synth.CONFIGS["tiny"].with_(topk=2049, window=32)
    with pytest.raises(B.SparseMLAError):
        B.sparse_mla_bwd_workspace(big.T, big.H, big.topk, big.num_kv)
