"""GPU parity of the CUDA path against the fp64 oracle (needs a GB300).

Every call goes through the C ABI (``sparse_mla_fwd_ex`` via the ctypes
binding).  Small workloads are compared in full; full-size workloads run at
their real size, in the launch configuration the benchmark uses, and are
compared on sampled tokens the oracle computes one by one.
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


def _sample_tokens(T, n=256, seed=0):
    rng = np.random.default_rng(seed)
    head = np.arange(min(T, 48))
    tail = np.arange(max(0, T - 48), T)
    mid = rng.choice(T, size=min(T, n), replace=False)
    return np.unique(np.concatenate([head, tail, mid]))


def _run(B, x, splits=0, trace=False, **dev_kw):
    q, kv, idx, sink, keep = to_dev(x, DEV, **dev_kw)
    tr = torch.full(idx.shape, -7, dtype=torch.int64, device=DEV) if trace else None
    out, lse = B.sparse_mla_fwd(q, kv, idx, sink, x["scale"], num_splits=splits, read_trace=tr)
    torch.cuda.synchronize()
    assert B.sparse_mla_device_status() == 0
    return out, lse, tr


# ------------------------------------------------------------ the workloads
@pytest.mark.parametrize("name", ["tiny", "sweep_k32", "sweep_k128", "sweep_k256", "sweep_k640",
                                  "sweep_k640_nosink"])
def test_config_full(B, name):
    cfg = synth.CONFIGS[name]
    x = synth.make_inputs(cfg)
    out, lse, _ = _run(B, x)
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"])
    compare(out, lse, O, L)


@pytest.mark.parametrize("name", ["small_head", "h128", "h128_long"])
def test_config_full_size_sampled(B, name):
    cfg = synth.CONFIGS[name]
    x = synth.make_inputs(cfg)
    kw = {}
    if cfg.kv_offset_bytes:
        # kv > 2 GiB into one allocation, NaN guard rows right after num_kv
        kw = dict(kv_offset_bytes=cfg.kv_offset_bytes, guard_rows=8, guard_value=0x7FC0)
    out, lse, _ = _run(B, x, **kw)
    toks = _sample_tokens(cfg.T)
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"], tokens=toks)
    compare(out, lse, O, L, tokens=toks)


# ------------------------------------------------------------ index handling
def _tiny_x(seed=0, sink=True, **cfg_kw):
    cfg = synth.CONFIGS["tiny"].with_(seed=seed, sink=sink, **cfg_kw)
    return cfg, synth.make_inputs(cfg)


HEADS = [16, 128]   # the small-head kernel and the tcgen05 H = 128 kernel


@pytest.mark.parametrize("H", HEADS)
@pytest.mark.parametrize("variant", ["shuffled", "dups", "oob32", "oob64", "nosink", "sinkneg"])
def test_tiny_variants(B, variant, H):
    cfg, x = _tiny_x(seed=31, sink=(variant != "nosink"), H=H)
    if variant == "shuffled":
        x["idx"] = synth.shuffle_rows(x["idx"], 1)
    elif variant == "dups":
        x["idx"] = synth.inject_duplicates(x["idx"], cfg.num_kv, 2, frac=0.25)
    elif variant == "oob32":
        x["idx"] = synth.inject_out_of_range(x["idx"], cfg.num_kv, 3, frac=0.3)
    elif variant == "oob64":
        x["idx"] = synth.inject_out_of_range(x["idx"].astype(np.int64), cfg.num_kv, 4, frac=0.3)
    elif variant == "sinkneg":
        x["sink"] = np.full_like(x["sink"], -np.inf)
    out, lse, _ = _run(B, x)
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"])
    compare(out, lse, O, L)


def _expected_trace(idx, num_kv, splits):
    """Rows read per token, in gather order: within each of the call's slot
    ranges (ceil(topk / splits) slots each), the valid slots' rows in slot
    order, then -1 for the rest of the range (validity from the oracle)."""
    T, K = idx.shape
    valid = orc.valid_slots(idx, num_kv)
    want = np.full((T, K), -1, dtype=np.int64)
    chunk = -(-K // splits) if K else 0
    for t in range(T):
        for s in range(splits):
            j0, j1 = min(K, s * chunk), min(K, (s + 1) * chunk)
            rows = idx[t, j0:j1][valid[t, j0:j1]].astype(np.int64)
            want[t, j0:j0 + len(rows)] = rows
    return want


@pytest.mark.parametrize("H", HEADS)
@pytest.mark.parametrize("dtype", [np.int32, np.int64])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_read_trace_bit_exact(B, dtype, splits, H):
    # The trace is written where each copy's source address is formed: the row
    # every gather actually reads, recovered from that address.  It must list
    # exactly the valid slots' rows (duplicates included, in slot order) and
    # nothing else.
    cfg, x = _tiny_x(seed=5, H=H)
    x["idx"] = synth.inject_out_of_range(x["idx"].astype(dtype), cfg.num_kv, 9, frac=0.35)
    x["idx"] = synth.inject_duplicates(x["idx"], cfg.num_kv, 10, frac=0.1)
    out, lse, tr = _run(B, x, splits=splits, trace=True)
    used = B.sparse_mla_plan(cfg.T, cfg.H, cfg.topk, splits)[1]
    want = _expected_trace(x["idx"], cfg.num_kv, used)
    np.testing.assert_array_equal(tr.cpu().numpy(), want)


@pytest.mark.parametrize("H", HEADS)
def test_poisoned_rows_and_guard_never_read(B, H):
    cfg, x = _tiny_x(seed=6, H=H)
    idx = x["idx"].copy()
    idx[idx == 0] = -1
    used = np.unique(idx[(idx >= 0) & (idx < cfg.num_kv)])
    poison = np.setdiff1d(np.arange(cfg.num_kv), used)
    assert 0 in poison and len(poison) >= 1
    kv_p = x["kv"].copy()
    kv_p[poison] = 0x7FC0                  # NaN rows no valid slot names
    x2 = dict(x, idx=synth.inject_out_of_range(idx, cfg.num_kv, 10, frac=0.2), kv=kv_p)
    out, lse, _ = _run(B, x2, guard_rows=16, guard_value=0x7FC0)
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x2["idx"], x["sink"], x["scale"])
    compare(out, lse, O, L)


@pytest.mark.parametrize("H", HEADS)
@pytest.mark.parametrize("sink", [True, False])
def test_all_invalid_rows(B, sink, H):
    cfg, x = _tiny_x(seed=7, sink=sink, H=H)
    x["idx"] = np.full_like(x["idx"], -1)
    x["idx"][::3, 5] = cfg.num_kv
    x["idx"][1::4, 0] = 2 ** 31 - 1
    out, lse, _ = _run(B, x)
    assert torch.all(out == 0)
    L = lse.cpu().numpy()
    if sink:
        np.testing.assert_allclose(L, np.broadcast_to(x["sink"], L.shape), rtol=0, atol=2e-6)
    else:
        assert np.all(np.isneginf(L))


@pytest.mark.parametrize("H", HEADS)
def test_mixed_empty_and_full_rows(B, H):
    cfg, x = _tiny_x(seed=8, H=H)
    x["idx"][::2] = -1                      # every other token fully masked
    for splits in (0, 1, 4):
        out, lse, _ = _run(B, x, splits=splits)
        O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"])
        compare(out, lse, O, L)


# ------------------------------------------------------------ split-TOPK path
@pytest.mark.parametrize("splits", [1, 2, 3, 4, 7, 16])
def test_forced_splits_match_oracle(B, splits):
    cfg = synth.CONFIGS["sweep_k640"].with_(T=256)
    x = synth.make_inputs(cfg)
    out, lse, _ = _run(B, x, splits=splits)
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"])
    compare(out, lse, O, L)


def test_split_vs_unsplit(B):
    cfg = synth.CONFIGS["small_head"].with_(T=512)
    x = synth.make_inputs(cfg)
    o1, l1, _ = _run(B, x, splits=1)
    o4, l4, _ = _run(B, x, splits=4)
    d = (o1.float() - o4.float()).abs().max().item()
    assert d <= 2e-2
    fin = torch.isfinite(l1)
    assert torch.equal(fin, torch.isfinite(l4))
    assert (l1[fin] - l4[fin]).abs().max().item() <= 5e-3


# ------------------------------------------------------------ shapes and edges
@pytest.mark.parametrize("H", [8, 16, 32, 64, 128])
def test_head_counts(B, H):
    cfg = synth.CONFIGS["tiny"].with_(H=H, T=96, pool=24, seed=12)
    x = synth.make_inputs(cfg)
    out, lse, _ = _run(B, x)
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"])
    compare(out, lse, O, L)


@pytest.mark.parametrize("idx64", [False, True])
@pytest.mark.parametrize("H", [16, 64])
def test_tokens_pipelined_per_cta(B, H, idx64):
    # More tokens than resident CTAs, so each small-head CTA walks several tokens
    # and compacts / gathers the next one while computing the current one; lists
    # of three 32-slot tiles and fully invalid tokens in between (a token
    # without tiles between tokens with tiles).
    cfg = synth.CONFIGS["tiny"].with_(T=700, H=H, pool=300, ratio=1, topk=96, window=40,
                                      index_dtype="int64" if idx64 else "int32", seed=17)
    x = synth.make_inputs(cfg)
    idx = x["idx"].copy()
    idx[3::7] = -1
    idx[5::11, ::2] = cfg.num_kv + 7
    x["idx"] = idx
    out, lse, _ = _run(B, x)
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"])
    compare(out, lse, O, L)


@pytest.mark.parametrize("H", [8, 16])
def test_small_head_token_mix_per_cta(B, H):
    # Each small-head CTA walks several tokens whose valid counts rotate through
    # none, one tile, a tile and one slot, two tiles and three tiles: a warp gathers
    # and reads only its own columns, so a tile starts on a warp-level sync, and a
    # token's second tile goes into the stage the previous token staged its output
    # in (ordered by one block barrier).  H = 8 also exercises the warps whose rows
    # are all past the head count.
    cfg = synth.CONFIGS["tiny"].with_(T=1400, H=H, pool=400, ratio=1, topk=96, window=64,
                                      seed=23 + H)
    x = synth.make_inputs(cfg)
    idx = x["idx"].copy()
    keep = np.array([0, 20, 32, 33, 64, 70, 96])[np.arange(cfg.T) % 7]
    idx[np.arange(cfg.topk)[None, :] >= keep[:, None]] = -1
    x["idx"] = idx
    out, lse, _ = _run(B, x)
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"])
    compare(out, lse, O, L)


@pytest.mark.parametrize("H", HEADS)
@pytest.mark.parametrize("topk,window", [(1, 1), (3, 2), (67, 40), (130, 64), (2048, 150),
                                         (2500, 200)])
def test_ragged_topk(B, topk, window, H):
    cfg = synth.CONFIGS["tiny"].with_(T=150, H=H, pool=2400, ratio=1, topk=topk, window=window,
                                      seed=13)
    x = synth.make_inputs(cfg)
    out, lse, _ = _run(B, x)
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"])
    compare(out, lse, O, L)


@pytest.mark.parametrize("H", HEADS)
def test_topk_zero_and_empty_pool(B, H):
    cfg, x = _tiny_x(seed=14, H=H)
    x0 = dict(x, idx=np.zeros((cfg.T, 0), dtype=np.int32))
    out, lse, _ = _run(B, x0)
    assert torch.all(out == 0)
    np.testing.assert_allclose(lse.cpu().numpy(), np.broadcast_to(x["sink"], (cfg.T, cfg.H)),
                               atol=2e-6)
    # empty pool: num_kv = 0, every slot invalid
    xe = dict(x, kv=np.zeros((0, 512), dtype=np.uint16))
    out, lse, _ = _run(B, xe)
    assert torch.all(out == 0)


@pytest.mark.parametrize("H", HEADS)
def test_single_token(B, H):
    cfg, x = _tiny_x(seed=15, H=H)
    x1 = dict(x, q=x["q"][40:41], idx=x["idx"][40:41])
    out, lse, _ = _run(B, x1)
    O, L = orc.sparse_mla_fwd(x1["q"], x1["kv"], x1["idx"], x1["sink"], x1["scale"])
    compare(out, lse, O, L)


@pytest.mark.parametrize("H", HEADS)
def test_out_buffer_bit_identical_to_allocating_call(B, H):
    cfg, x = _tiny_x(seed=16, H=H)
    q, kv, idx, sink, _ = to_dev(x, DEV)
    o1, l1 = B.sparse_mla_fwd(q, kv, idx, sink, x["scale"])
    out = torch.full_like(q, float("nan"))
    lse = torch.full((cfg.T, cfg.H), float("nan"), device=DEV)
    o2, l2 = B.sparse_mla_fwd(q, kv, idx, sink, x["scale"], out=out, lse=lse)
    torch.cuda.synchronize()
    assert o2.data_ptr() == out.data_ptr() and l2.data_ptr() == lse.data_ptr()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


def test_binding_rejections(B):
    cfg, x = _tiny_x(seed=17)
    q, kv, idx, sink, _ = to_dev(x, DEV)
    with pytest.raises(RuntimeError, match="kv dtype mismatch"):
        B.sparse_mla_fwd(q, kv.to(torch.float16), idx, sink)
    with pytest.raises(RuntimeError, match="bfloat16"):
        B.sparse_mla_fwd(q.float(), kv, idx, sink)
    with pytest.raises(RuntimeError, match="CUDA tensor"):
        B.sparse_mla_fwd(q, kv.cpu(), idx, sink)
    with pytest.raises(RuntimeError, match="contiguous"):
        out = torch.empty(cfg.T, cfg.H, 1024, dtype=torch.bfloat16, device=DEV)[..., ::2]
        B.sparse_mla_fwd(q, kv, idx, sink, out=out)
    with pytest.raises(RuntimeError, match="int32 or int64"):
        B.sparse_mla_fwd(q, kv, idx.to(torch.int16), sink)
    with pytest.raises(B.SparseMLAError):
        B.sparse_mla_fwd(q, kv, idx, sink, scale=float("nan"))


@pytest.mark.parametrize("name", ["sweep_k256", "h128"])
def test_deterministic(B, name):
    cfg = synth.CONFIGS[name].with_(T=512)
    x = synth.make_inputs(cfg)
    a, la, _ = _run(B, x)
    b, lb, _ = _run(B, x)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(la.view(torch.int32), lb.view(torch.int32))


def test_h128_uses_tcgen05_kernel(B):
    assert B.sparse_mla_plan(4096, 128, 512) == (1, 1, 1)
    assert B.sparse_mla_plan(8192, 128, 1024) == (1, 1, 1)
    assert B.sparse_mla_plan(64, 128, 2500)[0] == 0      # beyond its row list: split path


@pytest.mark.parametrize("T", [1, 2, 75, 77, 153, 1000])
def test_h128_token_counts(B, T):
    # fewer tokens than clusters, one per cluster, several per persistent cluster;
    # one split forces the tcgen05 kernel even where the library would split a
    # decode-sized call
    cfg = synth.CONFIGS["h128"].with_(T=T, pool=max(8, T // 4), seed=40 + T)
    x = synth.make_inputs(cfg)
    out, lse, _ = _run(B, x, splits=1)
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"])
    compare(out, lse, O, L)


def test_h128_short_and_empty_tokens(B):
    # Persistent clusters walking tokens with no valid slot (every third), one
    # valid slot, 65 valid slots (a one-slot ragged tile) and full lists: the
    # per-token Q loads and epilogues across runs of one-tile and empty tokens.
    cfg = synth.CONFIGS["h128"].with_(T=400, pool=100, seed=47)
    x = synth.make_inputs(cfg)
    idx = x["idx"].copy()
    valid = orc.valid_slots(idx, cfg.num_kv)
    for t in range(cfg.T):
        pos = np.flatnonzero(valid[t])
        if t % 3 == 0:
            idx[t] = -1
        elif t % 5 == 1:
            idx[t, pos[1:]] = -1
        elif t % 7 == 2:
            idx[t, pos[65:]] = -1
    x["idx"] = idx
    out, lse, _ = _run(B, x)
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"])
    compare(out, lse, O, L)


def _bf16_of(f):
    return synth.bf16_bits(np.asarray(f, np.float32))


@pytest.mark.parametrize("splits", [0, 2])
@pytest.mark.parametrize("case", ["q_times_4", "common_shift_25"])
def test_h128_large_logits(B, case, splits):
    # Logits well above the N(0,1) recipe's: q scaled by 4 (natural scores of
    # standard deviation 4), or a score component of about 25 shared by every
    # kv row of a token (a direction common to q and kv).  The tcgen05 kernel
    # rounds each half's partial scores to fp16 after taking the row's largest
    # off, so a shared component costs it no precision.
    cfg = synth.CONFIGS["h128"].with_(T=200, seed=43)
    x = synth.make_inputs(cfg)
    q = orc.bf16_to_f64(x["q"])
    if case == "q_times_4":
        x["q"] = _bf16_of(4.0 * q)          # exact: a power of two
    else:
        u = np.zeros(512)
        u[0::2] = 1.0 / np.sqrt(256.0)
        x["kv"] = _bf16_of(orc.bf16_to_f64(x["kv"]) + 4.0 * u)
        x["q"] = _bf16_of(q + (25.0 / 4.0) * np.sqrt(512.0) * u)
    out, lse, _ = _run(B, x, splits=splits)
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"])
    # Peaked softmax puts |O| up to about 5, where half a bf16 step of the
    # output alone is 2^-6: O is held to the bar plus one bf16 step of |O|
    # (output rounding and P's bf16 rounding); lse and the cosine to the bar.
    og = out.float().cpu().numpy().astype(np.float64)
    err = np.abs(og - O)
    print(f"large logits {case} splits={splits}: max|dO|={err.max():.3e} "
          f"max|O|={np.abs(O).max():.3f} max(|dO|/(2e-2+2^-8|O|))="
          f"{(err / (2e-2 + 2.0 ** -8 * np.abs(O))).max():.3f}")
    assert np.all(err <= 2e-2 + 2.0 ** -8 * np.abs(O))
    compare(out, lse, O, L, o_tol=np.inf)


@pytest.mark.parametrize("scale", [-1.0 / np.sqrt(512.0), -2.0 / np.sqrt(512.0), 0.0])
@pytest.mark.parametrize("H,splits", [(16, 0), (128, 0), (128, 2)])
def test_scale_sign_and_zero(B, H, splits, scale):
    # Scale is an argument and may be negative or zero (PR #6002 dropped the
    # positivity check).  A negative scale turns each row's smallest raw score
    # into its largest logit, which the H = 128 kernel's row maximum has to
    # follow; zero makes every score 0 (weights 1 / (n + e^sink)).  Lists of up
    # to 150 slots: several 64-slot tiles with a ragged last one.
    cfg = synth.CONFIGS["tiny"].with_(T=200, H=H, pool=200, ratio=1, topk=150, window=48, seed=23)
    x = synth.make_inputs(cfg)
    x["scale"] = float(scale)
    out, lse, _ = _run(B, x, splits=splits)
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"])
    compare(out, lse, O, L)


def test_h128_vs_split_path(B):
    cfg = synth.CONFIGS["h128"].with_(T=300, seed=41)
    x = synth.make_inputs(cfg)
    o1, l1, _ = _run(B, x, splits=0)     # tcgen05 kernel
    o2, l2, _ = _run(B, x, splits=2)     # small-head kernel, split-TOPK + combine
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    fin = torch.isfinite(l1)
    assert torch.equal(fin, torch.isfinite(l2))
    assert (l1[fin] - l2[fin]).abs().max().item() <= 5e-3


# ------------------------------------------------------------ decode-sized calls
@pytest.mark.parametrize("H", [8, 16, 128])
@pytest.mark.parametrize("T", [1, 2, 4, 8, 16])
def test_decode_sized_calls(B, H, T):
    # the last T tokens of an 8192-token context, with the library's split choice
    # (the split-TOPK path for these sizes, the tcgen05 kernel for H=128 at T=16)
    cfg = synth.CONFIGS[f"decode_h{H}_t{T}"]
    x = synth.make_inputs(cfg)
    out, lse, _ = _run(B, x)
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"])
    compare(out, lse, O, L)


def test_decode_plan():
    from sparse_mla_attention_token_gb300 import binding
    for H, want in ((8, 5), (16, 5), (128, 4)):
        for T in (1, 4, 8):
            cfg = synth.CONFIGS[f"decode_h{H}_t{T}"]
            assert binding.sparse_mla_plan(cfg.T, cfg.H, cfg.topk) == (0, want, 2)
    cfg = synth.CONFIGS["decode_h128_t16"]
    assert binding.sparse_mla_plan(cfg.T, cfg.H, cfg.topk) == (1, 1, 1)


def test_glm_shaped_call_sampled(B):
    # 16K tokens, 16 heads, top-k 2048, the sequence 2 GiB into a shared pool whose
    # other rows are NaN: sampled tokens against the oracle, no NaN anywhere
    cfg = synth.CONFIGS["glm_k2048"]
    x = synth.make_inputs(cfg)
    out, lse, _ = _run(B, x)
    toks = _sample_tokens(cfg.T, n=96)
    O, L = orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"], tokens=toks)
    compare(out, lse, O, L, tokens=toks)
    assert not torch.isnan(out).any()
