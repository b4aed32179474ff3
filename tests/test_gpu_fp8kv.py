"""GPU parity of the fp8-cache forward against the fp64 fp8-cache oracle (needs a GB300).

``sparse_mla_fwd_fp8kv`` through the C ABI: kv rows of e4m3 codes with one fp32
scale per 128-column block (the layout this library reads an fp8 cache in; the
pages leave the fp8 cache out of the prefill change), against
``oracle.fp8kv``, which decodes the codes exactly and applies the op's
definition.  Same bar as the bf16 op.
"""
import numpy as np
import pytest

from oracle import fp8kv
from sparse_mla_attention_token_gb300 import synth
from tests.parity import compare

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


def _run(B, x, kv8, sc, tokens=None):
    q = torch.from_numpy(x["q"].view(np.int16)).view(torch.bfloat16).to(DEV)
    k8 = torch.from_numpy(kv8).to(DEV)
    s = torch.from_numpy(sc).to(DEV)
    idx = torch.from_numpy(x["idx"]).to(DEV)
    sink = None if x["sink"] is None else torch.from_numpy(x["sink"]).to(DEV)
    out, lse = B.sparse_mla_fwd_fp8kv(q, k8, s, idx, sink, x["scale"])
    torch.cuda.synchronize()
    assert B.sparse_mla_device_status() == 0
    O, L = fp8kv.sparse_mla_fwd_fp8kv(x["q"], kv8, sc, x["idx"], x["sink"], x["scale"],
                                      tokens=tokens)
    return compare(out, lse, O, L, tokens=tokens)


@pytest.mark.parametrize("H", [8, 16, 128])
def test_fp8_tiny(B, H):
    cfg = synth.CONFIGS["tiny"].with_(H=H, T=96, pool=24, seed=400 + H)
    x = synth.make_inputs(cfg)
    _run(B, x, *synth.fp8_cache(x["kv"]))


@pytest.mark.parametrize("variant", ["oob64", "dups", "nosink", "empty_tokens", "nan_unused"])
def test_fp8_variants(B, variant):
    cfg = synth.CONFIGS["tiny"].with_(T=300, H=16, pool=200, ratio=1, topk=150, window=48,
                                      seed=410)
    x = synth.make_inputs(cfg)
    kv8, sc = synth.fp8_cache(x["kv"])
    if variant == "oob64":
        x["idx"] = synth.inject_out_of_range(x["idx"].astype(np.int64), cfg.num_kv, 3, frac=0.3)
    elif variant == "dups":
        x["idx"] = synth.inject_duplicates(x["idx"], cfg.num_kv, 4, frac=0.2)
    elif variant == "nosink":
        x["sink"] = None
    elif variant == "empty_tokens":
        x["idx"][::4] = -1
    elif variant == "nan_unused":
        used = np.unique(x["idx"][(x["idx"] >= 0) & (x["idx"] < cfg.num_kv)])
        unused = np.setdiff1d(np.arange(cfg.num_kv), used)
        kv8[unused] = 0x7F                 # NaN codes in rows no valid slot names
        sc[unused] = np.nan
    _run(B, x, kv8, sc)


@pytest.mark.parametrize("H", [8, 16])
def test_fp8_token_mix_per_cta(B, H):
    # Several tokens per CTA with valid counts rotating through none, one tile, a
    # tile and one slot, two and three tiles: each warp gathers, decodes and scales
    # its own columns (its block's scales in its own slot) and a token's first tile
    # waits for the previous token's staged output to be copied out.
    cfg = synth.CONFIGS["tiny"].with_(T=1400, H=H, pool=400, ratio=1, topk=96, window=64,
                                      seed=430 + H)
    x = synth.make_inputs(cfg)
    keep = np.array([0, 20, 32, 33, 64, 70, 96])[np.arange(cfg.T) % 7]
    x["idx"][np.arange(cfg.topk)[None, :] >= keep[:, None]] = -1
    _run(B, x, *synth.fp8_cache(x["kv"]))


@pytest.mark.parametrize("variant", ["wide_scales", "wide_scales_t4", "big_q", "tiny_q"])
def test_fp8_value_ranges(B, variant):
    # the fp16 operands' range handling: Q far outside fp16's range either way (the
    # softmax scale compensates, so the logits keep their size), and block scales that
    # differ by up to 2^12 between rows, so that the largest scale changes from tile to tile
    # (600 tokens: one launch without splits; wide_scales_t4: four tokens, a split launch
    # and the combine)
    cfg = synth.CONFIGS["tiny"].with_(T=4 if variant.endswith("t4") else 600, H=16, pool=400,
                                      ratio=1, topk=300, window=64, seed=430)
    x = synth.make_inputs(cfg)
    kv8, sc = synth.fp8_cache(x["kv"])
    if variant.startswith("wide_scales"):
        e = np.random.default_rng(431).integers(-6, 7, size=sc.shape)
        sc = (sc * np.exp2(e)).astype(np.float32)
    else:
        k = 20 if variant == "big_q" else -30
        q = synth.bf16_bits_to_f32(x["q"]) * np.float32(2.0 ** k)
        x["q"] = synth.bf16_bits(q.astype(np.float32))
        x["scale"] = float(np.float32(x["scale"] * 2.0 ** -k))
    q = torch.from_numpy(x["q"].view(np.int16)).view(torch.bfloat16).to(DEV)
    out, lse = B.sparse_mla_fwd_fp8kv(q, torch.from_numpy(kv8).to(DEV), torch.from_numpy(sc).to(DEV),
                                      torch.from_numpy(x["idx"]).to(DEV),
                                      torch.from_numpy(x["sink"]).to(DEV), x["scale"])
    torch.cuda.synchronize()
    O, L = fp8kv.sparse_mla_fwd_fp8kv(x["q"], kv8, sc, x["idx"], x["sink"], x["scale"])
    # bf16 output rounding grows with |O|: the O bar scales with the largest magnitude
    res = compare(out, lse, O, L, o_tol=2e-2 * max(1.0, float(np.abs(O).max())))
    print(variant, res, "max|O|", float(np.abs(O).max()))


@pytest.mark.parametrize("T", [1, 4, 16])
def test_fp8_decode_sized(B, T):
    cfg = synth.CONFIGS[f"decode_h16_t{T}"]
    x = synth.make_inputs(cfg)
    _run(B, x, *synth.fp8_cache(x["kv"]))


def test_fp8_sweep_k640_sampled(B):
    cfg = synth.CONFIGS["sweep_k640"]
    x = synth.make_inputs(cfg)
    toks = np.unique(np.concatenate([np.arange(40), np.arange(cfg.T - 40, cfg.T),
                                     np.random.default_rng(0).choice(cfg.T, 120, replace=False)]))
    _run(B, x, *synth.fp8_cache(x["kv"]), tokens=toks)


def test_fp8_rejections(B):
    cfg = synth.CONFIGS["tiny"].with_(seed=420)
    x = synth.make_inputs(cfg)
    kv8, sc = synth.fp8_cache(x["kv"])
    q = torch.from_numpy(x["q"].view(np.int16)).view(torch.bfloat16).to(DEV)
    idx = torch.from_numpy(x["idx"]).to(DEV)
    k8 = torch.from_numpy(kv8).to(DEV)
    with pytest.raises(RuntimeError, match="kv_scale"):
        B.sparse_mla_fwd_fp8kv(q, k8, torch.ones(cfg.num_kv, 2, device=DEV), idx)
    # the bf16 entry rejects an fp8 pool with a dtype error
    with pytest.raises(RuntimeError, match="kv dtype mismatch"):
        B.sparse_mla_fwd(q, k8.view(torch.float8_e4m3fn), idx)
