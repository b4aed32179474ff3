"""The oracle against the golden fixtures (CPU only).

The fixtures under ``tests/golden/`` hold small problems whose outputs follow
from the op's definition by hand algebra ("Sparse MLA training backward", aiter
PR #4766, section "Contract" and review notes; "Tuned sparse MLA prefill for
DSv4.1-Flash TP4; fix attn_sink in Triton fallback", aiter PR #6002,
description items "attn_sink", "int64 indices", "Invalid KV rows"), evaluated
at 50 digits.  The planted oracle mistakes of ``test_oracle_mutations`` must
also each fail against the fixtures alone.
"""
import numpy as np
import pytest

from oracle import oracle as orc
from tests.golden import fixtures
from tests.test_oracle_mutations import MUTANTS, _mutant_token_forward


def _oracle_agrees(fx) -> bool:
    O, L = orc.sparse_mla_fwd(fx["q"], fx["kv"], fx["idx"], fx["sink"], fx["scale"])
    fin = np.isfinite(fx["lse"])
    if not np.array_equal(fin, np.isfinite(L)):
        return False
    return bool(np.allclose(O, fx["O"], rtol=1e-12, atol=1e-14)
                and np.allclose(L[fin], fx["lse"][fin], rtol=1e-13, atol=1e-13))


@pytest.mark.parametrize("name", fixtures.NAMES)
def test_fixture_is_well_formed(name):
    fx = fixtures.load(name)
    T, H = fx["lse"].shape
    assert fx["q"].shape == (T, H, 512) and fx["O"].shape == (T, H, 512)
    assert fx["cite"] and fx["derivation"]
    # each O row is a weighted mean of kv rows with weights summing to at most 1
    kv = orc.bf16_to_f64(fx["kv"])
    bound = np.abs(kv).max(axis=0)
    assert np.all(np.abs(fx["O"]) <= bound[None, None, :] * (1 + 1e-12))


@pytest.mark.parametrize("name", fixtures.NAMES)
def test_oracle_matches_golden(name):
    assert _oracle_agrees(fixtures.load(name))


@pytest.mark.parametrize("kind", MUTANTS)
def test_golden_catches_planted_mistake(kind, monkeypatch):
    fxs = [fixtures.load(n) for n in fixtures.NAMES]
    monkeypatch.setattr(orc, "token_forward", _mutant_token_forward(kind))
    caught = []
    for fx in fxs:
        try:
            caught.append(not _oracle_agrees(fx))
        except Exception:
            caught.append(True)
    assert any(caught), f"golden fixtures miss the planted mistake {kind!r}"


@pytest.mark.parametrize("name", fixtures.NAMES)
def test_fixture_file_is_what_its_generator_writes(name):
    """The stored JSON is exactly the closed-form generator's output (no hand edits)."""
    pytest.importorskip("mpmath")
    import json
    import os
    from tests.golden import make_golden
    fx = getattr(make_golden, name)()
    with open(os.path.join(os.path.dirname(make_golden.__file__), name + ".json")) as f:
        stored = json.load(f)
    assert json.loads(json.dumps(fx)) == stored
