"""Pins for the oracle's greedy verification (the T -> 0 limit of the verify
step of [P1] "Speculative decoding: draft first, then verify").

  * The limit itself: with logits that differ by at least 1 and T = 1e-3,
    exp(-1/T) underflows to 0 in double, so the sampled oracle's softmax is
    exactly one-hot and it must give the greedy oracle's outputs for ANY draft
    probabilities and uniforms.
  * The argmax rule: numpy.argmax (first occurrence) on rows full of ties.
  * Special values, the early stop, and the output structure.
  * Planted mistakes in a copy of oracle.c are caught by these pins.
"""
import functools
import os

import numpy as np
import pytest

import oracle
import workloads

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")


def _distinct_rows(rng, B, K, V):
    """Rows that are permutations of 0..V-1: every gap between logits >= 1."""
    return np.stack([rng.permutation(V) for _ in range(B * (K + 1))]).reshape(B, K + 1, V)


def _tokens_near_argmax(rng, logits, K, p_hit=0.7):
    B, _, V = logits.shape
    a = logits[:, :K].argmax(-1)
    other = (a + 1 + rng.integers(0, V - 1, (B, K))) % V
    return np.where(rng.random((B, K)) < p_hit, a, other).astype(np.int32)


def check_limit(verify_greedy, dtype, V, K, B=400, seed=0):
    rng = np.random.default_rng(seed)
    vals = _distinct_rows(rng, B, K, V).astype(np.float32)
    logits = vals if dtype == "f32" else workloads.f32_to_bf16_bits(vals)
    x = _tokens_near_argmax(rng, vals, K)
    g = verify_greedy(logits, dtype, x)
    for trial in range(3):
        q = rng.dirichlet(np.full(V, 0.5), (B, K)).astype(np.float32)
        u = rng.random((B, K + 1), dtype=np.float32)
        s = oracle.verify(logits, dtype, q, x, u, 1e-3)
        for key in ("accept_len", "out_tokens", "accept_mask", "status"):
            if not np.array_equal(s[key], g[key]):
                b = int(np.nonzero(np.any((s[key] != g[key]).reshape(B, -1), axis=1))[0][0])
                raise AssertionError(f"{key} at {b}: sampled T->0 {s[key][b]} greedy {g[key][b]}")
    return g


def check_argmax_rule(verify_greedy, seed=1):
    rng = np.random.default_rng(seed)
    B, K, V = 300, 3, 12
    vals = rng.integers(0, 4, (B, K + 1, V)).astype(np.float32)   # many ties
    x = vals[:, :K].argmax(-1).astype(np.int32)                    # every draft accepted
    g = verify_greedy(vals, "f32", x)
    assert np.all(g["accept_len"] == K + 1)
    assert np.array_equal(g["row_argmax"], vals.argmax(-1))
    assert np.array_equal(g["out_tokens"][:, K], vals[:, K].argmax(-1))


def check_structure(verify_greedy, seed=2):
    rng = np.random.default_rng(seed)
    B, K, V = 500, 5, 9
    vals = rng.standard_normal((B, K + 1, V)).astype(np.float32)
    x = _tokens_near_argmax(rng, vals, K, p_hit=0.8)
    g = verify_greedy(vals, "f32", x)
    a = vals.argmax(-1)
    for b in range(B):
        n = int(g["accept_len"][b])
        j = n - 1
        acc = x[b] == a[b, :K]
        want_j = int(np.argmin(acc)) if not acc.all() else K
        assert j == want_j, (b, n, acc)
        assert np.array_equal(g["out_tokens"][b, :j], x[b, :j])
        assert g["out_tokens"][b, j] == a[b, j]
        assert np.all(g["out_tokens"][b, j + 1:] == -1)
        assert np.array_equal(g["accept_mask"][b], (np.arange(K) < j).astype(np.uint8))
        assert np.array_equal(g["row_argmax"][b, :j + 1], a[b, :j + 1])
        assert np.all(g["row_argmax"][b, j + 1:] == -1)


def _pins(verify_greedy):
    check_limit(verify_greedy, "f32", 64, 3)
    check_argmax_rule(verify_greedy)
    check_structure(verify_greedy)


@pytest.mark.parametrize("dtype,V,K", [("f32", 64, 3), ("f32", 500, 1), ("bf16", 200, 4),
                                       ("f32", 7, 0)])
def test_sampled_verify_at_tiny_temperature_is_greedy(dtype, V, K):
    g = check_limit(oracle.verify_greedy, dtype, V, K)
    assert 1 <= g["accept_len"].min() and g["accept_len"].max() <= K + 1


def test_argmax_is_the_first_occurrence():
    check_argmax_rule(oracle.verify_greedy)


def test_early_stop_and_output_structure():
    check_structure(oracle.verify_greedy)


def test_special_values():
    V, K = 6, 2
    base = np.tile(np.arange(V, dtype=np.float32), (1, K + 1, 1))
    x = np.array([[V - 1, V - 1]], np.int32)
    g = oracle.verify_greedy(base, "f32", x)
    assert g["accept_len"][0] == 3 and g["out_tokens"][0].tolist() == [V - 1, V - 1, V - 1]
    for bad in (np.nan, np.inf):
        lg = base.copy()
        lg[0, 1, 2] = bad
        g = oracle.verify_greedy(lg, "f32", x)
        assert g["status"][0] == oracle.NONFINITE and g["accept_len"][0] == 0
        assert np.all(g["out_tokens"][0] == -1) and np.all(g["row_argmax"][0] == -1)
    lg = base.copy()
    lg[0, 0] = -np.inf
    assert oracle.verify_greedy(lg, "f32", x)["status"][0] == oracle.NONFINITE
    lg = base.copy()
    lg[0, 0, :V - 2] = -np.inf                   # -inf entries are ordinary losers
    assert oracle.verify_greedy(lg, "f32", x)["accept_len"][0] == 3
    # a NaN in a row past the rejection is never read
    lg = base.copy()
    lg[0, 2, 0] = np.nan
    g = oracle.verify_greedy(lg, "f32", np.array([[0, V - 1]], np.int32))
    assert g["status"][0] == 0 and g["accept_len"][0] == 1 and g["out_tokens"][0, 0] == V - 1
    # a token outside [0, V) is an error even if the loop would stop before it
    g = oracle.verify_greedy(base, "f32", np.array([[0, V]], np.int32))
    assert g["status"][0] == oracle.TOKEN_RANGE and g["accept_len"][0] == 0


MUTANTS = {
    "last_occurrence": ("                if (l > best) {\n                    best = l;\n                    a = v;",
                        "                if (l >= best) {\n                    best = l;\n                    a = v;"),
    "emit_draft_on_reject": ("            ot[i] = (int32_t)a; /* the corrected token",
                             "            ot[i] = i < K ? tokens[(size_t)b * (size_t)K + (size_t)i] : (int32_t)a; /* the corrected token"),
    "no_stop_at_rejection": ("            len = i + 1;\n            break;\n        }\n        if (st != ORACLE_OK) {",
                             "            len = i + 1;\n        }\n        if (st != ORACLE_OK) {"),
    "length_off_by_one": ("            len = i + 1;\n            break;", "            len = i;\n            break;"),
    "max_of_wrong_row": ("((size_t)b * (size_t)(K + 1) + (size_t)i) *\n                                                        (size_t)V * es;",
                         "((size_t)b * (size_t)(K + 1) + (size_t)(i ? i - 1 : 0)) *\n                                                        (size_t)V * es;"),
}


@functools.lru_cache(maxsize=None)
def _mutant_lib(name, tmpdir):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = os.path.join(tmpdir, f"oracle_greedy_{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    return oracle.load_variant(path, os.path.join(tmpdir, f"lib_greedy_{name}.so"))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path_factory):
    lib = _mutant_lib(name, str(tmp_path_factory.getbasetemp()))
    with pytest.raises((AssertionError, ValueError, IndexError)):
        _pins(functools.partial(oracle.verify_greedy, lib=lib))
