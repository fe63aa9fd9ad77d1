"""Pins for the oracle's verification against a truncated target (top-p and
min-p, the production sampler settings named in [P2] "Two things that follow
from the math").

  * With both filters off the truncated verify is the verify.
  * Worked examples with hand-computed kept sets, including a tie at the top-p
    boundary (all tied tokens kept) and both filters together.
  * The limits: a vanishing top-p, or a min-p just below 1, keeps only the
    most probable token, so the truncated verify becomes the greedy verify.
  * The output law: rows built so that the kept set and p~ are known by
    construction; the emitted token at every reached position follows p~
    (chi-square) and acceptance at position 0 is sum min(p~, q).
  * Planted mistakes in a copy of oracle.c are caught.
"""
import functools
import os

import numpy as np
import pytest
import scipy.stats

import oracle
import workloads

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")


def _bonus_tokens(verify_t, p, top_p, min_p, us):
    """K = 0: the single draw from p~ of one row, at the given uniforms."""
    V = len(p)
    logits = np.log(np.asarray(p, np.float64)).astype(np.float32)
    M = len(us)
    out = verify_t(np.broadcast_to(logits, (M, 1, V)), "f32", np.zeros((M, 0, V), np.float32),
                   np.zeros((M, 0), np.int32), np.asarray(us, np.float32).reshape(M, 1), 1.0,
                   top_p, min_p)
    assert np.all(out["status"] == 0)
    return out["out_tokens"][:, 0].tolist()


def check_worked_examples(verify_t):
    # p = (.5, .3, .15, .05), top-p .9: mass above each token 0, .5, .8, .95, so
    # tokens 0..2 are kept, p~ = (.5, .3, .15)/.95 with cut points .526, .842
    assert _bonus_tokens(verify_t, [.5, .3, .15, .05], .9, 0.0, [.2, .6, .9, .999]) == [0, 1, 2, 2]
    # min-p .35: keep p >= .175, tokens 0, 1, p~ = (.625, .375)
    assert _bonus_tokens(verify_t, [.5, .3, .15, .05], 1.0, .35, [.6, .63, .99]) == [0, 1, 1]
    # a tie at the boundary: p = (.4, .2, .2, .2), top-p .5: the three tied
    # tokens have mass .4 above them, below .5, so all are kept (p~ = p) ...
    assert _bonus_tokens(verify_t, [.4, .2, .2, .2], .5, 0.0, [.3, .5, .7, .9]) == [0, 1, 2, 3]
    # ... and at top-p equal to the mass above them none of them is (the mass
    # above must be below top-p); the exact double comes from the softmax of
    # the same float32 logits, and one ulp more keeps them again
    lg = np.log(np.array([.4, .2, .2, .2])).astype(np.float32)
    st, p, _, _ = oracle.softmax_row(lg, "f32", 1.0)
    assert st == 0 and p[1] == p[2] == p[3]
    assert _bonus_tokens(verify_t, [.4, .2, .2, .2], p[0], 0.0, [.1, .9]) == [0, 0]
    assert _bonus_tokens(verify_t, [.4, .2, .2, .2], np.nextafter(p[0], 1.0), 0.0,
                         [.1, .9]) == [0, 3]
    # both: p = (.6, .25, .1, .04, .01), top-p .9 keeps tokens 0..2 (mass above
    # token 3 is .95), min-p .05 keeps p >= .03 (tokens 0..3): together 0..2,
    # p~ = (.6, .25, .1)/.95 with cut points .632, .895
    assert _bonus_tokens(verify_t, [.6, .25, .1, .04, .01], .9, .05,
                         [.5, .7, .95, .9999]) == [0, 1, 2, 2]


def check_greedy_limit(verify_t, seed=0):
    rng = np.random.default_rng(seed)
    B, K, V = 300, 3, 40
    vals = np.stack([rng.permutation(V) for _ in range(B * (K + 1))]).reshape(B, K + 1, V)
    vals = (0.5 * vals).astype(np.float32)                 # distinct, gaps 0.5
    a = vals[:, :K].argmax(-1)
    x = np.where(rng.random((B, K)) < 0.7, a, (a + 1) % V).astype(np.int32)
    g = oracle.verify_greedy(vals, "f32", x)
    q = rng.dirichlet(np.full(V, 0.5), (B, K)).astype(np.float32)
    u = rng.random((B, K + 1), dtype=np.float32)
    for top_p, min_p in ((1e-12, 0.0), (1.0, 0.999999)):
        t = verify_t(vals, "f32", q, x, u, 1.0, top_p, min_p)
        for key in ("accept_len", "out_tokens", "accept_mask", "status"):
            assert np.array_equal(t[key], g[key]), (top_p, min_p, key)


def law_rows(V, K, seed, keep=3, top_p=0.95, min_p=0.05):
    """Rows whose truncation is known by construction: `keep` tokens carry
    mass .97 (each at least .05 of it), the other tokens .01 each (V = keep +
    3).  Top-p .95 drops the small tokens (the mass above each is >= .97) and
    keeps the large ones (the mass above the smallest large one is < .95);
    min-p .05 drops the small ones too (.01 < .05 * p_max, p_max >= .97/keep).
    So p~ is the large part, renormalised."""
    assert V == keep + 3
    rng = np.random.Generator(np.random.Philox(seed))
    big = 0.05 + 0.97 * (1 - 0.05 * keep) * rng.dirichlet(np.ones(keep), K + 1) / 1.0
    big = big / big.sum(axis=1, keepdims=True) * 0.97
    p = np.concatenate([big, np.full((K + 1, 3), 0.01)], axis=1)
    perm = np.stack([rng.permutation(V) for _ in range(K + 1)])
    p = np.take_along_axis(p, perm, axis=1)
    pt = np.where(p > 0.02, p, 0.0)
    pt /= pt.sum(axis=1, keepdims=True)
    q = rng.dirichlet(np.full(V, 0.8), size=K).astype(np.float32)
    return np.log(p).astype(np.float32), q, pt


def check_output_law(verify_t, V=6, K=2, seed=3, trials=150000, pmin=1e-4):
    logits, q, pt = law_rows(V, K, seed)
    rng = np.random.Generator(np.random.Philox(seed + 99))
    x = np.zeros((trials, K), np.int32)
    for i in range(K):
        x[:, i] = workloads.sample_tokens(q[i], rng.random(trials))
    u = rng.random((trials, K + 1), dtype=np.float32)
    out = verify_t(np.broadcast_to(logits, (trials, K + 1, V)), "f32",
                   np.broadcast_to(q, (trials, K, V)), x, u, 1.0, 0.95, 0.05)
    assert np.all(out["status"] == 0)
    for n in range(K + 1):
        reached = out["accept_len"] >= n + 1
        N = int(reached.sum())
        tok = out["out_tokens"][reached, n]
        counts = np.bincount(tok, minlength=V)[:V].astype(np.float64)
        zero = pt[n] <= 0
        assert np.all(counts[zero] == 0), f"position {n}: a dropped token was emitted"
        _, pval = scipy.stats.chisquare(counts[~zero], pt[n][~zero] * N)
        assert pval > pmin, f"position {n}: chi-square p-value {pval:.2e}"
    acc0 = out["accept_mask"][:, 0].astype(np.float64)
    alpha0 = np.minimum(pt[0], q[0].astype(np.float64)).sum()
    assert abs(acc0.mean() - alpha0) < 4 * np.sqrt(alpha0 * (1 - alpha0) / trials)


def _pins(verify_t):
    check_worked_examples(verify_t)
    check_greedy_limit(verify_t)
    check_output_law(verify_t, trials=60000)


def test_filters_off_is_the_verify():
    for dtype, V in (("f32", 300), ("bf16", 1000)):
        inp = workloads.make_random(60, 4, V, dtype, seed=V)
        a = oracle.verify_inputs(inp)
        b = oracle.verify_truncated(inp.logits, inp.dtype, inp.q, inp.tokens, inp.uniforms, inp.T,
                                    1.0, 0.0)
        for key in a:
            assert np.array_equal(a[key], b[key], equal_nan=True), key
        assert np.all(np.isinf(b["trunc_margin"]))


def test_worked_examples():
    check_worked_examples(oracle.verify_truncated)


def test_greedy_limit():
    check_greedy_limit(oracle.verify_truncated)


@pytest.mark.parametrize("seed", [3, 4])
def test_output_law_is_the_truncated_target(seed):
    check_output_law(oracle.verify_truncated, seed=seed)


def test_draft_values_are_checked_where_the_residual_reads_them():
    """Against a truncated target the residual max(0, p~_j - q_j) is zero
    wherever p~_j is, so q_j is read, and checked, at the kept tokens only: a
    NaN at a dropped token changes nothing, a NaN at a kept one is an error
    (as for q(x_i) in the test).  With both filters off every entry is read."""
    V = 6
    logits = np.log(np.array([0.5, 0.3, 0.1, 0.05, 0.03, 0.02])).astype(np.float32)
    lg = np.broadcast_to(logits, (1, 2, V)).copy()
    q = np.full((1, 1, V), 1.0 / V, np.float32)
    x = np.array([[5]], np.int32)               # p(5) < q(5) u at u = 0.99: rejected
    u = np.array([[0.99, 0.5]], np.float32)
    base = oracle.verify_truncated(lg, "f32", q, x, u, 1.0, 0.95, 0.15)
    assert base["status"][0] == 0 and base["accept_len"][0] == 1
    kept = {0, 1, 2}                            # min-p 0.15: p >= 0.075
    for v in range(V):
        qq = q.copy()
        qq[0, 0, v] = np.nan
        out = oracle.verify_truncated(lg, "f32", qq, x, u, 1.0, 0.95, 0.15)
        if v in kept:
            assert out["status"][0] == oracle.NONFINITE, v
        elif v == 5:                            # q(x_0) itself, read by the test
            assert out["status"][0] == oracle.NONFINITE
        else:
            assert out["status"][0] == 0 and out["out_tokens"][0, 0] == base["out_tokens"][0, 0], v
        off = oracle.verify_truncated(lg, "f32", qq, x, u, 1.0, 1.0, 0.0)
        assert off["status"][0] == oracle.NONFINITE, v


def test_argument_checks():
    inp = workloads.make_random(2, 1, 50, "f32", seed=1)
    for top_p, min_p in ((0.0, 0.0), (0.5, 1.0), (np.nan, 0.0)):
        with pytest.raises(ValueError):
            oracle.verify_truncated(inp.logits, inp.dtype, inp.q, inp.tokens, inp.uniforms, 1.0,
                                    top_p, min_p)


MUTANTS = {
    "top_p_inclusive": ("            if (!(above < tr->top_p))", "            if (!(above <= tr->top_p))"),
    "top_p_counts_own_group": ("            if (!(above < tr->top_p))", "            if (!(above + gm < tr->top_p))"),
    "min_p_ignored": ("            if (!(p[v] >= tr->min_p * pmax))", "            if (!(p[v] >= 0.0))"),
    "not_renormalised": ("        p[v] = keep[v] ? p[v] / kept : 0.0;", "        p[v] = keep[v] ? p[v] : 0.0;"),
    "min_p_absolute": ("            if (!(p[v] >= tr->min_p * pmax))", "            if (!(p[v] >= tr->min_p))"),
}


@functools.lru_cache(maxsize=None)
def _mutant_lib(name, tmpdir):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = os.path.join(tmpdir, f"oracle_trunc_{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    return oracle.load_variant(path, os.path.join(tmpdir, f"lib_trunc_{name}.so"))


def test_pins_pass_on_the_oracle():
    _pins(oracle.verify_truncated)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path_factory):
    lib = _mutant_lib(name, str(tmp_path_factory.getbasetemp()))
    with pytest.raises((AssertionError, ValueError, IndexError)):
        _pins(functools.partial(oracle.verify_truncated, lib=lib))
