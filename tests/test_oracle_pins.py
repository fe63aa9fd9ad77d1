"""CPU tests that pin the fp64 oracle (oracle/) to the pages and the mathematics.

Citations as in tests/oracle_pins.py ([P1]-[P3], page title and section).
"""
import math

import numpy as np
import pytest
import scipy.optimize
import scipy.special

import oracle
import workloads
from tests import oracle_pins as pins


# ---------------------------------------------------------------- softmax -----

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1.0, 0.6, 2.5])
def test_softmax_matches_library_routine(dtype, T):
    """[P1]: p = softmax(logits / T).  Checked against scipy.special.softmax in
    float64 on the same stored values, and Sum p = 1."""
    rng = np.random.Generator(np.random.Philox(5))
    x = (3.0 * rng.standard_normal(1000)).astype(np.float32)
    row = workloads.f32_to_bf16_bits(x) if dtype == "bf16" else x
    st, p, m, s = oracle.softmax_row(row, dtype, T)
    assert st == oracle.OK
    ref = scipy.special.softmax(workloads.logits_as_f64(row, dtype) / T)
    np.testing.assert_allclose(p, ref, rtol=1e-12, atol=0)
    assert abs(p.sum() - 1.0) < 1e-12
    # exp(0) = 1 at the maximum, so p at the argmax is 1/s, and m = max/T
    k = int(np.argmax(p))
    assert abs(p[k] * s - 1.0) < 1e-12
    assert m == pytest.approx(workloads.logits_as_f64(row, dtype).max() / T, rel=1e-15)


def test_softmax_shift_invariance_and_two_point_closed_form():
    """Adding a constant to every logit leaves p unchanged; two logits a, b give
    p_0 = 1 / (1 + exp((b - a)/T))."""
    row = np.array([-3, 0, 2, 7, 1, -1], np.float32)
    _, p1, _, _ = oracle.softmax_row(row, "f32", 0.7)
    _, p2, _, _ = oracle.softmax_row(row + np.float32(64), "f32", 0.7)
    np.testing.assert_allclose(p1, p2, rtol=1e-13)
    two = np.array([1.0, 2.5], np.float32)
    _, p, _, _ = oracle.softmax_row(two, "f32", 0.5)
    assert p[0] == pytest.approx(1.0 / (1.0 + math.exp((2.5 - 1.0) / 0.5)), rel=1e-14)
    # bf16 bit patterns: 0x3F80 = 1.0, 0xC000 = -2.0
    _, p, m, _ = oracle.softmax_row(np.array([0x3F80, 0xC000], np.uint16), "bf16", 1.0)
    assert p[0] == pytest.approx(1.0 / (1.0 + math.exp(-3.0)), rel=1e-14)
    assert m == 1.0


def test_softmax_special_values():
    """-inf gives probability 0; NaN, +inf, or a row of all -inf is an error."""
    st, p, _, _ = oracle.softmax_row(np.array([0.0, -np.inf, 1.0], np.float32), "f32", 1.0)
    assert st == oracle.OK and p[1] == 0.0
    for bad in ([0.0, np.nan, 1.0], [0.0, np.inf], [-np.inf, -np.inf]):
        st, _, _, _ = oracle.softmax_row(np.array(bad, np.float32), "f32", 1.0)
        assert st == oracle.NONFINITE


# ------------------------------------------------------------ output law -----

@pytest.mark.parametrize("V,K,T,seed", [(4, 1, 1.0, 1), (6, 2, 0.7, 2), (8, 3, 1.3, 3)])
def test_output_law_brute_force(V, K, T, seed):
    """Enumerate drafts and trace every decision along its uniform on a grid of
    2e4 midpoints: accepted mass = min(p, q), corrected mass = max(0, p - q),
    bonus law = p_K, emitted-token law = p at every position."""
    pins.check_output_law(oracle.verify, V, K, T, seed)


@pytest.mark.parametrize("V,K", [(3, 2), (5, 1)])
def test_joint_output_law(V, K):
    """The whole law of (accepted length, tokens) against the analytic product law."""
    pins.joint_law(oracle.verify, V, K, 0.9, seed=21)


@pytest.mark.parametrize("V,K", [(4, 1), (6, 3), (8, 3)])
def test_chi_square_output_distribution(V, K):
    """[P2] "Speculative decoding": the output follows the target distribution.
    Fresh drafts x ~ q and fresh uniforms per trial; chi-square per position."""
    pins.check_chisq(oracle.verify, V, K, 1.0, seed=100 + V + K)


# ------------------------------------------------------- expected tokens -----

def test_table_matches_closed_form():
    """The printed table ([P2] "Speculative decoding") is the closed form
    (1 - a^(k+1)) / (1 - a) rounded to two decimals; so is [P1]'s 3.36."""
    for alpha, cells in pins.read_table():
        for k, printed in cells.items():
            assert round(pins.closed_form_tokens(alpha, k), 2) == pytest.approx(printed, abs=1e-9)
    assert round(pins.closed_form_tokens(0.8, 4), 2) == pytest.approx(3.36, abs=1e-9)


def test_consistency_check_inverse():
    """[P2] "Consistency check on my numbers": 1.8 and 2.0 tokens per pass at
    k = 3 correspond to acceptance about 0.47 and 0.54."""
    for tokens, want in ((1.8, 0.47), (2.0, 0.54)):
        a = scipy.optimize.brentq(lambda x: pins.closed_form_tokens(x, 3) - tokens, 0.01, 0.99)
        assert round(a, 2) == pytest.approx(want, abs=1e-9)


@pytest.mark.parametrize("K", [1, 3, 5])
@pytest.mark.parametrize("alpha", [0.35, 0.5, 0.6, 0.7, 0.8, 0.9])
def test_mean_tokens_per_pass(alpha, K):
    """Draft rows with overlap Sum min(p, q) = alpha at every position: the
    oracle's mean accepted length matches the closed form within 4 SE, and the
    printed table cell within 4 SE plus its rounding."""
    mean, se = pins.check_mean_tokens(oracle.verify, alpha, K)
    printed = dict(pins.read_table())[alpha][K]
    assert abs(mean - printed) < 4 * se + 0.005


# --------------------------------------------------------- special cases -----

def _tile(logits, q, B):
    return (np.ascontiguousarray(np.broadcast_to(logits, (B,) + logits.shape)),
            np.ascontiguousarray(np.broadcast_to(q, (B,) + q.shape)))


def test_q_equal_p_always_accepts():
    inp = workloads.make_random(200, 5, 50, seed=9)
    p = workloads.softmax64(workloads.logits_as_f64(inp.logits, "f32")[:, :5]).astype(np.float32)
    x = np.zeros((200, 5), np.int32)
    r = np.random.Generator(np.random.Philox(3)).random((200, 5))
    for b in range(200):
        for i in range(5):
            x[b, i] = workloads.sample_tokens(p[b, i], r[b, i:i + 1])[0]
    out = oracle.verify(inp.logits, "f32", p, x, inp.uniforms, 1.0)
    assert np.all(out["accept_len"] == 6)


def test_draft_on_target_zero_always_rejects_and_samples_p():
    """q one-hot on a token the target gives probability 0: the first test
    always rejects, and the corrected token follows p_0 (max(0, p - q) = p)."""
    V, M = 7, 20000
    logits = np.array([[0.5, -np.inf, 1.0, 0.0, -0.5, 2.0, 0.3],
                       [0.1, 0.2, 0.3, 0.4, 0.5, 0.6, 0.7]], np.float32)
    q = np.zeros((1, V), np.float32)
    q[0, 1] = 1.0
    L, Q = _tile(logits, q, M)
    u = np.zeros((M, 2), np.float32)
    u[:, 0] = np.random.Generator(np.random.Philox(1)).random(M, dtype=np.float32)
    u[:, 1] = ((np.arange(M) + 0.5) / M).astype(np.float32)
    out = oracle.verify(L, "f32", Q, np.ones((M, 1), np.int32), u, 1.0)
    assert np.all(out["accept_len"] == 1)
    law = np.bincount(out["out_tokens"][:, 0], minlength=V) / M
    np.testing.assert_allclose(law, pins.p_rows(logits, 1.0)[0], atol=2e-4)


def test_one_hot_target_is_deterministic():
    V = 9
    logits = np.full((3, V), -np.inf, np.float32)
    logits[:, 4] = 0.0
    rng = np.random.Generator(np.random.Philox(4))
    q = rng.dirichlet(np.ones(V), size=2).astype(np.float32)
    B = 500
    L, Q = _tile(logits, q, B)
    x = rng.integers(0, V, (B, 2)).astype(np.int32)
    u = rng.random((B, 3), dtype=np.float32)
    out = oracle.verify(L, "f32", Q, x, u, 1.0)
    al = out["accept_len"]
    assert np.all(out["out_tokens"][np.arange(B), al - 1] == 4)


def test_k0_is_plain_inverse_cdf_sampling():
    V, M = 6, 30000
    logits = np.array([[0.0, 1.0, -1.0, 2.0, 0.5, -3.0]], np.float32)
    L = np.ascontiguousarray(np.broadcast_to(logits, (M, 1, V)))
    u = ((np.arange(M) + 0.5) / M).astype(np.float32).reshape(M, 1)
    out = oracle.verify(L, "f32", np.zeros((M, 0, V), np.float32), np.zeros((M, 0), np.int32), u, 0.8)
    assert np.all(out["accept_len"] == 1)
    law = np.bincount(out["out_tokens"][:, 0], minlength=V) / M
    np.testing.assert_allclose(law, pins.p_rows(logits, 0.8)[0], atol=1e-4)


def test_zero_residual_falls_back_to_target_row():
    """An unnormalised draft row q = 1.01 p rejects with probability 1/101 and
    leaves max(0, p - q) = 0 everywhere; the draw then comes from p_j."""
    V, M = 5, 20000
    logits = np.array([[0.0, 1.0, 2.0, -1.0, 0.5], [0, 0, 0, 0, 0]], np.float32)
    p = pins.p_rows(logits, 1.0)
    q = (1.01 * p[:1]).astype(np.float32)
    L, Q = _tile(logits, q, M)
    u = np.zeros((M, 2), np.float32)
    u[:, 0] = np.float32(0.9999)
    u[:, 1] = ((np.arange(M) + 0.5) / M).astype(np.float32)
    out = oracle.verify(L, "f32", Q, np.full((M, 1), 2, np.int32), u, 1.0)
    assert np.all(out["accept_len"] == 1)
    law = np.bincount(out["out_tokens"][:, 0], minlength=V) / M
    np.testing.assert_allclose(law, p[0], atol=1e-4)


# ------------------------------------------------------------------ errors -----

def test_error_semantics():
    inp = workloads.make_random(6, 3, 40, seed=13)
    logits, q, x, u = inp.logits.copy(), inp.q.copy(), inp.tokens.copy(), inp.uniforms.copy()
    x[0, 2] = 40                      # out of range (even past the first rejection)
    x[1, 0] = -1
    u[2, 3] = np.float32(1.0)         # uniforms live in [0, 1)
    logits[3, 0, 7] = np.nan          # row 0 is always reached
    u[4, :3] = 0.0                    # accept everything at sequence 4 (q > 0 here)
    logits[4, 3, 5] = np.inf          # ... so the bonus row is reached
    out = oracle.verify(logits, "f32", q, x, u, 1.0)
    assert list(out["status"]) == [oracle.TOKEN_RANGE, oracle.TOKEN_RANGE, oracle.UNIFORM_RANGE,
                                   oracle.NONFINITE, oracle.NONFINITE, oracle.OK]
    bad = out["status"] != 0
    assert np.all(out["accept_len"][bad] == 0) and np.all(out["out_tokens"][bad] == -1)
    assert np.all(np.isnan(out["row_s"][bad]))


def test_rows_past_the_rejection_are_not_read():
    """[P1] loop stops at the first rejection: a NaN in a later row is never seen."""
    inp = workloads.make_random(1, 4, 30, seed=17)
    logits, u = inp.logits.copy(), inp.uniforms.copy()
    u[0, 0] = np.float32(0.99999994)
    q = inp.q.copy()
    q[0, 0] = 0.0
    q[0, 0, 3] = 1.0
    x = inp.tokens.copy()
    x[0, 0] = 3
    logits[0, 0, 3] = -np.inf         # p(x_0) = 0: rejected at 0 for sure
    logits[0, 2, 0] = np.nan
    out = oracle.verify(logits, "f32", q, x, u, 1.0)
    assert out["status"][0] == oracle.OK and out["accept_len"][0] == 1
    assert np.isnan(out["row_s"][0, 1:]).all() and not np.isnan(out["row_s"][0, 0])


def test_tie_margin_reports_the_neighbouring_token():
    """Weights 1/4, 1/4, 1/2 and u = 1/4 sit on the first boundary."""
    logits = np.array([[0.0, 0.0, math.log(2.0)]], np.float32)
    u = np.array([[0.25]], np.float32)
    out = oracle.verify(logits[None], "f32", np.zeros((1, 0, 3), np.float32),
                        np.zeros((1, 0), np.int32), u, 1.0)
    assert out["sample_margin"][0] < 1e-6
    assert {int(out["out_tokens"][0, 0]), int(out["sample_alt"][0])} == {0, 1}


def test_workload_recipes_have_the_stated_overlap():
    """The sweep's mixture gives Sum min(p, q) = alpha up to fp32 rounding of q."""
    cell = workloads.make_sweep_cell(0.7, 3, B=4, V=500, rounds=2)
    p = pins.p_rows(cell.logits, 1.0)
    ov = np.minimum(p[:, :3], cell.q.astype(np.float64)).sum(-1)
    np.testing.assert_allclose(ov, 0.7, atol=1e-6)


def test_inverse_transform_convention():
    """The draw maps u to the first token whose cumulative weight exceeds u
    (inverse-transform sampling over ascending ids): weights 0.1, 0.2, 0.3, 0.4
    have cumulative sums 0.1, 0.3, 0.6, 1.0."""
    logits = np.log(np.array([[0.1, 0.2, 0.3, 0.4]])).astype(np.float32)
    us = np.array([0.0, 0.05, 0.0999, 0.1001, 0.2999, 0.3001, 0.5999, 0.6001, 0.99999994], np.float32)
    want = [0, 0, 0, 1, 1, 2, 2, 3, 3]
    n = us.size
    out = oracle.verify(np.broadcast_to(logits, (n, 1, 4)), "f32", np.zeros((n, 0, 4), np.float32),
                        np.zeros((n, 0), np.int32), us.reshape(n, 1), 1.0)
    assert list(out["out_tokens"][:, 0]) == want
