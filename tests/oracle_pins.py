"""Checks that pin the fp64 oracle to what the pages and the mathematics fix.

Each check takes a ``verify`` callable with the signature of ``oracle.verify``
so the same checks can be pointed at a copy of the oracle with a planted
mistake (tests/test_oracle_mutants.py).  Nothing here re-types the oracle's
formulas: the references are closed forms of the method's output law (the
rejection-sampling theorem the pages rely on), library routines
(scipy.special.softmax), statistics (chi-square, standard errors) and values
the pages print (tests/golden/).

Citations: [P1] reactapp.top "Speculative decoding and early exit: speeding up
autoregressive decode", section "Speculative decoding: draft first, then
verify"; [P2] trefon.com "Decode is memory-bound: a ~59 tok/s ceiling on an RTX
4090 and how speculative decoding breaks it", sections "Speculative decoding"
and "Two things that follow from the math"; [P3] agentnet.co.il "New technical
post reveals how speculative decoding speeds up LLM inference without hurting
accuracy", section "How it works in practice".
"""
from __future__ import annotations

import os

import numpy as np
import scipy.special
import scipy.stats

import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


class PinFailure(AssertionError):
    pass


def check(cond, msg):
    if not cond:
        raise PinFailure(msg)


def p_rows(logits: np.ndarray, T: float) -> np.ndarray:
    """Target distributions by the library softmax of logits / T (float64).
    The temperature is a float32 argument of the verify call, so it is rounded
    to float32 here too."""
    return scipy.special.softmax(logits.astype(np.float64) / float(np.float32(T)), axis=-1)


def law_case(V: int, K: int, seed: int, zeros: bool = True):
    """Small target/draft rows with distinct rows per position.  With ``zeros``
    the draft puts no mass on a token the target likes, and the target puts no
    mass (a -inf logit) on a token the draft likes, to reach the edges."""
    rng = np.random.Generator(np.random.Philox(seed))
    logits = (1.5 * rng.standard_normal((K + 1, V))).astype(np.float32)
    q = rng.dirichlet(np.full(V, 0.8), size=K)
    if zeros and K:
        logits[0, 1] = -np.inf
        q[0, 1] = max(q[0, 1], 0.2)
        q[0, 2] = 0.0
        q[0] /= q[0].sum()
    return logits, q.astype(np.float32)


def _run(verify, logits, q, x, u, T):
    M = u.shape[0]
    K1, V = logits.shape
    return verify(np.broadcast_to(logits, (M, K1, V)), "f32",
                  np.broadcast_to(q, (M, K1 - 1, V)),
                  np.broadcast_to(np.asarray(x, np.int32), (M, K1 - 1)), u, T)


def structural(out: dict, tokens: np.ndarray, K: int):
    """[P3] 1 <= AL <= 1 + D; the accepted prefix is the drafts; mask marks it."""
    ok = out["status"] == 0
    al = out["accept_len"][ok]
    check(np.all((al >= 1) & (al <= K + 1)), f"accept_len outside [1, {K + 1}]")
    ot = out["out_tokens"][ok]
    mk = out["accept_mask"][ok]
    tk = np.broadcast_to(tokens, (out["status"].shape[0], K))[ok]
    for n in range(K + 1):
        rows = al == n + 1
        if not rows.any():
            continue
        if n:
            check(np.array_equal(ot[rows, :n], tk[rows, :n]), "prefix is not the drafts")
            check(np.all(mk[rows, :n] == 1), "mask misses an accepted position")
        check(np.all(ot[rows, n] >= 0), "missing sampled token")
        check(np.all(ot[rows, n + 1:] == -1), "padding after the sampled token")
        check(np.all(mk[rows, n:] == 0), "mask marks a position after the rejection")


def output_law(verify, logits, q, T, M=20000, margin=1e-9):
    """The oracle's exact decision functions on a midpoint grid of M uniforms.

    Returns (a, r, rK): a[i, y] = P(accept at i | x_i = y); r[j, y, c] = P(token
    c | rejection at j with x_j = y); rK[c] = P(bonus token c).  The tests at
    different positions use different uniforms ([P1] draws one per test), so
    each decision function is traced along its own uniform."""
    K1, V = logits.shape
    K = K1 - 1
    p = p_rows(logits, T)
    carrier = [int(np.argmax(p[i])) for i in range(K)]
    grid = ((np.arange(M) + 0.5) / M).astype(np.float32)
    a = np.zeros((K, V))
    r = np.zeros((K, V, V))
    for i in range(K):
        for y in range(V):
            x = list(carrier)
            x[i] = y
            u = np.zeros((M, K + 1), np.float32)
            u[:, i] = grid
            out = _run(verify, logits, q, x, u, T)
            check(np.all(out["status"] == 0), "unexpected error status")
            structural(out, np.asarray(x, np.int32), K)
            a[i, y] = out["accept_mask"][:, i].mean()
    for j in range(K):
        for y in range(V):
            pj, qj = p[j, y], float(q[j, y])
            if not pj < qj:
                continue  # min(1, p/q) = 1: a rejection here has probability 0
            # a float32 uniform just past p/q; the relative margin keeps it clear
            # of rounding differences between implementations (1e-9 between two
            # fp64 evaluations; the fp32 GPU path needs the 1e-6 tie band)
            if pj / qj > 1.0 - 10 * margin:
                continue  # rejection probability below 10*margin: no measurable mass
            uj = np.float32(pj / qj)
            while not float(uj) * qj >= pj * (1.0 + margin):
                uj = np.nextafter(uj, np.float32(1.0))
            x = list(carrier)
            x[j] = y
            u = np.zeros((M, K + 1), np.float32)
            u[:, j] = uj
            u[:, K] = grid
            out = _run(verify, logits, q, x, u, T)
            check(np.all(out["accept_len"] == j + 1), f"forced rejection at {j} not taken")
            r[j, y] = np.bincount(out["out_tokens"][:, j], minlength=V)[:V] / M
    u = np.zeros((M, K + 1), np.float32)
    u[:, K] = grid
    out = _run(verify, logits, q, carrier, u, T)
    check(np.all(out["accept_len"] == K + 1), "all-accept path not taken")
    rK = np.bincount(out["out_tokens"][:, K], minlength=V)[:V] / M
    return a, r, rK


def check_output_law(verify, V, K, T, seed, M=20000, tol=3e-4, margin=1e-9):
    """The rejection-sampling theorem ([P2] "Speculative decoding"; [P1]):
    per position, accepted mass q(y) * a(y) = min(p, q)(y); the rejection mass
    spread by the corrected-token law equals max(0, p - q); the bonus token
    follows p_K; so the token emitted at every reached position follows p."""
    logits, q = law_case(V, K, seed)
    p = p_rows(logits, T)
    a, r, rK = output_law(verify, logits, q, T, M, margin)
    for i in range(K):
        got = q[i].astype(np.float64) * a[i]
        want = np.minimum(p[i], q[i])
        check(np.max(np.abs(got - want)) < tol, f"accepted mass at {i}: {got} vs {want}")
        corr = np.einsum("y,yc->c", q[i].astype(np.float64) * (1.0 - a[i]), r[i])
        want_c = np.maximum(p[i] - q[i], 0.0)
        check(np.max(np.abs(corr - want_c)) < tol, f"corrected mass at {i}: {corr} vs {want_c}")
        check(np.max(np.abs(got + corr - p[i])) < 2 * tol, f"emitted token law at {i} is not p")
    check(np.max(np.abs(rK - p[K])) < tol, f"bonus law {rK} vs {p[K]}")
    return a, r, rK


def joint_law(verify, V, K, T, seed, M=20000):
    """Full law of (accepted length, tokens) from the traced decision functions,
    against the analytic law  prod_{i<n} min(p_i, q_i)(y_i) * max(0, p_n - q_n)(c)
    for n < K and  prod_{i<K} min(p_i, q_i)(y_i) * p_K(c)  for n = K."""
    logits, q = law_case(V, K, seed)
    p = p_rows(logits, T)
    a, r, rK = output_law(verify, logits, q, T, M)
    q64 = q.astype(np.float64)
    worst = 0.0
    total = 0.0
    for n in range(K + 1):
        for ys in np.ndindex(*([V] * n)):
            pre_got = np.prod([q64[i, y] * a[i, y] for i, y in enumerate(ys)]) if n else 1.0
            pre_want = np.prod([min(p[i, y], q64[i, y]) for i, y in enumerate(ys)]) if n else 1.0
            if n < K:
                tail_got = np.einsum("y,yc->c", q64[n] * (1.0 - a[n]), r[n])
                tail_want = np.maximum(p[n] - q64[n], 0.0)
            else:
                tail_got, tail_want = rK, p[K]
            got = pre_got * tail_got
            total += got.sum()
            worst = max(worst, float(np.max(np.abs(got - pre_want * tail_want))))
    check(abs(total - 1.0) < 1e-3, f"law does not sum to one ({total})")
    check(worst < 5e-4, f"joint law off by {worst}")
    return worst


def check_chisq(verify, V, K, T, seed, trials=200000, pmin=1e-4):
    """Monte Carlo with fresh drafts x ~ q and fresh uniforms in every trial:
    the token emitted at each reached position follows p_i (chi-square), and
    acceptance at position 0 happens at the rate sum_v min(p_0, q_0)
    ([P2] "Two things that follow from the math")."""
    logits, q = law_case(V, K, seed)
    p = p_rows(logits, T)
    rng = np.random.Generator(np.random.Philox(seed + 7777))
    x = np.zeros((trials, K), np.int32)
    for i in range(K):
        x[:, i] = workloads.sample_tokens(q[i], rng.random(trials))
    u = rng.random((trials, K + 1), dtype=np.float32)
    out = verify(np.broadcast_to(logits, (trials, K + 1, V)), "f32",
                 np.broadcast_to(q, (trials, K, V)), x, u, T)
    check(np.all(out["status"] == 0), "unexpected error status")
    structural(out, x, K)
    for n in range(K + 1):
        reached = out["accept_len"] >= n + 1
        N = int(reached.sum())
        if N < 1000:
            continue
        tok = out["out_tokens"][reached, n]  # the draft if accepted there, else the sample
        counts = np.bincount(tok, minlength=V)[:V].astype(np.float64)
        zero = p[n] <= 0
        check(np.all(counts[zero] == 0), f"position {n}: a zero-probability token was emitted")
        exp = p[n][~zero] * N
        stat, pval = scipy.stats.chisquare(counts[~zero], exp)
        check(pval > pmin, f"position {n}: chi-square p-value {pval:.2e}")
    if K:
        acc0 = out["accept_mask"][:, 0].astype(np.float64)
        alpha0 = np.minimum(p[0], q[0].astype(np.float64)).sum()
        se = np.sqrt(alpha0 * (1 - alpha0) / trials)
        check(abs(acc0.mean() - alpha0) < 4 * se + 1e-12,
              f"acceptance {acc0.mean():.5f} vs sum min(p, q) = {alpha0:.5f}")


def read_table():
    rows = []
    with open(os.path.join(GOLDEN, "tokens_per_pass.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                a, k1, k3, k5 = map(float, line.split())
                rows.append((a, {1: k1, 3: k3, 5: k5}))
    return rows


def closed_form_tokens(alpha: float, k: int) -> float:
    """E[tokens per pass] for i.i.d. acceptance alpha and k drafts ([P2])."""
    return (1.0 - alpha ** (k + 1)) / (1.0 - alpha)


def check_mean_tokens(verify, alpha, K, V=64, B=48, rounds=400, seed=11):
    """Drafts built with overlap exactly alpha at every position make each test
    an independent Bernoulli(alpha), so mean accepted length must match
    (1 - alpha^(K+1)) / (1 - alpha) within 4 standard errors, and the
    per-position acceptance among reached positions must be alpha."""
    cell = workloads.make_sweep_cell(alpha, K, B=B, V=V, rounds=rounds, seed=seed)
    n = B * rounds
    logits = np.broadcast_to(cell.logits[None], (rounds,) + cell.logits.shape).reshape(n, K + 1, V)
    q = np.broadcast_to(cell.q[None], (rounds,) + cell.q.shape).reshape(n, K, V)
    out = verify(logits, "f32", q, cell.tokens.reshape(n, K), cell.uniforms.reshape(n, K + 1), 1.0)
    check(np.all(out["status"] == 0), "unexpected error status")
    al = out["accept_len"].astype(np.float64)
    want = closed_form_tokens(alpha, K)
    se = al.std(ddof=1) / np.sqrt(n)
    check(abs(al.mean() - want) < 4 * se, f"alpha={alpha} K={K}: mean AL {al.mean():.4f} vs {want:.4f}")
    for i in range(K):
        reached = al >= i + 1
        acc = out["accept_mask"][reached, i].astype(np.float64)
        se_i = np.sqrt(alpha * (1 - alpha) / max(1, acc.size))
        check(abs(acc.mean() - alpha) < 4 * se_i + 1e-12,
              f"alpha={alpha} position {i}: acceptance {acc.mean():.4f}")
    return al.mean(), se
