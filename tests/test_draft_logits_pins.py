"""Pins for the oracle's verify with draft logits instead of draft
probabilities ([P1]'s loop forms q = softmax(draft_logits / T) itself).

  * It equals the verify fed with q = scipy.special.softmax(d / T_d) (a
    library routine) rounded to float32, outside the 1e-6 tie band, with and
    without the truncated target, at a draft temperature other than the
    target's.
  * The output law: drafts sampled from softmax(d / T_d); the emitted token at
    every reached position follows the target (chi-square).
  * A bad draft row is an error only when the loop reaches it.
"""
import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle
import workloads


def _q_from(dl, dtype, Td):
    return scipy.special.softmax(workloads.logits_as_f64(dl, dtype) / np.float32(Td),
                                 axis=-1).astype(np.float32)


@pytest.mark.parametrize("dtype,Td,top_p,min_p", [("f32", 1.0, 1.0, 0.0), ("bf16", 0.7, 1.0, 0.0),
                                                  ("bf16", 0.6, 0.95, 0.05), ("f32", 1.3, 0.9, 0.0)])
def test_equals_the_verify_with_library_softmax(dtype, Td, top_p, min_p):
    rng = np.random.default_rng(7)
    B, K, V = 200, 4, 300
    inp = workloads.make_random(B, K, V, dtype, T=0.8, seed=13)
    d64 = workloads.logits_as_f64(inp.logits[:, :K], dtype) + rng.standard_normal((B, K, V))
    dl = workloads._cast(d64, dtype)
    q = _q_from(dl, dtype, Td)
    x = workloads.sample_tokens(q, rng.random((B, K, 1)))[..., 0].astype(np.int32)
    f = oracle.verify_draft_logits(inp.logits, dtype, dl, x, inp.uniforms, inp.T, Td, top_p, min_p)
    r = oracle.verify_truncated(inp.logits, dtype, q, x, inp.uniforms, inp.T, top_p, min_p)
    tie = ((r["accept_margin"] < 1e-6) | (r["sample_margin"] < 1e-6) | (r["trunc_margin"] < 1e-6) |
           (f["accept_margin"] < 1e-6) | (f["sample_margin"] < 1e-6))
    assert tie.sum() < B // 10
    for key in ("accept_len", "out_tokens", "accept_mask", "status"):
        assert np.array_equal(f[key][~tie], r[key][~tie]), key
    assert np.allclose(f["row_s"][~tie], r["row_s"][~tie], rtol=0, atol=0, equal_nan=True)


def test_output_law_is_the_target():
    rng = np.random.Generator(np.random.Philox(21))
    V, K, M = 6, 2, 150000
    logits = (1.5 * rng.standard_normal((K + 1, V))).astype(np.float32)
    dl = (logits[:K] + rng.standard_normal((K, V))).astype(np.float32)
    q = scipy.special.softmax(dl.astype(np.float64), axis=-1)
    x = np.stack([workloads.sample_tokens(q[i], rng.random(M)) for i in range(K)], axis=1)
    u = rng.random((M, K + 1), dtype=np.float32)
    out = oracle.verify_draft_logits(np.broadcast_to(logits, (M, K + 1, V)), "f32",
                                     np.broadcast_to(dl, (M, K, V)), x, u, 1.0, 1.0)
    assert np.all(out["status"] == 0)
    p = scipy.special.softmax(logits.astype(np.float64), axis=-1)
    for n in range(K + 1):
        reached = out["accept_len"] >= n + 1
        tok = out["out_tokens"][reached, n]
        counts = np.bincount(tok, minlength=V).astype(np.float64)
        _, pval = scipy.stats.chisquare(counts, p[n] * reached.sum())
        assert pval > 1e-4, (n, pval)
    acc0 = out["accept_mask"][:, 0].mean()
    alpha0 = np.minimum(p[0], q[0]).sum()
    assert abs(acc0 - alpha0) < 4 * np.sqrt(alpha0 * (1 - alpha0) / M)


def test_bad_draft_rows():
    V, K = 50, 3
    logits = np.tile(np.arange(V, dtype=np.float32) / 10, (2, K + 1, 1))
    dl = np.tile(np.arange(V, dtype=np.float32) / 10, (2, K, 1))
    x = np.full((2, K), V - 1, np.int32)
    x[1, 0] = 0                    # sequence 1 is rejected at position 0:
    logits[1, 0, 0] = -20.0        # the target gives its draft token almost nothing
    u = np.full((2, K + 1), 0.99, np.float32)
    dl[:, 2, 7] = np.nan           # draft row 2: reached by sequence 0 only
    out = oracle.verify_draft_logits(logits, "f32", dl, x, u, 1.0, 1.0)
    assert out["status"][0] == oracle.NONFINITE and out["accept_len"][0] == 0
    assert out["status"][1] == 0 and out["accept_len"][1] == 1
    with pytest.raises(ValueError):
        oracle.verify_draft_logits(logits, "f32", dl, x, u, 1.0, 0.0)
