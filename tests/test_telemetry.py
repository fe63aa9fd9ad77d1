"""Acceptance telemetry and adaptive draft depth, on the CPU.

What the pages fix:
  * [P1] "Production perspective" and its checklist: ship the acceptance rate
    and the mean accepted length, record acceptance histograms;
  * [P2] "Speculative decoding": with i.i.d. acceptance alpha the number of
    accepted drafts is a geometric law cut at K, so P(AL = n) = alpha^(n-1)
    (1 - alpha) for n <= K and alpha^K for n = K + 1;
  * [P2] "Two things that follow from the math": cap the depth when the
    measured acceptance falls below 35 %.

The oracle's histogram and depth rule are pinned by those laws and by a worked
example; the library's host function spec_adapt must agree with the oracle's
on every histogram."""
import numpy as np
import pytest
import scipy.stats

import oracle
import workloads


@pytest.fixture(scope="module")
def sv():
    from speculative_decoding_verification_14_gb300 import build
    build.build()
    import speculative_decoding_verification_14_gb300 as pkg
    return pkg


def test_worked_example():
    # K = 4: lengths 1, 2, 3, 3, 5, 5, 5 and one error.  Tested drafts
    # 1+2+3+3+4+4+4 = 21, accepted 0+1+2+2+4+4+4 = 17; position 0 tested by all
    # 7, accepted by 6; position 2 tested by 5, accepted by 3.
    h = oracle.accept_hist(np.array([1, 2, 3, 3, 5, 5, 5, 0]), 4)
    assert h.tolist() == [1, 1, 1, 2, 0, 3]
    a = oracle.adapt(h, 4, 4)
    assert a["acceptance"] == pytest.approx(17 / 21, abs=1e-15)
    assert a["mean_accept_len"] == pytest.approx(24 / 7, abs=1e-15)
    assert a["pos_acceptance"].tolist() == pytest.approx([6 / 7, 5 / 6, 3 / 5, 3 / 3])
    with pytest.raises(ValueError):
        oracle.accept_hist(np.array([1, 6]), 4)


def _sweep_lengths(alpha, K, B=32, V=64, rounds=300, seed=21):
    cell = workloads.make_sweep_cell(alpha, K, B=B, V=V, rounds=rounds, seed=seed)
    n = B * rounds
    logits = np.broadcast_to(cell.logits[None], (rounds,) + cell.logits.shape).reshape(n, K + 1, V)
    q = np.broadcast_to(cell.q[None], (rounds,) + cell.q.shape).reshape(n, K, V)
    out = oracle.verify(logits, "f32", q, cell.tokens.reshape(n, K),
                        cell.uniforms.reshape(n, K + 1), 1.0)
    assert np.all(out["status"] == 0)
    return out["accept_len"]


@pytest.mark.parametrize("alpha,K", [(0.35, 3), (0.6, 5), (0.8, 3), (0.9, 1)])
def test_histogram_follows_the_truncated_geometric_law(alpha, K):
    al = _sweep_lengths(alpha, K)
    h = oracle.accept_hist(al, K).astype(np.float64)
    n = h.sum()
    law = np.array([alpha ** (m - 1) * (1 - alpha) for m in range(1, K + 1)] + [alpha ** K])
    assert law.sum() == pytest.approx(1.0)
    chi2 = ((h[1:] - n * law) ** 2 / (n * law)).sum()
    assert scipy.stats.chi2.sf(chi2, K) > 1e-4, (h, n * law)
    a = oracle.adapt(h.astype(np.uint64), K, K)
    tested = sum(h[m] * min(m, K) for m in range(1, K + 2))
    assert abs(a["acceptance"] - alpha) < 4 * np.sqrt(alpha * (1 - alpha) / tested)
    mean_want = (1 - alpha ** (K + 1)) / (1 - alpha)
    assert abs(a["mean_accept_len"] - mean_want) < 4 * al.std() / np.sqrt(n)
    for i in range(K):
        reached = h[i + 1:].sum()
        assert abs(a["pos_acceptance"][i] - alpha) < 4 * np.sqrt(alpha * (1 - alpha) / reached)


def test_depth_rule():
    K = 4
    # acceptance 0.23 < 0.35: capped; all accepted: full depth; too few tests: unchanged
    low = np.zeros(K + 2, np.uint64)
    low[1], low[2] = 70, 30     # tested 130, accepted 30 -> 0.23
    assert oracle.adapt(low, K, 6, K_floor=1)["next_K"] == 1
    high = np.zeros(K + 2, np.uint64)
    high[5] = 10                # every draft accepted
    assert oracle.adapt(high, K, 6, K_floor=1)["next_K"] == 6
    assert oracle.adapt(high, K, 6, K_floor=1, min_tested=1000)["next_K"] == 4
    assert oracle.adapt(high, 7, 6, K_floor=1, min_tested=1000)["next_K"] == 6
    # exactly at the threshold is not below it
    edge = np.zeros(K + 2, np.uint64)
    edge[1], edge[2] = 13, 7    # tested 1*13 + 2*7 = 27, accepted 7
    a = oracle.adapt(edge, K, 6, threshold=7 / 27)
    assert a["acceptance"] == 7 / 27 and a["next_K"] == 6


def test_library_matches_oracle(sv):
    rng = np.random.default_rng(5)
    cases = []
    for K in (0, 1, 3, 7, 32):
        for _ in range(20):
            h = rng.integers(0, 50, K + 2).astype(np.uint64)
            if rng.random() < 0.2:
                h[1:] = 0
            cases.append((h, K))
    for alpha, K in ((0.35, 3), (0.9, 1)):
        cases.append((oracle.accept_hist(_sweep_lengths(alpha, K, rounds=50), K), K))
    for h, K in cases:
        for K_max, K_floor, thr, mt in ((K, 0, 0.35, 0), (max(K, 5), 1, 0.5, 100), (32, 2, 0.9, 10)):
            o = oracle.adapt(h, K, K_max, K_floor, thr, mt)
            g = sv.spec_adapt(h.tolist(), K, K_max, K_floor, thr, mt)
            assert g["next_K"] == o["next_K"]
            for key in ("acceptance", "mean_accept_len"):
                assert (np.isnan(g[key]) and np.isnan(o[key])) or g[key] == o[key], key
            gp = np.array(g["pos_acceptance"][:K])
            assert np.array_equal(np.isnan(gp), np.isnan(o["pos_acceptance"]))
            assert np.allclose(gp[~np.isnan(gp)], o["pos_acceptance"][~np.isnan(gp)], rtol=0, atol=0)
            assert g["errors"] == int(h[0]) and g["sequences"] == int(h[1:].sum())
            assert all(np.isnan(g["pos_acceptance"][i]) for i in range(K, 32))


def test_library_argument_checks(sv):
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_adapt([0, 1, 2], 3, 3)          # bins < K + 2
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_adapt([0, 1, 2], 1, 3, K_floor=4)
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_adapt([0, 1, 2], 1, 33)
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_adapt([0, 1, 2], 1, 3, threshold=1.5)
    assert sv.spec_verify_set_telemetry(None, None, 0) == sv.SV_ERR_INVALID_ARG
