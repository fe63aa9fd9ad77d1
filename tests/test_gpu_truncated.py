"""GPU parity for verification against a truncated target (top-p, min-p): the
CUDA kernel through spec_verify_run_truncated against
oracle.verify_truncated on the same inputs.

Bar: as for the sampled verify (tests/gpu_helpers.py) -- bit-exact outside
the 1e-6 tie band, statuses exact, untruncated row statistics and p~(x)
within 1e-5 relative -- with one more kind of tie: a row the loop reaches
that lies within 1e-6 of a filter boundary (a token's log(p/p_max) within 1e-6
of log(min_p), or a mass-above value within 1e-6 of top_p), where float32 and
float64 may keep different sets; such sequences are counted and checked for
validity only."""
import json

import numpy as np
import pytest

import oracle
import workloads
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _gpu(inp, top_p, min_p, cluster=0):
    import torch
    v = gh.verifier()
    lg, qd, td, ud = gh.to_device(inp.logits, inp.dtype, inp.q, inp.tokens, inp.uniforms)
    if cluster:
        v.set_plan_override(cluster, 0, 0)
    try:
        out = v.run_truncated(lg, qd, td, ud, inp.T, top_p, min_p, stats=True)
        torch.cuda.synchronize()
    finally:
        if cluster:
            v.set_plan_override(0, 0, 0)
    res = {k: t.cpu().numpy() for k, t in out.items()}
    res["row_m"] = res["row_stats"][..., 0].astype(np.float64)
    res["row_s"] = res["row_stats"][..., 1].astype(np.float64)
    res["p_draft"] = res["p_draft"].astype(np.float64)
    return res


def _check(inp, top_p, min_p, label, cluster=0):
    o = oracle.verify_truncated(inp.logits, inp.dtype, inp.q, inp.tokens, inp.uniforms, inp.T,
                                top_p, min_p, lib=gh.oracle_lib())
    g = _gpu(inp, top_p, min_p, cluster)
    tt = o["trunc_margin"] < gh.TIE
    # truncation ties: validity only (folded into the acceptance-tie class),
    # and their p~(x) is not compared
    o = dict(o)
    o["accept_margin"] = np.where(tt, 0.0, o["accept_margin"])
    o["p_draft"] = np.where(tt[:, None], np.nan, o["p_draft"])
    g["p_draft"] = np.where(tt[:, None], np.nan, g["p_draft"])
    info = gh.compare(g, o, inp.K, label=label)
    info["trunc_ties"] = int(tt.sum())
    return info, o


@pytest.mark.parametrize("name", ["b8_k4_v32000_bf16_peaked", "b64_k3_v151936_bf16",
                                  "b1_k4_v32000_f32"])
def test_workloads_at_the_production_settings(name):
    """Each workload at its own temperature with top-p 0.95 and min-p 0.05."""
    inp = workloads.make_config(name)
    info, _ = _check(inp, 0.95, 0.05, name)
    assert info["exact"] + info["accept_ties"] + info["draw_ties"] == inp.B


def test_b256_full_at_the_production_settings():
    """All 256 sequences of the 256 x 8 x 128256 bf16 workload, at [P2]'s
    production sampler settings (top-p 0.95, min-p 0.05), under the plan the
    planner picks for that size (the one the benchmark times).  Every sequence
    is exact or a counted tie; the ties stay below 8 % of the batch."""
    inp = workloads.make_config("b256_k7_v128256_bf16_zipf")
    info, _ = _check(inp, 0.95, 0.05, "b256 full")
    ties = info["accept_ties"] + info["draw_ties"] + info["trunc_ties"]
    print("truncated b256 full: " + json.dumps(info))
    assert info["exact"] + info["accept_ties"] + info["draw_ties"] == inp.B
    assert ties <= 0.08 * inp.B


@pytest.mark.parametrize("cluster", [0, 1, 2, 4, 8])
@pytest.mark.parametrize("dtype,V,T", [("bf16", 32000, 0.6), ("f32", 4099, 1.0),
                                       ("bf16", 1001, 0.6), ("f32", 64, 0.8)])
@pytest.mark.parametrize("top_p,min_p", [(0.95, 0.05), (0.9, 0.0), (1.0, 0.1), (1.0, 0.0)])
def test_random_shapes(dtype, V, T, top_p, min_p, cluster):
    inp = workloads.make_random(16, 4, V, dtype, T=T, sigma=3.0, seed=V % 97 + cluster)
    _check(inp, top_p, min_p, f"{dtype} V={V} T={T} p={top_p} m={min_p} C={cluster}", cluster)


def test_filters_off_match_the_sampled_kernel():
    inp = workloads.make_config("b64_k3_v151936_bf16")
    g = _gpu(inp, 1.0, 0.0)
    s = gh.gpu_verify_inputs(inp)
    o = oracle.verify_inputs(inp)
    tie = (o["accept_margin"] < gh.TIE) | (o["sample_margin"] < gh.TIE)
    assert np.array_equal(g["accept_len"][~tie], s["accept_len"][~tie])
    assert np.array_equal(g["out_tokens"][~tie], s["out_tokens"][~tie])


def test_errors_and_special_values():
    import speculative_decoding_verification_14_gb300 as sv
    v = gh.verifier()
    v.error()
    inp = workloads.make_random(6, 3, 3000, "f32", T=0.6, seed=9)
    lg = inp.logits.copy()
    lg[1, 0, 5] = np.nan
    lg[2, :, :2000] = -np.inf                 # -inf entries: weight 0, never kept
    x = inp.tokens.copy()
    x[3, 1] = 3000                            # out of range
    bad = workloads.Inputs(inp.name, inp.B, inp.K, inp.V, inp.dtype, inp.T, lg, inp.q, x,
                           inp.uniforms)
    info, o = _check(bad, 0.95, 0.05, "errors")
    assert o["status"][1] == oracle.NONFINITE and o["status"][3] == oracle.TOKEN_RANGE
    rc, mask = v.error()
    assert mask == (1 << sv.SV_ERR_NONFINITE) | (1 << sv.SV_ERR_TOKEN_RANGE)
    import torch
    with pytest.raises(sv.SpecVerifyError):
        lgd, qd, td, ud = gh.to_device(inp.logits, inp.dtype, inp.q, inp.tokens, inp.uniforms)
        v.run_truncated(lgd, qd, td, ud, inp.T, 0.0, 0.05)
    torch.cuda.synchronize()


@pytest.mark.parametrize("entry", ["truncated", "draft_logits"])
def test_repeated_runs_with_filters_are_bit_identical(entry):
    """With top-p < 1 and min-p > 0 two runs give the same bits: the top-p
    histograms add fixed-point integers, so the order in which warps add their
    weights cannot move a cut.  The rows hold many equal logits, so that
    top-p masses land on bin boundaries."""
    import torch
    v = gh.verifier()
    if entry == "truncated":
        inp = workloads.make_random(12, 4, 5000, "bf16", T=0.7, sigma=1.0, seed=41)
    else:
        inp = workloads.make_random_draft_logits(12, 4, 5000, "bf16", T=0.7, T_draft=0.9,
                                                 sigma=1.0, seed=41)
    lg = inp.logits.copy()
    lg[:, :, ::3] = lg[:, :, :1]                 # a third of every row ties the first entry
    inp.logits = lg
    runs = []
    for _ in range(3):
        if entry == "truncated":
            lgd, qd, td, ud = gh.to_device(inp.logits, inp.dtype, inp.q, inp.tokens, inp.uniforms)
            out = v.run_truncated(lgd, qd, td, ud, inp.T, 0.9, 0.05, stats=True)
        else:
            lgd, _, td, ud = gh.to_device(inp.logits, inp.dtype, np.zeros(1, np.float32),
                                          inp.tokens, inp.uniforms)
            dld = torch.from_numpy(np.ascontiguousarray(inp.dlogits).view(np.int16)).cuda().view(
                torch.bfloat16)
            out = v.run_draft_logits(lgd, dld, td, ud, inp.T, inp.T_draft, 0.9, 0.05, stats=True)
        torch.cuda.synchronize()
        runs.append({k: t.cpu().numpy().copy() for k, t in out.items()})
    for r in runs[1:]:
        for k in runs[0]:
            np.testing.assert_array_equal(runs[0][k], r[k], err_msg=k)


def test_draft_values_checked_at_kept_tokens_only():
    """Against the truncated target q_j is read, and checked, where p~_j > 0:
    a NaN at a dropped token of the rejected row leaves the sequence as it
    was, a NaN at a kept token makes it an error -- on the survivor-list path
    (min-p on) and on the row path (top-p alone)."""
    import torch
    inp = workloads.make_random(8, 3, 4000, "bf16", T=0.7, sigma=3.0, seed=52)
    for top_p, min_p in ((0.95, 0.05), (0.9, 0.0)):
        base = oracle.verify_truncated(inp.logits, inp.dtype, inp.q, inp.tokens, inp.uniforms,
                                       inp.T, top_p, min_p)
        rej = [b for b in range(inp.B) if base["status"][b] == 0 and base["accept_len"][b] <= inp.K]
        assert len(rej) >= 2
        lgf = (inp.logits.astype(np.uint32) << 16).view(np.float32)
        q = inp.q.copy()
        b0, b1 = rej[0], rej[1]
        j0, j1 = base["accept_len"][b0] - 1, base["accept_len"][b1] - 1
        q[b0, j0, int(np.argmin(lgf[b0, j0]))] = np.nan   # dropped by either filter
        q[b1, j1, int(np.argmax(lgf[b1, j1]))] = np.nan   # always kept
        bad = workloads.Inputs(inp.name, inp.B, inp.K, inp.V, inp.dtype, inp.T, inp.logits, q,
                               inp.tokens, inp.uniforms)
        info, o = _check(bad, top_p, min_p, f"q NaN p={top_p} m={min_p}")
        assert o["status"][b0] == 0 and o["status"][b1] == oracle.NONFINITE
        np.testing.assert_array_equal(o["out_tokens"][b0], base["out_tokens"][b0])
    torch.cuda.synchronize()
