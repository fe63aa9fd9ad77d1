"""GPU parity for verification with draft logits: the CUDA kernel through
spec_verify_run_draft_logits against oracle.verify_draft_logits on the same
inputs (q_i = softmax(d_i / T_d), formed by each side on its own).

Bar: as for the sampled verify (tests/gpu_helpers.py) -- bit-exact outside the
1e-6 tie band, statuses exact, row statistics and p(x) within 1e-5 relative --
and, with a truncated target, the truncated test's extra tie class (a reached
row within 1e-6 of a filter boundary: validity only)."""
import json

import numpy as np
import pytest

import oracle
import workloads
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _to_dev(a, dtype):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _gpu(inp, top_p=1.0, min_p=0.0, cluster=0, dl_dev=None, tokens=None):
    import torch
    v = gh.verifier()
    lg = _to_dev(inp.logits, inp.dtype)
    dl = _to_dev(inp.dlogits, inp.dtype) if dl_dev is None else dl_dev
    x = torch.from_numpy(np.ascontiguousarray(inp.tokens if tokens is None else tokens,
                                              dtype=np.int32)).cuda()
    u = torch.from_numpy(np.ascontiguousarray(inp.uniforms, dtype=np.float32)).cuda()
    if cluster:
        v.set_plan_override(cluster, 0, 0)
    try:
        out = v.run_draft_logits(lg, dl, x, u, inp.T, inp.T_draft, top_p, min_p, stats=True)
        torch.cuda.synchronize()
    finally:
        if cluster:
            v.set_plan_override(0, 0, 0)
    res = {k: t.cpu().numpy() for k, t in out.items()}
    res["row_m"] = res["row_stats"][..., 0].astype(np.float64)
    res["row_s"] = res["row_stats"][..., 1].astype(np.float64)
    res["p_draft"] = res["p_draft"].astype(np.float64)
    return res


def _check(inp, top_p=1.0, min_p=0.0, label="", cluster=0, dl_dev=None, tokens=None,
           dlogits=None):
    o = oracle.verify_draft_logits(inp.logits, inp.dtype,
                                   inp.dlogits if dlogits is None else dlogits,
                                   inp.tokens if tokens is None else tokens, inp.uniforms, inp.T,
                                   inp.T_draft, top_p, min_p, lib=gh.oracle_lib())
    g = _gpu(inp, top_p, min_p, cluster, dl_dev, tokens)
    tt = o["trunc_margin"] < gh.TIE
    o = dict(o)
    o["accept_margin"] = np.where(tt, 0.0, o["accept_margin"])
    o["p_draft"] = np.where(tt[:, None], np.nan, o["p_draft"])
    g["p_draft"] = np.where(tt[:, None], np.nan, g["p_draft"])
    info = gh.compare(g, o, inp.K, label=label)
    info["trunc_ties"] = int(tt.sum())
    return info, o, g


@pytest.mark.parametrize("name", ["b1_k4_v32000_f32", "b8_k4_v32000_bf16_peaked",
                                  "b64_k3_v151936_bf16", "b256_k7_v128256_bf16_zipf"])
def test_workloads_full_size(name):
    """Each workload at full size with the drafter's logits (draft = target +
    noise, stored in the target's dtype, T_d = T)."""
    inp = workloads.with_draft_logits(name)
    info, o, _ = _check(inp, label=name)
    assert info["exact"] + info["accept_ties"] + info["draw_ties"] == inp.B
    assert info["exact"] >= 0.8 * inp.B


@pytest.mark.parametrize("name", ["b64_k3_v151936_bf16", "b256_k7_v128256_bf16_zipf"])
def test_workloads_truncated_target(name):
    """Draft logits with [P2]'s production sampler settings (top-p 0.95, min-p
    0.05) on the target side, every sequence of the workload, under the
    planner's own plan.  Every sequence is exact or a counted tie; the ties stay
    below 8 % of the batch."""
    inp = workloads.with_draft_logits(name)
    info, _, _ = _check(inp, 0.95, 0.05, label=name + " top-p/min-p")
    print("draft logits, truncated target: " + json.dumps({"case": name, **info}))
    assert info["exact"] + info["accept_ties"] + info["draw_ties"] == inp.B
    assert info["accept_ties"] + info["draw_ties"] + info["trunc_ties"] <= 0.08 * inp.B


@pytest.mark.parametrize("cluster", [0, 1, 2, 4, 8, 16])
@pytest.mark.parametrize("dtype,V,T,Td", [("bf16", 32000, 0.6, 0.6), ("f32", 4099, 1.0, 1.3),
                                          ("bf16", 1001, 0.7, 0.5), ("f32", 64, 0.8, 0.8)])
@pytest.mark.parametrize("top_p,min_p", [(1.0, 0.0), (0.95, 0.05)])
def test_random_shapes(dtype, V, T, Td, top_p, min_p, cluster):
    if cluster == 16 and (top_p < 1.0 or min_p > 0.0):
        pytest.skip("the truncated kernel's clusters stop at 8 CTAs")
    inp = workloads.make_random_draft_logits(16, 4, V, dtype, T=T, T_draft=Td, sigma=3.0,
                                             seed=V % 89 + cluster)
    _check(inp, top_p, min_p, f"{dtype} V={V} T={T} Td={Td} p={top_p} m={min_p} C={cluster}",
           cluster)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_large_batch_on_three_stage_rings(dtype):
    """Batches too large for the six-stage rings, one CTA per sequence: the
    draft-logit form of the 128-thread kernel with three stages per warp."""
    inp = workloads.make_random_draft_logits(800, 3, 3000, dtype, T=0.9, T_draft=1.2, seed=41)
    p = gh.verifier().plan_draft_logits(inp.B, inp.K, inp.V, 1 if dtype == "bf16" else 0, 0)
    assert p["stages"] == 3 and p["threads"] == 128 and p["group"] == 1
    info, _, _ = _check(inp, label=f"{dtype} three stages")
    assert info["exact"] + info["accept_ties"] + info["draw_ties"] == inp.B


@pytest.mark.parametrize("K", [0, 1, 32])
def test_depths(K):
    inp = workloads.make_random_draft_logits(12, K, 2048, "bf16", T=0.9, T_draft=1.1, seed=K + 5)
    info, _, _ = _check(inp, label=f"K={K}")
    assert info["exact"] + info["accept_ties"] + info["draw_ties"] == inp.B


def test_unaligned_draft_rows_take_the_element_path():
    """A draft tensor that starts 2 bytes past a 16-byte boundary."""
    import torch
    inp = workloads.make_random_draft_logits(8, 3, 4096, "bf16", T=0.8, T_draft=0.8, seed=31)
    flat = np.concatenate([np.zeros(1, np.uint16), inp.dlogits.reshape(-1)])
    buf = _to_dev(flat, "bf16")
    dl = buf[1:].view(inp.B, inp.K, inp.V)
    assert dl.data_ptr() % 16 == 2
    info, _, _ = _check(inp, label="unaligned draft", dl_dev=dl)
    assert info["exact"] + info["accept_ties"] + info["draw_ties"] == inp.B
    torch.cuda.synchronize()


def test_errors_and_special_values():
    import speculative_decoding_verification_14_gb300 as sv
    v = gh.verifier()
    v.error()
    inp = workloads.make_random_draft_logits(8, 3, 3000, "f32", T=0.6, T_draft=0.6, seed=9)
    dl = inp.dlogits.copy()
    dl[1, 0, 7] = np.nan                  # a reached draft row: error
    dl[2, 0, :] = -np.inf                 # a reached draft row of only -inf: error
    dl[4, 2, 11] = np.inf                 # row 2 of sequence 4: an error only if reached
    dl[5, 0, :1500] = -np.inf             # -inf entries: q = 0 there (legal)
    x = inp.tokens.copy()
    x[3, 1] = 3000                        # out of range
    bad = workloads.DraftLogitInputs(inp.name, inp.B, inp.K, inp.V, inp.dtype, inp.T, inp.T_draft,
                                     inp.logits, dl, inp.q, x, inp.uniforms)
    info, o, g = _check(bad, label="errors", dlogits=dl, tokens=x)
    assert o["status"][1] == oracle.NONFINITE and o["status"][2] == oracle.NONFINITE
    assert o["status"][3] == oracle.TOKEN_RANGE
    assert o["status"][5] == oracle.OK
    rc, mask = v.error()
    assert mask == (1 << sv.SV_ERR_NONFINITE) | (1 << sv.SV_ERR_TOKEN_RANGE)
    import torch
    lg = _to_dev(inp.logits, "f32")
    dd = _to_dev(inp.dlogits, "f32")
    xd = torch.from_numpy(inp.tokens).cuda()
    ud = torch.from_numpy(inp.uniforms).cuda()
    for T_draft, top_p in ((0.0, 1.0), (float("nan"), 1.0), (1.0, 0.0)):
        with pytest.raises(sv.SpecVerifyError):
            v.run_draft_logits(lg, dd, xd, ud, inp.T, T_draft, top_p, 0.0)
    torch.cuda.synchronize()


def test_agrees_with_the_q_kernel_fed_the_softmax():
    """The same verify through spec_verify_run with q = softmax(d / T_d)
    rounded to float32: equal outside the tie bands of both oracles."""
    inp = workloads.with_draft_logits("b64_k3_v151936_bf16")
    g = _gpu(inp)
    s = gh.gpu_verify(inp.logits, inp.dtype, inp.q, inp.tokens, inp.uniforms, inp.T)
    o = oracle.verify_draft_logits(inp.logits, inp.dtype, inp.dlogits, inp.tokens, inp.uniforms,
                                   inp.T, inp.T_draft)
    r = oracle.verify(inp.logits, inp.dtype, inp.q, inp.tokens, inp.uniforms, inp.T)
    tie = ((o["accept_margin"] < 1e-5) | (o["sample_margin"] < 1e-5) |
           (r["accept_margin"] < 1e-5) | (r["sample_margin"] < 1e-5))
    assert np.array_equal(g["accept_len"][~tie], s["accept_len"][~tie])
    assert np.array_equal(g["out_tokens"][~tie], s["out_tokens"][~tie])


@pytest.mark.parametrize("top_p,min_p", [(1.0, 0.0), (0.95, 0.05)])
def test_telemetry_counts(top_p, min_p):
    """The accepted-length counters of the draft-logit kernel: twice the
    histogram of its own accepted lengths after two calls, errors in bin 0."""
    import torch
    v = gh.verifier()
    inp = workloads.make_random_draft_logits(40, 5, 3000, "bf16", T=0.7, T_draft=0.9, seed=17)
    x = inp.tokens.copy()
    x[3, 2] = -1                                   # sequence 3 errors
    hist = torch.zeros(inp.K + 2, dtype=torch.int32, device="cuda")
    lg, dl = _to_dev(inp.logits, "bf16"), _to_dev(inp.dlogits, "bf16")
    xd = torch.from_numpy(x).cuda()
    ud = torch.from_numpy(inp.uniforms).cuda()
    v.set_telemetry(hist)
    try:
        o1 = v.run_draft_logits(lg, dl, xd, ud, inp.T, inp.T_draft, top_p, min_p)
        o2 = v.run_draft_logits(lg, dl, xd, ud, inp.T, inp.T_draft, top_p, min_p)
        torch.cuda.synchronize()
    finally:
        v.set_telemetry(None)
    v.error()
    al1, al2 = o1["accept_len"].cpu().numpy(), o2["accept_len"].cpu().numpy()
    assert np.array_equal(al1, al2) and al1[3] == 0
    h = hist.cpu().numpy().astype(np.int64)
    expect = np.bincount(al1, minlength=inp.K + 2)
    assert np.array_equal(h, 2 * expect)


def test_repeated_runs_are_bit_identical_and_outputs_stay_in_bounds():
    """Two runs give the same bits; guard regions around every output keep
    their fill (no write outside [B], [B, K+1], [B, K], [B, K+1, 2])."""
    import torch
    v = gh.verifier()
    inp = workloads.make_random_draft_logits(9, 4, 3000, "bf16", T=0.8, T_draft=0.8, seed=23)
    B, K = inp.B, inp.K
    lg, dl = _to_dev(inp.logits, "bf16"), _to_dev(inp.dlogits, "bf16")
    xd = torch.from_numpy(inp.tokens).cuda()
    ud = torch.from_numpy(inp.uniforms).cuda()
    guard = 64
    runs = []
    for _ in range(2):
        fences, out = [], {}
        for name, shape, dtype, fill in (("accept_len", (B,), torch.int32, 0x5A5A5A5A),
                                         ("out_tokens", (B, K + 1), torch.int32, 0x5A5A5A5A),
                                         ("accept_mask", (B, K), torch.uint8, 0xA5),
                                         ("row_stats", (B, K + 1, 2), torch.float32, 12345.0),
                                         ("p_draft", (B, K), torch.float32, 12345.0),
                                         ("status", (B,), torch.int32, 0x5A5A5A5A)):
            n = int(np.prod(shape))
            full = torch.full((n + 2 * guard,), fill, dtype=dtype, device="cuda")
            fences.append((name, full, n, fill))
            out[name] = full[guard:guard + n].view(shape)
        v.run_draft_logits(lg, dl, xd, ud, inp.T, inp.T_draft, out=out)
        torch.cuda.synchronize()
        for name, full, n, fill in fences:
            assert torch.all(full[:guard] == fill) and torch.all(full[guard + n:] == fill), name
        runs.append({k: t.cpu().numpy().copy() for k, t in out.items()})
    for k in runs[0]:
        np.testing.assert_array_equal(runs[0][k], runs[1][k], err_msg=k)
    assert np.all(runs[0]["status"] == 0)
