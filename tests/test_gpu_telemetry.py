"""GPU: the verify kernel's accepted-length counters ([P1] "Production
perspective": record acceptance histograms) against the oracle's histogram of
the same inputs, accumulated over calls, and the library's depth rule read off
them."""
import numpy as np
import pytest

import oracle
import workloads
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _run(v, inp, hist):
    import torch
    lg, qd, td, ud = gh.to_device(inp.logits, inp.dtype, inp.q, inp.tokens, inp.uniforms)
    v.set_telemetry(hist)
    try:
        out = v.run(lg, qd, td, ud, inp.T, status=True)
        torch.cuda.synchronize()
    finally:
        v.set_telemetry(None)
    return {k: t.cpu().numpy() for k, t in out.items()}


@pytest.mark.parametrize("name", ["b64_k3_v151936_bf16", "b8_k4_v32000_bf16_peaked"])
def test_counts_match_the_oracle_histogram(name):
    import torch
    import speculative_decoding_verification_14_gb300 as sv
    inp = workloads.make_config(name)
    o = oracle.verify_inputs(inp)
    v = gh.verifier()
    hist = torch.zeros(inp.K + 2, dtype=torch.int32, device="cuda")
    g1 = _run(v, inp, hist)
    g2 = _run(v, inp, hist)
    h = hist.cpu().numpy().astype(np.uint64)
    # the counters are exactly the call's own accepted lengths, twice
    assert np.array_equal(g1["accept_len"], g2["accept_len"])
    assert np.array_equal(h, 2 * oracle.accept_hist(g1["accept_len"], inp.K))
    # and the oracle's histogram, up to the sequences in the tie band
    info = gh.compare(g1, o, inp.K, label=name)
    ho = oracle.accept_hist(o["accept_len"], inp.K).astype(np.int64)
    ties = info["accept_ties"] + info["draw_ties"]
    assert info["exact"] + ties == inp.B
    assert np.abs(h.astype(np.int64) // 2 - ho).sum() <= 2 * ties
    a_g = sv.spec_adapt((h // 2).tolist(), inp.K, inp.K)
    a_o = oracle.adapt(h // 2, inp.K, inp.K)
    assert a_g["next_K"] == a_o["next_K"] and a_g["acceptance"] == a_o["acceptance"]


def test_errors_land_in_bin_zero_and_bins_are_checked():
    import torch
    import speculative_decoding_verification_14_gb300 as sv
    inp = workloads.make_random(6, 3, 5000, "f32", seed=3)
    tokens = inp.tokens.copy()
    tokens[2, 1] = 5000                      # out of range: sequence 2 errors
    bad = workloads.Inputs(inp.name, inp.B, inp.K, inp.V, inp.dtype, inp.T, inp.logits, inp.q,
                           tokens, inp.uniforms)
    v = gh.verifier()
    v.error()                                # clear the sticky error word
    hist = torch.zeros(inp.K + 2, dtype=torch.int32, device="cuda")
    g = _run(v, bad, hist)
    h = hist.cpu().numpy()
    assert g["accept_len"][2] == 0 and h[0] == 1 and h.sum() == inp.B
    assert np.array_equal(h, np.bincount(g["accept_len"], minlength=inp.K + 2))
    assert v.error()[0] == sv.SV_ERR_TOKEN_RANGE
    small = torch.zeros(inp.K + 1, dtype=torch.int32, device="cuda")
    lg, qd, td, ud = gh.to_device(inp.logits, inp.dtype, inp.q, inp.tokens, inp.uniforms)
    v.set_telemetry(small)
    try:
        with pytest.raises(sv.SpecVerifyError) as e:
            v.run(lg, qd, td, ud, inp.T)
        assert e.value.code == sv.SV_ERR_INVALID_ARG
    finally:
        v.set_telemetry(None)
    torch.cuda.synchronize()
    assert small.sum().item() == 0
