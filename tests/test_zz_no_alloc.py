"""spec_verify_run_noalloc: the context-free, allocation-free entry point.

It must give the same outputs as spec_verify_run on the same inputs, call
after call (its scratch is a static device array that nothing resets), and
reject sizes beyond its limits before launching.  This file is collected last
so that the GPU test also runs after every other test in the same process.
"""
from __future__ import annotations

import numpy as np
import pytest

import workloads
from tests.gpu_helpers import to_device, verifier


def _ptr(t):
    return None if t is None else t.data_ptr()


def _outputs(torch, B, K, dev):
    return {
        "accept_len": torch.full((B,), -7, dtype=torch.int32, device=dev),
        "out_tokens": torch.full((B, K + 1), -7, dtype=torch.int32, device=dev),
        "accept_mask": torch.full((B, max(K, 1)), 7, dtype=torch.uint8, device=dev),
        "row_stats": torch.full((B, K + 1, 2), -7.0, dtype=torch.float32, device=dev),
        "p_draft": torch.full((B, max(K, 1)), -7.0, dtype=torch.float32, device=dev),
        "status": torch.full((B,), -7, dtype=torch.int32, device=dev),
    }


def _run_noalloc(sv, torch, inp, lg, qd, td, ud, stream):
    B, K, V = inp.B, inp.K, inp.V
    out = _outputs(torch, B, K, lg.device)
    rc = sv.spec_verify_run_noalloc(
        lg.device.index, lg.data_ptr(), sv.SV_BF16 if inp.dtype == "bf16" else sv.SV_F32,
        qd.data_ptr() if K else None, td.data_ptr() if K else None, ud.data_ptr(), B, K, V, inp.T,
        _ptr(out["accept_len"]), _ptr(out["out_tokens"]), _ptr(out["accept_mask"]) if K else None,
        _ptr(out["row_stats"]), _ptr(out["p_draft"]) if K else None, _ptr(out["status"]), stream)
    return rc, out


def _same(ref, got, K):
    np.testing.assert_array_equal(got["accept_len"], ref["accept_len"])
    np.testing.assert_array_equal(got["out_tokens"], ref["out_tokens"])
    np.testing.assert_array_equal(got["status"], ref["status"])
    if K:
        np.testing.assert_array_equal(got["accept_mask"][:, :K], ref["accept_mask"][:, :K])
        np.testing.assert_allclose(got["p_draft"][:, :K], ref["p_draft"][:, :K], rtol=1e-6,
                                   equal_nan=True)
    np.testing.assert_allclose(got["row_stats"], ref["row_stats"], rtol=1e-6, equal_nan=True)


CASES = [
    lambda: workloads.make_config("b8_k4_v32000_bf16_peaked"),
    lambda: workloads.make_random(5, 3, 4099, "f32", T=0.9, seed=11),   # rows not 16-byte multiples
    lambda: workloads.make_random(3, 0, 1000, "bf16", T=1.3, seed=12),  # K = 0: bonus draw only
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", range(len(CASES)))
def test_noalloc_matches_the_context_entry_twice_in_a_row(case):
    torch = pytest.importorskip("torch")
    import speculative_decoding_verification_14_gb300 as sv
    inp = CASES[case]()
    B, K = inp.B, inp.K
    lg, qd, td, ud = to_device(inp.logits, inp.dtype, inp.q, inp.tokens, inp.uniforms)
    ref = verifier().run(lg, qd, td, ud, inp.T, stats=True, status=True)
    torch.cuda.synchronize()
    ref = {k: t.cpu().numpy() for k, t in ref.items()}
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        rc, out = _run_noalloc(sv, torch, inp, lg, qd, td, ud, stream)
        assert rc == sv.SV_OK, sv.spec_verify_strerror(rc)
        torch.cuda.synchronize()
        _same(ref, {k: t.cpu().numpy() for k, t in out.items()}, K)
    assert (ref["status"] == 0).all() and (ref["accept_len"] >= 1).all()


@pytest.mark.gpu
def test_noalloc_rejects_sizes_beyond_its_limits():
    torch = pytest.importorskip("torch")
    import speculative_decoding_verification_14_gb300 as sv
    inp = workloads.make_random(2, 2, 64, "f32", seed=13)
    lg, qd, td, ud = to_device(inp.logits, inp.dtype, inp.q, inp.tokens, inp.uniforms)
    out = _outputs(torch, 2, 2, lg.device)
    args = lambda B, K, V: (lg.device.index, lg.data_ptr(), sv.SV_F32, qd.data_ptr(), td.data_ptr(),
                            ud.data_ptr(), B, K, V, 1.0, _ptr(out["accept_len"]),
                            _ptr(out["out_tokens"]), _ptr(out["accept_mask"]), None, None,
                            _ptr(out["status"]), None)
    assert sv.spec_verify_run_noalloc(*args(2, 33, 64)) == sv.SV_ERR_INVALID_ARG
    assert sv.spec_verify_run_noalloc(*args((1 << 20) + 1, 2, 64)) == sv.SV_ERR_INVALID_ARG
    assert sv.spec_verify_run_noalloc(*args(2, 2, (1 << 31) + 1)) == sv.SV_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert (out["accept_len"].cpu().numpy() == -7).all()  # nothing was launched


def test_noalloc_rejects_a_bad_device_without_cuda():
    import speculative_decoding_verification_14_gb300 as sv
    for dev in (-1, 64):
        assert sv.spec_verify_run_noalloc(dev, None, 0, None, None, None, 1, 0, 1, 1.0, None, None,
                                          None) == sv.SV_ERR_INVALID_ARG


@pytest.mark.gpu
def test_noalloc_error_paths_mark_only_their_sequence():
    """Planted faults -- a draft token outside [0, V), a NaN in a row the loop
    reaches, a uniform of 1.0 -- mark only their own sequence: its status
    carries the error, accept_len is 0 and its tokens are -1, as with
    spec_verify_run and the oracle.  A clean call right after still matches
    spec_verify_run."""
    torch = pytest.importorskip("torch")
    import oracle
    import speculative_decoding_verification_14_gb300 as sv
    inp = workloads.make_random(6, 4, 3001, "f32", T=0.8, seed=21)
    lg, x, u = inp.logits.copy(), inp.tokens.copy(), inp.uniforms.copy()
    x[1, 2] = inp.V                 # token out of range
    lg[3, 0, 1234] = np.nan         # row 0 is always reached
    u[4, 1] = np.float32(1.0)       # uniform outside [0, 1)
    inp.logits, inp.tokens, inp.uniforms = lg, x, u
    want = oracle.verify_inputs(inp)
    assert list(want["status"]) == [0, sv.SV_ERR_TOKEN_RANGE, 0, sv.SV_ERR_NONFINITE,
                                    sv.SV_ERR_UNIFORM_RANGE, 0]
    d = to_device(inp.logits, inp.dtype, inp.q, inp.tokens, inp.uniforms)
    ref = verifier().run(*d, inp.T, stats=True, status=True)
    torch.cuda.synchronize()
    ref = {k: t.cpu().numpy() for k, t in ref.items()}
    stream = torch.cuda.current_stream().cuda_stream
    rc, out = _run_noalloc(sv, torch, inp, *d, stream)
    assert rc == sv.SV_OK, sv.spec_verify_strerror(rc)
    torch.cuda.synchronize()
    got = {k: t.cpu().numpy() for k, t in out.items()}
    _same(ref, got, inp.K)
    np.testing.assert_array_equal(got["status"], want["status"])
    bad = want["status"] != 0
    assert (got["accept_len"][bad] == 0).all()
    assert (got["out_tokens"][bad] == -1).all()
    assert (got["accept_mask"][bad] == 0).all()
    np.testing.assert_array_equal(got["accept_len"][~bad], want["accept_len"][~bad])
    # a clean call after the faulty one: the same outputs as the context entry
    clean = workloads.make_random(6, 4, 3001, "f32", T=0.8, seed=22)
    dc = to_device(clean.logits, clean.dtype, clean.q, clean.tokens, clean.uniforms)
    ref = verifier().run(*dc, clean.T, stats=True, status=True)
    torch.cuda.synchronize()
    ref = {k: t.cpu().numpy() for k, t in ref.items()}
    rc, out = _run_noalloc(sv, torch, clean, *dc, stream)
    assert rc == sv.SV_OK
    torch.cuda.synchronize()
    _same(ref, {k: t.cpu().numpy() for k, t in out.items()}, clean.K)
    assert (ref["status"] == 0).all()
