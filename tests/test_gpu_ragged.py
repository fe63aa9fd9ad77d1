"""GPU parity for ragged batches (per-sequence draft depth K_b, packed rows):
the CUDA library through spec_verify_run_ragged against oracle.verify_ragged
on the same inputs.  Same bar as the uniform verify (tests/gpu_helpers.py):
bit-exact outside the 1e-6 tie band, statuses exact, row statistics within
1e-5 relative."""
import numpy as np
import pytest

import oracle
import workloads
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _gpu(rg, plan=None, offsets=None, v=None):
    import torch
    v = v or gh.verifier()
    if rg.dtype == "bf16":
        lg = torch.from_numpy(rg.logits.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        lg = torch.from_numpy(rg.logits).cuda()
    q = torch.from_numpy(rg.q).cuda()
    x = torch.from_numpy(rg.tokens).cuda()
    u = torch.from_numpy(rg.uniforms).cuda()
    off = torch.from_numpy(rg.offsets if offsets is None else offsets).cuda()
    if plan:
        v.set_plan_override(*plan)
    try:
        out = v.run_ragged(lg, q, x, u, off, rg.K_max, rg.T, stats=True)
        torch.cuda.synchronize()
    finally:
        if plan:
            v.set_plan_override(0, 0, 0)
    return {k: t.cpu().numpy() for k, t in out.items()}


def _compare(g, o, offsets, label):
    B = o["accept_len"].size
    assert np.array_equal(g["status"], o["status"]), label
    ok = o["status"] == 0
    tie = (o["accept_margin"] < gh.TIE) | (o["sample_margin"] < gh.TIE)
    exact = ok & ~tie
    for b in range(B):
        r0, r1 = int(offsets[b]), int(offsets[b + 1])
        if not ok[b]:
            assert g["accept_len"][b] == 0, f"{label}: error row {b}"
            continue
        n = int(g["accept_len"][b])
        assert 1 <= n <= r1 - r0, f"{label}: row {b} length {n}"
        if exact[b]:
            assert n == o["accept_len"][b], f"{label}: row {b} length {n} vs {o['accept_len'][b]}"
            assert np.array_equal(g["out_tokens"][r0:r1], o["out_tokens"][r0:r1]), f"{label}: {b}"
            d0, d1 = r0 - b, r1 - b - 1
            assert np.array_equal(g["accept_mask"][d0:d1], o["accept_mask"][d0:d1]), f"{label}: {b}"
    both = ~np.isnan(g["row_stats"][:, 1]) & ~np.isnan(o["row_s"])
    rows_exact = np.zeros(offsets[-1], bool)
    for b in np.nonzero(exact)[0]:
        rows_exact[offsets[b]:offsets[b + 1]] = True
    assert np.array_equal(np.isnan(g["row_stats"][rows_exact, 1]), np.isnan(o["row_s"][rows_exact]))
    if both.any():
        rel = np.abs(g["row_stats"][both, 1] - o["row_s"][both]) / np.abs(o["row_s"][both])
        assert rel.max() < gh.RTOL, f"{label}: normaliser rel err {rel.max():.2e}"
    return int(exact.sum()), int((ok & tie).sum())


def test_full_size_mixed_depths():
    """The 256-sequence, V = 128256 bf16 workload with K_b drawn from 0..7."""
    inp = workloads.make_config("b256_k7_v128256_bf16_zipf")
    Ks = np.random.default_rng(0).integers(0, 8, inp.B)
    rg = workloads.ragged_from(inp, Ks)
    o = oracle.verify_ragged(rg.logits, rg.dtype, rg.q, rg.tokens, rg.uniforms, rg.offsets,
                             rg.K_max, rg.T)
    g = _gpu(rg)
    exact, ties = _compare(g, o, rg.offsets, "b256 ragged")
    # draw ties (a uniform within 1e-6 of a CDF boundary) are frequent on these
    # long flat rows; they are checked for validity, not counted as exact
    assert exact + ties == inp.B and exact >= 0.85 * inp.B


@pytest.mark.parametrize("plan", [None, (1, 0, 0), (4, 1, 0), (8, 2, 0), (16, 0, 0), (2, 3, 256)])
@pytest.mark.parametrize("dtype,V", [("bf16", 32000), ("f32", 4099), ("bf16", 1001)])
def test_random_shapes_every_plan(dtype, V, plan):
    inp = workloads.make_random(20, 6, V, dtype, seed=V % 89)
    Ks = np.random.default_rng(V).integers(0, 7, inp.B)
    Ks[:2] = (0, 6)
    rg = workloads.ragged_from(inp, Ks)
    o = oracle.verify_ragged(rg.logits, rg.dtype, rg.q, rg.tokens, rg.uniforms, rg.offsets,
                             rg.K_max, rg.T)
    _compare(_gpu(rg, plan), o, rg.offsets, f"{dtype} V={V} plan={plan}")


def test_equal_depths_match_the_uniform_entry_point():
    inp = workloads.make_config("b64_k3_v151936_bf16")
    rg = workloads.ragged_from(inp, np.full(inp.B, inp.K))
    g = _gpu(rg)
    u = gh.gpu_verify_inputs(inp)
    assert np.array_equal(g["accept_len"], u["accept_len"])
    assert np.array_equal(g["out_tokens"], u["out_tokens"].reshape(-1))
    assert np.array_equal(g["row_stats"], u["row_stats"].reshape(-1, 2), equal_nan=True)


def test_bad_offsets_mark_only_their_sequence():
    import speculative_decoding_verification_14_gb300 as sv
    v = gh.verifier()
    v.error()
    inp = workloads.make_random(6, 3, 3000, "bf16", seed=7)
    rg = workloads.ragged_from(inp, np.array([3, 1, 2, 0, 3, 2]))
    good = _gpu(rg)
    for bad_b, edit in ((1, lambda o: o.__setitem__(2, o[1])),
                        (2, lambda o: o.__setitem__(3, o[2] + 9)),
                        (0, lambda o: o.__setitem__(0, -1)),
                        (5, lambda o: o.__setitem__(6, rg.R + 1))):
        off = rg.offsets.copy()
        edit(off)
        o = oracle.verify_ragged(rg.logits, rg.dtype, rg.q, rg.tokens, rg.uniforms, off,
                                 rg.K_max, rg.T)
        g = _gpu(rg, offsets=off)
        assert np.array_equal(g["status"], o["status"])
        assert g["status"][bad_b] == sv.SV_ERR_BAD_OFFSETS and g["accept_len"][bad_b] == 0
        for b in range(rg.B):
            if g["status"][b] == 0:
                assert g["accept_len"][b] == good["accept_len"][b]
        assert v.error()[0] == sv.SV_ERR_BAD_OFFSETS
