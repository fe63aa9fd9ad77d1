"""Pins for the oracle's ragged batches (per-sequence draft depth K_b, packed
rows).  [P1]'s loop verifies one sequence at a time, so a ragged batch must
give, sequence by sequence, what the uniform verify gives for that sequence
alone; the packing arithmetic is checked against slices cut here, and
offsets that describe no packing mark only their own sequence."""
import numpy as np
import pytest

import oracle
import workloads


def _ragged_vs_uniform(inp, Ks):
    rg = workloads.ragged_from(inp, Ks)
    o = oracle.verify_ragged(rg.logits, rg.dtype, rg.q, rg.tokens, rg.uniforms, rg.offsets,
                             inp.K, rg.T)
    for b, k in enumerate(Ks):
        r0, r1 = rg.offsets[b], rg.offsets[b + 1]
        d0, d1 = r0 - b, r1 - b - 1
        ref = oracle.verify(inp.logits[b:b + 1, :k + 1], inp.dtype, inp.q[b:b + 1, :k],
                            inp.tokens[b:b + 1, :k], inp.uniforms[b:b + 1, :k + 1], inp.T)
        assert o["accept_len"][b] == ref["accept_len"][0]
        assert o["status"][b] == ref["status"][0]
        assert np.array_equal(o["out_tokens"][r0:r1], ref["out_tokens"][0])
        assert np.array_equal(o["accept_mask"][d0:d1], ref["accept_mask"][0])
        assert np.array_equal(o["row_s"][r0:r1], ref["row_s"][0], equal_nan=True)
        assert np.array_equal(o["p_draft"][d0:d1], ref["p_draft"][0], equal_nan=True)
        assert o["sample_margin"][b] == ref["sample_margin"][0]
    return o


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_mixed_depths_match_each_sequence_alone(dtype):
    inp = workloads.make_random(40, 7, 300, dtype, seed=12)
    Ks = np.random.default_rng(1).integers(0, 8, 40)
    Ks[:3] = (0, 7, 0)
    o = _ragged_vs_uniform(inp, Ks)
    assert np.all((o["accept_len"] >= 1) & (o["accept_len"] <= Ks + 1))


def test_equal_depths_are_the_uniform_batch():
    inp = workloads.make_random(16, 4, 500, "f32", seed=3)
    rg = workloads.ragged_from(inp, np.full(16, 4))
    o = oracle.verify_ragged(rg.logits, rg.dtype, rg.q, rg.tokens, rg.uniforms, rg.offsets, 4,
                             rg.T)
    u = oracle.verify_inputs(inp)
    assert np.array_equal(o["accept_len"], u["accept_len"])
    assert np.array_equal(o["out_tokens"], u["out_tokens"].reshape(-1))
    assert np.array_equal(o["accept_mask"], u["accept_mask"].reshape(-1))
    assert np.array_equal(o["row_s"], u["row_s"].reshape(-1), equal_nan=True)


def test_bad_offsets_mark_only_their_sequence():
    inp = workloads.make_random(6, 3, 200, "f32", seed=5)
    rg = workloads.ragged_from(inp, np.array([3, 1, 2, 0, 3, 2]))
    good = oracle.verify_ragged(rg.logits, rg.dtype, rg.q, rg.tokens, rg.uniforms, rg.offsets, 3,
                                rg.T)
    for bad_b, off in ((1, lambda o: o.__setitem__(2, o[1])),          # K_1 = -1
                       (2, lambda o: o.__setitem__(3, o[2] + 9)),      # K_2 = 8 > K_max
                       (0, lambda o: o.__setitem__(0, -1))):           # before the array
        o = rg.offsets.copy()
        off(o)
        res = oracle.verify_ragged(rg.logits, rg.dtype, rg.q, rg.tokens, rg.uniforms, o, 3, rg.T)
        assert res["status"][bad_b] == oracle.BAD_OFFSETS and res["accept_len"][bad_b] == 0
        for b in range(6):
            if res["status"][b] == oracle.BAD_OFFSETS:
                continue
            assert res["accept_len"][b] == good["accept_len"][b]
    # the last sequence running past the packed rows
    o = rg.offsets.copy()
    o[-1] = rg.R + 1
    res = oracle.verify_ragged(rg.logits, rg.dtype, rg.q, rg.tokens, rg.uniforms, o, 3, rg.T)
    assert res["status"][-1] == oracle.BAD_OFFSETS
    assert np.array_equal(res["accept_len"][:-1], good["accept_len"][:-1])
