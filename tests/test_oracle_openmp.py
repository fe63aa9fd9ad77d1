"""The OpenMP build of the oracle (the same oracle.c with -fopenmp, sequences
spread over host threads) gives results identical to the plain build: each
sequence's arithmetic is unchanged, only which thread runs it differs.  The
benchmark's all-core CPU baseline times this build."""
import numpy as np
import pytest

import oracle
import workloads


@pytest.fixture(scope="module")
def omp():
    try:
        return oracle.load_openmp(threads=4)
    except Exception as e:  # no OpenMP runtime for this compiler
        pytest.skip(f"OpenMP build unavailable: {e}")


def same(a, b):
    for k in a:
        if a[k].dtype.kind == "f":
            assert np.array_equal(a[k], b[k], equal_nan=True), k
        else:
            assert np.array_equal(a[k], b[k]), k


def test_thread_count(omp):
    assert omp.oracle_threads() == 4


@pytest.mark.parametrize("dtype,V", [("bf16", 3001), ("f32", 257)])
def test_sampled_verify_identical(omp, dtype, V):
    inp = workloads.make_random(37, 5, V, dtype, seed=V)
    same(oracle.verify_inputs(inp), oracle.verify_inputs(inp, lib=omp))


def test_truncated_and_draft_logits_identical(omp):
    inp = workloads.make_random(23, 4, 2049, "bf16", seed=5)
    a = oracle.verify_truncated(inp.logits, inp.dtype, inp.q, inp.tokens, inp.uniforms, inp.T,
                                0.9, 0.05)
    b = oracle.verify_truncated(inp.logits, inp.dtype, inp.q, inp.tokens, inp.uniforms, inp.T,
                                0.9, 0.05, lib=omp)
    same(a, b)
    dl = inp.logits[:, :-1].copy()
    a = oracle.verify_draft_logits(inp.logits, inp.dtype, dl, inp.tokens, inp.uniforms, inp.T,
                                   1.3, 0.95, 0.0)
    b = oracle.verify_draft_logits(inp.logits, inp.dtype, dl, inp.tokens, inp.uniforms, inp.T,
                                   1.3, 0.95, 0.0, lib=omp)
    same(a, b)


def test_greedy_and_ragged_identical(omp):
    inp = workloads.make_random(29, 3, 1001, "f32", seed=11)
    a = oracle.verify_greedy(inp.logits, inp.dtype, inp.tokens)
    b = oracle.verify_greedy(inp.logits, inp.dtype, inp.tokens, lib=omp)
    same(a, b)
    rg = workloads.ragged_from(inp, np.random.default_rng(2).integers(0, inp.K + 1, inp.B))
    a = oracle.verify_ragged(rg.logits, rg.dtype, rg.q, rg.tokens, rg.uniforms, rg.offsets,
                             rg.K_max, rg.T)
    b = oracle.verify_ragged(rg.logits, rg.dtype, rg.q, rg.tokens, rg.uniforms, rg.offsets,
                             rg.K_max, rg.T, lib=omp)
    same(a, b)
