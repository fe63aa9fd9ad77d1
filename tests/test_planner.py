"""CPU tests of the launch planner (spec_verify_plan_for): one cluster per
sequence, vocabulary slices that cover every row, shared memory within the
device limit, and the overrides honoured."""
import itertools

import pytest

GB300 = dict(num_sms=152, smem=232448, max_cluster=16)


@pytest.fixture(scope="module")
def sv():
    from speculative_decoding_verification_14_gb300 import build
    build.build()
    import speculative_decoding_verification_14_gb300 as pkg
    return pkg


def plan(sv, B, K, V, dtype, oc=0, og=0, ot=0, dev=GB300):
    return sv.spec_verify_plan_for(dev["num_sms"], dev["smem"], dev["max_cluster"], B, K, V, dtype,
                                   oc, og, ot)


@pytest.mark.parametrize("B,K,V,dtype", list(itertools.product(
    [1, 3, 8, 32, 64, 256, 5000], [0, 1, 4, 7, 32], [1, 7, 1000, 4099, 32000, 128256, 151936, 1 << 20],
    [0, 1])))
def test_plan_invariants(sv, B, K, V, dtype):
    rc, p = plan(sv, B, K, V, dtype)
    es = 2 if dtype == 1 else 4
    if -(-V // 16) * es > GB300["smem"] - 4096:
        # one CTA holds its whole slice of a row in shared memory: past 16
        # slices of ~223 KB the shape has no plan
        assert rc == sv.SV_ERR_UNSUPPORTED
        return
    assert rc == sv.SV_OK
    C, slice_ = p["cluster"], p["slice"]
    assert 1 <= C <= 16
    assert slice_ % 8 == 0 and slice_ * C >= V and slice_ * (C - 1) < V + 8 * C
    assert p["grid"] == B * C
    assert 1 <= p["group"] <= K + 1
    assert p["smem_bytes"] <= GB300["smem"]
    assert p["bulk_copy"] == int((V * es) % 16 == 0)
    assert p["threads"] in (128, 256, 512)


def test_workload_plans(sv):
    # big batches read rows one at a time; small ones load every row at once
    assert plan(sv, 256, 7, 128256, 1)[1]["group"] == 1
    assert plan(sv, 256, 7, 128256, 1)[1]["cluster"] == 8
    assert plan(sv, 1, 4, 32000, 0)[1]["group"] == 5
    assert plan(sv, 1, 4, 32000, 0)[1]["cluster"] == 16
    assert plan(sv, 64, 3, 151936, 1)[1]["group"] == 1


def test_overrides(sv):
    rc, p = plan(sv, 4, 5, 50000, 1, oc=4, og=3, ot=512)
    assert rc == 0 and (p["cluster"], p["group"], p["threads"]) == (4, 3, 512)
    rc, p = plan(sv, 4, 2, 50000, 1, og=9)
    assert rc == 0 and p["group"] == 3
    assert plan(sv, 4, 2, 1000, 1, ot=100)[0] == sv.SV_ERR_INVALID_ARG
    assert plan(sv, 4, 2, 1000, 1, oc=17)[0] == sv.SV_ERR_INVALID_ARG
    small = dict(GB300, max_cluster=8)
    assert plan(sv, 4, 2, 1000, 1, oc=16, dev=small)[0] == sv.SV_ERR_UNSUPPORTED


def test_shared_memory_limit(sv):
    # a slice that cannot fit even one row: unsupported
    tiny = dict(GB300, smem=48 * 1024)
    assert plan(sv, 1, 1, 1 << 22, 0, dev=tiny)[0] == sv.SV_ERR_UNSUPPORTED
    # groups shrink before the cluster grows
    rc, p = plan(sv, 1, 32, 1 << 20, 1)
    assert rc == 0 and p["smem_bytes"] <= GB300["smem"] and p["group"] < 33


def test_bad_arguments(sv):
    assert plan(sv, 0, 1, 100, 0)[0] == sv.SV_ERR_INVALID_ARG
    assert plan(sv, 1, 33, 100, 0)[0] == sv.SV_ERR_INVALID_ARG
    assert plan(sv, 1, 1, 0, 0)[0] == sv.SV_ERR_INVALID_ARG
    assert plan(sv, 1, 1, 100, 2)[0] == sv.SV_ERR_INVALID_ARG
