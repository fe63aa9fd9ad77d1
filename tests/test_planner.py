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
    assert rc == sv.SV_OK
    es = 2 if dtype == 1 else 4
    C, slice_ = p["cluster"], p["slice"]
    assert C in (1, 2, 4, 8, 16)
    assert slice_ % 8 == 0 and slice_ * C >= V and slice_ * (C - 1) < V + 8 * C
    assert p["grid"] == B * C
    assert 1 <= p["group"] <= K + 1
    assert p["smem_bytes"] <= GB300["smem"]
    assert p["bulk_copy"] == int((V * es) % 16 == 0)
    assert p["threads"] == 128
    assert p["prefetch_next"] == int(p["group"] == 1)
    # the batch is resident at once whenever a cluster of one CTA per sequence fits
    per_sm = min(896 // p["threads"], 233472 // (p["smem_bytes"] + 1024))
    if B <= 152 * per_sm:
        assert B * C <= 152 * per_sm or C == 1


def test_workload_plans(sv):
    # 256 sequences: four CTAs each keep the whole batch resident, one row per step
    p = plan(sv, 256, 7, 128256, 1)[1]
    assert (p["cluster"], p["group"]) == (4, 1)
    # one sequence: the largest cluster, every row at once
    p = plan(sv, 1, 4, 32000, 0)[1]
    assert (p["cluster"], p["group"]) == (16, 5)
    # 64 sequences fill the GPU already with eight CTAs each; sixteen would
    # leave each warp fewer than four ring stages per row
    p = plan(sv, 64, 3, 151936, 1)[1]
    assert (p["cluster"], p["group"]) == (8, 1)


@pytest.mark.parametrize("B,K,V,dtype", list(itertools.product(
    [1, 8, 64, 128, 152, 256, 1024], [0, 3, 7], [32000, 128256, 151936], [0, 1])))
def test_ring_depth(sv, B, K, V, dtype):
    """Six ring stages exactly when the plan has 128 threads and its CTAs are
    all resident at the deep kernels' occupancy (at most four per SM, as the
    deeper rings' shared memory allows); three otherwise."""
    rc, p = plan(sv, B, K, V, dtype)
    assert rc == sv.SV_OK
    assert p["stages"] in (3, 6)
    if p["stages"] == 6:
        per_sm = min(4, 233472 // (p["smem_bytes"] + 1024))
        assert p["threads"] == 128 and p["grid"] <= per_sm * 152
    else:
        # with three more stages per warp the plan's CTAs would not all be
        # resident at the deep kernels' occupancy (or the plan is wider)
        per_sm = min(4, 233472 // (p["smem_bytes"] + 3 * 4 * 2048 + 1024))
        assert p["threads"] != 128 or p["grid"] > per_sm * 152


def test_workload_ring_depths(sv):
    assert plan(sv, 256, 7, 128256, 1)[1]["stages"] == 3     # 1024 CTAs: seven per SM
    assert plan(sv, 64, 3, 151936, 1)[1]["stages"] == 6      # 512 CTAs
    assert plan(sv, 8, 4, 32000, 1)[1]["stages"] == 6
    assert plan(sv, 1, 4, 32000, 0)[1]["stages"] == 6


def test_overrides(sv):
    rc, p = plan(sv, 4, 5, 50000, 1, oc=4, og=3, ot=512)
    assert rc == 0 and (p["cluster"], p["group"], p["threads"]) == (4, 3, 512)
    rc, p = plan(sv, 4, 2, 50000, 1, og=9)
    assert rc == 0 and p["group"] == 3
    assert plan(sv, 4, 2, 1000, 1, ot=100)[0] == sv.SV_ERR_INVALID_ARG
    assert plan(sv, 4, 2, 1000, 1, oc=17)[0] == sv.SV_ERR_INVALID_ARG
    small = dict(GB300, max_cluster=8)
    assert plan(sv, 4, 2, 1000, 1, oc=16, dev=small)[0] == sv.SV_ERR_UNSUPPORTED


def test_shared_memory_does_not_grow_with_the_vocabulary(sv):
    """The rings are fixed and the exchange slots follow the cluster (at most
    16 CTAs); only the draw's tile arrays (a total and an offset per 512
    entries of a CTA's slice) follow V."""
    small = plan(sv, 1, 1, 32000, 1)[1]
    huge = plan(sv, 1, 1, 1 << 24, 1)[1]
    tiles = lambda p: 2 * 4 * 4 * -(-p["slice"] // (4 * 512))  # [2][warps][tiles] floats
    slots = lambda p: 2 * p["group"] * p["cluster"] * 4 * 16   # [2][group][C x warps] partials
    grow = huge["smem_bytes"] - small["smem_bytes"]
    assert grow <= tiles(huge) - tiles(small) + slots(huge) - slots(small) + 64
    assert tiles(huge) <= 16 * 1024 + 64
    tiny = dict(GB300, smem=8 * 1024)
    assert plan(sv, 1, 1, 32000, 0, dev=tiny)[0] == sv.SV_ERR_UNSUPPORTED


def test_bad_arguments(sv):
    assert plan(sv, 0, 1, 100, 0)[0] == sv.SV_ERR_INVALID_ARG
    assert plan(sv, 1, 33, 100, 0)[0] == sv.SV_ERR_INVALID_ARG
    assert plan(sv, 1, 1, 0, 0)[0] == sv.SV_ERR_INVALID_ARG
    assert plan(sv, 1, 1, 100, 2)[0] == sv.SV_ERR_INVALID_ARG
    assert plan(sv, 1, 1, (1 << 31) + 1, 0)[0] == sv.SV_ERR_INVALID_ARG


# ------------------------------------------------------------ greedy -----

def gplan(sv, B, K, V, dtype, oc=0, dev=GB300):
    return sv.spec_verify_plan_greedy_for(dev["num_sms"], dev["max_cluster"], B, K, V, dtype, oc)


@pytest.mark.parametrize("B,K,V,dtype", list(itertools.product(
    [1, 8, 64, 256, 5000], [0, 4, 32], [1, 7, 32000, 128256, 151936, 1 << 20], [0, 1])))
def test_greedy_plan_invariants(sv, B, K, V, dtype):
    rc, p = gplan(sv, B, K, V, dtype)
    assert rc == sv.SV_OK
    es = 2 if dtype == 1 else 4
    C, slice_ = p["cluster"], p["slice"]
    assert C in (1, 2, 4, 8, 16)
    assert slice_ % 8 == 0 and slice_ * C >= V and slice_ * (C - 1) < V + 8 * C
    assert p["grid"] == B * C and p["group"] == 1 and p["threads"] == 128
    assert p["bulk_copy"] == int((V * es) % 16 == 0)
    # the batch stays resident (eight CTAs per SM) whenever one CTA per sequence fits
    if B <= 152 * 8:
        assert B * C <= 152 * 8


def test_greedy_workload_plans(sv):
    assert gplan(sv, 256, 7, 128256, 1)[1]["cluster"] == 4
    assert gplan(sv, 64, 3, 151936, 1)[1]["cluster"] == 8
    assert gplan(sv, 8, 4, 32000, 1)[1]["cluster"] == 16
    assert gplan(sv, 1, 4, 32000, 0)[1]["cluster"] == 16
    assert gplan(sv, 4, 2, 50000, 1, oc=2)[1]["cluster"] == 2
    assert gplan(sv, 4, 2, 50000, 1, oc=16, dev=dict(GB300, max_cluster=8))[0] == sv.SV_ERR_UNSUPPORTED
    assert gplan(sv, 0, 2, 50000, 1)[0] == sv.SV_ERR_INVALID_ARG
    assert gplan(sv, 1, 33, 50000, 1)[0] == sv.SV_ERR_INVALID_ARG


# ------------------------------------------------------- draft logits -----

def dplan(sv, B, K, V, dtype, filters, oc=0, dev=GB300):
    return sv.spec_verify_plan_draft_logits_for(dev["num_sms"], dev["max_cluster"], B, K, V, dtype,
                                                filters, oc)


@pytest.mark.parametrize("B,K,V,dtype,filters", list(itertools.product(
    [1, 8, 64, 256, 5000], [0, 7], [1, 7, 32000, 128256], [0, 1], [0, 1])))
def test_draft_logits_plan_invariants(sv, B, K, V, dtype, filters):
    rc, p = dplan(sv, B, K, V, dtype, filters)
    assert rc == sv.SV_OK
    es = 2 if dtype == 1 else 4
    C, slice_ = p["cluster"], p["slice"]
    assert C in ((1, 2, 4, 8) if filters else (1, 2, 4, 8, 16))
    assert slice_ % 8 == 0 and slice_ * C >= V and slice_ * (C - 1) < V + 8 * C
    assert p["grid"] == B * C and p["threads"] == 128
    assert p["bulk_copy"] == int((V * es) % 16 == 0)
    per_sm = 4 if filters else 7  # resident CTAs per SM (launch bounds)
    if B <= 152 * per_sm:
        assert B * C <= 152 * per_sm
    # with a filter on, the plan is the truncated kernel's; without, the
    # sampled verify's mapping with room for the draft rows' partials
    if filters:
        assert p == sv.spec_verify_plan_truncated_for(152, 16, B, K, V, dtype, 0)[1]
    else:
        q = sv.spec_verify_plan_for(152, 232448, 16, B, K, V, dtype, 0, 0, 0)[1]
        for k in ("cluster", "slice", "grid", "threads", "bulk_copy", "stages"):
            assert p[k] == q[k], k
        assert p["group"] <= q["group"] and p["smem_bytes"] >= q["smem_bytes"]
        assert p["smem_bytes"] <= 232448


def test_draft_logits_workload_plans(sv):
    assert dplan(sv, 256, 7, 128256, 1, 0)[1]["cluster"] == 4
    assert dplan(sv, 256, 7, 128256, 1, 1)[1]["cluster"] == 2
    assert dplan(sv, 256, 7, 128256, 1, 0)[1]["stages"] == 3
    assert dplan(sv, 64, 3, 151936, 1, 0)[1]["cluster"] == 8
    assert dplan(sv, 64, 3, 151936, 1, 0)[1]["stages"] == 6
    assert dplan(sv, 1, 4, 32000, 0, 0)[1]["cluster"] == 16
    assert dplan(sv, 8, 4, 32000, 1, 0)[1]["cluster"] == 8
    assert dplan(sv, 8, 4, 32000, 1, 1)[1]["cluster"] == 8
    assert dplan(sv, 1, 4, 32000, 0, 0, dev=dict(GB300, max_cluster=8))[1]["cluster"] == 8
    assert dplan(sv, 4, 2, 50000, 1, 0, oc=16, dev=dict(GB300, max_cluster=8))[0] == \
        sv.SV_ERR_UNSUPPORTED
    assert dplan(sv, 4, 2, 50000, 1, 1, oc=16)[0] == sv.SV_ERR_INVALID_ARG
    assert dplan(sv, 0, 2, 50000, 1, 0)[0] == sv.SV_ERR_INVALID_ARG
