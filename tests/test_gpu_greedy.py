"""GPU parity for greedy verification (the T -> 0 limit of [P1]'s verify step):
the CUDA kernel through the C ABI against oracle.verify_greedy on the same
inputs.  Both sides compare the same stored logits, so every output --
accepted lengths, tokens, masks, statuses and the per-row argmax -- must match
bit for bit (no tie band: the lowest-index rule decides equal maxima)."""
import numpy as np
import pytest

import oracle
import workloads
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

KEYS = ("accept_len", "out_tokens", "accept_mask", "status", "row_argmax")


def _gpu(logits, dtype, tokens, cluster=0, v=None, offset=0):
    """Run the greedy kernel; `offset` > 0 shifts the logits base pointer by
    that many elements (an unaligned base takes the element path)."""
    import torch
    v = v or gh.verifier()
    B, K1, V = logits.shape
    K = K1 - 1
    flat = np.ascontiguousarray(logits).reshape(-1)
    if offset:
        flat = np.concatenate([np.zeros(offset, flat.dtype), flat])
    if dtype == "bf16":
        lg = torch.from_numpy(flat.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        lg = torch.from_numpy(flat.astype(np.float32)).cuda()
    lg = lg[offset:].view(B, K1, V)
    td = torch.from_numpy(np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, K)).cuda()
    if cluster:
        v.set_plan_override(cluster, 0, 0)
    try:
        out = v.run_greedy(lg, td, argmax=True)
        torch.cuda.synchronize()
    finally:
        if cluster:
            v.set_plan_override(0, 0, 0)
    return {k: t.cpu().numpy() for k, t in out.items()}


def _check(logits, dtype, tokens, label, **kw):
    o = oracle.verify_greedy(logits, dtype, tokens)
    g = _gpu(logits, dtype, tokens, **kw)
    for k in KEYS:
        if not np.array_equal(g[k], o[k]):
            B = o["accept_len"].shape[0]
            b = int(np.nonzero(np.any((g[k] != o[k]).reshape(B, -1), axis=1))[0][0])
            raise AssertionError(f"{label}: {k} differs at sequence {b}: gpu {g[k][b]} "
                                 f"oracle {o[k][b]}")
    return o


@pytest.mark.parametrize("name", workloads.CONFIG_ORDER)
def test_config_parity_full_size(name):
    """The four workloads at full size with a greedy drafter, default plan."""
    inp = workloads.greedy_drafts(workloads.make_config(name))
    o = _check(inp.logits, inp.dtype, inp.tokens, name)
    assert o["accept_len"].min() >= 1


@pytest.mark.parametrize("cluster", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("dtype,V", [("bf16", 32000), ("f32", 4099), ("bf16", 1001), ("f32", 64),
                                     ("bf16", 7), ("f32", 151936)])
def test_random_shapes_every_cluster(dtype, V, cluster):
    rng = np.random.default_rng(V + cluster)
    B, K = 24, 5
    inp = workloads.make_random(B, K, V, dtype, seed=V % 97 + cluster)
    vals = workloads.logits_as_f64(inp.logits, dtype)
    a = vals[:, :K].argmax(-1)
    x = np.where(rng.random((B, K)) < 0.75, a, rng.integers(0, V, (B, K))).astype(np.int32)
    _check(inp.logits, dtype, x, f"{dtype} V={V} C={cluster}", cluster=cluster)


@pytest.mark.parametrize("cluster", [0, 4, 16])
def test_ties_across_lanes_warps_and_ctas(cluster):
    """Integer logits with the maximum repeated at many places: the lowest index wins."""
    rng = np.random.default_rng(3)
    B, K, V = 16, 6, 20000
    vals = rng.integers(0, 40, (B, K + 1, V)).astype(np.float32)
    for b in range(B):                       # the max appears late, and again later
        for i in range(K + 1):
            pos = np.sort(rng.choice(V, 3, replace=False))
            vals[b, i, pos] = 50.0
    x = vals[:, :K].argmax(-1).astype(np.int32)
    x[::3, 3] = (x[::3, 3] + 1) % V           # some rejections
    for dtype in ("f32", "bf16"):
        logits = vals if dtype == "f32" else workloads.f32_to_bf16_bits(vals)
        _check(logits, dtype, x, f"ties {dtype} C={cluster}", cluster=cluster)


def test_k0_and_k32_and_one_entry_rows():
    rng = np.random.default_rng(4)
    for B, K, V in ((5, 0, 3000), (3, 32, 2048), (9, 2, 1)):
        vals = rng.standard_normal((B, K + 1, V)).astype(np.float32)
        x = vals[:, :K].argmax(-1).astype(np.int32) if K else np.zeros((B, 0), np.int32)
        o = _check(vals, "f32", x, f"B={B} K={K} V={V}")
        assert np.all(o["accept_len"] == K + 1)


def test_unaligned_base_takes_the_element_path():
    rng = np.random.default_rng(5)
    B, K, V = 6, 3, 5000
    for dtype in ("f32", "bf16"):
        inp = workloads.make_random(B, K, V, dtype, seed=8)
        vals = workloads.logits_as_f64(inp.logits, dtype)
        x = np.where(rng.random((B, K)) < 0.7, vals[:, :K].argmax(-1), 0).astype(np.int32)
        _check(inp.logits, dtype, x, f"offset {dtype}", offset=1)


def test_special_values_and_errors():
    import speculative_decoding_verification_14_gb300 as sv
    v = gh.verifier()
    v.error()
    B, K, V = 6, 3, 3000
    vals = np.tile(np.arange(V, dtype=np.float32), (B, K + 1, 1))
    x = np.full((B, K), V - 1, np.int32)
    vals[1, 1, 17] = np.nan                  # error at row 1
    vals[2, 0, 2999] = np.inf                # error at row 0
    vals[3, 2] = -np.inf                     # an all -inf row
    vals[4, 0, :2990] = -np.inf              # -inf entries are ordinary losers
    x[5, 0] = 0                              # rejected at 0: later NaN never read
    vals[5, 1, 5] = np.nan
    o = _check(vals, "f32", x, "special values")
    assert o["status"].tolist() == [0, 5, 5, 5, 0, 0]
    rc, mask = v.error()
    assert rc == sv.SV_ERR_NONFINITE and mask == 1 << sv.SV_ERR_NONFINITE
    x2 = x.copy()
    x2[0, 2] = V                             # out of range
    o = _check(vals, "f32", x2, "token range")
    assert o["status"][0] == sv.SV_ERR_TOKEN_RANGE
    assert v.error()[0] == sv.SV_ERR_TOKEN_RANGE


def test_telemetry_counts_greedy_runs():
    import torch
    inp = workloads.greedy_drafts(workloads.make_config("b8_k4_v32000_bf16_peaked"))
    o = oracle.verify_greedy(inp.logits, inp.dtype, inp.tokens)
    v = gh.verifier()
    hist = torch.zeros(inp.K + 2, dtype=torch.int32, device="cuda")
    v.set_telemetry(hist)
    try:
        _gpu(inp.logits, inp.dtype, inp.tokens, v=v)
        _gpu(inp.logits, inp.dtype, inp.tokens, v=v)
    finally:
        v.set_telemetry(None)
    h = hist.cpu().numpy().astype(np.uint64)
    assert np.array_equal(h, 2 * oracle.accept_hist(o["accept_len"], inp.K))
