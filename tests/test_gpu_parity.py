"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle on
the same seeded inputs and the same uniforms.  Bar and tie band: see
tests/gpu_helpers.py."""
import json

import numpy as np
import pytest

import oracle
import workloads
from tests import gpu_helpers as gh
from tests import oracle_pins as pins

pytestmark = pytest.mark.gpu

def _record(name, info):
    """Print a line per parity case (tie counts, stat errors): pytest shows it
    with -rP or -s."""
    print("parity case " + json.dumps({"case": name, **info}))


# ----------------------------------------------------------- workloads -----

@pytest.mark.parametrize("name", workloads.CONFIG_ORDER)
def test_config_parity_full_size(name):
    """The four named workloads at full size, default launch plan (the plan
    bench.py times): every sequence against the oracle."""
    inp = workloads.make_config(name)
    o = oracle.verify_inputs(inp)
    g = gh.gpu_verify_inputs(inp)
    info = gh.compare(g, o, inp.K, label=name)
    info.update(gh.stat_errors(g, o))
    info["mean_accept_len"] = float(np.mean(o["accept_len"]))
    _record(name, info)
    assert info["exact"] + info["accept_ties"] + info["draw_ties"] == inp.B


@pytest.mark.parametrize("name", ["b1_k4_v32000_f32", "b8_k4_v32000_bf16_peaked"])
def test_config_parity_many_seeds(name):
    """The two small workloads over 40 seeds each (fresh logits, drafts, uniforms)."""
    total = {"B": 0, "exact": 0, "accept_ties": 0, "draw_ties": 0, "errors": 0}
    for seed in range(100, 140):
        inp = workloads.make_config(name, seed=seed)
        info = gh.compare(gh.gpu_verify_inputs(inp), oracle.verify_inputs(inp), inp.K,
                          label=f"{name}/seed{seed}")
        for k in total:
            total[k] += info[k]
    _record(name + "_seeds", total)


# ----------------------------------------------- random shapes x plans -----

SHAPES = [  # B, K, V, dtype, T
    (3, 4, 1000, "f32", 1.0),
    (5, 3, 4099, "bf16", 0.6),      # V*2 not a multiple of 16: element-wise path
    (2, 7, 20011, "f32", 1.3),      # odd V, ragged last slice
    (4, 2, 50000, "bf16", 0.8),
    (1, 32, 2048, "bf16", 1.0),     # largest K
    (6, 0, 3000, "f32", 1.0),       # K = 0: one draw from row 0
    (9, 1, 7, "bf16", 1.0),         # tiny V
    (4, 3, 1, "f32", 1.0),          # V = 1
    (2, 5, 257, "f32", 0.9),
]
PLANS = [None, (1, 1, 128), (2, 2, 256), (4, 1, 512), (8, 0, 256), (16, 1, 128), (16, 0, 512),
         (3, 3, 256)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B{}_K{}_V{}_{}".format(*s[:4]))
@pytest.mark.parametrize("plan", PLANS, ids=lambda p: "auto" if p is None else "c{}g{}t{}".format(*p))
def test_random_shapes_every_plan(shape, plan):
    B, K, V, dtype, T = shape
    inp = workloads.make_random(B, K, V, dtype=dtype, T=T, seed=B * 1000 + K * 10 + V % 97)
    o = oracle.verify_inputs(inp)
    g = gh.gpu_verify_inputs(inp, plan=plan)
    gh.compare(g, o, K, label=f"{shape}/{plan}")


def test_f32_batch_on_three_stage_rings():
    """A float32 batch too large for the six-stage rings: the 128-thread
    kernel with three stages per warp (one CTA per sequence)."""
    inp = workloads.make_random(800, 3, 3000, dtype="f32", T=0.9, seed=31)
    p = gh.verifier().plan(inp.B, inp.K, inp.V, 0)
    assert p["stages"] == 3 and p["threads"] == 128 and p["group"] == 1
    info = gh.compare(gh.gpu_verify_inputs(inp), oracle.verify_inputs(inp), inp.K,
                      label="f32 three stages")
    _record("f32_three_stages", info)


def test_many_small_sequences_all_positions():
    """A batch large enough that every accepted length 1..K+1 occurs."""
    inp = workloads.make_random(3000, 6, 300, dtype="bf16", T=1.0, sigma=1.0, sigma_draft=0.3,
                                seed=77)
    o = oracle.verify_inputs(inp)
    g = gh.gpu_verify_inputs(inp)
    info = gh.compare(g, o, 6, label="many_small")
    assert set(np.unique(o["accept_len"])) == set(range(1, 8))
    _record("many_small", info)


# ------------------------------------------------------------ edge cases -----

def test_q_equal_p_accepts_everything_and_draws_bonus():
    inp = workloads.make_random(64, 5, 5000, dtype="f32", seed=3)
    p = workloads.softmax64(workloads.logits_as_f64(inp.logits, "f32")[:, :5]).astype(np.float32)
    inp.q = p
    o = oracle.verify_inputs(inp)
    g = gh.gpu_verify_inputs(inp)
    gh.compare(g, o, 5, label="q=p")
    assert np.all(g["accept_len"] == 6)


def test_neg_inf_logits_and_one_hot_target():
    inp = workloads.make_random(16, 3, 4000, dtype="bf16", seed=5)
    lg = inp.logits.copy()
    lg[:, :, ::3] = 0xFF80                       # -inf in a third of the vocabulary
    lg[8:, :, :] = 0xFF80
    lg[8:, :, 1234] = workloads.f32_to_bf16_bits(np.array([0.5], np.float32))[0]  # one-hot rows
    inp.logits = lg
    o = oracle.verify_inputs(inp)
    g = gh.gpu_verify_inputs(inp)
    gh.compare(g, o, 3, label="neg_inf")
    n = g["accept_len"][8:]
    assert np.all(g["out_tokens"][np.arange(8, 16), n - 1] == 1234)


def test_zero_residual_falls_back_to_target_row():
    """q = 1.01 p (unnormalised): rejection leaves max(0, p - q) = 0 everywhere."""
    inp = workloads.make_random(32, 2, 3000, dtype="f32", seed=8)
    p = workloads.softmax64(workloads.logits_as_f64(inp.logits, "f32")[:, :2])
    inp.q = (1.01 * p).astype(np.float32)
    u = inp.uniforms.copy()
    u[:, 0] = np.float32(0.9999)                 # rejects at position 0 (ratio 1/1.01)
    inp.uniforms = u
    o = oracle.verify_inputs(inp)
    g = gh.gpu_verify_inputs(inp)
    gh.compare(g, o, 2, label="zero_residual")
    assert np.all(g["accept_len"] == 1)


def test_unaligned_pointers_take_the_element_path():
    """Logits starting 2 bytes past a 16-byte boundary cannot use bulk copies."""
    import torch
    inp = workloads.make_random(4, 3, 8192, dtype="bf16", seed=9)
    o = oracle.verify_inputs(inp)
    v = gh.verifier()
    flat = torch.from_numpy(inp.logits.view(np.int16).reshape(-1)).cuda()
    buf = torch.empty(flat.numel() + 8, dtype=torch.int16, device="cuda")
    buf[1:1 + flat.numel()] = flat
    lg = buf[1:1 + flat.numel()].view(torch.bfloat16).view(inp.logits.shape)
    assert lg.data_ptr() % 16 != 0
    _, qd, td, ud = gh.to_device(inp.logits, "bf16", inp.q, inp.tokens, inp.uniforms)
    out = v.run(lg, qd, td, ud, inp.T, stats=True)
    g = {k: t.cpu().numpy() for k, t in out.items()}
    g["row_m"] = g["row_stats"][..., 0].astype(np.float64)
    g["row_s"] = g["row_stats"][..., 1].astype(np.float64)
    g["p_draft"] = g["p_draft"].astype(np.float64)
    gh.compare(g, o, 3, label="unaligned")


def test_large_vocab_small_batch():
    inp = workloads.make_random(2, 3, 1 << 20, dtype="bf16", seed=10)
    gh.compare(gh.gpu_verify_inputs(inp), oracle.verify_inputs(inp), 3, label="V=2^20")


# ---------------------------------------------------------------- errors -----

def test_device_errors_mark_only_their_sequence_and_clear():
    import speculative_decoding_verification_14_gb300 as sv
    inp = workloads.make_random(6, 3, 2000, dtype="f32", seed=13)
    lg, x, u = inp.logits.copy(), inp.tokens.copy(), inp.uniforms.copy()
    x[0, 2] = 2000
    x[1, 0] = -5
    u[2, 3] = np.float32(1.0)
    lg[3, 0, 17] = np.nan
    u[4, :3] = 0.0
    lg[4, 3, 5] = np.inf
    inp.logits, inp.tokens, inp.uniforms = lg, x, u
    o = oracle.verify_inputs(inp)
    v = gh.verifier()
    v.error()  # clear
    g = gh.gpu_verify_inputs(inp)
    gh.compare(g, o, 3, label="errors")
    assert list(g["status"]) == [sv.SV_ERR_TOKEN_RANGE, sv.SV_ERR_TOKEN_RANGE,
                                 sv.SV_ERR_UNIFORM_RANGE, sv.SV_ERR_NONFINITE,
                                 sv.SV_ERR_NONFINITE, sv.SV_OK]
    code, mask = v.error()
    assert code == sv.SV_ERR_TOKEN_RANGE
    assert mask == (1 << 4) | (1 << 5) | (1 << 7)
    # the next clean call succeeds and the word is clear
    clean = workloads.make_random(6, 3, 2000, dtype="f32", seed=14)
    gh.compare(gh.gpu_verify_inputs(clean), oracle.verify_inputs(clean), 3, label="after")
    assert v.error() == (sv.SV_OK, 0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("stats", [True, False])
def test_nan_of_either_sign_is_nonfinite(dtype, stats):
    """A NaN in a reached row is a sequence error whatever its sign bit (the
    kernel's warp maxima order floats by integer keys); rows that are all
    negative keep their ordinary parity."""
    import speculative_decoding_verification_14_gb300 as sv
    inp = workloads.make_random(5, 3, 4096, dtype=dtype, seed=21)
    lg = inp.logits.copy()
    if dtype == "f32":
        bits = lg.view(np.uint32)
        bits[0, 0, 100] = 0xFFC00000       # negative quiet NaN
        bits[1, 0, 4095] = 0x7FC00000      # positive quiet NaN
        bits[2, 0, 9] = 0xFF800001         # negative signalling NaN
        lg[3] = lg[3] - np.float32(1e4)    # every logit negative
    else:
        lg[0, 0, 100] = 0xFFC0
        lg[1, 0, 4095] = 0x7FC0
        lg[2, 0, 9] = 0xFF81
        f = workloads.logits_as_f64(lg[3:4], "bf16") - 1e4
        lg[3:4] = workloads.f32_to_bf16_bits(f.astype(np.float32))
    inp.logits = lg
    o = oracle.verify_inputs(inp)
    g = gh.gpu_verify_inputs(inp, stats=stats)
    gh.compare(g, o, 3, check_stats=stats, label=f"nan {dtype} stats={stats}")
    assert list(g["status"][:3]) == [sv.SV_ERR_NONFINITE] * 3
    assert list(g["status"][3:]) == [sv.SV_OK] * 2
    gh.verifier().error()  # clear the sticky word


@pytest.mark.parametrize("name", workloads.CONFIG_ORDER)
def test_without_row_stats_nothing_changes(name):
    """Without row_stats the kernel drops the exact running max from its fold
    and moves an offset on a chunk-sum bound instead; that changes rounding
    only, so on these workloads lengths, tokens, masks and statuses are the
    same bits as with row_stats, and still match the oracle."""
    inp = workloads.make_config(name)
    on = gh.gpu_verify_inputs(inp, stats=True)
    off = gh.gpu_verify_inputs(inp, stats=False)
    for k in ("accept_len", "out_tokens", "accept_mask", "status"):
        np.testing.assert_array_equal(off[k], on[k], err_msg=k)
    info = gh.compare(off, oracle.verify_inputs(inp), inp.K, check_stats=False, label=name + "/no_stats")
    assert info["exact"] + info["accept_ties"] + info["draw_ties"] == inp.B


def test_rebase_without_row_stats():
    """Spikes far above the bulk of a row sit in later chunks of many lanes, so
    offsets move mid-row -- without row_stats through the chunk-sum bound --
    and the outputs still match the oracle and the run with row_stats."""
    inp = workloads.make_random(2, 3, 300000, dtype="bf16", seed=16)
    lg = inp.logits.copy()
    lg[:, :, 4095::4096] = 0x41C8                # bf16 25.0 every 4096 entries
    inp.logits = lg
    on = gh.gpu_verify_inputs(inp, stats=True)
    off = gh.gpu_verify_inputs(inp, stats=False)
    for k in ("accept_len", "out_tokens", "accept_mask", "status"):
        np.testing.assert_array_equal(off[k], on[k], err_msg=k)
    info = gh.compare(off, oracle.verify_inputs(inp), inp.K, check_stats=False, label="rebase_no_stats")
    assert info["exact"] + info["accept_ties"] + info["draw_ties"] == inp.B


def test_special_values_without_row_stats():
    """NaN, +inf and all -inf rows are still caught when the running max is not kept."""
    import speculative_decoding_verification_14_gb300 as sv
    inp = workloads.make_random(6, 3, 3000, dtype="bf16", seed=15)
    lg = inp.logits.copy()
    lg[0, 1, 2900] = 0x7FC0                      # NaN late in row 1
    lg[1, 0, 5] = 0x7F80                         # +inf early in row 0
    lg[2, 0, :] = 0xFF80                         # row 0 entirely -inf
    lg[3, :, ::2] = 0xFF80                       # -inf in half the vocabulary: still valid
    inp.logits = lg
    o = oracle.verify_inputs(inp)
    g = gh.gpu_verify_inputs(inp, stats=False)
    gh.compare(g, o, 3, check_stats=False, label="special_no_stats")
    assert g["status"][1] == sv.SV_ERR_NONFINITE and g["status"][2] == sv.SV_ERR_NONFINITE
    gh.verifier().error()  # clear the sticky word for the tests after this one


def test_host_side_validation_launches_nothing():
    import speculative_decoding_verification_14_gb300 as sv
    import torch
    v = gh.verifier()
    inp = workloads.make_random(2, 2, 100, seed=1)
    lg, qd, td, ud = gh.to_device(inp.logits, "f32", inp.q, inp.tokens, inp.uniforms)
    for T in (0.0, -1.0, float("nan"), float("inf")):
        with pytest.raises(sv.SpecVerifyError) as e:
            v.run(lg, qd, td, ud, T)
        assert e.value.code == sv.SV_ERR_INVALID_ARG
    big = torch.zeros(2, 34, 100, device="cuda")
    with pytest.raises(sv.SpecVerifyError):
        v.run(big, torch.zeros(2, 33, 100, device="cuda"), torch.zeros(2, 33, dtype=torch.int32,
                                                                          device="cuda"),
              torch.zeros(2, 34, device="cuda"), 1.0)
    rc = sv.spec_verify_run(v.ctx, None, 0, None, None, None, 1, 0, 10, 1.0, None, None, None)
    assert rc == sv.SV_ERR_INVALID_ARG


# ------------------------------------------------------ determinism etc. -----

def test_repeated_runs_are_bit_identical():
    inp = workloads.make_config("b8_k4_v32000_bf16_peaked")
    a = gh.gpu_verify_inputs(inp)
    b = gh.gpu_verify_inputs(inp)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


def test_outputs_leave_neighbouring_memory_untouched():
    """Guard regions around every output keep their fill; the outputs between
    them still match the oracle."""
    import torch
    inp = workloads.make_random(7, 4, 3000, dtype="bf16", seed=21)
    lg, qd, td, ud = gh.to_device(inp.logits, "bf16", inp.q, inp.tokens, inp.uniforms)
    B, K = 7, 4
    guard = 64

    def fenced(n, dtype, fill):
        t = torch.full((n + 2 * guard,), fill, dtype=dtype, device="cuda")
        return t, t[guard:guard + n]

    fences = []
    out = {}
    for name, shape, dtype, fill in (("accept_len", (B,), torch.int32, 0x5A5A5A5A),
                                     ("out_tokens", (B, K + 1), torch.int32, 0x5A5A5A5A),
                                     ("accept_mask", (B, K), torch.uint8, 0xA5),
                                     ("row_stats", (B, K + 1, 2), torch.float32, 12345.0),
                                     ("p_draft", (B, K), torch.float32, 12345.0),
                                     ("status", (B,), torch.int32, 0x5A5A5A5A)):
        n = int(np.prod(shape))
        full, inner = fenced(n, dtype, fill)
        fences.append((name, full, n, fill))
        out[name] = inner.view(shape)
    gh.verifier().run(lg, qd, td, ud, inp.T, out=out)
    torch.cuda.synchronize()
    for name, full, n, fill in fences:
        assert torch.all(full[:guard] == fill) and torch.all(full[guard + n:] == fill), name
    g = {k: t.cpu().numpy() for k, t in out.items()}
    g["row_m"] = g["row_stats"][..., 0].astype(np.float64)
    g["row_s"] = g["row_stats"][..., 1].astype(np.float64)
    g["p_draft"] = g["p_draft"].astype(np.float64)
    gh.compare(g, oracle.verify_inputs(inp), K, label="fenced")


def test_cuda_graph_replay_matches_eager():
    import torch
    inp = workloads.make_config("b1_k4_v32000_f32")
    lg, qd, td, ud = gh.to_device(inp.logits, "f32", inp.q, inp.tokens, inp.uniforms)
    v = gh.verifier()
    eager = {k: t.clone() for k, t in v.run(lg, qd, td, ud, inp.T).items()}
    out = {k: torch.empty_like(t) for k, t in eager.items()}
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        v.run(lg, qd, td, ud, inp.T, out=out)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    for t in out.values():
        t.fill_(-7)
    with torch.cuda.graph(graph):
        v.run(lg, qd, td, ud, inp.T, out=out)
    for _ in range(3):
        for t in out.values():
            t.fill_(-7)
        graph.replay()
        torch.cuda.synchronize()
        for k in eager:
            assert torch.equal(out[k], eager[k]), k


def test_host_buffer_entry_matches_device_entry():
    import speculative_decoding_verification_14_gb300 as sv
    inp = workloads.make_config("b8_k4_v32000_bf16_peaked")
    g = gh.gpu_verify_inputs(inp)
    v = gh.verifier()
    B, K = inp.B, inp.K
    out = {"accept_len": np.empty(B, np.int32), "out_tokens": np.empty((B, K + 1), np.int32),
           "accept_mask": np.empty((B, K), np.uint8), "row_stats": np.empty((B, K + 1, 2), np.float32),
           "p_draft": np.empty((B, K), np.float32), "status": np.empty(B, np.int32)}
    rc = v.run_host(inp.logits, sv.SV_BF16, inp.q, inp.tokens, inp.uniforms, inp.T, out)
    assert rc == sv.SV_OK
    for k in ("accept_len", "out_tokens", "accept_mask", "row_stats", "status"):
        np.testing.assert_array_equal(out[k], g[k], err_msg=k)


# ------------------------------------- the method's laws through the GPU -----

@pytest.mark.parametrize("V,K,T,seed", [(4, 1, 1.0, 1), (8, 3, 1.3, 3)])
def test_gpu_output_law(V, K, T, seed):
    pins.check_output_law(gh.gpu_verify, V, K, T, seed, margin=2e-6)


@pytest.mark.parametrize("V,K", [(4, 1), (6, 3), (8, 3)])
def test_gpu_chi_square(V, K):
    pins.check_chisq(gh.gpu_verify, V, K, 1.0, seed=100 + V + K)


@pytest.mark.parametrize("K", [1, 3, 5])
@pytest.mark.parametrize("alpha", workloads.SWEEP_ALPHAS)
def test_acceptance_sweep_full_size(alpha, K):
    """The sweep workload: B = 32, V = 32000, draft overlap alpha at every
    position, 10^4 rounds with fresh drafts and uniforms.  Mean accepted length
    matches (1 - alpha^(K+1)) / (1 - alpha) within 4 SE, the printed table cell
    within 4 SE plus rounding, and the first rounds match the oracle exactly."""
    import torch
    cell = workloads.make_sweep_cell(alpha, K)
    v = gh.verifier()
    lg = torch.from_numpy(cell.logits).cuda()
    qd = torch.from_numpy(cell.q).cuda()
    td = torch.from_numpy(cell.tokens).cuda()
    ud = torch.from_numpy(cell.uniforms).cuda()
    R, B = cell.tokens.shape[0], cell.B
    lens = torch.empty(R, B, dtype=torch.int32, device="cuda")
    out = None
    for r in range(R):
        out = v.run(lg, qd, td[r], ud[r], 1.0, out=out)
        lens[r].copy_(out["accept_len"])
    al = lens.cpu().numpy().astype(np.float64).reshape(-1)
    want = pins.closed_form_tokens(alpha, K)
    se = al.std(ddof=1) / np.sqrt(al.size)
    assert abs(al.mean() - want) < 4 * se, (al.mean(), want, se)
    printed = dict(pins.read_table())[alpha][K]
    assert abs(al.mean() - printed) < 4 * se + 0.005
    for r in range(3):
        inp = cell.round_inputs(r)
        gh.compare(gh.gpu_verify_inputs(inp), oracle.verify_inputs(inp), K, label=f"sweep{alpha}/{K}/{r}")
    _record(f"sweep_a{alpha}_k{K}", {"mean_accept_len": float(al.mean()), "se": float(se),
                                     "closed_form": want, "printed": printed})
