"""GPU-side helpers for the parity tests: run the CUDA library through its C ABI
(via the ctypes binding) on numpy inputs, and compare with the oracle.

Parity bar:
 * accepted lengths, tokens and masks bit-exact, except sequences whose oracle
   decision lies within TIE = 1e-6 of its uniform (an acceptance test with
   |u - p/q| < 1e-6, or the draw with u within 1e-6 of a normalised CDF
   boundary next to the drawn token); those are counted, checked for validity,
   and for draw ties the GPU token must be one of the two tokens bordering the
   boundary;
 * statuses bit-exact;
 * softmax statistics and p(x) within 1e-5 relative (fp32 and bf16 inputs
   alike: both sides read the same stored values).
"""
from __future__ import annotations

import numpy as np

TIE = 1e-6
RTOL = 1e-5

_verifiers = {}
_oracle_lib = []


def oracle_lib():
    """The OpenMP build of the oracle on every core this process may use
    (results identical to the plain build: tests/test_oracle_openmp.py), or
    None -- the plain build -- where no OpenMP runtime is available."""
    if not _oracle_lib:
        import oracle
        try:
            _oracle_lib.append(oracle.load_openmp())
        except Exception:
            _oracle_lib.append(None)
    return _oracle_lib[0]


def verifier(max_B=1 << 20, max_K=32, max_V=1 << 21):
    import speculative_decoding_verification_14_gb300 as sv
    key = (max_B, max_K, max_V)
    if key not in _verifiers:
        _verifiers[key] = sv.Verifier(max_B, max_K, max_V)
    return _verifiers[key]


def to_device(inp_logits, dtype, q, tokens, uniforms):
    import torch
    if dtype == "bf16":
        lg = torch.from_numpy(np.ascontiguousarray(inp_logits).view(np.int16)).cuda().view(torch.bfloat16)
    else:
        lg = torch.from_numpy(np.ascontiguousarray(inp_logits, dtype=np.float32)).cuda()
    return (lg, torch.from_numpy(np.ascontiguousarray(q, dtype=np.float32)).cuda(),
            torch.from_numpy(np.ascontiguousarray(tokens, dtype=np.int32)).cuda(),
            torch.from_numpy(np.ascontiguousarray(uniforms, dtype=np.float32)).cuda())


def gpu_verify(logits, dtype, q, tokens, uniforms, T, plan=None, stats=True, v=None):
    """Same signature and keys as oracle.verify (minus the margin keys)."""
    import torch
    v = v or verifier()
    B, K1, V = logits.shape
    K = K1 - 1
    q = np.ascontiguousarray(np.broadcast_to(q, (B, K, V)))
    tokens = np.ascontiguousarray(np.broadcast_to(tokens, (B, K)))
    lg, qd, td, ud = to_device(np.ascontiguousarray(np.broadcast_to(logits, (B, K1, V))), dtype, q,
                               tokens, uniforms)
    if plan:
        v.set_plan_override(*plan)
    try:
        out = v.run(lg, qd, td, ud, T, stats=stats, status=True)
        torch.cuda.synchronize()
    finally:
        if plan:
            v.set_plan_override(0, 0, 0)
    res = {k: t.cpu().numpy() for k, t in out.items()}
    if "row_stats" in res:
        res["row_m"] = res["row_stats"][..., 0].astype(np.float64)
        res["row_s"] = res["row_stats"][..., 1].astype(np.float64)
    if "p_draft" in res:
        res["p_draft"] = res["p_draft"].astype(np.float64)
    return res


def gpu_verify_inputs(inp, plan=None, stats=True):
    return gpu_verify(inp.logits, inp.dtype, inp.q, inp.tokens, inp.uniforms, inp.T, plan, stats)


def _rel(a, b):
    return np.abs(a - b) / np.maximum(np.abs(b), 1e-300)


def compare(g: dict, o: dict, K: int, check_stats: bool = True, label: str = "") -> dict:
    """Element-by-element comparison.  Returns counts for reporting; raises
    AssertionError on any mismatch outside the tie band."""
    B = o["accept_len"].shape[0]
    np.testing.assert_array_equal(g["status"], o["status"], err_msg=f"{label}: status")
    ok = o["status"] == 0
    acc_tie = ok & (o["accept_margin"] < TIE)
    smp_tie = ok & ~acc_tie & (o["sample_margin"] < TIE)
    exact = ok & ~acc_tie & ~smp_tie
    # exact rows
    for key in ("accept_len", "out_tokens", "accept_mask"):
        gg, oo = g[key][exact], o[key][exact]
        if not np.array_equal(gg, oo):
            bad = np.nonzero(~np.all((g[key] == o[key]).reshape(B, -1), axis=1) & exact)[0]
            b = int(bad[0])
            raise AssertionError(
                f"{label}: {key} differs outside the tie band at sequence {b} of {len(bad)}: "
                f"gpu {g[key][b]} oracle {o[key][b]} (accept margin {o['accept_margin'][b]:.3e}, "
                f"sample margin {o['sample_margin'][b]:.3e}, len g/o {g['accept_len'][b]}/"
                f"{o['accept_len'][b]})")
    # error rows report the sentinel
    bad_rows = ~ok
    assert np.all(g["accept_len"][bad_rows] == 0)
    assert np.all(g["out_tokens"][bad_rows] == -1)
    # draw ties: same length and prefix, token one of the two bordering tokens
    for b in np.nonzero(smp_tie)[0]:
        n = int(o["accept_len"][b])
        assert g["accept_len"][b] == n, f"{label}: draw-tie row {b} length"
        assert np.array_equal(g["out_tokens"][b, :n - 1], o["out_tokens"][b, :n - 1])
        assert g["out_tokens"][b, n - 1] in (o["out_tokens"][b, n - 1], o["sample_alt"][b]), \
            f"{label}: draw-tie row {b}: gpu token {g['out_tokens'][b, n - 1]} not in " \
            f"{{{o['out_tokens'][b, n - 1]}, {o['sample_alt'][b]}}}"
    # acceptance ties: only validity
    for b in np.nonzero(acc_tie)[0]:
        n = int(g["accept_len"][b])
        assert 1 <= n <= K + 1
    if check_stats and "row_m" in g:
        # rows both sides computed; on exact rows the NaN pattern must agree
        both = ~np.isnan(o["row_s"]) & ~np.isnan(g["row_s"])
        ex = exact[:, None] & np.ones_like(both)
        np.testing.assert_array_equal(np.isnan(g["row_s"])[ex], np.isnan(o["row_s"])[ex],
                                      err_msg=f"{label}: rows reached")
        if both.any():
            assert np.max(_rel(g["row_s"][both], o["row_s"][both])) < RTOL, \
                f"{label}: softmax normaliser rel err {np.max(_rel(g['row_s'][both], o['row_s'][both])):.2e}"
            dm = np.abs(g["row_m"][both] - o["row_m"][both]) / np.maximum(1.0, np.abs(o["row_m"][both]))
            assert np.max(dm) < 1e-6, f"{label}: softmax max err {np.max(dm):.2e}"
        if K:
            bp = ~np.isnan(o["p_draft"]) & ~np.isnan(g["p_draft"])
            if bp.any():
                err = np.max(np.abs(g["p_draft"][bp] - o["p_draft"][bp]) /
                             np.maximum(np.abs(o["p_draft"][bp]), 1e-30))
                assert err < RTOL, f"{label}: p(x) rel err {err:.2e}"
    return {"B": int(B), "exact": int(exact.sum()), "accept_ties": int(acc_tie.sum()),
            "draw_ties": int(smp_tie.sum()), "errors": int((~ok).sum())}


def stat_errors(g: dict, o: dict) -> dict:
    """Largest relative errors of the GPU's softmax normaliser and p(x)."""
    both = ~np.isnan(o["row_s"]) & ~np.isnan(g["row_s"])
    res = {"row_s_rel": float(np.max(_rel(g["row_s"][both], o["row_s"][both]))) if both.any() else 0.0}
    if o["p_draft"].size and "p_draft" in g:
        bp = ~np.isnan(o["p_draft"]) & ~np.isnan(g["p_draft"])
        res["p_draft_rel"] = float(np.max(_rel(g["p_draft"][bp], o["p_draft"][bp]))) if bp.any() else 0.0
    return res
