"""CPU tests of the benchmark's algorithmic byte counts (the numerator of the
reported roofline fraction) against a per-sequence count written from the
definition of what each verify must move, and host-side argument checks of the
draft-logit entry point (no GPU needed)."""
import types

import numpy as np
import pytest

import bench


def _inp(B, K, V, dtype):
    return types.SimpleNamespace(B=B, K=K, V=V, dtype=dtype,
                                 logit_bytes=2 if dtype == "bf16" else 4)


def _per_sequence(K, V, es, n, kind):
    """One sequence with accepted length n (rows 0..n-1 reached)."""
    tokens, uniforms = K * 4, (K + 1) * 4
    outputs = 4 + (K + 1) * 4 + K                 # accept_len, out_tokens, accept_mask
    rows = n * V * es                             # target rows the loop reaches
    if kind == "greedy":                          # no q, no uniforms
        return rows + tokens + outputs
    if kind == "draft_logits":                    # every tested draft row, whole
        return rows + min(n, K) * V * es + tokens + uniforms + outputs
    rejected = V * 4 if n <= K else 0             # the rejected row of q
    if kind == "truncated_min_p":                 # q_j read at kept tokens only
        rejected = 0
    gathered = min(n, K) * 4                      # q(x) of each test
    return rows + rejected + gathered + tokens + uniforms + outputs


@pytest.mark.parametrize("kind", ["sampled", "greedy", "draft_logits", "truncated_min_p",
                                  "truncated_top_p"])
@pytest.mark.parametrize("B,K,V,dtype", [(256, 7, 128256, "bf16"), (1, 4, 32000, "f32"),
                                         (5, 0, 1000, "bf16"), (3, 32, 7, "f32")])
def test_uniform_batches(kind, B, K, V, dtype):
    inp = _inp(B, K, V, dtype)
    rng = np.random.default_rng(B + K + V)
    for al in (rng.integers(1, K + 2, B), np.ones(B, np.int64), np.full(B, K + 1)):
        al = al.astype(np.int32)
        want = sum(_per_sequence(K, V, inp.logit_bytes, int(n),
                                 "sampled" if kind == "truncated_top_p" else kind) for n in al)
        fn = {"sampled": bench.algorithmic_bytes, "greedy": bench.algorithmic_bytes_greedy,
              "draft_logits": bench.algorithmic_bytes_draft_logits,
              "truncated_min_p": lambda i, a: bench.algorithmic_bytes_truncated(i, a, 0.05),
              "truncated_top_p": lambda i, a: bench.algorithmic_bytes_truncated(i, a, 0.0)}[kind]
        assert fn(inp, al) == want


def test_ragged_batch():
    rng = np.random.default_rng(3)
    B, K, V = 40, 7, 5000
    Ks = rng.integers(0, K + 1, B)
    offsets = np.zeros(B + 1, np.int32)
    offsets[1:] = np.cumsum(Ks + 1)
    rg = types.SimpleNamespace(B=B, V=V, logit_bytes=2, offsets=offsets)
    al = np.array([rng.integers(1, k + 2) for k in Ks], np.int32)
    want = sum(_per_sequence(int(k), V, 2, int(n), "sampled") for k, n in zip(Ks, al))
    assert bench.algorithmic_bytes_ragged(rg, al) == want + (B + 1) * 4


def test_draft_logit_entry_rejects_a_null_context_without_cuda():
    from speculative_decoding_verification_14_gb300 import build
    build.build()
    import speculative_decoding_verification_14_gb300 as sv
    assert sv.spec_verify_run_draft_logits(None, None, 0, None, None, None, 1, 1, 10, 1.0, 1.0,
                                           1.0, 0.0, None, None, None) == sv.SV_ERR_INVALID_ARG
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_get_plan_draft_logits(None, 1, 1, 10, sv.SV_BF16, 0)
    # the pure planner refuses what the entry point refuses
    assert sv.spec_verify_plan_draft_logits_for(152, 16, 1, 33, 1000, sv.SV_BF16, 0)[0] == \
        sv.SV_ERR_INVALID_ARG
    assert sv.spec_verify_plan_draft_logits_for(152, 16, 1, 3, 1000, 7, 0)[0] == \
        sv.SV_ERR_INVALID_ARG

