"""Seeded synthetic inputs for batched draft verification.

This module serves both sides of every parity check: the CUDA library and the
fp64 oracle read the very same arrays.  It draws random numbers and builds the
*inputs* of the verify step (target logits, draft distributions, draft tokens,
uniforms).  It holds none of the verification arithmetic: no acceptance test,
no residual distribution, no inverse-CDF sampling of the corrected or bonus
token.  The draft side (``q = softmax(draft_logits / T)`` and ``x ~ q``) is part
of producing inputs, exactly as the draft model produces them before the target
verifies (see the pages' draft loop in "Speculative decoding: draft first, then
verify").

Random streams: ``numpy.random.Generator(PCG64(SeedSequence(key)))`` with one key
per field and sequence: [seed, k, b] for the named workloads (k = 0 target
logits, 1 draft noise, 2 boost positions, 3 draft tokens; b the sequence) and
[seed, 4] for the uniforms; the first workload takes its uniforms from
``Philox(0)`` as its recipe states.  Uniforms are float32 in [0, 1).

bf16 logits are produced by rounding the fp64 draw to fp32 (round to nearest
even) and then to bf16 (round to nearest even).  Both sides read the rounded
values; the oracle upcasts them exactly.
"""
from __future__ import annotations

import dataclasses
import os
from typing import Optional

import numpy as np

__all__ = [
    "Inputs", "SweepCell", "CONFIGS", "SWEEP_ALPHAS", "SWEEP_KS",
    "make_config", "make_random", "make_sweep_cell", "sample_tokens",
    "softmax64", "f32_to_bf16_bits", "bf16_bits_to_f32", "logits_as_f64",
    "draft_from_target", "uniforms",
]


# ----------------------------------------------------------------------------
# dtype helpers
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    # the largest finite or infinite pattern plus the rounding bias stays below 2^32
    lsb = (bits >> 16) & np.uint32(1)
    lsb += np.uint32(0x7FFF)
    lsb += bits
    lsb >>= 16
    out = lsb.astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def logits_as_f64(logits: np.ndarray, dtype: str) -> np.ndarray:
    """The stored logits as exact float64 values."""
    if dtype == "bf16":
        return bf16_bits_to_f32(logits).astype(np.float64)
    return np.asarray(logits, dtype=np.float32).astype(np.float64)


def _cast(x64: np.ndarray, dtype: str) -> np.ndarray:
    x32 = x64.astype(np.float32)
    return f32_to_bf16_bits(x32) if dtype == "bf16" else x32


def softmax64(z: np.ndarray) -> np.ndarray:
    """Row-wise softmax in float64, used to build draft distributions."""
    z = np.asarray(z, dtype=np.float64)
    m = np.max(z, axis=-1, keepdims=True)
    e = np.exp(z - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def _rng(seed: int, k: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, k])))


def _rng3(seed: int, k: int, b: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, k, b])))


# ----------------------------------------------------------------------------
# the input bundle
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class Inputs:
    """One verify call's inputs, host-resident.

    logits   [B, K+1, V]  float32, or uint16 bf16 bit patterns when dtype == "bf16"
    q        [B, K, V]    float32 draft probabilities
    tokens   [B, K]       int32 draft tokens
    uniforms [B, K+1]     float32 in [0, 1): u[b, i] for the test at position i,
                          u[b, K] for the one corrected-or-bonus sample
    """
    name: str
    B: int
    K: int
    V: int
    dtype: str
    T: float
    logits: np.ndarray
    q: np.ndarray
    tokens: np.ndarray
    uniforms: np.ndarray

    @property
    def logit_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def nominal_bytes(self) -> int:
        """Logits + all of q + tokens + uniforms + outputs, read/written once."""
        B, K, V = self.B, self.K, self.V
        return (B * (K + 1) * V * self.logit_bytes + B * K * V * 4 + B * K * 4
                + B * (K + 1) * 4 + B * 4 + B * (K + 1) * 4 + B * K)


# ----------------------------------------------------------------------------
# the five workloads of the verify step
# ----------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    B: int
    K: int
    V: int
    dtype: str
    T: float
    sigma: float           # target logits ~ N(0, sigma^2)
    sigma_draft: float     # draft logits = target + N(0, sigma_draft^2)
    boost_frac: float = 0.0
    boost: float = 0.0
    zipf_s: float = 0.0    # additive bias -s * ln(v + 1) over token ids
    seed: int = 0


CONFIGS = {
    "b1_k4_v32000_f32": Config("b1_k4_v32000_f32", 1, 4, 32000, "f32", 1.0, 2.0, 1.0, seed=0),
    "b8_k4_v32000_bf16_peaked": Config("b8_k4_v32000_bf16_peaked", 8, 4, 32000, "bf16", 0.6,
                                       3.0, 0.5, boost_frac=0.01, boost=8.0, seed=1),
    "b64_k3_v151936_bf16": Config("b64_k3_v151936_bf16", 64, 3, 151936, "bf16", 0.6, 2.5, 0.8,
                                  seed=2),
    "b256_k7_v128256_bf16_zipf": Config("b256_k7_v128256_bf16_zipf", 256, 7, 128256, "bf16", 1.0,
                                        2.0, 0.7, zipf_s=1.1, seed=3),
}
CONFIG_ORDER = list(CONFIGS)
SWEEP_ALPHAS = (0.35, 0.5, 0.6, 0.7, 0.8, 0.9)
SWEEP_KS = (1, 3, 5)


def sample_tokens(q_rows: np.ndarray, r: np.ndarray) -> np.ndarray:
    """Draft tokens x ~ q by inverse CDF: first v whose running sum exceeds r * total.

    q_rows [..., V] float32; r [..., n] float64 in [0, 1) -> int32 [..., n].
    This is the draft model's own sampler, part of producing the inputs.
    """
    q_rows = np.asarray(q_rows)
    lead = q_rows.shape[:-1]
    V = q_rows.shape[-1]
    qf = q_rows.reshape(-1, V)
    rf = np.asarray(r, dtype=np.float64).reshape(qf.shape[0], -1)
    out = np.empty(rf.shape, dtype=np.int32)
    for row in range(qf.shape[0]):
        cum = np.cumsum(qf[row].astype(np.float64))
        idx = np.searchsorted(cum, rf[row] * cum[-1], side="right")
        out[row] = np.minimum(idx, V - 1)
    return out.reshape(lead + (rf.shape[1],))


def draft_from_target(target_f64: np.ndarray, sigma_draft: float, T: float,
                      rng: np.random.Generator) -> np.ndarray:
    """q = softmax((target + N(0, sigma_draft^2)) / T), computed in fp64, rounded to fp32."""
    d = target_f64 + sigma_draft * rng.standard_normal(target_f64.shape)
    return softmax64(d / T).astype(np.float32)


def uniforms(seed: int, B: int, K: int) -> np.ndarray:
    return _rng(seed, 4).random((B, K + 1), dtype=np.float32)


def _sequences_into(name: str, seed: int, b0: int, b1: int, logits, q, tokens):
    """Fill logits, draft rows and draft tokens of sequences b0..b1-1 (arrays
    indexed by sequence).  Every sequence has its own streams, so any split of
    the batch gives the same arrays."""
    cfg = CONFIGS[name]
    K, V, T = cfg.K, cfg.V, cfg.T
    bias = -cfg.zipf_s * np.log(np.arange(V, dtype=np.float64) + 1.0) if cfg.zipf_s else None
    n_boost = int(np.floor(cfg.boost_frac * V))
    for b in range(b0, b1):
        rt, rn, rb, rx = (_rng3(seed, k, b) for k in range(4))
        t = cfg.sigma * rt.standard_normal((K + 1, V))
        if n_boost:
            for i in range(K + 1):
                t[i, rb.choice(V, size=n_boost, replace=False)] += cfg.boost
        if bias is not None:
            t += bias
        logits[b] = _cast(t, cfg.dtype)
        if K:
            up = logits_as_f64(logits[b, :K], cfg.dtype)
            q[b] = draft_from_target(up, cfg.sigma_draft, T, rn)
            tokens[b] = sample_tokens(q[b], rx.random((K, 1)))[:, 0]


def _worker(args):
    from multiprocessing import shared_memory
    name, seed, b0, b1, B, shm_names = args
    cfg = CONFIGS[name]
    shapes = _shapes(cfg, B)
    blocks = [shared_memory.SharedMemory(name=n) for n in shm_names]
    try:
        arrs = [np.ndarray(shp, dtype=dt, buffer=blk.buf) for (shp, dt), blk in zip(shapes, blocks)]
        _sequences_into(name, seed, b0, b1, *arrs)
        del arrs
    finally:
        for blk in blocks:
            blk.close()
    return b1 - b0


def _shapes(cfg, B):
    store = np.uint16 if cfg.dtype == "bf16" else np.float32
    return [((B, cfg.K + 1, cfg.V), store), ((B, cfg.K, cfg.V), np.float32), ((B, cfg.K), np.int32)]


def make_config(name: str, seed: Optional[int] = None, B: Optional[int] = None,
                workers: Optional[int] = None) -> Inputs:
    """Build one of the named workloads.  ``seed`` overrides the config's seed;
    ``B`` builds only the first B sequences (a prefix of the full batch).
    Large batches are generated by a spawn-started process pool writing into
    shared memory; the arrays do not depend on the number of workers."""
    cfg = CONFIGS[name]
    seed = cfg.seed if seed is None else seed
    B_full = cfg.B
    B = B_full if B is None else min(B, B_full)
    K, V, T = cfg.K, cfg.V, cfg.T
    shapes = _shapes(cfg, B)
    if workers is None:
        workers = min(16, os.cpu_count() or 1) if B * (2 * K + 1) * V > 50_000_000 else 1
    if workers > 1 and B > 1:
        import concurrent.futures
        import multiprocessing
        from multiprocessing import shared_memory
        blocks = [shared_memory.SharedMemory(create=True, size=max(1, int(np.prod(shp)) * np.dtype(dt).itemsize))
                  for shp, dt in shapes]
        try:
            step = -(-B // workers)
            jobs = [(name, seed, lo, min(B, lo + step), B, [b.name for b in blocks])
                    for lo in range(0, B, step)]
            with concurrent.futures.ProcessPoolExecutor(
                    max_workers=len(jobs), mp_context=multiprocessing.get_context("spawn")) as ex:
                assert sum(ex.map(_worker, jobs)) == B
            logits, q, tokens = (np.ndarray(shp, dtype=dt, buffer=blk.buf).copy()
                                 for (shp, dt), blk in zip(shapes, blocks))
        finally:
            for blk in blocks:
                blk.close()
                blk.unlink()
    else:
        logits, q, tokens = (np.empty(shp, dtype=dt) for shp, dt in shapes)
        _sequences_into(name, seed, 0, B, logits, q, tokens)
    # the first workload takes its uniforms from Philox seed 0 itself
    ru = np.random.Generator(np.random.Philox(0)) if name == "b1_k4_v32000_f32" and seed == 0 \
        else _rng(seed, 4)
    u = ru.random((B_full, K + 1), dtype=np.float32)[:B]
    return Inputs(name, B, K, V, cfg.dtype, T, logits, q, tokens, np.ascontiguousarray(u))


@dataclasses.dataclass
class RaggedInputs:
    """A ragged batch: sequence b owns packed target rows offsets[b] ..
    offsets[b+1]-1, i.e. K_b + 1 rows with its own draft depth K_b.

    logits [R, V], q [R-B, V], tokens [R-B], uniforms [R], offsets [B+1] int32.
    """
    name: str
    B: int
    K_max: int
    V: int
    dtype: str
    T: float
    logits: np.ndarray
    q: np.ndarray
    tokens: np.ndarray
    uniforms: np.ndarray
    offsets: np.ndarray

    @property
    def R(self) -> int:
        return int(self.offsets[-1])

    @property
    def logit_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4


def ragged_from(inp: Inputs, Ks) -> RaggedInputs:
    """Pack the first K_b + 1 target rows, K_b draft rows, K_b tokens and
    K_b + 1 uniforms of every sequence of a uniform batch (K_b <= K)."""
    Ks = np.asarray(Ks, dtype=np.int64)
    assert Ks.shape == (inp.B,) and Ks.min() >= 0 and Ks.max() <= inp.K
    offsets = np.zeros(inp.B + 1, np.int32)
    offsets[1:] = np.cumsum(Ks + 1)
    lg = np.concatenate([inp.logits[b, :k + 1] for b, k in enumerate(Ks)])
    q = (np.concatenate([inp.q[b, :k] for b, k in enumerate(Ks)]) if Ks.sum()
         else np.zeros((0, inp.V), np.float32))
    x = (np.concatenate([inp.tokens[b, :k] for b, k in enumerate(Ks)]) if Ks.sum()
         else np.zeros(0, np.int32))
    u = np.concatenate([inp.uniforms[b, :k + 1] for b, k in enumerate(Ks)])
    return RaggedInputs(inp.name + "_ragged", inp.B, inp.K, inp.V, inp.dtype, inp.T,
                        np.ascontiguousarray(lg), np.ascontiguousarray(q, dtype=np.float32),
                        np.ascontiguousarray(x, dtype=np.int32),
                        np.ascontiguousarray(u, dtype=np.float32), offsets)


@dataclasses.dataclass
class DraftLogitInputs:
    """A workload whose drafter hands over its logits: dlogits [B, K, V] in the
    target's dtype, draft tokens sampled from softmax(dlogits / T_draft), and q
    [B, K, V] = that softmax rounded to float32 (for reference)."""
    name: str
    B: int
    K: int
    V: int
    dtype: str
    T: float
    T_draft: float
    logits: np.ndarray
    dlogits: np.ndarray
    q: np.ndarray
    tokens: np.ndarray
    uniforms: np.ndarray


def with_draft_logits(name: str, seed: Optional[int] = None, B: Optional[int] = None) -> DraftLogitInputs:
    """One of the named workloads with the draft logits themselves: the same
    target rows and the same draft noise stream as make_config (d = target +
    N(0, sigma_draft^2)), d stored in the target's dtype, and draft tokens drawn
    from softmax(d_stored / T) with the same token stream."""
    cfg = CONFIGS[name]
    seed = cfg.seed if seed is None else seed
    inp = make_config(name, seed=seed, B=B)
    Bn, K, V, T = inp.B, cfg.K, cfg.V, cfg.T
    d_st = np.empty((Bn, K, V), dtype=inp.logits.dtype)
    q = np.empty((Bn, K, V), dtype=np.float32)
    tokens = np.empty((Bn, K), dtype=np.int32)
    for b in range(Bn):
        rn, rx = _rng3(seed, 1, b), _rng3(seed, 3, b)
        if not K:
            continue
        up = logits_as_f64(inp.logits[b, :K], cfg.dtype)
        d = up + cfg.sigma_draft * rn.standard_normal(up.shape)
        d_st[b] = _cast(d, cfg.dtype)
        qd = softmax64(logits_as_f64(d_st[b], cfg.dtype) / T)
        q[b] = qd.astype(np.float32)
        tokens[b] = sample_tokens(qd, rx.random((K, 1)))[:, 0]
    return DraftLogitInputs(name + "_dlogits", Bn, K, V, cfg.dtype, T, T, inp.logits, d_st, q,
                            tokens, inp.uniforms)


def make_random_draft_logits(B: int, K: int, V: int, dtype: str = "f32", T: float = 1.0,
                             T_draft: float = 1.0, sigma: float = 2.0, sigma_draft: float = 1.0,
                             seed: int = 0) -> DraftLogitInputs:
    """Small random instance whose drafter hands over its logits: target rows as
    make_random, d = target + N(0, sigma_draft^2) stored in the target's dtype,
    draft tokens drawn from softmax(d_stored / T_draft)."""
    inp = make_random(B, K, V, dtype, T=T, sigma=sigma, sigma_draft=sigma_draft, seed=seed)
    rn, rx = _rng(seed, 11), _rng(seed, 13)
    up = logits_as_f64(inp.logits[:, :K], dtype)
    d_st = _cast(up + sigma_draft * rn.standard_normal(up.shape), dtype)
    q64 = softmax64(logits_as_f64(d_st, dtype) / float(np.float32(T_draft))) if K else \
        np.zeros((B, 0, V))
    tokens = (sample_tokens(q64, rx.random((B, K, 1)))[..., 0] if K
              else np.zeros((B, 0), np.int32))
    return DraftLogitInputs(f"random_dlogits_{B}x{K}x{V}", B, K, V, dtype, T, T_draft, inp.logits,
                            np.ascontiguousarray(d_st), q64.astype(np.float32),
                            np.ascontiguousarray(tokens.astype(np.int32)), inp.uniforms)


def greedy_drafts(inp: Inputs) -> Inputs:
    """The same workload with a greedy drafter: x_i = argmax_v q[b, i, v] (lowest
    id among equal maxima) instead of a draw from q.  Used for greedy
    verification, where the target side is greedy too."""
    tokens = (np.argmax(inp.q, axis=-1).astype(np.int32) if inp.K
              else np.zeros((inp.B, 0), np.int32))
    return Inputs(inp.name + "_greedy", inp.B, inp.K, inp.V, inp.dtype, inp.T, inp.logits, inp.q,
                  np.ascontiguousarray(tokens), inp.uniforms)


def make_random(B: int, K: int, V: int, dtype: str = "f32", T: float = 1.0, sigma: float = 2.0,
                sigma_draft: float = 1.0, seed: int = 0, name: str = "random") -> Inputs:
    """Small random instance with the value distribution of the first workload."""
    rt, rn, rx, ru = _rng(seed, 0), _rng(seed, 1), _rng(seed, 3), _rng(seed, 4)
    t = sigma * rt.standard_normal((B, K + 1, V))
    logits = _cast(t, dtype)
    up = logits_as_f64(logits, dtype)
    q = draft_from_target(up[:, :K], sigma_draft, T, rn) if K else np.zeros((B, 0, V), np.float32)
    tokens = sample_tokens(q, rx.random((B, K, 1)))[..., 0] if K else np.zeros((B, 0), np.int32)
    u = ru.random((B, K + 1), dtype=np.float32)
    return Inputs(name, B, K, V, dtype, T, np.ascontiguousarray(logits), np.ascontiguousarray(q),
                  np.ascontiguousarray(tokens.astype(np.int32)), u)


# ----------------------------------------------------------------------------
# acceptance sweep: draft rows with a controlled overlap alpha = sum_v min(p, q)
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class SweepCell:
    """Fixed target logits and draft rows for one (alpha, K) cell, plus `rounds`
    fresh draws of draft tokens and uniforms.

    logits [B, K+1, V] f32, q [B, K, V] f32, tokens [R, B, K], uniforms [R, B, K+1].
    """
    alpha: float
    B: int
    K: int
    V: int
    T: float
    logits: np.ndarray
    q: np.ndarray
    tokens: np.ndarray
    uniforms: np.ndarray

    def round_inputs(self, r: int) -> Inputs:
        return Inputs(f"sweep_a{self.alpha}_k{self.K}_r{r}", self.B, self.K, self.V, "f32", self.T,
                      self.logits, self.q, np.ascontiguousarray(self.tokens[r]),
                      np.ascontiguousarray(self.uniforms[r]))


def make_sweep_cell(alpha: float, K: int, B: int = 32, V: int = 32000, rounds: int = 10 ** 4,
                    seed: int = 4, sigma: float = 2.0, dirichlet: float = 0.1) -> SweepCell:
    """Target rows softmax(N(0, sigma^2)) at T = 1; each draft row is the mixture
    (1 - w) p + w r with r ~ Dirichlet(dirichlet) and w = (1 - alpha) / TV(p, r),
    so that sum_v min(p, q) = 1 - w * TV(p, r) = alpha (r is redrawn while
    TV(p, r) < 1 - alpha).  Draft tokens and uniforms are fresh in every round."""
    cell_seed = seed * 1000 + int(round(alpha * 100)) * 10 + K
    rt, rm, rx, ru = _rng(cell_seed, 0), _rng(cell_seed, 2), _rng(cell_seed, 3), _rng(cell_seed, 4)
    logits = (sigma * rt.standard_normal((B, K + 1, V))).astype(np.float32)
    p = softmax64(logits.astype(np.float64))
    q = np.empty((B, K, V), dtype=np.float32)
    for b in range(B):
        for i in range(K):
            while True:
                g = rm.standard_gamma(dirichlet, V)
                s = g.sum()
                if s <= 0:
                    continue
                r = g / s
                tv = np.maximum(p[b, i] - r, 0.0).sum()
                if tv >= 1.0 - alpha:
                    break
            w = (1.0 - alpha) / tv
            q[b, i] = ((1.0 - w) * p[b, i] + w * r).astype(np.float32)
    tokens = np.empty((rounds, B, K), dtype=np.int32)
    if K:
        draws = rx.random((B, K, rounds))
        tokens[:] = np.moveaxis(sample_tokens(q, draws), -1, 0)
    u = ru.random((rounds, B, K + 1), dtype=np.float32)
    return SweepCell(alpha, B, K, V, 1.0, logits, q, tokens, u)
