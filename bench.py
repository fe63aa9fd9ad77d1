#!/usr/bin/env python
"""Benchmark of the batched draft-verification step on GB300.

One step = one spec_verify_run call over one batch of the workload (the whole
hot path: row softmax statistics, accept tests, first-rejection scan, residual
or bonus draw).  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Metric: verified rows/s, rows = B*(K+1) per step, with inputs resident in HBM
(value), plus tokens/s, algorithmic HBM GB/s and its fraction of the measured
copy bandwidth (roofline), the fp64 CPU oracle on a bounded sample
(cpu_baseline), and the same metric through the host-buffer entry point with
the copies inside the timed region (e2e).  Several copies of the inputs are
rotated so that no step finds the previous step's data in L2 (each copy is
larger than L2).  Under torchrun every rank verifies its own batch (weak
scaling, no collective besides the timing barrier and max).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "verified rows/s and HBM GB/s (% of GB300 peak) for B×(K+1)×V verify"
DEFAULT_WORKLOAD = "b256_k7_v128256_bf16_zipf"
L2_BYTES = 129 * 1024 * 1024
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=workloads.CONFIG_ORDER)
    ap.add_argument("--mode", choices=["sampled", "greedy", "ragged", "truncated",
                                       "draft_logits"],
                    default="sampled",
                    help="sampled: spec_verify_run at the workload's temperature; greedy: "
                         "spec_verify_run_greedy (T -> 0) with a greedy drafter; ragged: "
                         "spec_verify_run_ragged with per-sequence depths K_b ~ U{0..K}; "
                         "truncated: spec_verify_run_truncated with --top-p / --min-p; "
                         "draft_logits: spec_verify_run_draft_logits with the drafter's "
                         "logits (T_d = T, untruncated target)")
    ap.add_argument("--top-p", type=float, default=0.95)
    ap.add_argument("--min-p", type=float, default=0.05)
    ap.add_argument("--sets", type=int, default=3, help="input copies rotated between steps")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph-launches", type=int, default=30,
                    help="steps captured in one CUDA graph for the graph-replay timing (0 = skip)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--stat-launches", type=int, default=100,
                    help="launches timed one by one for the median / p95 per launch")
    ap.add_argument("--clock-window", type=float, default=2.0,
                    help="seconds of untimed load, sampled for clocks, before the timed steps")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, dist, device: str = "cuda") -> float:
    """The largest of every rank's x (the job takes as long as its slowest rank)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_inputs(workload: str, rank: int):
    """Weak scaling: every rank verifies a batch of its own, the workload's
    recipe with the seed moved by the rank (sequences are independent, so the
    ranks exchange nothing)."""
    cfg = workloads.CONFIGS[workload]
    return workloads.make_config(workload, seed=cfg.seed + rank)


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


_CSRC = "speculative_decoding_verification_14_gb300/csrc/"
# the sources each mode's kernel and launch path are built from (every entry
# point's host side lives in spec_verify.cu)
KERNEL_SOURCES = {
    "sampled": ("spec_verify.cu", "sv_internal.h", "planner.cpp"),
    "ragged": ("spec_verify.cu", "sv_internal.h", "planner.cpp"),
    "greedy": ("greedy.cu", "spec_verify.cu", "sv_internal.h", "planner.cpp"),
    "truncated": ("truncated.cu", "spec_verify.cu", "sv_internal.h", "planner.cpp"),
    "draft_logits": ("spec_verify.cu", "sv_internal.h", "planner.cpp"),
}


def kernel_source_hash(mode: str = "sampled") -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[mode]:
        with open(os.path.join(ROOT, _CSRC + rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profile_traffic(workload: str, mode: str):
    """DRAM bytes per launch from the committed ncu summary, if it covers this
    workload and mode and was taken on the current sources of that mode's
    kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    key = workload + ("" if mode == "sampled" else "_" + mode)
    try:
        with open(path) as f:
            e = json.load(f).get(key)
        if not e or e.get("kernel_source_sha256") != kernel_source_hash(mode):
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


# ------------------------------------------------------------ byte counts -----

def algorithmic_bytes(inp, accept_len: np.ndarray) -> int:
    """Bytes the method must move for one verify, from its outputs.

    Per sequence b with accepted length n = accept_len[b] (rows 0..n-1 reached):
      n rows of logits (V * sizeof(logit) each)             -- the test loop reads
                                                               rows in order and
                                                               stops at the first
                                                               rejection
      + V * 4 for the draft row q_j when a draft was rejected (n <= K)
      + 4 per test that ran (q(x_i) gathered), min(n, K) tests
      + K * 4 (draft tokens) + (K + 1) * 4 (uniforms)
      + outputs: 4 + (K + 1) * 4 + K
    The method needs row j once: the draw's second read of it (and rows read
    before a rejection was known) are traffic, not algorithmic bytes.
    """
    B, K, V, es = inp.B, inp.K, inp.V, inp.logit_bytes
    n = accept_len.astype(np.int64)
    rows = int(n.sum())
    rejected = int((n <= K).sum())
    tests = int(np.minimum(n, K).sum())
    return (rows * V * es + rejected * V * 4 + tests * 4 + B * K * 4 + B * (K + 1) * 4
            + B * (4 + (K + 1) * 4 + K))


def algorithmic_bytes_truncated(inp, accept_len: np.ndarray, min_p: float) -> int:
    """As algorithmic_bytes, except that with min-p on the residual reads q_j
    only at the kept tokens (max(0, p~ - q) is zero elsewhere): the rejected
    draft row's V * 4 bytes drop out (its few kept entries, 4-byte gathers,
    are not counted).  With min-p off the draw streams q_j whole."""
    full = algorithmic_bytes(inp, accept_len)
    if min_p <= 0.0:
        return full
    rejected = int((accept_len.astype(np.int64) <= inp.K).sum())
    return full - rejected * inp.V * 4


def algorithmic_bytes_ragged(rg, accept_len: np.ndarray) -> int:
    """Ragged batch: the per-sequence count of algorithmic_bytes with each
    sequence's own depth K_b, plus the row offsets."""
    V, es = rg.V, rg.logit_bytes
    Ks = np.diff(rg.offsets.astype(np.int64)) - 1
    n = accept_len.astype(np.int64)
    per = (n * V * es + (n <= Ks) * V * 4 + np.minimum(n, Ks) * 4 + Ks * 4 + (Ks + 1) * 4
           + 4 + (Ks + 1) * 4 + Ks)
    return int(per.sum()) + (rg.B + 1) * 4


def algorithmic_bytes_draft_logits(inp, accept_len: np.ndarray) -> int:
    """Verify with draft logits: per sequence with accepted length n, the n
    target rows reached and the min(n, K) draft rows tested (each row's
    normaliser needs all of it; the residual re-uses the rejected draft row),
    plus tokens, uniforms and outputs as algorithmic_bytes."""
    B, K, V = inp.B, inp.K, inp.V
    es = 2 if inp.dtype == "bf16" else 4
    n = accept_len.astype(np.int64)
    rows = int(n.sum()) + int(np.minimum(n, K).sum())
    return rows * V * es + B * K * 4 + B * (K + 1) * 4 + B * (4 + (K + 1) * 4 + K)


def algorithmic_bytes_greedy(inp, accept_len: np.ndarray) -> int:
    """Greedy verification: n rows of logits per sequence (rows 0..n-1, read in
    order up to the first rejection), the K draft tokens, and the outputs."""
    B, K, V, es = inp.B, inp.K, inp.V, inp.logit_bytes
    rows = int(accept_len.astype(np.int64).sum())
    return rows * V * es + B * K * 4 + B * (4 + (K + 1) * 4 + K)


# ---------------------------------------------------------------- clocks -----

class ClockSampler:
    def __init__(self, device: int):
        self.device = device
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.device)], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# -------------------------------------------------------------- our arm -----

def run_ours(args):
    import torch
    import speculative_decoding_verification_14_gb300 as sv

    world, rank, local = dist_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.cuda.current_device()

    cfg = workloads.CONFIGS[args.workload]
    inp = rank_inputs(args.workload, rank)
    greedy = args.mode == "greedy"
    ragged = args.mode == "ragged"
    trunc = args.mode == "truncated"
    dlog = args.mode == "draft_logits"
    if greedy:
        inp = workloads.greedy_drafts(inp)
    if dlog:
        inp = workloads.with_draft_logits(args.workload, seed=cfg.seed + rank)
    rg = None
    if ragged:  # each sequence keeps its first K_b + 1 rows, K_b ~ U{0..K}
        Ks = np.random.default_rng(1000 + cfg.seed + rank).integers(0, inp.K + 1, inp.B)
        rg = workloads.ragged_from(inp, Ks)
    B, K, V, T = inp.B, inp.K, inp.V, inp.T
    dcode = sv.SV_BF16 if inp.dtype == "bf16" else sv.SV_F32
    per_set = (inp.logits.nbytes + inp.tokens.nbytes if greedy else
               rg.logits.nbytes + rg.q.nbytes if ragged else
               inp.logits.nbytes + inp.dlogits.nbytes + inp.tokens.nbytes + inp.uniforms.nbytes
               if dlog else inp.nominal_bytes())
    nsets = max(1, args.sets)

    def dev_logits(src=None):
        src = inp.logits if src is None else src
        if inp.dtype == "bf16":
            return torch.from_numpy(src.view(np.int16)).cuda().view(torch.bfloat16)
        return torch.from_numpy(src).cuda()

    sets = []
    for s in range(nsets):
        if greedy:  # the greedy step reads no draft probabilities and no uniforms
            sets.append((dev_logits(), None, torch.from_numpy(inp.tokens).cuda(), None))
        elif dlog:  # the drafter's logits take q's place
            sets.append((dev_logits(), dev_logits(inp.dlogits), torch.from_numpy(inp.tokens).cuda(),
                         torch.from_numpy(inp.uniforms).cuda()))
        elif ragged:
            sets.append((dev_logits(rg.logits), torch.from_numpy(rg.q).cuda(),
                         torch.from_numpy(rg.tokens).cuda(), torch.from_numpy(rg.uniforms).cuda(),
                         torch.from_numpy(rg.offsets).cuda()))
        else:
            sets.append((dev_logits(), torch.from_numpy(inp.q).cuda(),
                         torch.from_numpy(inp.tokens).cuda(), torch.from_numpy(inp.uniforms).cuda()))
    rows_per_step = rg.R if ragged else B * (K + 1)
    outs = {"accept_len": torch.empty(B, dtype=torch.int32, device="cuda"),
            "out_tokens": torch.empty(rows_per_step, dtype=torch.int32, device="cuda"),
            "accept_mask": torch.empty(rows_per_step - B, dtype=torch.uint8, device="cuda")}
    verifier = sv.Verifier(B, K, V)
    stream = torch.cuda.current_stream()
    lib = sv.library()
    calls = []
    for st in sets:
        lg, q, x, u = st[:4]
        if ragged:
            calls.append((verifier.ctx, lg.data_ptr(), dcode, q.data_ptr(), x.data_ptr(),
                          u.data_ptr(), st[4].data_ptr(), rg.R, B, K, V, ctypes.c_float(T),
                          outs["accept_len"].data_ptr(), outs["out_tokens"].data_ptr(),
                          outs["accept_mask"].data_ptr(), None, None, None))
        elif dlog:
            calls.append((verifier.ctx, lg.data_ptr(), dcode, q.data_ptr(), x.data_ptr(),
                          u.data_ptr(), B, K, V, ctypes.c_float(T), ctypes.c_float(inp.T_draft),
                          ctypes.c_double(1.0), ctypes.c_double(0.0),
                          outs["accept_len"].data_ptr(), outs["out_tokens"].data_ptr(),
                          outs["accept_mask"].data_ptr(), None, None, None))
        elif trunc:
            calls.append((verifier.ctx, lg.data_ptr(), dcode, q.data_ptr(), x.data_ptr(),
                          u.data_ptr(), B, K, V, ctypes.c_float(T), ctypes.c_double(args.top_p),
                          ctypes.c_double(args.min_p), outs["accept_len"].data_ptr(),
                          outs["out_tokens"].data_ptr(), outs["accept_mask"].data_ptr(), None,
                          None, None))
        elif greedy:
            calls.append((verifier.ctx, lg.data_ptr(), dcode, x.data_ptr(), B, K, V,
                          outs["accept_len"].data_ptr(), outs["out_tokens"].data_ptr(),
                          outs["accept_mask"].data_ptr(), None, None))
        else:
            calls.append((verifier.ctx, lg.data_ptr(), dcode, q.data_ptr(), x.data_ptr(),
                          u.data_ptr(), B, K, V, ctypes.c_float(T), outs["accept_len"].data_ptr(),
                          outs["out_tokens"].data_ptr(), outs["accept_mask"].data_ptr(), None,
                          None, None))
    run = (lib.spec_verify_run_greedy if greedy else lib.spec_verify_run_ragged if ragged
           else lib.spec_verify_run_truncated if trunc
           else lib.spec_verify_run_draft_logits if dlog else lib.spec_verify_run)

    def step(k, s=None):
        rc = run(*calls[k % nsets], stream.cuda_stream if s is None else s)
        if rc != 0:
            raise sv.SpecVerifyError(rc, f"verify ({args.mode})")

    def barrier():
        if dist is not None:
            dist.barrier()

    # warm-up, then an untimed sampled window for the clock record
    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize()
    clocks = ClockSampler(dev)
    clocks.start()
    t_end = time.time() + args.clock_window
    k = 0
    while time.time() < t_end:
        for _ in range(64):
            step(k)
            k += 1
        torch.cuda.synchronize()

    # Inputs larger than L2 (several copies rotated): K back-to-back steps
    # between two events on the launch stream (events between the launches
    # would add their own gaps).  Inputs that fit in L2: every step is preceded
    # by a write of twice the L2 size, and the step alone is timed between two
    # events, so each step starts with its inputs in HBM only.
    flush = per_set <= L2_BYTES
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda") if flush else None
    barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if flush:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        t0.record(stream)
        for k in range(args.steps):
            flush_buf.zero_()
            evs[k][0].record(stream)
            step(k)
            evs[k][1].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
        total_ms = sum(a.elapsed_time(b) for a, b in evs)
    else:
        t0.record(stream)
        for k in range(args.steps):
            step(k)
        t1.record(stream)
        torch.cuda.synchronize()
        total_ms = t0.elapsed_time(t1)
    barrier()
    clk = clocks.stop()
    local_ms = total_ms
    total_ms = max_over_ranks(total_ms, dist)

    # per-launch statistics: an event after every launch (flushed inputs: an
    # event pair around every launch); the event adds its own small gap
    stats = None
    if args.stat_launches > 0:
        n_st = args.stat_launches
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_st + 1)]
        per = []
        if flush:
            for k in range(n_st):
                flush_buf.zero_()
                ev[0].record(stream)
                step(k)
                ev[1].record(stream)
                torch.cuda.synchronize()
                per.append(ev[0].elapsed_time(ev[1]) * 1e3)
        else:
            ev[0].record(stream)
            for k in range(n_st):
                step(k)
                ev[k + 1].record(stream)
            torch.cuda.synchronize()
            per = [ev[k].elapsed_time(ev[k + 1]) * 1e3 for k in range(n_st)]
        per = np.sort(np.asarray(per))
        stats = {"median_us": float(np.median(per)), "p95_us": float(np.percentile(per, 95)),
                 "mean_us": float(per.mean()), "min_us": float(per[0]), "n": n_st,
                 "method": ("an event pair around each launch, L2 flushed before it" if flush else
                            "an event recorded after each of n back-to-back launches (the events "
                            "add their own gaps)")}

    # the same steps replayed from a CUDA graph: no host launch cost between
    # kernels, so small workloads show their device time
    graph = None
    if args.graph_launches > 0:
        n_in = args.graph_launches
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step(0, side.cuda_stream)  # outside the capture: the library is set up
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=side):
                for k in range(n_in):
                    step(k, side.cuda_stream)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        reps = max(3, min(50, int(2e5 / max(1.0, local_ms * 1e3 / args.steps * n_in))))
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(reps):
            g.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        graph = {"us_per_launch": g0.elapsed_time(g1) * 1e3 / (reps * n_in),
                 "launches_per_graph": n_in, "replays": reps}
        del g

    err, _ = verifier.error()
    if err != sv.SV_OK:
        raise sv.SpecVerifyError(err, "device error during the benchmark")
    acc = outs["accept_len"].cpu().numpy()
    alg = (algorithmic_bytes_greedy(inp, acc) if greedy else
           algorithmic_bytes_ragged(rg, acc) if ragged else
           algorithmic_bytes_draft_logits(inp, acc) if dlog else
           algorithmic_bytes_truncated(inp, acc, args.min_p) if trunc else algorithmic_bytes(inp, acc))
    avg_launch_s = local_ms / args.steps / 1e3  # this rank's average launch duration
    value = world * rows_per_step * args.steps / (total_ms / 1e3)
    tokens_per_step = int(acc.sum())
    peak, peak_kind = measured_peak()
    achieved = alg / avg_launch_s / 1e9
    plan = (verifier.plan_greedy(B, K, V, dcode) if greedy else
            verifier.plan_truncated(B, K, V, dcode) if trunc else
            verifier.plan_draft_logits(B, K, V, dcode, 0) if dlog else verifier.plan(B, K, V, dcode))

    # end to end through the host-buffer entry point, copies inside the region
    e2e = None
    if greedy and not args.no_e2e and args.e2e_steps > 0:
        e2e = e2e_greedy(args, inp, verifier, acc, dist, world, rows_per_step)
    elif ragged and not args.no_e2e and args.e2e_steps > 0:
        e2e = e2e_ragged(args, rg, verifier, acc, dist, world)
    elif trunc and not args.no_e2e and args.e2e_steps > 0:
        e2e = e2e_truncated(args, inp, verifier, acc, dist, world, rows_per_step)
    elif dlog and not args.no_e2e and args.e2e_steps > 0:
        e2e = e2e_draft_logits(args, inp, verifier, acc, dist, world, rows_per_step)
    elif not args.no_e2e and args.e2e_steps > 0:
        def pinned(a):
            t = torch.empty(a.shape, dtype={np.float32: torch.float32, np.uint16: torch.int16,
                                            np.int32: torch.int32, np.uint8: torch.uint8}[a.dtype.type],
                            pin_memory=True)
            arr = t.numpy()
            arr[...] = a.view(arr.dtype) if a.dtype != arr.dtype else a
            return t, arr
        keep = []
        h = {}
        for name, a in (("logits", inp.logits), ("q", inp.q), ("tokens", inp.tokens),
                        ("uniforms", inp.uniforms)):
            t, arr = pinned(a)
            keep.append(t)
            h[name] = arr
        hout = {}
        for name, shape, dt in (("accept_len", (B,), np.int32), ("out_tokens", (B, K + 1), np.int32),
                                ("accept_mask", (B, K), np.uint8)):
            t, arr = pinned(np.zeros(shape, dt))
            keep.append(t)
            hout[name] = arr
        rc = verifier.run_host(h["logits"], dcode, h["q"], h["tokens"], h["uniforms"], T, hout,
                               stream=stream.cuda_stream)  # first call allocates staging
        assert rc == sv.SV_OK, sv.spec_verify_strerror(rc)
        barrier()
        ts = time.perf_counter()
        for _ in range(args.e2e_steps):
            rc = verifier.run_host(h["logits"], dcode, h["q"], h["tokens"], h["uniforms"], T, hout,
                                   stream=stream.cuda_stream)
            assert rc == sv.SV_OK
        el = time.perf_counter() - ts
        el = max_over_ranks(el, dist)
        assert np.array_equal(hout["accept_len"], acc)
        h2d = inp.logits.nbytes + inp.q.nbytes + inp.tokens.nbytes + inp.uniforms.nbytes
        d2h = hout["accept_len"].nbytes + hout["out_tokens"].nbytes + hout["accept_mask"].nbytes + 4
        e2e = {"value": world * rows_per_step * args.e2e_steps / el, "unit": "rows/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "steps": args.e2e_steps, "api": "spec_verify_run_host (pinned host buffers)"}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = (cpu_baseline_ragged(rg, args.cpu_seconds) if ragged
               else cpu_baseline(inp, args.cpu_seconds, greedy=greedy,
                                 trunc=(args.top_p, args.min_p) if trunc else None, dlog=dlog))

    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload + (" with a greedy drafter, greedy verify (T -> 0)"
                                                if greedy else
                                                " as a ragged batch, K_b ~ U{0..K}, packed rows"
                                                if ragged else
                                                f" against the truncated target (top-p "
                                                f"{args.top_p}, min-p {args.min_p})"
                                                if trunc else
                                                " with the drafter's logits (bf16/f32 like the "
                                                "target, T_d = T), untruncated target"
                                                if dlog else ""),
                   "rows": rows_per_step,
                   "B": B, "K": K, "V": V, "logits_dtype": inp.dtype,
                   "T": 0.0 if greedy else T,
                   "l2": (f"L2 flushed before every step ({2 * L2_BYTES >> 20} MB written; inputs "
                          f"{per_set / 1e6:.1f} MB), each step timed alone between two events"
                          if flush else
                          f"{nsets} input copies of {per_set / 1e9:.2f} GB rotated "
                          f"(each larger than the {L2_BYTES >> 20} MB L2)"),
                   "plan": plan},
        "tokens_per_s": world * tokens_per_step * args.steps / (total_ms / 1e3),
        "mean_accept_len": float(acc.mean()),
        "hbm_gbs_algorithmic": achieved,
        "per_launch": stats,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": profile_traffic(args.workload, args.mode),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind ==
                     "measured" else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": alg, "avg_launch_us": avg_launch_s * 1e6},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "graph_replay": graph,
        "clocks": clk,
    }
    return line


def host_cores() -> dict:
    """The host threads this process may run on, and lscpu's CPU count."""
    info = {"affinity": len(os.sched_getaffinity(0))}
    try:
        out = subprocess.run(["lscpu"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                             text=True, timeout=10).stdout
        for line in out.splitlines():
            k, _, v = line.partition(":")
            if k.strip() in ("CPU(s)", "Model name", "Thread(s) per core"):
                info["lscpu " + k.strip()] = v.strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return info


def _time_oracle(one, B: int, seconds: float, rows_per_seq: float, par: int = 1):
    """Whole passes of one(n) over the first n sequences until `seconds` of
    wall time have passed; n is sized from a first call on min(B, par)
    sequences so that a pass takes about a quarter of `seconds`."""
    m = min(B, par)
    t = time.perf_counter()
    one(m)
    rate = m / max(time.perf_counter() - t, 1e-6)  # sequences per second
    n = int(min(B, max(m, rate * seconds / 4)))
    reps = 0
    t = time.perf_counter()
    while True:
        one(n)
        reps += 1
        el = time.perf_counter() - t
        if el >= seconds:
            break
    return (reps * n * rows_per_seq / el,
            f"{reps} pass(es) over the first {n} of {B} sequences ({el:.1f} s)")


def _oracle_call(inp, lib, greedy=False, trunc=None, dlog=False):
    import oracle

    def one(n):
        if greedy:
            oracle.verify_greedy(inp.logits[:n], inp.dtype, inp.tokens[:n], lib=lib)
        elif dlog:
            oracle.verify_draft_logits(inp.logits[:n], inp.dtype, inp.dlogits[:n], inp.tokens[:n],
                                       inp.uniforms[:n], inp.T, inp.T_draft, lib=lib)
        elif trunc is not None:
            oracle.verify_truncated(inp.logits[:n], inp.dtype, inp.q[:n], inp.tokens[:n],
                                    inp.uniforms[:n], inp.T, trunc[0], trunc[1], lib=lib)
        else:
            oracle.verify(inp.logits[:n], inp.dtype, inp.q[:n], inp.tokens[:n], inp.uniforms[:n],
                          inp.T, lib=lib)
    return one


def cpu_baseline(inp, seconds: float, greedy: bool = False, trunc=None, dlog=False) -> dict:
    """The oracle as it stands on the host cores: the OpenMP build of oracle.c
    (sequences spread over every core this process may use) and, beside it, the
    plain build on one thread, each on whole passes over the first sequences of
    the workload until `seconds` have passed."""
    import oracle
    oracle.build()
    cores = host_cores()
    v1, s1 = _time_oracle(_oracle_call(inp, None, greedy, trunc, dlog), inp.B, seconds, inp.K + 1)
    single = {"value": v1, "unit": "rows/s", "cores": 1, "kind": "oracle", "sample": s1,
              "build": "oracle.c, plain"}
    try:
        omp = oracle.load_openmp(cores["affinity"])
        nth = omp.oracle_threads()
    except Exception as e:  # no OpenMP runtime: the single-thread figure alone
        single["host"] = cores
        single["openmp"] = f"unavailable: {e}"
        return single
    vn, sn = _time_oracle(_oracle_call(inp, omp, greedy, trunc, dlog), inp.B, seconds, inp.K + 1,
                          par=nth)
    return {"value": vn, "unit": "rows/s", "cores": nth, "kind": "oracle", "sample": sn,
            "build": f"oracle.c with -fopenmp, sequences over {nth} threads",
            "host": cores, "single_thread": single}


def cpu_baseline_ragged(rg, seconds: float) -> dict:
    """The ragged oracle as it stands: OpenMP build on every core, and the
    plain build on one thread beside it, whole passes over the batch."""
    import oracle
    oracle.build()
    cores = host_cores()

    def timed(lib):
        t = time.perf_counter()
        reps = 0
        while True:
            oracle.verify_ragged(rg.logits, rg.dtype, rg.q, rg.tokens, rg.uniforms, rg.offsets,
                                 rg.K_max, rg.T, lib=lib)
            reps += 1
            el = time.perf_counter() - t
            if el >= seconds:
                break
        return reps * rg.R / el, f"{reps} pass(es) over all {rg.B} sequences ({rg.R} rows, {el:.1f} s)"
    v1, s1 = timed(None)
    single = {"value": v1, "unit": "rows/s", "cores": 1, "kind": "oracle", "sample": s1,
              "build": "oracle.c, plain"}
    try:
        omp = oracle.load_openmp(cores["affinity"])
        nth = omp.oracle_threads()
    except Exception as e:
        single["host"] = cores
        single["openmp"] = f"unavailable: {e}"
        return single
    vn, sn = timed(omp)
    return {"value": vn, "unit": "rows/s", "cores": nth, "kind": "oracle", "sample": sn,
            "build": f"oracle.c with -fopenmp, sequences over {nth} threads",
            "host": cores, "single_thread": single}


def e2e_ragged(args, rg, verifier, acc, dist, world) -> dict:
    """Ragged batch end to end through the public API: pinned host copies of
    the packed inputs to the device, spec_verify_run_ragged, outputs back, all
    inside the timed region."""
    import torch
    h = {"logits": torch.from_numpy(rg.logits.view(np.int16) if rg.dtype == "bf16"
                                    else rg.logits).pin_memory(),
         "q": torch.from_numpy(rg.q).pin_memory(), "tokens": torch.from_numpy(rg.tokens).pin_memory(),
         "uniforms": torch.from_numpy(rg.uniforms).pin_memory(),
         "offsets": torch.from_numpy(rg.offsets).pin_memory()}
    d = {k: torch.empty(t.shape, dtype=t.dtype, device="cuda") for k, t in h.items()}
    R, B = rg.R, rg.B
    h_out = {k: torch.empty(n, dtype=dt).pin_memory() for k, n, dt in
             (("accept_len", B, torch.int32), ("out_tokens", R, torch.int32),
              ("accept_mask", R - B, torch.uint8))}

    def once():
        for k in h:
            d[k].copy_(h[k], non_blocking=True)
        lg = d["logits"].view(torch.bfloat16) if rg.dtype == "bf16" else d["logits"]
        out = verifier.run_ragged(lg, d["q"], d["tokens"], d["uniforms"], d["offsets"], rg.K_max,
                                  rg.T, status=False)
        for k, t in h_out.items():
            t.copy_(out[k], non_blocking=True)
        torch.cuda.current_stream().synchronize()
    once()
    if dist is not None:
        dist.barrier()
    ts = time.perf_counter()
    for _ in range(args.e2e_steps):
        once()
    el = time.perf_counter() - ts
    el = max_over_ranks(el, dist)
    assert np.array_equal(h_out["accept_len"].numpy(), acc)
    return {"value": world * R * args.e2e_steps / el, "unit": "rows/s",
            "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in h.values())),
            "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in h_out.values())),
            "steps": args.e2e_steps,
            "api": "Verifier.run_ragged (spec_verify_run_ragged) with pinned host copies"}


def e2e_truncated(args, inp, verifier, acc, dist, world, rows_per_step) -> dict:
    """Truncated-target verify end to end through the public API: pinned host
    inputs copied to the device, spec_verify_run_truncated, outputs copied
    back, all inside the timed region."""
    import torch
    B, K = inp.B, inp.K
    h = {"logits": torch.from_numpy(inp.logits.view(np.int16) if inp.dtype == "bf16"
                                    else inp.logits).pin_memory(),
         "q": torch.from_numpy(inp.q).pin_memory(), "tokens": torch.from_numpy(inp.tokens).pin_memory(),
         "uniforms": torch.from_numpy(inp.uniforms).pin_memory()}
    d = {k: torch.empty(t.shape, dtype=t.dtype, device="cuda") for k, t in h.items()}
    h_out = {k: torch.empty(shape, dtype=dt).pin_memory() for k, shape, dt in
             (("accept_len", (B,), torch.int32), ("out_tokens", (B, K + 1), torch.int32),
              ("accept_mask", (B, K), torch.uint8))}

    def once():
        for k in h:
            d[k].copy_(h[k], non_blocking=True)
        lg = d["logits"].view(torch.bfloat16) if inp.dtype == "bf16" else d["logits"]
        out = verifier.run_truncated(lg, d["q"], d["tokens"], d["uniforms"], inp.T, args.top_p,
                                     args.min_p, status=False)
        for k, t in h_out.items():
            t.copy_(out[k], non_blocking=True)
        torch.cuda.current_stream().synchronize()
    once()
    if dist is not None:
        dist.barrier()
    ts = time.perf_counter()
    for _ in range(args.e2e_steps):
        once()
    el = max_over_ranks(time.perf_counter() - ts, dist)
    assert np.array_equal(h_out["accept_len"].numpy(), acc)
    return {"value": world * rows_per_step * args.e2e_steps / el, "unit": "rows/s",
            "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in h.values())),
            "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in h_out.values())),
            "steps": args.e2e_steps,
            "api": "Verifier.run_truncated (spec_verify_run_truncated) with pinned host copies"}


def e2e_draft_logits(args, inp, verifier, acc, dist, world, rows_per_step) -> dict:
    """Draft-logit verify end to end through the public API: pinned host target
    and draft logits, tokens and uniforms copied to the device,
    spec_verify_run_draft_logits, outputs copied back, all inside the timed
    region."""
    import torch
    B, K = inp.B, inp.K

    def host(a):
        return torch.from_numpy(a.view(np.int16) if inp.dtype == "bf16" else a).pin_memory()
    h = {"logits": host(inp.logits), "dlogits": host(inp.dlogits),
         "tokens": torch.from_numpy(inp.tokens).pin_memory(),
         "uniforms": torch.from_numpy(inp.uniforms).pin_memory()}
    d = {k: torch.empty(t.shape, dtype=t.dtype, device="cuda") for k, t in h.items()}
    h_out = {k: torch.empty(shape, dtype=dt).pin_memory() for k, shape, dt in
             (("accept_len", (B,), torch.int32), ("out_tokens", (B, K + 1), torch.int32),
              ("accept_mask", (B, K), torch.uint8))}

    def once():
        for k in h:
            d[k].copy_(h[k], non_blocking=True)
        lg, dl = ((d["logits"].view(torch.bfloat16), d["dlogits"].view(torch.bfloat16))
                  if inp.dtype == "bf16" else (d["logits"], d["dlogits"]))
        out = verifier.run_draft_logits(lg, dl, d["tokens"], d["uniforms"], inp.T, inp.T_draft,
                                        status=False)
        for k, t in h_out.items():
            t.copy_(out[k], non_blocking=True)
        torch.cuda.current_stream().synchronize()
    once()
    if dist is not None:
        dist.barrier()
    ts = time.perf_counter()
    for _ in range(args.e2e_steps):
        once()
    el = max_over_ranks(time.perf_counter() - ts, dist)
    assert np.array_equal(h_out["accept_len"].numpy(), acc)
    return {"value": world * rows_per_step * args.e2e_steps / el, "unit": "rows/s",
            "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in h.values())),
            "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in h_out.values())),
            "steps": args.e2e_steps,
            "api": "Verifier.run_draft_logits (spec_verify_run_draft_logits) with pinned host copies"}


def e2e_greedy(args, inp, verifier, acc, dist, world, rows_per_step) -> dict:
    """Greedy verification end to end through the public API: pinned host
    logits and tokens copied to the device, spec_verify_run_greedy, outputs
    copied back, all inside the timed region."""
    import torch
    B, K = inp.B, inp.K
    h_lg = torch.from_numpy(inp.logits.view(np.int16) if inp.dtype == "bf16" else inp.logits)
    h_lg = h_lg.pin_memory()
    h_x = torch.from_numpy(inp.tokens).pin_memory()
    d_lg = torch.empty(h_lg.shape, dtype=h_lg.dtype, device="cuda")
    d_x = torch.empty(h_x.shape, dtype=h_x.dtype, device="cuda")
    h_out = {k: torch.empty(shape, dtype=dt).pin_memory() for k, shape, dt in
             (("accept_len", (B,), torch.int32), ("out_tokens", (B, K + 1), torch.int32),
              ("accept_mask", (B, K), torch.uint8))}

    def once():
        d_lg.copy_(h_lg, non_blocking=True)
        d_x.copy_(h_x, non_blocking=True)
        lg = d_lg.view(torch.bfloat16) if inp.dtype == "bf16" else d_lg
        out = verifier.run_greedy(lg, d_x, status=False)
        for k, t in h_out.items():
            t.copy_(out[k], non_blocking=True)
        torch.cuda.current_stream().synchronize()
    once()
    if dist is not None:
        dist.barrier()
    ts = time.perf_counter()
    for _ in range(args.e2e_steps):
        once()
    el = time.perf_counter() - ts
    el = max_over_ranks(el, dist)
    assert np.array_equal(h_out["accept_len"].numpy(), acc)
    return {"value": world * rows_per_step * args.e2e_steps / el, "unit": "rows/s",
            "h2d_bytes_per_step": int(inp.logits.nbytes + inp.tokens.nbytes),
            "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in h_out.values())),
            "steps": args.e2e_steps,
            "api": "Verifier.run_greedy (spec_verify_run_greedy) with pinned host copies"}


# -------------------------------------------------------- reference arm -----

def run_reference(args):
    """The oracle (fp64 CPU) timed as the reference arm on a bounded sample of
    the same workload per step: the OpenMP build of oracle.c on every core
    this process may use (the plain build on one thread if OpenMP is
    unavailable)."""
    world, rank, local = dist_env()
    if rank != 0:
        return None
    import oracle
    oracle.build()
    cores = host_cores()
    try:
        lib = oracle.load_openmp(cores["affinity"])
        nth = lib.oracle_threads()
        build = f"oracle.c with -fopenmp, sequences over {nth} threads"
    except Exception as e:
        lib, nth, build = None, 1, f"oracle.c, plain (OpenMP unavailable: {e})"
    inp = workloads.make_config(args.workload)

    def one(n):
        oracle.verify(inp.logits[:n], inp.dtype, inp.q[:n], inp.tokens[:n], inp.uniforms[:n],
                      inp.T, lib=lib)
    m = min(inp.B, nth)
    t = time.perf_counter()
    one(m)
    rate = m / max(time.perf_counter() - t, 1e-6)
    budget = 120.0 / max(1, args.steps + args.warmup)   # whole run within ~2 minutes
    n = int(min(inp.B, max(m, rate * budget)))
    for _ in range(args.warmup):
        one(n)
    t = time.perf_counter()
    for _ in range(args.steps):
        one(n)
    el = time.perf_counter() - t
    value = args.steps * n * (inp.K + 1) / el
    sample = f"first {n} of {inp.B} sequences per step"
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": args.workload, "B": inp.B, "K": inp.K,
                                            "V": inp.V, "logits_dtype": inp.dtype, "T": inp.T},
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": nth, "kind": "oracle",
                             "sample": sample, "build": build, "host": cores},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main():
    args = parse_args()
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
