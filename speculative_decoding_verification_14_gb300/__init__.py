"""Python binding of libspecverify (batched speculative-decoding verification
on GB300).  Argument marshalling only: every step of the verify runs in the
library's CUDA kernels.  The functions carry the C-ABI names of
include/spec_verify.h; ``Verifier`` is a convenience wrapper over them that
takes torch CUDA tensors (torch provides device memory and streams only).

There is no fallback: if the library is missing or no GPU is present, calls
raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libspecverify.so")

SV_F32, SV_BF16 = 0, 1
(SV_OK, SV_ERR_INVALID_ARG, SV_ERR_UNSUPPORTED, SV_ERR_CUDA, SV_ERR_TOKEN_RANGE, SV_ERR_NONFINITE,
 SV_ERR_TIMEOUT, SV_ERR_UNIFORM_RANGE, SV_ERR_BAD_OFFSETS) = range(9)


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {spec_verify_strerror(code)} (code {code})" if what else
                         f"{spec_verify_strerror(code)} (code {code})")


class sv_plan(ctypes.Structure):
    _fields_ = [("cluster", ctypes.c_int), ("group", ctypes.c_int), ("threads", ctypes.c_int),
                ("smem_bytes", ctypes.c_int), ("slice", ctypes.c_int64), ("grid", ctypes.c_int64),
                ("bulk_copy", ctypes.c_int), ("prefetch_next", ctypes.c_int), ("stages", ctypes.c_int)]

    def as_dict(self) -> dict:
        return {f: getattr(self, f) for f, _ in self._fields_}


class sv_adapt(ctypes.Structure):
    _fields_ = [("sequences", ctypes.c_uint64), ("errors", ctypes.c_uint64),
                ("tested", ctypes.c_uint64), ("accepted", ctypes.c_uint64),
                ("acceptance", ctypes.c_double), ("mean_accept_len", ctypes.c_double),
                ("pos_tested", ctypes.c_uint64 * 32), ("pos_acceptance", ctypes.c_double * 32),
                ("next_K", ctypes.c_int)]

    def as_dict(self) -> dict:
        d = {f: getattr(self, f) for f, _ in self._fields_}
        d["pos_tested"] = list(self.pos_tested)
        d["pos_acceptance"] = list(self.pos_acceptance)
        return d


_lib: Optional[ctypes.CDLL] = None
P = ctypes.c_void_p


def library() -> ctypes.CDLL:
    """Load libspecverify.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libspecverify.so is not built ({LIB_PATH}); run "
                              "`python -m speculative_decoding_verification_14_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        run_args = [P, P, ctypes.c_int, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                    ctypes.c_float, P, P, P, P, P, P, P]
        sigs = {
            "spec_verify_init": (ctypes.c_int, [ctypes.POINTER(P), ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int64]),
            "spec_verify_run": (ctypes.c_int, run_args),
            "spec_verify_run_host": (ctypes.c_int, run_args),
            "spec_verify_run_noalloc": (ctypes.c_int, [ctypes.c_int] + run_args[1:]),
            "spec_verify_get_error": (ctypes.c_int, [P, P, ctypes.POINTER(ctypes.c_uint32)]),
            "spec_verify_get_plan": (ctypes.c_int, [P, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                                    ctypes.c_int, ctypes.POINTER(sv_plan)]),
            "spec_verify_set_plan_override": (ctypes.c_int, [P, ctypes.c_int, ctypes.c_int,
                                                             ctypes.c_int]),
            "spec_verify_plan_for": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                                    ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_int, ctypes.POINTER(sv_plan)]),
            "spec_verify_run_truncated": (ctypes.c_int, [P, P, ctypes.c_int, P, P, P,
                                                         ctypes.c_int, ctypes.c_int,
                                                         ctypes.c_int64, ctypes.c_float,
                                                         ctypes.c_double, ctypes.c_double, P, P, P,
                                                         P, P, P, P]),
            "spec_verify_get_plan_truncated": (ctypes.c_int, [P, ctypes.c_int, ctypes.c_int,
                                                              ctypes.c_int64, ctypes.c_int,
                                                              ctypes.POINTER(sv_plan)]),
            "spec_verify_plan_truncated_for": (ctypes.c_int, [ctypes.c_int, ctypes.c_int,
                                                              ctypes.c_int, ctypes.c_int,
                                                              ctypes.c_int64, ctypes.c_int,
                                                              ctypes.c_int,
                                                              ctypes.POINTER(sv_plan)]),
            "spec_verify_run_draft_logits": (ctypes.c_int, [P, P, ctypes.c_int, P, P, P,
                                                            ctypes.c_int, ctypes.c_int,
                                                            ctypes.c_int64, ctypes.c_float,
                                                            ctypes.c_float, ctypes.c_double,
                                                            ctypes.c_double, P, P, P, P, P, P,
                                                            P]),
            "spec_verify_get_plan_draft_logits": (ctypes.c_int, [P, ctypes.c_int, ctypes.c_int,
                                                                 ctypes.c_int64, ctypes.c_int,
                                                                 ctypes.c_int,
                                                                 ctypes.POINTER(sv_plan)]),
            "spec_verify_plan_draft_logits_for": (ctypes.c_int, [ctypes.c_int, ctypes.c_int,
                                                                 ctypes.c_int, ctypes.c_int,
                                                                 ctypes.c_int64, ctypes.c_int,
                                                                 ctypes.c_int, ctypes.c_int,
                                                                 ctypes.POINTER(sv_plan)]),
            "spec_verify_run_ragged": (ctypes.c_int, [P, P, ctypes.c_int, P, P, P, P,
                                                      ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                                      ctypes.c_int64, ctypes.c_float, P, P, P, P,
                                                      P, P, P]),
            "spec_verify_run_greedy": (ctypes.c_int, [P, P, ctypes.c_int, P, ctypes.c_int,
                                                      ctypes.c_int, ctypes.c_int64, P, P, P, P,
                                                      P, P]),
            "spec_verify_get_plan_greedy": (ctypes.c_int, [P, ctypes.c_int, ctypes.c_int,
                                                           ctypes.c_int64, ctypes.c_int,
                                                           ctypes.POINTER(sv_plan)]),
            "spec_verify_plan_greedy_for": (ctypes.c_int, [ctypes.c_int, ctypes.c_int,
                                                           ctypes.c_int, ctypes.c_int,
                                                           ctypes.c_int64, ctypes.c_int,
                                                           ctypes.c_int, ctypes.POINTER(sv_plan)]),
            "spec_verify_set_telemetry": (ctypes.c_int, [P, P, ctypes.c_int]),
            "spec_verify_selftest_wait": (ctypes.c_int, [ctypes.c_int, ctypes.c_ulonglong,
                                                         ctypes.c_int,
                                                         ctypes.POINTER(ctypes.c_int),
                                                         ctypes.POINTER(ctypes.c_ulonglong)]),
            "spec_adapt": (ctypes.c_int, [P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_double, ctypes.c_uint64,
                                          ctypes.POINTER(sv_adapt)]),
            "spec_verify_destroy": (ctypes.c_int, [P]),
            "spec_verify_strerror": (ctypes.c_char_p, [ctypes.c_int]),
            "spec_verify_version": (ctypes.c_int, []),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


# ------------------------------------------------- C-ABI names, 1:1 -----

def spec_verify_strerror(code: int) -> str:
    return library().spec_verify_strerror(int(code)).decode()


def spec_verify_version() -> int:
    return library().spec_verify_version()


def spec_verify_init(device: int, max_B: int, max_K: int, max_V: int) -> int:
    ctx = P()
    rc = library().spec_verify_init(ctypes.byref(ctx), device, max_B, max_K, max_V)
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_verify_init")
    return ctx.value


def spec_verify_destroy(ctx: int) -> int:
    return library().spec_verify_destroy(ctx)


def spec_verify_run(ctx, logits_ptr, dtype, q_ptr, tokens_ptr, uniforms_ptr, B, K, V, T,
                    accept_len_ptr, out_tokens_ptr, accept_mask_ptr, row_stats_ptr=None,
                    p_draft_ptr=None, status_ptr=None, stream=None) -> int:
    return library().spec_verify_run(ctx, logits_ptr, dtype, q_ptr, tokens_ptr, uniforms_ptr, B, K,
                                     V, float(T), accept_len_ptr, out_tokens_ptr, accept_mask_ptr,
                                     row_stats_ptr, p_draft_ptr, status_ptr, stream)


def spec_verify_run_host(ctx, logits_ptr, dtype, q_ptr, tokens_ptr, uniforms_ptr, B, K, V, T,
                         accept_len_ptr, out_tokens_ptr, accept_mask_ptr, row_stats_ptr=None,
                         p_draft_ptr=None, status_ptr=None, stream=None) -> int:
    return library().spec_verify_run_host(ctx, logits_ptr, dtype, q_ptr, tokens_ptr, uniforms_ptr,
                                          B, K, V, float(T), accept_len_ptr, out_tokens_ptr,
                                          accept_mask_ptr, row_stats_ptr, p_draft_ptr, status_ptr,
                                          stream)


def spec_verify_run_noalloc(device, logits_ptr, dtype, q_ptr, tokens_ptr, uniforms_ptr, B, K, V, T,
                            accept_len_ptr, out_tokens_ptr, accept_mask_ptr, row_stats_ptr=None,
                            p_draft_ptr=None, status_ptr=None, stream=None) -> int:
    return library().spec_verify_run_noalloc(int(device), logits_ptr, dtype, q_ptr, tokens_ptr,
                                             uniforms_ptr, B, K, V, float(T), accept_len_ptr,
                                             out_tokens_ptr, accept_mask_ptr, row_stats_ptr,
                                             p_draft_ptr, status_ptr, stream)


def spec_verify_run_truncated(ctx, logits_ptr, dtype, q_ptr, tokens_ptr, uniforms_ptr, B, K, V,
                              T, top_p, min_p, accept_len_ptr, out_tokens_ptr, accept_mask_ptr,
                              row_stats_ptr=None, p_draft_ptr=None, status_ptr=None,
                              stream=None) -> int:
    return library().spec_verify_run_truncated(ctx, logits_ptr, dtype, q_ptr, tokens_ptr,
                                               uniforms_ptr, B, K, V, float(T), float(top_p),
                                               float(min_p), accept_len_ptr, out_tokens_ptr,
                                               accept_mask_ptr, row_stats_ptr, p_draft_ptr,
                                               status_ptr, stream)


def spec_verify_get_plan_truncated(ctx, B, K, V, dtype) -> dict:
    plan = sv_plan()
    rc = library().spec_verify_get_plan_truncated(ctx, B, K, V, dtype, ctypes.byref(plan))
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_verify_get_plan_truncated")
    return plan.as_dict()


def spec_verify_plan_truncated_for(num_sms, max_cluster, B, K, V, dtype, ovr_cluster=0):
    plan = sv_plan()
    rc = library().spec_verify_plan_truncated_for(num_sms, max_cluster, B, K, V, dtype,
                                                  ovr_cluster, ctypes.byref(plan))
    return rc, plan.as_dict()


def spec_verify_run_draft_logits(ctx, logits_ptr, dtype, dlogits_ptr, tokens_ptr, uniforms_ptr, B,
                                 K, V, T, T_draft, top_p, min_p, accept_len_ptr, out_tokens_ptr,
                                 accept_mask_ptr, row_stats_ptr=None, p_draft_ptr=None,
                                 status_ptr=None, stream=None) -> int:
    return library().spec_verify_run_draft_logits(ctx, logits_ptr, dtype, dlogits_ptr, tokens_ptr,
                                                  uniforms_ptr, B, K, V, float(T), float(T_draft),
                                                  float(top_p), float(min_p), accept_len_ptr,
                                                  out_tokens_ptr, accept_mask_ptr, row_stats_ptr,
                                                  p_draft_ptr, status_ptr, stream)


def spec_verify_get_plan_draft_logits(ctx, B, K, V, dtype, filters) -> dict:
    plan = sv_plan()
    rc = library().spec_verify_get_plan_draft_logits(ctx, B, K, V, dtype, int(filters),
                                                     ctypes.byref(plan))
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_verify_get_plan_draft_logits")
    return plan.as_dict()


def spec_verify_plan_draft_logits_for(num_sms, max_cluster, B, K, V, dtype, filters,
                                      ovr_cluster=0):
    plan = sv_plan()
    rc = library().spec_verify_plan_draft_logits_for(num_sms, max_cluster, B, K, V, dtype,
                                                     int(filters), ovr_cluster,
                                                     ctypes.byref(plan))
    return rc, plan.as_dict()


def spec_verify_run_ragged(ctx, logits_ptr, dtype, q_ptr, tokens_ptr, uniforms_ptr, offsets_ptr,
                           total_rows, B, K_max, V, T, accept_len_ptr, out_tokens_ptr,
                           accept_mask_ptr, row_stats_ptr=None, p_draft_ptr=None, status_ptr=None,
                           stream=None) -> int:
    return library().spec_verify_run_ragged(ctx, logits_ptr, dtype, q_ptr, tokens_ptr,
                                            uniforms_ptr, offsets_ptr, total_rows, B, K_max, V,
                                            float(T), accept_len_ptr, out_tokens_ptr,
                                            accept_mask_ptr, row_stats_ptr, p_draft_ptr,
                                            status_ptr, stream)


def spec_verify_run_greedy(ctx, logits_ptr, dtype, tokens_ptr, B, K, V, accept_len_ptr,
                           out_tokens_ptr, accept_mask_ptr, row_argmax_ptr=None, status_ptr=None,
                           stream=None) -> int:
    return library().spec_verify_run_greedy(ctx, logits_ptr, dtype, tokens_ptr, B, K, V,
                                            accept_len_ptr, out_tokens_ptr, accept_mask_ptr,
                                            row_argmax_ptr, status_ptr, stream)


def spec_verify_get_plan_greedy(ctx, B, K, V, dtype) -> dict:
    plan = sv_plan()
    rc = library().spec_verify_get_plan_greedy(ctx, B, K, V, dtype, ctypes.byref(plan))
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_verify_get_plan_greedy")
    return plan.as_dict()


def spec_verify_plan_greedy_for(num_sms, max_cluster, B, K, V, dtype, ovr_cluster=0):
    plan = sv_plan()
    rc = library().spec_verify_plan_greedy_for(num_sms, max_cluster, B, K, V, dtype, ovr_cluster,
                                               ctypes.byref(plan))
    return rc, plan.as_dict()


def spec_verify_selftest_wait(device: int, limit_ns: int, arrive: bool):
    """Returns (status, completed, elapsed_ns) of the bounded-wait self-test."""
    done = ctypes.c_int(-1)
    el = ctypes.c_ulonglong(0)
    rc = library().spec_verify_selftest_wait(int(device), int(limit_ns), 1 if arrive else 0,
                                             ctypes.byref(done), ctypes.byref(el))
    return rc, done.value, el.value


def spec_verify_set_telemetry(ctx, hist_ptr, bins) -> int:
    return library().spec_verify_set_telemetry(ctx, hist_ptr, int(bins))


def spec_adapt(hist, K: int, K_max: int, K_floor: int = 1, threshold: float = 0.35,
               min_tested: int = 0) -> dict:
    """`hist`: host sequence of accepted-length counts (bin 0 = errors) taken
    at draft depth K.  Returns the sv_adapt fields as a dict."""
    arr = (ctypes.c_uint32 * len(hist))(*[int(h) for h in hist])
    out = sv_adapt()
    rc = library().spec_adapt(arr, len(hist), K, K_max, K_floor, float(threshold),
                              int(min_tested), ctypes.byref(out))
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_adapt")
    return out.as_dict()


def spec_verify_get_error(ctx, stream=None):
    mask = ctypes.c_uint32(0)
    rc = library().spec_verify_get_error(ctx, stream, ctypes.byref(mask))
    return rc, mask.value


def spec_verify_get_plan(ctx, B, K, V, dtype) -> dict:
    plan = sv_plan()
    rc = library().spec_verify_get_plan(ctx, B, K, V, dtype, ctypes.byref(plan))
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_verify_get_plan")
    return plan.as_dict()


def spec_verify_set_plan_override(ctx, cluster=0, group=0, threads=0) -> int:
    return library().spec_verify_set_plan_override(ctx, cluster, group, threads)


def spec_verify_plan_for(num_sms, smem_per_cta, max_cluster, B, K, V, dtype, ovr_cluster=0,
                         ovr_group=0, ovr_threads=0):
    plan = sv_plan()
    rc = library().spec_verify_plan_for(num_sms, smem_per_cta, max_cluster, B, K, V, dtype,
                                        ovr_cluster, ovr_group, ovr_threads, ctypes.byref(plan))
    return rc, plan.as_dict()


# ------------------------------------------------------ torch wrapper -----

def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return SV_F32
    if t.dtype == torch.bfloat16:
        return SV_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


class Verifier:
    """Owns one library context on one CUDA device.

    ``run`` takes CUDA tensors: logits [B, K+1, V] (float32 or bfloat16), q
    [B, K, V] float32, tokens [B, K] int32, uniforms [B, K+1] float32, and a
    temperature; it returns a dict of CUDA tensors accept_len [B], out_tokens
    [B, K+1], accept_mask [B, K] (uint8), and optionally row_stats [B, K+1, 2],
    p_draft [B, K], status [B].  The launch goes on torch's current stream."""

    def __init__(self, max_B: int, max_K: int, max_V: int, device: Optional[int] = None):
        import torch
        if not torch.cuda.is_available():
            raise RuntimeError("speculative_decoding_verification_14_gb300 needs a CUDA GPU")
        self.device = torch.cuda.current_device() if device is None else int(device)
        self.ctx = spec_verify_init(self.device, max_B, max_K, max_V)

    def close(self):
        if getattr(self, "ctx", None):
            spec_verify_destroy(self.ctx)
            self.ctx = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def plan(self, B, K, V, dtype=SV_BF16) -> dict:
        return spec_verify_get_plan(self.ctx, B, K, V, dtype)

    def set_plan_override(self, cluster=0, group=0, threads=0):
        rc = spec_verify_set_plan_override(self.ctx, cluster, group, threads)
        if rc != SV_OK:
            raise SpecVerifyError(rc, "spec_verify_set_plan_override")

    def error(self, stream=None):
        return spec_verify_get_error(self.ctx, stream)

    def set_telemetry(self, hist) -> None:
        """Count accepted lengths of every later run into `hist`, a uint32
        CUDA tensor of at least K + 2 counters (zeroed by the caller); None
        stops counting.  The tensor must stay alive while it is set."""
        if hist is None:
            rc = spec_verify_set_telemetry(self.ctx, None, 0)
        else:
            import torch
            if hist.dtype != torch.int32 and hist.dtype != getattr(torch, "uint32", None):
                raise TypeError("telemetry counters must be a 32-bit integer tensor")
            if not hist.is_cuda or not hist.is_contiguous():
                raise ValueError("telemetry counters must be a contiguous CUDA tensor")
            rc = spec_verify_set_telemetry(self.ctx, hist.data_ptr(), hist.numel())
        if rc != SV_OK:
            raise SpecVerifyError(rc, "spec_verify_set_telemetry")
        self._telemetry = hist

    def run(self, logits, q, tokens, uniforms, temperature: float, out: Optional[dict] = None,
            stats: bool = False, status: bool = True, stream=None) -> dict:
        import torch
        B, K1, V = logits.shape
        K = K1 - 1
        dev = logits.device
        if out is None:
            out = {
                "accept_len": torch.empty(B, dtype=torch.int32, device=dev),
                "out_tokens": torch.empty(B, K + 1, dtype=torch.int32, device=dev),
                "accept_mask": torch.empty(B, max(K, 1), dtype=torch.uint8, device=dev)[:, :K],
            }
            if stats:
                out["row_stats"] = torch.empty(B, K + 1, 2, dtype=torch.float32, device=dev)
                out["p_draft"] = torch.empty(B, max(K, 1), dtype=torch.float32, device=dev)[:, :K]
            if status:
                out["status"] = torch.empty(B, dtype=torch.int32, device=dev)
        s = stream if stream is not None else torch.cuda.current_stream(dev).cuda_stream

        def ptr(name):
            t = out.get(name)
            return None if t is None else t.data_ptr()

        rc = spec_verify_run(self.ctx, logits.data_ptr(), _dtype_code(logits),
                             q.data_ptr() if K else None, tokens.data_ptr() if K else None,
                             uniforms.data_ptr(), B, K, V, temperature, ptr("accept_len"),
                             ptr("out_tokens"), ptr("accept_mask") if K else None,
                             ptr("row_stats"), ptr("p_draft") if K else None, ptr("status"), s)
        if rc != SV_OK:
            raise SpecVerifyError(rc, "spec_verify_run")
        return out

    def run_greedy(self, logits, tokens, out: Optional[dict] = None, argmax: bool = False,
                   status: bool = True, stream=None) -> dict:
        """Greedy (T -> 0) verification: logits [B, K+1, V] (float32 or bfloat16)
        and tokens [B, K] int32 CUDA tensors.  Returns accept_len, out_tokens,
        accept_mask and optionally row_argmax [B, K+1] and status."""
        import torch
        B, K1, V = logits.shape
        K = K1 - 1
        dev = logits.device
        if out is None:
            out = {
                "accept_len": torch.empty(B, dtype=torch.int32, device=dev),
                "out_tokens": torch.empty(B, K + 1, dtype=torch.int32, device=dev),
                "accept_mask": torch.empty(B, max(K, 1), dtype=torch.uint8, device=dev)[:, :K],
            }
            if argmax:
                out["row_argmax"] = torch.empty(B, K + 1, dtype=torch.int32, device=dev)
            if status:
                out["status"] = torch.empty(B, dtype=torch.int32, device=dev)
        s = stream if stream is not None else torch.cuda.current_stream(dev).cuda_stream

        def ptr(name):
            t = out.get(name)
            return None if t is None else t.data_ptr()

        rc = spec_verify_run_greedy(self.ctx, logits.data_ptr(), _dtype_code(logits),
                                    tokens.data_ptr() if K else None, B, K, V, ptr("accept_len"),
                                    ptr("out_tokens"), ptr("accept_mask") if K else None,
                                    ptr("row_argmax"), ptr("status"), s)
        if rc != SV_OK:
            raise SpecVerifyError(rc, "spec_verify_run_greedy")
        return out

    def run_ragged(self, logits, q, tokens, uniforms, offsets, K_max: int, temperature: float,
                   out: Optional[dict] = None, stats: bool = False, status: bool = True,
                   stream=None) -> dict:
        """Ragged batch: logits [R, V], q [R-B, V], tokens [R-B], uniforms [R],
        offsets [B+1] int32 CUDA tensors (sequence b owns rows offsets[b] ..
        offsets[b+1]-1).  Returns packed accept_len [B], out_tokens [R],
        accept_mask [R-B], optionally row_stats [R, 2], p_draft [R-B], status [B]."""
        import torch
        R, V = logits.shape
        B = offsets.numel() - 1
        nd = R - B
        dev = logits.device
        if out is None:
            out = {"accept_len": torch.empty(B, dtype=torch.int32, device=dev),
                   "out_tokens": torch.empty(R, dtype=torch.int32, device=dev),
                   "accept_mask": torch.empty(max(nd, 1), dtype=torch.uint8, device=dev)[:nd]}
            if stats:
                out["row_stats"] = torch.empty(R, 2, dtype=torch.float32, device=dev)
                out["p_draft"] = torch.empty(max(nd, 1), dtype=torch.float32, device=dev)[:nd]
            if status:
                out["status"] = torch.empty(B, dtype=torch.int32, device=dev)
        s = stream if stream is not None else torch.cuda.current_stream(dev).cuda_stream

        def ptr(name):
            t = out.get(name)
            return None if t is None else t.data_ptr()

        rc = spec_verify_run_ragged(self.ctx, logits.data_ptr(), _dtype_code(logits),
                                    q.data_ptr() if nd else None,
                                    tokens.data_ptr() if nd else None, uniforms.data_ptr(),
                                    offsets.data_ptr(), R, B, K_max, V, temperature,
                                    ptr("accept_len"), ptr("out_tokens"),
                                    ptr("accept_mask") if nd else None, ptr("row_stats"),
                                    ptr("p_draft") if nd else None, ptr("status"), s)
        if rc != SV_OK:
            raise SpecVerifyError(rc, "spec_verify_run_ragged")
        return out

    def run_truncated(self, logits, q, tokens, uniforms, temperature: float, top_p: float,
                      min_p: float, out: Optional[dict] = None, stats: bool = False,
                      status: bool = True, stream=None) -> dict:
        """run() against the truncated target (top-p, min-p)."""
        import torch
        B, K1, V = logits.shape
        K = K1 - 1
        dev = logits.device
        if out is None:
            out = {
                "accept_len": torch.empty(B, dtype=torch.int32, device=dev),
                "out_tokens": torch.empty(B, K + 1, dtype=torch.int32, device=dev),
                "accept_mask": torch.empty(B, max(K, 1), dtype=torch.uint8, device=dev)[:, :K],
            }
            if stats:
                out["row_stats"] = torch.empty(B, K + 1, 2, dtype=torch.float32, device=dev)
                out["p_draft"] = torch.empty(B, max(K, 1), dtype=torch.float32, device=dev)[:, :K]
            if status:
                out["status"] = torch.empty(B, dtype=torch.int32, device=dev)
        s = stream if stream is not None else torch.cuda.current_stream(dev).cuda_stream

        def ptr(name):
            t = out.get(name)
            return None if t is None else t.data_ptr()

        rc = spec_verify_run_truncated(self.ctx, logits.data_ptr(), _dtype_code(logits),
                                       q.data_ptr() if K else None,
                                       tokens.data_ptr() if K else None, uniforms.data_ptr(), B,
                                       K, V, temperature, top_p, min_p, ptr("accept_len"),
                                       ptr("out_tokens"), ptr("accept_mask") if K else None,
                                       ptr("row_stats"), ptr("p_draft") if K else None,
                                       ptr("status"), s)
        if rc != SV_OK:
            raise SpecVerifyError(rc, "spec_verify_run_truncated")
        return out

    def run_draft_logits(self, logits, dlogits, tokens, uniforms, temperature: float,
                         draft_temperature: float, top_p: float = 1.0, min_p: float = 0.0,
                         out: Optional[dict] = None, stats: bool = False, status: bool = True,
                         stream=None) -> dict:
        """run() with the drafter's logits dlogits [B, K, V] (the target's dtype)
        in place of q; top_p < 1 / min_p > 0 truncate the target."""
        import torch
        B, K1, V = logits.shape
        K = K1 - 1
        if K and (dlogits.dtype != logits.dtype or tuple(dlogits.shape) != (B, K, V)):
            raise ValueError("dlogits must be [B, K, V] in the target's dtype")
        dev = logits.device
        if out is None:
            out = {
                "accept_len": torch.empty(B, dtype=torch.int32, device=dev),
                "out_tokens": torch.empty(B, K + 1, dtype=torch.int32, device=dev),
                "accept_mask": torch.empty(B, max(K, 1), dtype=torch.uint8, device=dev)[:, :K],
            }
            if stats:
                out["row_stats"] = torch.empty(B, K + 1, 2, dtype=torch.float32, device=dev)
                out["p_draft"] = torch.empty(B, max(K, 1), dtype=torch.float32, device=dev)[:, :K]
            if status:
                out["status"] = torch.empty(B, dtype=torch.int32, device=dev)
        s = stream if stream is not None else torch.cuda.current_stream(dev).cuda_stream

        def ptr(name):
            t = out.get(name)
            return None if t is None else t.data_ptr()

        rc = spec_verify_run_draft_logits(self.ctx, logits.data_ptr(), _dtype_code(logits),
                                          dlogits.data_ptr() if K else None,
                                          tokens.data_ptr() if K else None, uniforms.data_ptr(),
                                          B, K, V, temperature, draft_temperature, top_p, min_p,
                                          ptr("accept_len"), ptr("out_tokens"),
                                          ptr("accept_mask") if K else None, ptr("row_stats"),
                                          ptr("p_draft") if K else None, ptr("status"), s)
        if rc != SV_OK:
            raise SpecVerifyError(rc, "spec_verify_run_draft_logits")
        return out

    def plan_draft_logits(self, B, K, V, dtype=SV_BF16, filters=0) -> dict:
        return spec_verify_get_plan_draft_logits(self.ctx, B, K, V, dtype, filters)

    def plan_truncated(self, B, K, V, dtype=SV_BF16) -> dict:
        return spec_verify_get_plan_truncated(self.ctx, B, K, V, dtype)

    def plan_greedy(self, B, K, V, dtype=SV_BF16) -> dict:
        return spec_verify_get_plan_greedy(self.ctx, B, K, V, dtype)

    def run_host(self, logits, dtype: int, q, tokens, uniforms, temperature: float,
                 out: dict, stream=None) -> int:
        """Host-buffer entry: numpy (ideally pinned) arrays in, numpy arrays out.
        Returns the status of the call (launch status or lowest device error)."""
        B, K1, V = logits.shape
        K = K1 - 1

        def ptr(a):
            return None if a is None else a.ctypes.data

        return spec_verify_run_host(self.ctx, ptr(logits), dtype, ptr(q) if K else None,
                                    ptr(tokens) if K else None, ptr(uniforms), B, K, V, temperature,
                                    ptr(out["accept_len"]), ptr(out["out_tokens"]),
                                    ptr(out.get("accept_mask")) if K else None,
                                    ptr(out.get("row_stats")), ptr(out.get("p_draft")),
                                    ptr(out.get("status")), stream)
