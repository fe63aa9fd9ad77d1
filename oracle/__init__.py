"""fp64 CPU oracle for batched speculative-decoding verification.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg (and its reference arm) may import this package.
The product library never imports, links or executes it, and the two share no
code: this side is plain C in ``oracle.c`` compiled with gcc.

Citations ([P1]-[P3], page title and section) are listed in ``oracle.h``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_LIB_OMP = os.path.join(_HERE, "liboracle_omp.so")

OK, TOKEN_RANGE, NONFINITE, UNIFORM_RANGE, BAD_OFFSETS = 0, 4, 5, 7, 8

_lib: Optional[ctypes.CDLL] = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB, openmp: bool = False) -> str:
    """Compile an oracle source into a shared library (skipped when up to date).
    ``openmp``: the same source with -fopenmp, so that a batch's sequences are
    verified on several host threads."""
    newest = max(os.path.getmtime(src), os.path.getmtime(_HDR))
    if force or not os.path.exists(out) or os.path.getmtime(out) < newest:
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-std=gnu99", "-Wall"] +
                              (["-fopenmp"] if openmp else []) +
                              ["-I", _HERE, "-shared", "-fPIC", "-o", tmp, src, "-lm"])
        os.replace(tmp, out)
    return out


def load_openmp(threads: Optional[int] = None) -> ctypes.CDLL:
    """The OpenMP build of oracle.c, bound like the plain one, set to
    ``threads`` host threads (default: the cores this process may run on)."""
    lib = _bind(build(src=_SRC, out=_LIB_OMP, openmp=True))
    lib.oracle_threads.restype = ctypes.c_int
    lib.oracle_threads.argtypes = []
    lib.oracle_set_threads.restype = ctypes.c_int
    lib.oracle_set_threads.argtypes = [ctypes.c_int]
    lib.oracle_set_threads(int(threads or len(os.sched_getaffinity(0))))
    return lib


def _bind(path: str) -> ctypes.CDLL:
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    lib.oracle_verify.restype = ctypes.c_int
    lib.oracle_verify.argtypes = [P, ctypes.c_int, P, P, P, ctypes.c_int64, ctypes.c_int,
                                  ctypes.c_int64, ctypes.c_float] + [P] * 10
    lib.oracle_verify_truncated.restype = ctypes.c_int
    lib.oracle_verify_truncated.argtypes = [P, ctypes.c_int, P, P, P, ctypes.c_int64, ctypes.c_int,
                                            ctypes.c_int64, ctypes.c_float, ctypes.c_double,
                                            ctypes.c_double] + [P] * 11
    lib.oracle_verify_draft_logits.restype = ctypes.c_int
    lib.oracle_verify_draft_logits.argtypes = [P, ctypes.c_int, P, P, P, ctypes.c_int64,
                                               ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                               ctypes.c_float, ctypes.c_double, ctypes.c_double] + [P] * 11
    lib.oracle_verify_ragged.restype = ctypes.c_int
    lib.oracle_verify_ragged.argtypes = [P, ctypes.c_int, P, P, P, P, ctypes.c_int64, ctypes.c_int,
                                         ctypes.c_int64, ctypes.c_int64, ctypes.c_float] + [P] * 10
    lib.oracle_verify_greedy.restype = ctypes.c_int
    lib.oracle_verify_greedy.argtypes = [P, ctypes.c_int, P, ctypes.c_int64, ctypes.c_int,
                                         ctypes.c_int64, P, P, P, P, P]
    lib.oracle_accept_hist.restype = ctypes.c_int
    lib.oracle_accept_hist.argtypes = [P, ctypes.c_int64, ctypes.c_int, P]
    lib.oracle_adapt.restype = ctypes.c_int
    lib.oracle_adapt.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                 ctypes.c_uint64, P, P, P, P]
    lib.oracle_softmax_row.restype = ctypes.c_int
    lib.oracle_softmax_row.argtypes = [P, ctypes.c_int, ctypes.c_int64, ctypes.c_double,
                                       P, P, P]
    return lib


def _load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = _bind(build())
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(dtype: str) -> int:
    if dtype not in ("f32", "bf16"):
        raise ValueError(f"unknown logits dtype {dtype!r}")
    return 0 if dtype == "f32" else 1


def softmax_row(row: np.ndarray, dtype: str, T: float):
    """(status, p, m, s) for one stored logits row."""
    lib = _load()
    row = np.ascontiguousarray(row, dtype=np.float32 if dtype == "f32" else np.uint16)
    V = row.shape[-1]
    p = np.empty(V, dtype=np.float64)
    m = ctypes.c_double()
    s = ctypes.c_double()
    st = lib.oracle_softmax_row(_ptr(row), _dtype_code(dtype), V, float(T), _ptr(p),
                                ctypes.byref(m), ctypes.byref(s))
    return st, p, m.value, s.value


def verify(logits: np.ndarray, dtype: str, q: np.ndarray, tokens: np.ndarray,
           uniforms: np.ndarray, T: float, lib: Optional[ctypes.CDLL] = None) -> dict:
    """Run the oracle over a batch.  Shapes: logits [B, K+1, V] (float32, or uint16
    bf16 bits), q [B, K, V] float32, tokens [B, K] int32, uniforms [B, K+1] float32.

    Returns a dict of numpy arrays: accept_len, out_tokens, accept_mask, status,
    row_m, row_s, p_draft, accept_margin, sample_margin, sample_alt.
    ``lib`` selects another build of the oracle (used to show that the pins
    catch planted mistakes); by default the oracle next to this file."""
    lib = lib or _load()
    logits = np.ascontiguousarray(logits, dtype=np.float32 if dtype == "f32" else np.uint16)
    B, K1, V = logits.shape
    K = K1 - 1
    q = np.ascontiguousarray(q, dtype=np.float32).reshape(B, K, V)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, K)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, K + 1)
    out = {
        "accept_len": np.empty(B, np.int32),
        "out_tokens": np.empty((B, K + 1), np.int32),
        "accept_mask": np.empty((B, K), np.uint8),
        "status": np.empty(B, np.int32),
        "row_m": np.empty((B, K + 1), np.float64),
        "row_s": np.empty((B, K + 1), np.float64),
        "p_draft": np.empty((B, K), np.float64),
        "accept_margin": np.empty(B, np.float64),
        "sample_margin": np.empty(B, np.float64),
        "sample_alt": np.empty(B, np.int32),
    }
    rc = lib.oracle_verify(_ptr(logits), _dtype_code(dtype), _ptr(q), _ptr(tokens),
                           _ptr(uniforms), B, K, V, float(T), _ptr(out["accept_len"]),
                           _ptr(out["out_tokens"]), _ptr(out["accept_mask"]),
                           _ptr(out["status"]), _ptr(out["row_m"]), _ptr(out["row_s"]),
                           _ptr(out["p_draft"]), _ptr(out["accept_margin"]),
                           _ptr(out["sample_margin"]), _ptr(out["sample_alt"]))
    if rc != 0:
        raise ValueError(f"oracle_verify rejected its arguments (rc={rc})")
    return out


def verify_ragged(logits: np.ndarray, dtype: str, q: np.ndarray, tokens: np.ndarray,
                  uniforms: np.ndarray, offsets: np.ndarray, K_max: int, T: float,
                  lib: Optional[ctypes.CDLL] = None) -> dict:
    """Ragged batch.  logits [R, V] packed target rows (sequence b owns rows
    offsets[b]..offsets[b+1]-1), q [R-B, V], tokens [R-B], uniforms [R],
    offsets [B+1] int32.  Returns packed accept_len [B], out_tokens [R],
    accept_mask [R-B], status [B], row_m/row_s [R], p_draft [R-B] and the
    margins [B]."""
    lib = lib or _load()
    logits = np.ascontiguousarray(logits, dtype=np.float32 if dtype == "f32" else np.uint16)
    R, V = logits.shape
    offsets = np.ascontiguousarray(offsets, dtype=np.int32)
    B = offsets.size - 1
    nd = max(R - B, 0)
    q = np.ascontiguousarray(q, dtype=np.float32).reshape(nd, V)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(nd)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(R)
    out = {
        "accept_len": np.empty(B, np.int32), "out_tokens": np.full(R, -1, np.int32),
        "accept_mask": np.zeros(max(nd, 1), np.uint8)[:nd], "status": np.empty(B, np.int32),
        "row_m": np.full(R, np.nan), "row_s": np.full(R, np.nan), "p_draft": np.full(nd, np.nan),
        "accept_margin": np.empty(B), "sample_margin": np.empty(B),
        "sample_alt": np.empty(B, np.int32),
    }
    rc = lib.oracle_verify_ragged(_ptr(logits), _dtype_code(dtype), _ptr(q), _ptr(tokens),
                                  _ptr(uniforms), _ptr(offsets), B, K_max, R, V, float(T),
                                  _ptr(out["accept_len"]), _ptr(out["out_tokens"]),
                                  _ptr(out["accept_mask"]), _ptr(out["status"]),
                                  _ptr(out["row_m"]), _ptr(out["row_s"]), _ptr(out["p_draft"]),
                                  _ptr(out["accept_margin"]), _ptr(out["sample_margin"]),
                                  _ptr(out["sample_alt"]))
    if rc != 0:
        raise ValueError(f"oracle_verify_ragged rejected its arguments (rc={rc})")
    return out


def verify_greedy(logits: np.ndarray, dtype: str, tokens: np.ndarray,
                  lib: Optional[ctypes.CDLL] = None) -> dict:
    """Greedy (T -> 0) verification.  logits [B, K+1, V] (float32, or uint16
    bf16 bits), tokens [B, K] int32.  Returns accept_len, out_tokens,
    accept_mask, status, row_argmax."""
    lib = lib or _load()
    logits = np.ascontiguousarray(logits, dtype=np.float32 if dtype == "f32" else np.uint16)
    B, K1, V = logits.shape
    K = K1 - 1
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, K)
    out = {
        "accept_len": np.empty(B, np.int32),
        "out_tokens": np.empty((B, K + 1), np.int32),
        "accept_mask": np.empty((B, K), np.uint8),
        "status": np.empty(B, np.int32),
        "row_argmax": np.empty((B, K + 1), np.int32),
    }
    rc = lib.oracle_verify_greedy(_ptr(logits), _dtype_code(dtype), _ptr(tokens), B, K, V,
                                  _ptr(out["accept_len"]), _ptr(out["out_tokens"]),
                                  _ptr(out["accept_mask"]), _ptr(out["status"]),
                                  _ptr(out["row_argmax"]))
    if rc != 0:
        raise ValueError(f"oracle_verify_greedy rejected its arguments (rc={rc})")
    return out


def accept_hist(accept_len: np.ndarray, K: int) -> np.ndarray:
    """Counts of accepted lengths 0..K+1 (uint64)."""
    lib = _load()
    al = np.ascontiguousarray(accept_len, dtype=np.int32)
    hist = np.zeros(K + 2, np.uint64)
    if lib.oracle_accept_hist(_ptr(al), al.size, K, _ptr(hist)) != 0:
        raise ValueError("accepted length outside [0, K+1]")
    return hist


def adapt(hist, K: int, K_max: int, K_floor: int = 1, threshold: float = 0.35,
          min_tested: int = 0) -> dict:
    """Acceptance rate, mean accepted length, per-position acceptance and the
    next draft depth of a histogram taken at depth K."""
    lib = _load()
    h = np.zeros(max(K + 2, len(hist)), np.uint64)
    h[:len(hist)] = np.asarray(hist, dtype=np.uint64)
    acc, mlen = ctypes.c_double(), ctypes.c_double()
    pos = np.full(max(K, 1), np.nan)
    nk = ctypes.c_int()
    if lib.oracle_adapt(_ptr(h), K, K_max, K_floor, float(threshold), int(min_tested),
                        ctypes.byref(acc), ctypes.byref(mlen), _ptr(pos), ctypes.byref(nk)) != 0:
        raise ValueError("oracle_adapt rejected its arguments")
    return {"acceptance": acc.value, "mean_accept_len": mlen.value, "pos_acceptance": pos[:K],
            "next_K": nk.value}


def verify_truncated(logits: np.ndarray, dtype: str, q: np.ndarray, tokens: np.ndarray,
                     uniforms: np.ndarray, T: float, top_p: float, min_p: float,
                     lib: Optional[ctypes.CDLL] = None) -> dict:
    """verify() against the truncated target (top-p, min-p; see oracle.h).
    Adds trunc_margin [B]: the distance of the rows reached from a filter
    boundary."""
    lib = lib or _load()
    logits = np.ascontiguousarray(logits, dtype=np.float32 if dtype == "f32" else np.uint16)
    B, K1, V = logits.shape
    K = K1 - 1
    q = np.ascontiguousarray(q, dtype=np.float32).reshape(B, K, V)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, K)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, K + 1)
    out = {
        "accept_len": np.empty(B, np.int32), "out_tokens": np.empty((B, K + 1), np.int32),
        "accept_mask": np.empty((B, K), np.uint8), "status": np.empty(B, np.int32),
        "row_m": np.empty((B, K + 1)), "row_s": np.empty((B, K + 1)), "p_draft": np.empty((B, K)),
        "accept_margin": np.empty(B), "sample_margin": np.empty(B),
        "sample_alt": np.empty(B, np.int32), "trunc_margin": np.empty(B),
    }
    rc = lib.oracle_verify_truncated(_ptr(logits), _dtype_code(dtype), _ptr(q), _ptr(tokens),
                                     _ptr(uniforms), B, K, V, float(T), float(top_p), float(min_p),
                                     _ptr(out["accept_len"]), _ptr(out["out_tokens"]),
                                     _ptr(out["accept_mask"]), _ptr(out["status"]),
                                     _ptr(out["row_m"]), _ptr(out["row_s"]), _ptr(out["p_draft"]),
                                     _ptr(out["accept_margin"]), _ptr(out["sample_margin"]),
                                     _ptr(out["sample_alt"]), _ptr(out["trunc_margin"]))
    if rc != 0:
        raise ValueError(f"oracle_verify_truncated rejected its arguments (rc={rc})")
    return out


def verify_draft_logits(logits: np.ndarray, dtype: str, dlogits: np.ndarray, tokens: np.ndarray,
                        uniforms: np.ndarray, T: float, T_draft: float, top_p: float = 1.0,
                        min_p: float = 0.0, lib: Optional[ctypes.CDLL] = None) -> dict:
    """verify_truncated() with draft logits dlogits [B, K, V] (same dtype as the
    target) instead of q: q_i = softmax(d_i / T_draft) in float64."""
    lib = lib or _load()
    st = np.float32 if dtype == "f32" else np.uint16
    logits = np.ascontiguousarray(logits, dtype=st)
    B, K1, V = logits.shape
    K = K1 - 1
    dlogits = np.ascontiguousarray(dlogits, dtype=st).reshape(B, K, V)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, K)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, K + 1)
    out = {
        "accept_len": np.empty(B, np.int32), "out_tokens": np.empty((B, K + 1), np.int32),
        "accept_mask": np.empty((B, K), np.uint8), "status": np.empty(B, np.int32),
        "row_m": np.empty((B, K + 1)), "row_s": np.empty((B, K + 1)), "p_draft": np.empty((B, K)),
        "accept_margin": np.empty(B), "sample_margin": np.empty(B),
        "sample_alt": np.empty(B, np.int32), "trunc_margin": np.empty(B),
    }
    rc = lib.oracle_verify_draft_logits(_ptr(logits), _dtype_code(dtype), _ptr(dlogits),
                                        _ptr(tokens), _ptr(uniforms), B, K, V, float(T),
                                        float(T_draft), float(top_p), float(min_p),
                                        _ptr(out["accept_len"]), _ptr(out["out_tokens"]),
                                        _ptr(out["accept_mask"]), _ptr(out["status"]),
                                        _ptr(out["row_m"]), _ptr(out["row_s"]),
                                        _ptr(out["p_draft"]), _ptr(out["accept_margin"]),
                                        _ptr(out["sample_margin"]), _ptr(out["sample_alt"]),
                                        _ptr(out["trunc_margin"]))
    if rc != 0:
        raise ValueError(f"oracle_verify_draft_logits rejected its arguments (rc={rc})")
    return out


def verify_inputs(inp, lib: Optional[ctypes.CDLL] = None) -> dict:
    """verify() on a workloads.Inputs bundle."""
    return verify(inp.logits, inp.dtype, inp.q, inp.tokens, inp.uniforms, inp.T, lib=lib)


def load_variant(src_path: str, out_path: str) -> ctypes.CDLL:
    """Build and bind another oracle source (a copy with a planted mistake)."""
    return _bind(build(force=True, src=src_path, out=out_path))
