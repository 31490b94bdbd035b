"""TEST INFRASTRUCTURE ONLY: the CPU oracle of the SFI decode-attention path.

Loads ``liboracle.so`` (compiled from ``sfi_oracle.c`` with gcc on first use, or by the
package's build step) and exposes its functions on numpy arrays. Only the tests, the
smoke check and the benchmark's CPU-baseline leg may import this package.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sfi_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-pthread"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, no contraction, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def load(path: str | None = None):
    lib = C.CDLL(path or build())
    P = C.c_void_p
    i32, f64 = C.c_int, C.c_double
    lib.sfi_oracle_attend.argtypes = [i32, i32, P, P, P, P, i32, P, P]
    lib.sfi_oracle_attend_split.argtypes = [i32, i32, P, P, P, i32, i32, P]
    lib.sfi_oracle_evidence.argtypes = [i32, i32, P, P]
    lib.sfi_oracle_evidence.restype = None
    lib.sfi_oracle_num_candidates.argtypes = [i32, i32, i32]
    lib.sfi_oracle_prior_norm.argtypes = [i32, i32]
    lib.sfi_oracle_prior_norm.restype = f64
    lib.sfi_oracle_fused_scores.argtypes = [i32, i32, i32, i32, f64, P, P]
    lib.sfi_oracle_topk.argtypes = [i32, P, i32, P]
    lib.sfi_oracle_select.argtypes = [i32, i32, i32, i32, i32, f64, P, P]
    lib.sfi_oracle_sparse_rows.argtypes = [i32, i32, i32, i32, P, i32, P]
    lib.sfi_oracle_schedule.argtypes = [i32, P, i32, P]
    lib.sfi_oracle_schedule.restype = None
    lib.sfi_oracle_schedule_tokens.argtypes = [i32, P, P, i32, i32, P]
    lib.sfi_oracle_schedule_tokens.restype = None
    lib.sfi_oracle_log2f.argtypes = [C.c_float]
    lib.sfi_oracle_log2f.restype = C.c_float
    lib.sfi_oracle_refine_scores.argtypes = [i32, i32, i32, i32, i32, f64, i32, C.c_float, P, i32,
                                             C.c_float, C.c_float, C.c_float, P, P]
    lib.sfi_oracle_key_norms.argtypes = [i32, i32, P, P]
    lib.sfi_oracle_key_norms.restype = None
    lib.sfi_oracle_attend_batch.argtypes = [i32, i32, i32, i32, P, P, P, P, i32, P, P, P, i32]
    return lib


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = load()
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def attend(q, k, v, rows=None, want_p: bool = False):
    """Attention of q [G][D] over rows of k, v [n][D] (bf16 bits). Returns (o, p)."""
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    G, D = q.shape
    if rows is None:
        n = k.shape[0]
        rp = None
    else:
        rows = _c(rows, np.int32)
        n = rows.shape[0]
        rp = _p(rows)
    o = np.zeros((G, D), dtype=np.float64)
    p = np.zeros((G, n), dtype=np.float64) if want_p else None
    rc = lib().sfi_oracle_attend(G, D, _p(q), _p(k), _p(v), rp, n, _p(o),
                                 _p(p) if want_p else None)
    if rc != 0:
        raise ValueError("oracle attend failed")
    return o, p


def attend_split(q, k, v, split: int):
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    G, D = q.shape
    o = np.zeros((G, D), dtype=np.float64)
    if lib().sfi_oracle_attend_split(G, D, _p(q), _p(k), _p(v), k.shape[0], split, _p(o)):
        raise ValueError("oracle attend_split failed")
    return o


def evidence(p):
    p = _c(p, np.float64)
    G, L = p.shape
    f = np.zeros(L, dtype=np.float64)
    lib().sfi_oracle_evidence(G, L, _p(p), _p(f))
    return f


def num_candidates(L, S, W):
    return lib().sfi_oracle_num_candidates(L, S, W)


def prior_norm(n_cand, tau):
    return lib().sfi_oracle_prior_norm(n_cand, tau)


def fused_scores(L, S, W, tau, lam, f32):
    f32 = _c(f32, np.float32)
    n = max(0, L - W - S)
    s = np.zeros(max(n, 1), dtype=np.float32)
    n = lib().sfi_oracle_fused_scores(L, S, W, tau, lam, _p(f32), _p(s))
    return s[:n]


def topk(s, K):
    s = _c(s, np.float32)
    out = np.zeros(max(1, min(K, s.shape[0])), dtype=np.int32)
    n = lib().sfi_oracle_topk(s.shape[0], _p(s), K, _p(out))
    return out[:n]


def select(L, S, W, K, tau, lam, f32):
    f32 = _c(f32, np.float32)
    out = np.zeros(max(1, K), dtype=np.int32)
    n = lib().sfi_oracle_select(L, S, W, K, tau, lam, _p(f32), _p(out))
    if n < 0:
        raise ValueError("oracle select failed")
    return out[:n]


def sparse_rows(L_slow, L_now, S, W, sel):
    sel = _c(sel, np.int32)
    rows = np.zeros(S + len(sel) + W + 1, dtype=np.int32)
    n = lib().sfi_oracle_sparse_rows(L_slow, L_now, S, W, _p(sel), len(sel), _p(rows))
    return rows[:n]


def schedule(mask, t_max):
    mask = _c(mask, np.uint8)
    slow = np.zeros(mask.shape[0], dtype=np.uint8)
    lib().sfi_oracle_schedule(mask.shape[0], _p(mask), t_max, _p(slow))
    return slow


def schedule_tokens(tokens, trigger_ids, t_max):
    tokens = _c(tokens, np.int32)
    trig = _c(trigger_ids, np.int32)
    slow = np.zeros(tokens.shape[0], dtype=np.uint8)
    lib().sfi_oracle_schedule_tokens(tokens.shape[0], _p(tokens), _p(trig), trig.shape[0], t_max,
                                     _p(slow))
    return slow


def log2f(x: float) -> float:
    return lib().sfi_oracle_log2f(x)


def refine_scores(L, S, W, tau, lam, f32, geometric=False, nu=0.0, knorm=None, radius=0,
                  gamma=1.0, mu=0.0, delta=0.0):
    """Refined Selector scores of the H heads of one (layer, sequence): f32 [H][L] evidence,
    knorm [H][L] key norms (or None); Soft-NMS over `radius` neighbours with factor `gamma`
    and similarity limit `delta` (0: none). Returns fp32 [H][n_C]."""
    f32 = _c(f32, np.float32)
    H = f32.shape[0]
    n = max(0, L - W - S)
    out = np.zeros((H, max(n, 1)), dtype=np.float32)
    kn = None if knorm is None else _c(knorm, np.float32)
    n = lib().sfi_oracle_refine_scores(H, L, S, W, tau, lam, 1 if geometric else 0, nu,
                                       None if kn is None else _p(kn), radius, gamma, delta, mu,
                                       _p(f32), _p(out))
    if n < 0:
        raise ValueError("oracle refine failed")
    return out[:, :n]


def key_norms(k):
    k = _c(k, np.uint16)
    out = np.zeros(k.shape[0], dtype=np.float32)
    lib().sfi_oracle_key_norms(k.shape[0], k.shape[1], _p(k), _p(out))
    return out


def attend_batch(q, k, v, n_rows, rows=None, want_f: bool = False, threads: int = 0):
    """q [U][G][D], k/v [U][lmax][D] (bf16 bits), n_rows [U]; rows [U][rmax] or None.
    Returns (o [U][G][D] double, f [U][lmax] double or None)."""
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    n_rows = _c(n_rows, np.int32)
    U, G, D = q.shape
    lmax = k.shape[1]
    o = np.zeros((U, G, D), dtype=np.float64)
    f = np.zeros((U, lmax), dtype=np.float64) if want_f else None
    if rows is not None:
        rows = _c(rows, np.int32)
        rp, rmax = _p(rows), rows.shape[1]
    else:
        rp, rmax = None, 0
    threads = threads or os.cpu_count() or 1
    rc = lib().sfi_oracle_attend_batch(U, G, D, lmax, _p(q), _p(k), _p(v), rp, rmax,
                                       _p(n_rows), _p(o), _p(f) if want_f else None, threads)
    if rc != 0:
        raise ValueError("oracle attend_batch failed")
    return o, f
