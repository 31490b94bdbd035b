"""SFI (Slow-Fast Inference) decode attention for GB300 (sm_103a).

Thin ctypes binding of ``libsfi.so`` (C ABI in include/sfi.h). Every function here only
marshals arguments; all computation runs in the library's CUDA kernels. The library must
have been built (``python -c "import __graft_entry__ as g; g.build()"``): there is no CPU
fallback, and calling any entry point without it raises ``RuntimeError``.
"""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsfi.so")

SFI_OK = 0
SFI_ERR_INVALID_ARG = 1
SFI_ERR_UNSUPPORTED = 2
SFI_ERR_CAPACITY = 3
SFI_ERR_WORKSPACE = 4
SFI_ERR_CUDA = 5
SFI_ERR_DEVICE = 6

SFI_DEVERR_PAGE_RANGE = 0x1
SFI_DEVERR_CAPACITY = 0x2
SFI_DEVERR_TIMEOUT = 0x4
SFI_DEVERR_LENGTH = 0x8

ENTRY_POINTS = (
    "sfi_status_string", "sfi_version", "sfi_workspace_bytes", "sfi_workspace_init",
    "sfi_append_kv", "sfi_dense_decode_attn", "sfi_select", "sfi_compact", "sfi_key_norms",
    "sfi_refine_scores",
    "sfi_sparse_decode_attn", "sfi_fast_decode_step", "sfi_sparse_decode_attn_static",
    "sfi_schedule",
    "sfi_schedule_tokens", "sfi_decode_run", "sfi_read_error", "sfi_clear_error",
    "sfi_test_inject_stall",
)


class SfiKvCache(C.Structure):
    _fields_ = [
        ("n_layers", C.c_int32), ("batch", C.c_int32), ("n_q_heads", C.c_int32),
        ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("capacity", C.c_int32),
        ("page_size", C.c_int32), ("n_pages", C.c_int32), ("max_pages_per_seq", C.c_int32),
        ("max_len", C.c_int32), ("k", C.c_void_p), ("v", C.c_void_p),
        ("page_table", C.c_void_p), ("seq_len", C.c_void_p), ("err", C.c_void_p),
    ]


class SfiBudget(C.Structure):
    _fields_ = [("n_sink", C.c_int32), ("n_window", C.c_int32), ("n_select", C.c_int32),
                ("prior_tau", C.c_int32), ("lambda_", C.c_double), ("nms_radius", C.c_int32),
                ("nms_gamma", C.c_float), ("excl_mu", C.c_float), ("norm_nu", C.c_float),
                ("geometric", C.c_int32), ("nms_delta", C.c_float)]


class SfiSparseMem(C.Structure):
    _fields_ = [("kc", C.c_void_p), ("vc", C.c_void_p), ("sel_idx", C.c_void_p),
                ("sel_cnt", C.c_void_p), ("rows", C.c_void_p)]


class SfiDecodePlan(C.Structure):
    _fields_ = [("n_steps", C.c_int32), ("slow", C.c_void_p), ("q", C.c_void_p),
                ("k_new", C.c_void_p), ("v_new", C.c_void_p), ("out", C.c_void_p),
                ("out_fp32", C.c_int32), ("out_per_step", C.c_int32), ("scores_f", C.c_void_p),
                ("masks", C.c_void_p), ("len_start", C.c_int32), ("dense_only", C.c_int32),
                ("events", C.c_void_p), ("side_stream", C.c_void_p), ("fork_event", C.c_void_p),
                ("join_event", C.c_void_p), ("pipeline_group", C.c_int32),
                ("concurrent_fast", C.c_int32)]


class SfiError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


_lib = None


def lib():
    """The loaded library; raises RuntimeError when it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        l = C.CDLL(LIB_PATH)
        P, I32, SZ = C.c_void_p, C.c_int32, C.c_size_t
        KV, BD, MEM = C.POINTER(SfiKvCache), C.POINTER(SfiBudget), C.POINTER(SfiSparseMem)
        sig = {
            "sfi_status_string": (C.c_char_p, [C.c_int]),
            "sfi_version": (C.c_char_p, []),
            "sfi_workspace_bytes": (SZ, [KV, BD]),
            "sfi_workspace_init": (C.c_int, [P, SZ, P]),
            "sfi_append_kv": (C.c_int, [KV, P, P, P, P]),
            "sfi_dense_decode_attn": (C.c_int, [KV, P, P, I32, P, P, P, SZ, P]),
            "sfi_select": (C.c_int, [KV, P, BD, MEM, P, P]),
            "sfi_compact": (C.c_int, [KV, BD, MEM, P, P]),
            "sfi_key_norms": (C.c_int, [KV, P, P, P]),
            "sfi_refine_scores": (C.c_int, [KV, P, P, BD, P, P, P]),
            "sfi_sparse_decode_attn": (C.c_int, [KV, MEM, BD, P, P, I32, P, P, SZ, P]),
            "sfi_fast_decode_step": (C.c_int, [KV, MEM, BD, P, P, P, P, I32, P, P, SZ, P]),
            "sfi_sparse_decode_attn_static": (C.c_int, [KV, MEM, BD, P, P, I32, P, P]),
            "sfi_schedule": (C.c_int, [I32, P, I32, P]),
            "sfi_schedule_tokens": (C.c_int, [I32, P, P, I32, I32, P]),
            "sfi_decode_run": (C.c_int, [KV, BD, MEM, C.POINTER(SfiDecodePlan), P, SZ, P]),
            "sfi_read_error": (C.c_int, [KV, C.POINTER(C.c_uint32), P]),
            "sfi_clear_error": (C.c_int, [KV, P]),
            "sfi_test_inject_stall": (C.c_int, [I32]),
        }
        for name, (res, args) in sig.items():
            f = getattr(l, name)
            f.restype, f.argtypes = res, args
        _lib = l
    return _lib


def _ptr(x):
    """Device/host address of a torch tensor, numpy array, int or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x).__name__}")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(fn: str, status: int):
    if status != SFI_OK:
        raise SfiError(fn, status)


def status_string(status: int) -> str:
    return lib().sfi_status_string(status).decode()


def sfi_version() -> str:
    return lib().sfi_version().decode()


def sfi_workspace_bytes(kv: SfiKvCache, budget: SfiBudget | None = None) -> int:
    n = lib().sfi_workspace_bytes(C.byref(kv), C.byref(budget) if budget is not None else None)
    if n == 0:
        raise SfiError("sfi_workspace_bytes", SFI_ERR_INVALID_ARG)
    return n


def sfi_workspace_init(ws, ws_bytes: int, stream=None):
    _check("sfi_workspace_init", lib().sfi_workspace_init(_ptr(ws), ws_bytes, _stream(stream)))


def sfi_append_kv(kv: SfiKvCache, k_new, v_new, active=None, stream=None):
    _check("sfi_append_kv", lib().sfi_append_kv(C.byref(kv), _ptr(k_new), _ptr(v_new),
                                                _ptr(active), _stream(stream)))


def sfi_dense_decode_attn(kv: SfiKvCache, q, out, out_fp32: bool, scores_f, ws, ws_bytes: int,
                          active=None, stream=None):
    _check("sfi_dense_decode_attn", lib().sfi_dense_decode_attn(
        C.byref(kv), _ptr(q), _ptr(out), 1 if out_fp32 else 0, _ptr(scores_f), _ptr(active),
        _ptr(ws), ws_bytes, _stream(stream)))


def sfi_select(kv: SfiKvCache, scores_f, budget: SfiBudget, mem: SfiSparseMem, active=None,
               stream=None):
    _check("sfi_select", lib().sfi_select(C.byref(kv), _ptr(scores_f), C.byref(budget),
                                          C.byref(mem), _ptr(active), _stream(stream)))


def sfi_key_norms(kv: SfiKvCache, norms, active=None, stream=None):
    _check("sfi_key_norms", lib().sfi_key_norms(C.byref(kv), _ptr(norms), _ptr(active),
                                                _stream(stream)))


def sfi_refine_scores(kv: SfiKvCache, scores_f, key_norms, budget: SfiBudget, refined,
                      active=None, stream=None):
    _check("sfi_refine_scores", lib().sfi_refine_scores(
        C.byref(kv), _ptr(scores_f), _ptr(key_norms), C.byref(budget), _ptr(refined),
        _ptr(active), _stream(stream)))


def sfi_compact(kv: SfiKvCache, budget: SfiBudget, mem: SfiSparseMem, active=None, stream=None):
    _check("sfi_compact", lib().sfi_compact(C.byref(kv), C.byref(budget), C.byref(mem),
                                            _ptr(active), _stream(stream)))


def sfi_sparse_decode_attn(kv: SfiKvCache, mem: SfiSparseMem, budget: SfiBudget, q, out,
                           out_fp32: bool, ws, ws_bytes: int, active=None, stream=None):
    _check("sfi_sparse_decode_attn", lib().sfi_sparse_decode_attn(
        C.byref(kv), C.byref(mem), C.byref(budget), _ptr(q), _ptr(out), 1 if out_fp32 else 0,
        _ptr(active), _ptr(ws), ws_bytes, _stream(stream)))


def sfi_fast_decode_step(kv: SfiKvCache, mem: SfiSparseMem, budget: SfiBudget, k_new, v_new, q,
                         out, out_fp32: bool, ws, ws_bytes: int, active=None, stream=None):
    """Append of k_new/v_new and the fast step's attention in one launch; kv.max_len bounds
    seq_len before the append."""
    _check("sfi_fast_decode_step", lib().sfi_fast_decode_step(
        C.byref(kv), C.byref(mem), C.byref(budget), _ptr(k_new), _ptr(v_new), _ptr(q), _ptr(out),
        1 if out_fp32 else 0, _ptr(active), _ptr(ws), ws_bytes, _stream(stream)))


def sfi_sparse_decode_attn_static(kv: SfiKvCache, mem: SfiSparseMem, budget: SfiBudget, q, out,
                                  out_fp32: bool, active=None, stream=None):
    """The fast step without a workspace: its scratch is a fixed device array inside the
    library (for callers that cannot allocate device memory). Overlapping calls race."""
    _check("sfi_sparse_decode_attn_static", lib().sfi_sparse_decode_attn_static(
        C.byref(kv), C.byref(mem), C.byref(budget), _ptr(q), _ptr(out), 1 if out_fp32 else 0,
        _ptr(active), _stream(stream)))


def sfi_schedule(mask, t_max: int):
    """Trigger policy on a host uint8 mask (numpy); returns the uint8 slow-step flags."""
    import numpy as np
    mask = np.ascontiguousarray(mask, dtype=np.uint8)
    slow = np.zeros(mask.shape[0], dtype=np.uint8)
    _check("sfi_schedule", lib().sfi_schedule(mask.shape[0], mask.ctypes.data, t_max,
                                              slow.ctypes.data))
    return slow


def sfi_schedule_tokens(tokens, trigger_ids, t_max: int):
    """Trigger policy on a host int32 token stream; returns the uint8 slow-step flags."""
    import numpy as np
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    trig = np.ascontiguousarray(trigger_ids, dtype=np.int32)
    slow = np.zeros(tokens.shape[0], dtype=np.uint8)
    _check("sfi_schedule_tokens", lib().sfi_schedule_tokens(
        tokens.shape[0], tokens.ctypes.data, trig.ctypes.data, trig.shape[0], t_max,
        slow.ctypes.data))
    return slow


def sfi_decode_run(kv: SfiKvCache, budget: SfiBudget, mem: SfiSparseMem, plan: SfiDecodePlan,
                   ws, ws_bytes: int, stream=None):
    _check("sfi_decode_run", lib().sfi_decode_run(C.byref(kv), C.byref(budget), C.byref(mem),
                                                  C.byref(plan), _ptr(ws), ws_bytes,
                                                  _stream(stream)))


def sfi_read_error(kv: SfiKvCache, stream=None) -> int:
    bits = C.c_uint32(0)
    st = lib().sfi_read_error(C.byref(kv), C.byref(bits), _stream(stream))
    if st not in (SFI_OK, SFI_ERR_DEVICE):
        raise SfiError("sfi_read_error", st)
    return bits.value


def sfi_clear_error(kv: SfiKvCache, stream=None):
    _check("sfi_clear_error", lib().sfi_clear_error(C.byref(kv), _stream(stream)))


def sfi_test_inject_stall(on: bool = True):
    """Test hook: the next attention launch waits on a barrier that never completes, so its
    bounded waits give up and report SFI_DEVERR_TIMEOUT."""
    _check("sfi_test_inject_stall", lib().sfi_test_inject_stall(1 if on else 0))
