"""The C-ABI library loads and exports every entry point include/sfi.h declares; its
host-only paths (status strings, argument checks that fail before any CUDA call, the
trigger-policy scheduler) work without a GPU."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import oracle
import sparse_long_context_sfi_gb300 as sfi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return sfi.lib()


def declared():
    src = open(os.path.join(ROOT, "include", "sfi.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sfi_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared()
    assert "sfi_dense_decode_attn" in names and "sfi_select" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in sfi.h but not exported"
    assert sorted(sfi.ENTRY_POINTS) == names


def test_status_strings(lib):
    for s in range(7):
        assert sfi.status_string(s)
    assert "sm_103a" in sfi.sfi_version()


def test_argument_errors_return_before_any_launch(lib):
    kv = sfi.SfiKvCache()  # all zero: null pointers
    st = lib.sfi_append_kv(C.byref(kv), None, None, None, None)
    assert st == sfi.SFI_ERR_INVALID_ARG
    dummy = 1 << 20  # never dereferenced: the checks fail first
    kv = sfi.SfiKvCache(n_layers=1, batch=1, n_q_heads=8, n_kv_heads=2, head_dim=64, capacity=16,
                        max_len=4, k=dummy, v=dummy, seq_len=dummy, err=dummy)
    assert lib.sfi_append_kv(C.byref(kv), dummy, dummy, None, None) == sfi.SFI_ERR_UNSUPPORTED
    kv.head_dim = 128
    kv.n_q_heads = 12  # group 6
    assert lib.sfi_append_kv(C.byref(kv), dummy, dummy, None, None) == sfi.SFI_ERR_UNSUPPORTED
    kv.n_q_heads = 8
    kv.max_len = 16    # no room to append
    assert lib.sfi_append_kv(C.byref(kv), dummy, dummy, None, None) == sfi.SFI_ERR_CAPACITY
    kv.max_len = 4
    kv.k = dummy + 8   # misaligned
    assert lib.sfi_append_kv(C.byref(kv), dummy, dummy, None, None) == sfi.SFI_ERR_INVALID_ARG
    kv.k = dummy
    kv.page_size = 16  # paged without a page table
    assert lib.sfi_append_kv(C.byref(kv), dummy, dummy, None, None) == sfi.SFI_ERR_INVALID_ARG
    kv.page_size = 0
    bad = sfi.SfiBudget(n_sink=4, n_window=64, n_select=16, prior_tau=48, lambda_=0.1)
    mem = sfi.SfiSparseMem(kc=dummy, vc=dummy, sel_idx=dummy, sel_cnt=dummy, rows=dummy)
    assert lib.sfi_select(C.byref(kv), dummy, C.byref(bad), C.byref(mem), None, None) == \
        sfi.SFI_ERR_INVALID_ARG  # tau not a power of two
    bad.prior_tau, bad.lambda_ = 64, 1.5
    assert lib.sfi_compact(C.byref(kv), C.byref(bad), C.byref(mem), None, None) == \
        sfi.SFI_ERR_INVALID_ARG  # lambda outside [0, 1]
    bad.lambda_, bad.nms_radius, bad.nms_gamma = 0.1, 1, 0.5
    for delta in (-1e-3, float("nan")):  # Soft-NMS similarity limit negative or NaN
        bad.nms_delta = delta
        assert lib.sfi_refine_scores(C.byref(kv), dummy, None, C.byref(bad), dummy, None,
                                     None) == sfi.SFI_ERR_INVALID_ARG


def test_static_fast_step_rejects_units_beyond_its_scratch(lib):
    """The allocation-free fast step has scratch for 16384 units; more give SFI_ERR_CAPACITY
    before any device call (the pointers are never dereferenced)."""
    dummy = 1 << 20
    bud = sfi.SfiBudget(n_sink=4, n_window=64, n_select=256, prior_tau=64, lambda_=0.1)
    mem = sfi.SfiSparseMem(kc=dummy, vc=dummy, sel_idx=dummy, sel_cnt=dummy, rows=dummy)
    kv = sfi.SfiKvCache(n_layers=65, batch=32, n_q_heads=32, n_kv_heads=8, head_dim=128,
                        capacity=1024, max_len=4, k=dummy, v=dummy, seq_len=dummy, err=dummy)
    assert lib.sfi_sparse_decode_attn_static(C.byref(kv), C.byref(mem), C.byref(bud), dummy,
                                             dummy, 1, None, None) == sfi.SFI_ERR_CAPACITY


@pytest.mark.parametrize("t_max", [0, 1, 5, 64])
def test_native_scheduler_matches_oracle(lib, t_max):
    rng = np.random.default_rng(t_max)
    for _ in range(20):
        m = (rng.random(rng.integers(1, 200)) < 0.15).astype(np.uint8)
        np.testing.assert_array_equal(sfi.sfi_schedule(m, t_max), oracle.schedule(m, t_max))


def test_decode_plan_layout_matches_header(lib):
    """ctypes structs mirror the C layouts (field offsets of the 64-bit ABI)."""
    assert C.sizeof(sfi.SfiKvCache) == 10 * 4 + 5 * 8
    assert C.sizeof(sfi.SfiBudget) == 4 * 4 + 8 + 6 * 4
    assert sfi.SfiBudget.lambda_.offset == 16 and sfi.SfiBudget.nms_delta.offset == 44
    assert C.sizeof(sfi.SfiSparseMem) == 5 * 8
    assert sfi.SfiDecodePlan.masks.offset == 64 and sfi.SfiDecodePlan.events.offset == 80
    assert sfi.SfiDecodePlan.side_stream.offset == 88 and sfi.SfiDecodePlan.join_event.offset == 104
    assert sfi.SfiDecodePlan.pipeline_group.offset == 112
    assert sfi.SfiDecodePlan.concurrent_fast.offset == 116
    assert C.sizeof(sfi.SfiDecodePlan) == 120


def test_layer_pipeline_needs_both_events(lib):
    """A decode run with a side stream but without its fork and join events is refused
    before any CUDA call."""
    dummy = 1 << 20  # never dereferenced: the checks fail first
    kv = sfi.SfiKvCache(n_layers=2, batch=1, n_q_heads=8, n_kv_heads=2, head_dim=128, capacity=64,
                        max_len=8, k=dummy, v=dummy, seq_len=dummy, err=dummy)
    bud = sfi.SfiBudget(n_sink=4, n_window=16, n_select=8, prior_tau=16, lambda_=0.1)
    mem = sfi.SfiSparseMem(kc=dummy, vc=dummy, sel_idx=dummy, sel_cnt=dummy, rows=dummy)
    slow = np.ones(4, np.uint8)
    plan = sfi.SfiDecodePlan(n_steps=4, slow=slow.ctypes.data, q=dummy, k_new=dummy, v_new=dummy,
                             out=dummy, out_fp32=1, out_per_step=1, scores_f=dummy, len_start=8,
                             side_stream=dummy, fork_event=dummy)
    assert lib.sfi_decode_run(C.byref(kv), C.byref(bud), C.byref(mem), C.byref(plan), dummy,
                              1 << 30, None) == sfi.SFI_ERR_INVALID_ARG
    plan.fork_event, plan.join_event = None, dummy
    assert lib.sfi_decode_run(C.byref(kv), C.byref(bud), C.byref(mem), C.byref(plan), dummy,
                              1 << 30, None) == sfi.SFI_ERR_INVALID_ARG


def test_concurrent_fast_needs_side_stream_and_events(lib):
    """concurrent_fast without a side stream, or without its fork or join event, is refused
    before any CUDA call."""
    dummy = 1 << 20  # never dereferenced: the checks fail first
    kv = sfi.SfiKvCache(n_layers=1, batch=2, n_q_heads=8, n_kv_heads=2, head_dim=128, capacity=64,
                        max_len=8, k=dummy, v=dummy, seq_len=dummy, err=dummy)
    bud = sfi.SfiBudget(n_sink=4, n_window=16, n_select=8, prior_tau=16, lambda_=0.1)
    mem = sfi.SfiSparseMem(kc=dummy, vc=dummy, sel_idx=dummy, sel_cnt=dummy, rows=dummy)
    slow = np.array([[1, 1], [1, 0]], np.uint8)
    plan = sfi.SfiDecodePlan(n_steps=2, slow=slow.ctypes.data, q=dummy, k_new=dummy, v_new=dummy,
                             out=dummy, out_fp32=1, out_per_step=1, scores_f=dummy, masks=dummy,
                             len_start=8, concurrent_fast=1)
    for side, fork, join in ((None, dummy, dummy), (dummy, None, dummy), (dummy, dummy, None)):
        plan.side_stream, plan.fork_event, plan.join_event = side, fork, join
        assert lib.sfi_decode_run(C.byref(kv), C.byref(bud), C.byref(mem), C.byref(plan), dummy,
                                  1 << 30, None) == sfi.SFI_ERR_INVALID_ARG


@pytest.mark.parametrize("t_max", [0, 7, 64])
def test_native_token_scheduler_matches_oracle(lib, t_max):
    from synth import gen
    key = gen.key_from_seed(11)
    trig = np.array(gen.TRIGGER_TOKENS, np.int32)
    for b in range(5):
        toks = gen.token_stream(key, 500, b=b, mean_span=9.0)
        np.testing.assert_array_equal(sfi.sfi_schedule_tokens(toks, trig, t_max),
                                      oracle.schedule_tokens(toks, trig, t_max))
