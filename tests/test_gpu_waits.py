"""Bounded waits on the GPU. With the test hook sfi_test_inject_stall, the first CTA of the
next attention launch waits on a barrier that never completes; the kernel must give up after
about a second, report SFI_DEVERR_TIMEOUT through the error word, drain and return, and the
context must stay usable: after clearing the error and re-initialising the workspace, the
next steps match a run that never stalled."""
import time

import numpy as np
import pytest
import torch

from synth import device as sdev
from synth.configs import WORKLOADS
from synth.workload import HostWorkload

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2


@pytest.mark.parametrize("case", [dict(ctx=3000, batch=2), dict(ctx=1300, batch=3, n_layers=5)],
                         ids=["clustered", "tile_ranges"])
def test_stalled_barrier_times_out_and_context_survives(case):
    import __graft_entry__
    __graft_entry__.build()
    import sparse_long_context_sfi_gb300 as sfi
    n = 6
    wl = HostWorkload(WORKLOADS["llama8b_ctx32k_b4"].scaled(steps=n, **case))
    cfg = wl.cfg
    a = sdev.make_state(wl)   # stalls at step 1
    b = sdev.make_state(wl)   # never stalls
    ins = sdev.DeviceInputs(wl, n, a.k.device)
    shape = (cfg.n_layers, cfg.batch, cfg.n_q_heads, cfg.head_dim)
    oa = torch.zeros(shape, dtype=torch.float32, device=a.k.device)
    ob = torch.zeros_like(oa)
    slow0 = np.ones(cfg.batch, bool)
    fast = np.zeros(cfg.batch, bool)
    a.step(ins.q[0], ins.k_new[0], ins.v_new[0], slow0, oa)
    b.step(ins.q[0], ins.k_new[0], ins.v_new[0], slow0, ob)
    torch.cuda.synchronize()
    assert sfi.sfi_read_error(a.kv) == 0

    sfi.sfi_test_inject_stall(True)
    t0 = time.time()
    a.step(ins.q[1], ins.k_new[1], ins.v_new[1], fast, oa)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    b.step(ins.q[1], ins.k_new[1], ins.v_new[1], fast, ob)
    torch.cuda.synchronize()
    bits = sfi.sfi_read_error(a.kv)
    assert bits & sfi.SFI_DEVERR_TIMEOUT
    assert elapsed < 30.0
    assert sfi.sfi_read_error(b.kv) == 0
    # the lengths still advanced (every CTA counts itself, stalled or not)
    assert torch.equal(a.seq_len, b.seq_len)

    # Recover: clear the error, re-initialise the workspace, take the cache state of the
    # run that never stalled (a timed-out step's outputs and appends are not guaranteed),
    # and continue: the library and the context work as before.
    sfi.sfi_clear_error(a.kv)
    sfi.sfi_workspace_init(a.ws, a.ws_bytes)
    for name in ("k", "v", "kc", "vc", "sel_idx", "sel_cnt", "rows"):
        getattr(a, name).copy_(getattr(b, name))
    for t in range(2, n):
        a.step(ins.q[t], ins.k_new[t], ins.v_new[t], fast, oa)
        b.step(ins.q[t], ins.k_new[t], ins.v_new[t], fast, ob)
        torch.cuda.synchronize()
        assert sfi.sfi_read_error(a.kv) == 0
        ga, gb = oa.cpu().numpy().astype(np.float64), ob.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(ga - gb) <= ATOL + RTOL * np.abs(gb)), f"step {t}"
