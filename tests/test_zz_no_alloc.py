"""The allocation-free fast step, sfi_sparse_decode_attn_static, against the workspace
version sfi_sparse_decode_attn.

Callers that cannot allocate device memory (a plug-in that only receives its input and
output buffers, a decode loop that must not call cudaMalloc) use the static variant, whose
scratch is a fixed device array inside the library. This checks, through the C ABI, that two
calls in a row give the same outputs as the workspace version within the parity tolerance
of the other GPU tests (|a - b| <= 2e-3 + 1e-2 |b|). The file name sorts last so that a run
stopping at the first failure has already run every other test; it also passes alone in a
fresh process.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_static_scratch_fast_step_matches_workspace_version():
    import __graft_entry__
    __graft_entry__.build()
    import sparse_long_context_sfi_gb300 as sfi
    from synth import device as sdev
    from synth.configs import WORKLOADS
    from synth.workload import HostWorkload

    cfg = WORKLOADS["llama8b_ctx32k_b4"].scaled(ctx=3000, batch=3, steps=4)
    wl = HostWorkload(cfg)
    st = sdev.make_state(wl)
    ins = sdev.DeviceInputs(wl, 3, st.k.device)
    shape = (cfg.n_layers, cfg.batch, cfg.n_q_heads, cfg.head_dim)
    dev = st.k.device
    # slow step 0 fills the packed sparse memory
    st.step(ins.q[0], ins.k_new[0], ins.v_new[0], np.ones(cfg.batch, bool),
            torch.zeros(shape, dtype=torch.float32, device=dev))
    for t in (1, 2):                      # two calls in a row, each after its append
        st.kv.max_len = int(st.len0.max()) + t          # lengths before this append
        sfi.sfi_append_kv(st.kv, ins.k_new[t], ins.v_new[t])
        st.kv.max_len += 1
        assert sfi.sfi_read_error(st.kv) == 0
        ref = torch.zeros(shape, dtype=torch.float32, device=dev)
        got = torch.full(shape, float("nan"), dtype=torch.float32, device=dev)
        sfi.sfi_sparse_decode_attn(st.kv, st.mem, st.budget, ins.q[t], ref, True, st.ws,
                                   st.ws_bytes)
        sfi.sfi_sparse_decode_attn_static(st.kv, st.mem, st.budget, ins.q[t], got, True)
        torch.cuda.synchronize()
        r, g = ref.cpu().numpy().astype(np.float64), got.cpu().numpy().astype(np.float64)
        assert np.isfinite(g).all()
        assert (np.abs(g - r) <= 2e-3 + 1e-2 * np.abs(r)).all(), \
            f"call {t}: max abs diff {np.abs(g - r).max()}"
    assert sfi.sfi_read_error(st.kv) == 0
