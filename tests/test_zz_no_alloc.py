"""The allocation-free fast step, sfi_sparse_decode_attn_static, against the workspace
version sfi_sparse_decode_attn and against the oracle.

Callers that cannot allocate device memory (a plug-in that only receives its input and
output buffers, a decode loop that must not call cudaMalloc) use the static variant, whose
scratch is a fixed device array inside the library. This checks, through the C ABI, that two
calls in a row give the same outputs as the workspace version, and as the oracle's attention
over the same sparse rows, within the parity tolerance of the other GPU tests
(|a - b| <= 2e-3 + 1e-2 |b|). The shapes cover group 4 with split units, group 8 (the
largest partials) and more units than CTAs (every CTA leaves partials in the shared array).
The file name sorts last so that a run stopping at the first failure has already run every
other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2


@pytest.mark.parametrize("shape", [
    dict(ctx=3000, batch=3),                        # 24 units, group 4
    dict(ctx=1100, batch=2, n_q_heads=64),          # 16 units, group 8
    dict(ctx=1200, batch=12),                       # 96 units
], ids=["group4", "group8", "96_units"])
def test_static_scratch_fast_step_matches_workspace_version_and_oracle(shape):
    import __graft_entry__
    __graft_entry__.build()
    import oracle
    import sparse_long_context_sfi_gb300 as sfi
    from synth import device as sdev
    from synth.configs import WORKLOADS
    from synth.workload import HostWorkload

    cfg = WORKLOADS["llama8b_ctx32k_b4"].scaled(steps=4, **shape)
    wl = HostWorkload(cfg)
    st = sdev.make_state(wl)
    ins = sdev.DeviceInputs(wl, 3, st.k.device)
    shp = (cfg.n_layers, cfg.batch, cfg.n_q_heads, cfg.head_dim)
    dev = st.k.device
    G, S, W = cfg.group, cfg.n_sink, cfg.n_window
    # slow step 0 fills the packed sparse memory
    st.step(ins.q[0], ins.k_new[0], ins.v_new[0], np.ones(cfg.batch, bool),
            torch.zeros(shp, dtype=torch.float32, device=dev))
    torch.cuda.synchronize()
    sel = [st.sel_idx[u, :int(st.sel_cnt[u])].cpu().numpy() for u in range(st.n_units)]
    for t in (1, 2):                      # two calls in a row, each after its append
        st.kv.max_len = int(st.len0.max()) + t          # lengths before this append
        sfi.sfi_append_kv(st.kv, ins.k_new[t], ins.v_new[t])
        st.kv.max_len += 1
        assert sfi.sfi_read_error(st.kv) == 0
        ref = torch.zeros(shp, dtype=torch.float32, device=dev)
        got = torch.full(shp, float("nan"), dtype=torch.float32, device=dev)
        sfi.sfi_sparse_decode_attn(st.kv, st.mem, st.budget, ins.q[t], ref, True, st.ws,
                                   st.ws_bytes)
        sfi.sfi_sparse_decode_attn_static(st.kv, st.mem, st.budget, ins.q[t], got, True)
        torch.cuda.synchronize()
        r, g = ref.cpu().numpy().astype(np.float64), got.cpu().numpy().astype(np.float64)
        assert np.isfinite(g).all()
        assert (np.abs(g - r) <= ATOL + RTOL * np.abs(r)).all(), \
            f"call {t}: max abs diff to the workspace version {np.abs(g - r).max()}"
        for u in range(st.n_units):
            b, kvh = (u // cfg.n_kv_heads) % cfg.batch, u % cfg.n_kv_heads
            Ls = int(wl.len0[b]) + 1
            rows = oracle.sparse_rows(Ls, Ls + t, S, W, sel[u])
            k = wl.rows("k", 0, b, kvh, np.arange(Ls + t))
            v = wl.rows("v", 0, b, kvh, np.arange(Ls + t))
            o, _ = oracle.attend(wl.query(t, 0, b)[kvh * G:(kvh + 1) * G], k, v, rows)
            gu = g[0, b, kvh * G:(kvh + 1) * G]
            assert (np.abs(gu - o) <= ATOL + RTOL * np.abs(o)).all(), \
                f"call {t} unit {u}: max abs err to the oracle {np.abs(gu - o).max()}"
    assert sfi.sfi_read_error(st.kv) == 0
