"""GPU parity of the Selector refinements and key norms (C ABI) against the oracle.

Both sides evaluate the same fp32 recipes, so given the same evidence (the GPU's own, as
for sfi_select) the refined scores and the selections are compared bit for bit. Key norms
are compared bit for bit against the oracle on the cache rows.
"""
import numpy as np
import pytest
import torch

import oracle
from synth import device as sdev
from synth.configs import WORKLOADS
from synth.workload import HostWorkload

pytestmark = pytest.mark.gpu

OPTIONS = [
    dict(nms_radius=2, nms_gamma=0.5),
    dict(excl_mu=0.4),
    dict(norm_nu=16.0),
    dict(geometric=1),
    dict(geometric=1, nms_radius=1, nms_gamma=0.25, excl_mu=0.3, norm_nu=14.0),
    dict(nms_radius=3, nms_gamma=0.5, nms_delta=2e-4),
    dict(geometric=1, nms_radius=2, nms_gamma=0.25, nms_delta=1.0, excl_mu=0.3),
]


@pytest.fixture(scope="module")
def slow_state():
    import __graft_entry__
    __graft_entry__.build()
    cfg = WORKLOADS["llama8b_ctx32k_b4"].scaled(ctx=2500, batch=2, n_layers=2, steps=2)
    wl = HostWorkload(cfg)
    st = sdev.make_state(wl)
    ins = sdev.DeviceInputs(wl, 1, st.k.device)
    out = torch.zeros((cfg.n_layers, cfg.batch, cfg.n_q_heads, cfg.head_dim), device=st.k.device)
    st.step(ins.q[0], ins.k_new[0], ins.v_new[0], np.ones(cfg.batch, bool), out)
    torch.cuda.synchronize()
    return wl, st


def test_key_norms_bit_exact(slow_state):
    import sparse_long_context_sfi_gb300 as sfi
    wl, st = slow_state
    cfg = wl.cfg
    norms = torch.zeros_like(st.scores)
    sfi.sfi_key_norms(st.kv, norms)
    torch.cuda.synchronize()
    got = norms.cpu().numpy()
    for u in range(st.n_units):
        layer, b, kvh = u // (cfg.n_kv_heads * cfg.batch), (u // cfg.n_kv_heads) % cfg.batch, u % cfg.n_kv_heads
        L = int(wl.len0[b]) + 1
        ref = oracle.key_norms(wl.rows("k", layer, b, kvh, np.arange(L)))
        np.testing.assert_array_equal(got[u, :L], ref)


@pytest.mark.parametrize("opt", OPTIONS, ids=lambda o: "-".join(f"{k}{v}" for k, v in o.items()))
def test_refined_scores_and_selection_bit_exact(slow_state, opt):
    import sparse_long_context_sfi_gb300 as sfi
    wl, st = slow_state
    cfg = wl.cfg
    norms = torch.zeros_like(st.scores)
    sfi.sfi_key_norms(st.kv, norms)
    bud = sfi.SfiBudget(n_sink=cfg.n_sink, n_window=cfg.n_window, n_select=cfg.n_select,
                        prior_tau=cfg.prior_tau, lambda_=cfg.lam, **opt)
    refined = torch.full_like(st.scores, float("nan"))
    sfi.sfi_refine_scores(st.kv, st.scores, norms, bud, refined)
    # selection on the refined scores: lambda = 0 keeps them as they are
    sel_bud = sfi.SfiBudget(n_sink=cfg.n_sink, n_window=cfg.n_window, n_select=cfg.n_select,
                            prior_tau=cfg.prior_tau, lambda_=0.0)
    sfi.sfi_select(st.kv, refined, sel_bud, st.mem)
    torch.cuda.synchronize()
    assert sfi.sfi_read_error(st.kv) == 0
    f = st.scores.cpu().numpy()
    kn = norms.cpu().numpy()
    r_gpu = refined.cpu().numpy()
    sel = st.sel_idx.cpu().numpy()
    cnt = st.sel_cnt.cpu().numpy()
    H = cfg.n_kv_heads
    S, W, K = cfg.n_sink, cfg.n_window, cfg.n_select
    for layer in range(cfg.n_layers):
        for b in range(cfg.batch):
            L = int(wl.len0[b]) + 1
            u0 = (layer * cfg.batch + b) * H
            ref = oracle.refine_scores(L, S, W, cfg.prior_tau, cfg.lam, f[u0:u0 + H, :L],
                                       geometric=bool(opt.get("geometric", 0)),
                                       nu=opt.get("norm_nu", 0.0), knorm=kn[u0:u0 + H, :L],
                                       radius=opt.get("nms_radius", 0),
                                       gamma=opt.get("nms_gamma", 1.0), mu=opt.get("excl_mu", 0.0),
                                       delta=opt.get("nms_delta", 0.0))
            n = L - W - S
            np.testing.assert_array_equal(r_gpu[u0:u0 + H, S:S + n].view(np.uint32),
                                          ref.view(np.uint32))
            for h in range(H):
                want = oracle.topk(ref[h], K) + S
                np.testing.assert_array_equal(sel[u0 + h, :cnt[u0 + h]], want)
