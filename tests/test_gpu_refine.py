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


@pytest.mark.parametrize("opt", [
    dict(nms_radius=2, nms_gamma=0.5, nms_delta=3e-4, excl_mu=0.2, norm_nu=15.0),
    dict(geometric=1, nms_radius=3, nms_gamma=0.25, nms_delta=0.5),
], ids=["arithmetic", "geometric"])
def test_refinement_on_paged_ragged_cache_with_inactive_sequences(opt):
    """Key norms, refined scores and the Selector over them on a paged cache (16-row pages)
    with ragged lengths (some with fewer candidates than the budget), for a subset of the
    sequences: active ones bit-exact against the oracle, inactive ones left untouched. The
    Soft-NMS similarity limit is chosen so that it changes some refined scores against both
    the unlimited rule and Soft-NMS off."""
    import __graft_entry__
    __graft_entry__.build()
    import sparse_long_context_sfi_gb300 as sfi
    cfg = WORKLOADS["ragged_paged_b32"].scaled(batch=5, ctx=2600, ctx_lo=300, steps=2)
    wl = HostWorkload(cfg)
    st = sdev.make_state(wl)
    dev = st.k.device
    ins = sdev.DeviceInputs(wl, 1, dev)
    out = torch.zeros((cfg.n_layers, cfg.batch, cfg.n_q_heads, cfg.head_dim), device=dev)
    st.step(ins.q[0], ins.k_new[0], ins.v_new[0], np.ones(cfg.batch, bool), out)
    torch.cuda.synchronize()
    act = np.array([1, 0, 1, 1, 0], np.uint8)
    active = torch.from_numpy(act).to(dev)
    sel_before = st.sel_idx.cpu().numpy().copy()
    cnt_before = st.sel_cnt.cpu().numpy().copy()
    norms = torch.full_like(st.scores, float("nan"))
    sfi.sfi_key_norms(st.kv, norms, active)
    bud = sfi.SfiBudget(n_sink=cfg.n_sink, n_window=cfg.n_window, n_select=cfg.n_select,
                        prior_tau=cfg.prior_tau, lambda_=cfg.lam, **opt)
    refined = torch.full_like(st.scores, float("nan"))
    sfi.sfi_refine_scores(st.kv, st.scores, norms, bud, refined, active)
    sel_bud = sfi.SfiBudget(n_sink=cfg.n_sink, n_window=cfg.n_window, n_select=cfg.n_select,
                            prior_tau=cfg.prior_tau, lambda_=0.0)
    sfi.sfi_select(st.kv, refined, sel_bud, st.mem, active)
    torch.cuda.synchronize()
    assert sfi.sfi_read_error(st.kv) == 0
    f, kn, r_gpu = st.scores.cpu().numpy(), norms.cpu().numpy(), refined.cpu().numpy()
    sel, cnt = st.sel_idx.cpu().numpy(), st.sel_cnt.cpu().numpy()
    H, S, W, K = cfg.n_kv_heads, cfg.n_sink, cfg.n_window, cfg.n_select
    differs_from_unlimited = differs_from_off = False
    kw = dict(geometric=bool(opt.get("geometric", 0)), nu=opt.get("norm_nu", 0.0),
              gamma=opt["nms_gamma"], mu=opt.get("excl_mu", 0.0))
    for b in range(cfg.batch):
        u0 = b * H
        L = int(wl.len0[b]) + 1
        if not act[b]:
            assert np.isnan(kn[u0:u0 + H]).all() and np.isnan(r_gpu[u0:u0 + H]).all()
            np.testing.assert_array_equal(sel[u0:u0 + H], sel_before[u0:u0 + H])
            np.testing.assert_array_equal(cnt[u0:u0 + H], cnt_before[u0:u0 + H])
            continue
        for h in range(H):
            want = oracle.key_norms(wl.rows("k", 0, b, h, np.arange(L)))
            np.testing.assert_array_equal(kn[u0 + h, :L], want)
        args = (L, S, W, cfg.prior_tau, cfg.lam, f[u0:u0 + H, :L])
        ref = oracle.refine_scores(*args, knorm=kn[u0:u0 + H, :L], radius=opt["nms_radius"],
                                   delta=opt["nms_delta"], **kw)
        n = L - W - S
        np.testing.assert_array_equal(r_gpu[u0:u0 + H, S:S + n].view(np.uint32),
                                      ref.view(np.uint32))
        for h in range(H):
            np.testing.assert_array_equal(sel[u0 + h, :cnt[u0 + h]], oracle.topk(ref[h], K) + S,
                                          err_msg=f"sequence {b} head {h}, L={L}")
        unlimited = oracle.refine_scores(*args, knorm=kn[u0:u0 + H, :L],
                                         radius=opt["nms_radius"], **kw)
        off = oracle.refine_scores(*args, knorm=kn[u0:u0 + H, :L], radius=0, **kw)
        differs_from_unlimited |= not np.array_equal(ref, unlimited)
        differs_from_off |= not np.array_equal(ref, off)
    assert differs_from_unlimited and differs_from_off
