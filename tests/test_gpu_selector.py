"""Selector bit-exactness on both Selector kernels, against the oracle.

sfi_select runs a cluster of CTAs per unit when the launch stays within about two waves
(few units), and one 1024-thread CTA per unit otherwise: with the evidence of the unit's
candidates staged in shared memory when they fit (up to 36,864), streamed from global
memory when they do not. The ragged and multi-layer workloads run the one-CTA kernel in
both modes, the 32K batch-4 workload the clustered one; each is held to the same bar:
given identical evidence the selected positions equal the oracle's bit for bit (Top-K by
fused score, ties to the lower position, written ascending; gist.science technical
summary, section 2B).

The evidence is written straight into the score buffer, in distributions that stress the
radix select: heavy-tailed, all equal, two-valued, coarsely quantised (many ties at the
threshold) and signed with NaNs (the key order puts NaN lowest, negatives below zero).
Sequences of different lengths share a launch, including lengths with fewer candidates than
the budget and with exactly as many.
"""
import numpy as np
import pytest
import torch

import oracle
from synth.configs import WORKLOADS

pytestmark = pytest.mark.gpu

BATCH = 12                     # 12 sequences x 8 kv heads = 96 units: more than the clustered
                               # Selector takes on a 152-SM part (76)
CL_BATCH = 4                   # 32 units: the clustered Selector (4 CTAs per unit)


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def evidence(kind: str, L: int, rng) -> np.ndarray:
    if kind == "heavy":
        return (rng.random(L) ** 6 / L).astype(np.float32)
    if kind == "tie":
        return np.full(L, 1.0 / L, np.float32)
    if kind == "two":
        return np.where(rng.random(L) < 0.1, 3.0 / L, 1.0 / L).astype(np.float32)
    if kind == "quant":
        return (rng.integers(0, 40, L) / (40.0 * L)).astype(np.float32)
    if kind == "signed":
        x = rng.standard_normal(L).astype(np.float32)
        x[rng.integers(0, L, 25)] = np.nan
        x[rng.integers(0, L, 25)] = -0.0
        x[rng.integers(0, L, 25)] = 0.0
        return x
    raise ValueError(kind)


KINDS = ["heavy", "tie", "two", "quant", "signed"]


def make_state(lo: int, hi: int, n_select: int, seed: int, batch: int = BATCH):
    from sparse_long_context_sfi_gb300.engine import SfiState
    cfg = WORKLOADS["llama8b_ctx32k_b4"].scaled(batch=batch, ctx=hi, ctx_lo=lo, steps=2,
                                                 n_select=n_select)
    rng = np.random.default_rng(seed)
    len0 = rng.integers(lo, hi + 1, batch)
    S, W, K = cfg.n_sink, cfg.n_window, cfg.n_select
    len0[1] = S + W + K - 3      # fewer candidates than the budget: all kept
    len0[2] = S + W + K          # exactly as many
    len0[3] = hi                 # the launch's bound
    st = SfiState(cfg, len0, device="cuda")
    st.kv.max_len = int(len0.max())
    return cfg, st, rng


def run_select(cfg, st, rng, budget=None, scores=None):
    """Fill the evidence, select on the GPU; returns (f, sel, cnt) on the host."""
    import sparse_long_context_sfi_gb300 as sfi
    H = cfg.n_kv_heads
    f = np.zeros((st.n_units, st.capacity), np.float32)
    for u in range(st.n_units):
        L = int(st.len0[u // H])
        f[u, :L] = evidence(KINDS[u % len(KINDS)], L, rng)
    st.scores.copy_(torch.from_numpy(f))
    sfi.sfi_select(st.kv, st.scores if scores is None else scores, budget or st.budget, st.mem)
    torch.cuda.synchronize()
    assert sfi.sfi_read_error(st.kv) == 0
    return f, st.sel_idx.cpu().numpy(), st.sel_cnt.cpu().numpy()


@pytest.mark.parametrize("lo,hi,n_select,batch", [
    (12000, 36000, 1980, BATCH),      # one CTA per unit, staged: candidates in shared memory
    (37000, 41000, 1980, BATCH),      # one CTA per unit, streamed: more than 36,864 candidates
    (8192, 32768, 956, BATCH),        # the ragged workload's budget and length range (staged)
    (12000, 36000, 1980, CL_BATCH),   # clustered: threshold-bin lists, or radix on many ties
    (37000, 41000, 956, CL_BATCH),    # clustered, long units
], ids=["staged", "streaming", "ragged_budget", "clustered", "clustered_long"])
def test_selector_bit_exact(lo, hi, n_select, batch):
    """Both Selector kernels against the oracle on evidence of every distribution: heavy
    tails (the clustered kernel exchanges the threshold bin's keys as lists), all equal and
    two-valued (its fallback to radix passes over the cluster's histograms)."""
    cfg, st, rng = make_state(lo, hi, n_select, seed=lo + batch, batch=batch)
    f, sel, cnt = run_select(cfg, st, rng)
    S, W, K = cfg.n_sink, cfg.n_window, cfg.n_select
    H = cfg.n_kv_heads
    for u in range(st.n_units):
        L = int(st.len0[u // H])
        want = oracle.select(L, S, W, K, cfg.prior_tau, cfg.lam, f[u, :L])
        assert cnt[u] == len(want), f"unit {u} ({KINDS[u % len(KINDS)]}, L={L})"
        np.testing.assert_array_equal(sel[u, :cnt[u]], want,
                                      err_msg=f"unit {u} ({KINDS[u % len(KINDS)]}, L={L})")


@pytest.mark.parametrize("lo,hi", [(12000, 36000), (37000, 41000)], ids=["staged", "streaming"])
def test_single_cta_selector_on_refined_scores_bit_exact(lo, hi):
    """Soft-NMS, cross-head exclusivity and the key-norm prior term (sfi_refine_scores), then
    Top-K on the refined scores (lambda = 0 keeps them as they are), both on the one-CTA
    Selector; compared with the oracle's refinement and Top-K bit for bit."""
    import sparse_long_context_sfi_gb300 as sfi
    cfg, st, rng = make_state(lo, hi, 1980, seed=hi)
    H, S, W, K = cfg.n_kv_heads, cfg.n_sink, cfg.n_window, cfg.n_select
    st.k.copy_((torch.randn(st.k.shape, device="cuda") * 1.5).to(torch.bfloat16))
    norms = torch.zeros_like(st.scores)
    sfi.sfi_key_norms(st.kv, norms)
    f = np.zeros((st.n_units, st.capacity), np.float32)
    for u in range(st.n_units):
        L = int(st.len0[u // H])
        f[u, :L] = evidence("heavy" if u % 2 else "quant", L, rng)
    st.scores.copy_(torch.from_numpy(f))
    opt = dict(nms_radius=2, nms_gamma=0.5, excl_mu=0.3, norm_nu=15.0)
    bud = sfi.SfiBudget(n_sink=S, n_window=W, n_select=K, prior_tau=cfg.prior_tau,
                        lambda_=cfg.lam, **opt)
    refined = torch.full_like(st.scores, float("nan"))
    sfi.sfi_refine_scores(st.kv, st.scores, norms, bud, refined)
    sel_bud = sfi.SfiBudget(n_sink=S, n_window=W, n_select=K, prior_tau=cfg.prior_tau,
                            lambda_=0.0)
    sfi.sfi_select(st.kv, refined, sel_bud, st.mem)
    torch.cuda.synchronize()
    assert sfi.sfi_read_error(st.kv) == 0
    kn = norms.cpu().numpy()
    r_gpu = refined.cpu().numpy()
    sel, cnt = st.sel_idx.cpu().numpy(), st.sel_cnt.cpu().numpy()
    for b in range(cfg.batch):
        L = int(st.len0[b])
        u0 = b * H
        ref = oracle.refine_scores(L, S, W, cfg.prior_tau, cfg.lam, f[u0:u0 + H, :L],
                                   nu=opt["norm_nu"], knorm=kn[u0:u0 + H, :L],
                                   radius=opt["nms_radius"], gamma=opt["nms_gamma"],
                                   mu=opt["excl_mu"])
        n = max(0, L - W - S)
        np.testing.assert_array_equal(r_gpu[u0:u0 + H, S:S + n].view(np.uint32),
                                      ref.view(np.uint32))
        for h in range(H):
            want = oracle.topk(ref[h], K) + S
            np.testing.assert_array_equal(sel[u0 + h, :cnt[u0 + h]], want,
                                          err_msg=f"sequence {b} head {h}, L={L}")


@pytest.mark.parametrize("batch", [BATCH, CL_BATCH], ids=["single_cta", "clustered"])
def test_length_beyond_bound_sets_error_and_skips_unit(batch):
    """A sequence whose length exceeds the launch's bound (kv.max_len, which sizes the
    shared-memory staging) gets no selection and raises SFI_DEVERR_LENGTH, on both Selector
    kernels; the other sequences' selections still equal the oracle's bit for bit."""
    import sparse_long_context_sfi_gb300 as sfi
    cfg, st, rng = make_state(12000, 30000, 1980, seed=11 + batch, batch=batch)
    S, W, K, H = cfg.n_sink, cfg.n_window, cfg.n_select, cfg.n_kv_heads
    f = np.zeros((st.n_units, st.capacity), np.float32)
    for u in range(st.n_units):
        L = int(st.len0[u // H])
        f[u, :L] = evidence(KINDS[u % len(KINDS)], L, rng)
    st.scores.copy_(torch.from_numpy(f))
    lens = st.len0.astype(np.int32).copy()
    lens[0] = st.kv.max_len + 100
    st.seq_len.copy_(torch.from_numpy(lens))
    st.sel_cnt.fill_(-7)
    sfi.sfi_select(st.kv, st.scores, st.budget, st.mem)
    torch.cuda.synchronize()
    assert sfi.sfi_read_error(st.kv) == 0x8
    sfi.sfi_clear_error(st.kv)
    sel, cnt = st.sel_idx.cpu().numpy(), st.sel_cnt.cpu().numpy()
    for u in range(st.n_units):
        if u // H == 0:
            assert cnt[u] == -7, f"unit {u}: selected beyond the bound"
            continue
        L = int(lens[u // H])
        want = oracle.select(L, S, W, K, cfg.prior_tau, cfg.lam, f[u, :L])
        assert cnt[u] == len(want)
        np.testing.assert_array_equal(sel[u, :cnt[u]], want, err_msg=f"unit {u}")
