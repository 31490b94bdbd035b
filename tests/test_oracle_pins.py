"""Pins of the CPU oracle against things other than itself: library routines it must
reduce to, closed forms, invariants and brute force on tiny inputs (no GPU).

Sources: "Slow-Fast Inference: Training-Free Inference Acceleration via Within-Sentence
Support Stability" -- the blog "How SFI Works" section (slow = dense attention, fast =
attention over the kept support), and the gist.science technical summary, sections 2A
(sparse state), 2B (Selector: evidence, prior, closed-form fusion, Top-K), 2C (trigger
policy) and 3 (packed sparse buffer, recent tokens from the cache).
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from synth import gen

D = 128


def rand_bf16(rng, *shape, scale=1.0):
    return gen.f32_to_bf16((rng.standard_normal(shape) * scale).astype(np.float32))


def f64(b):
    return gen.bf16_to_f32(b).astype(np.float64)


# ------------------------------------------------------------------------------ attention

@pytest.mark.parametrize("G,L", [(1, 1), (4, 37), (8, 300)])
def test_attend_matches_library_sdpa(G, L):
    """Dense attention equals torch's scaled_dot_product_attention in fp64."""
    rng = np.random.default_rng(G * 1000 + L)
    q, k, v = rand_bf16(rng, G, D), rand_bf16(rng, L, D, scale=2.0), rand_bf16(rng, L, D)
    o, p = oracle.attend(q, k, v, want_p=True)
    tq = torch.from_numpy(f64(q))[:, None, :]           # [G, 1, D]
    tk = torch.from_numpy(f64(k))[None].expand(G, L, D)
    tv = torch.from_numpy(f64(v))[None].expand(G, L, D)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)[:, 0].numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)
    # Attention weights: the same routine with V = identity returns the weights themselves.
    eye = torch.eye(L, dtype=torch.float64)[None].expand(G, L, L)
    w = torch.nn.functional.scaled_dot_product_attention(tq, tk, eye)[:, 0].numpy()
    np.testing.assert_allclose(p, w, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)


def test_attend_closed_forms():
    rng = np.random.default_rng(1)
    G, L = 4, 50
    q = rand_bf16(rng, G, D)
    # identical keys: uniform weights, o = mean of V rows
    k = np.repeat(rand_bf16(rng, 1, D), L, axis=0)
    v = rand_bf16(rng, L, D)
    o, _ = oracle.attend(q, k, v)
    np.testing.assert_allclose(o, np.repeat(f64(v).mean(axis=0)[None], G, 0), rtol=0, atol=1e-13)
    # one row: o = v_0
    o, _ = oracle.attend(q, k[:1], v[:1])
    np.testing.assert_array_equal(o, np.repeat(f64(v[:1]), G, 0))
    # equal V rows: o = that row whatever the weights
    k = rand_bf16(rng, L, D, scale=3.0)
    v = np.repeat(rand_bf16(rng, 1, D), L, axis=0)
    o, _ = oracle.attend(q, k, v)
    np.testing.assert_allclose(o, np.repeat(f64(v[:1]), G, 0), rtol=1e-14, atol=1e-14)


def test_attend_row_subset_is_attention_over_subset():
    rng = np.random.default_rng(2)
    q, k, v = rand_bf16(rng, 4, D), rand_bf16(rng, 80, D), rand_bf16(rng, 80, D)
    rows = np.array([3, 0, 17, 79, 40, 41], dtype=np.int32)
    o1, _ = oracle.attend(q, k, v, rows)
    o2, _ = oracle.attend(q, k[rows], v[rows])
    np.testing.assert_array_equal(o1, o2)


@pytest.mark.parametrize("split", [1, 3, 16, 64, 200, 1000])
def test_split_merge_equals_unsplit(split):
    rng = np.random.default_rng(3)
    q, k, v = rand_bf16(rng, 4, D), rand_bf16(rng, 200, D, scale=2.0), rand_bf16(rng, 200, D)
    o, _ = oracle.attend(q, k, v)
    np.testing.assert_allclose(oracle.attend_split(q, k, v, split), o, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------------------- evidence

def test_evidence_is_group_mean_of_weights():
    rng = np.random.default_rng(4)
    G, L = 4, 120
    q, k, v = rand_bf16(rng, G, D), rand_bf16(rng, L, D, scale=2.0), rand_bf16(rng, L, D)
    _, p = oracle.attend(q, k, v, want_p=True)
    f = oracle.evidence(p)
    assert abs(f.sum() - 1.0) < 1e-12
    np.testing.assert_allclose(f, p.mean(axis=0), rtol=1e-15, atol=0)
    # G = 1: the evidence is that head's softmax
    _, p1 = oracle.attend(q[:1], k, v, want_p=True)
    np.testing.assert_array_equal(oracle.evidence(p1), p1[0])


# ------------------------------------------------------------------------ prior and fusion

@pytest.mark.parametrize("n,tau", [(0, 64), (1, 64), (10, 64), (63, 64), (64, 64), (65, 64),
                                   (5000, 64), (131000, 128), (7, 1)])
def test_prior_norm_closed_form(n, tau):
    z = oracle.prior_norm(n, tau)
    if n >= tau:
        closed = (tau + 1) / 2.0 + (n - tau)
    else:
        closed = n * (n + 1) / (2.0 * tau)
    assert z == closed


def test_fused_scores_lambda0_is_evidence():
    rng = np.random.default_rng(5)
    L, S, W = 500, 4, 64
    f = rng.random(L).astype(np.float32)
    s = oracle.fused_scores(L, S, W, 64, 0.0, f)
    np.testing.assert_array_equal(s, f[S:L - W])


def test_fused_scores_lambda1_is_prior_distribution():
    L, S, W, tau = 1000, 4, 64, 64
    n = L - W - S
    s = oracle.fused_scores(L, S, W, tau, 1.0, np.zeros(L, np.float32)).astype(np.float64)
    d = (L - W) - np.arange(S, L - W)
    ramp = np.minimum(1.0, d / tau)
    # the prior is a distribution over the candidates ...
    assert abs(s.sum() - 1.0) < 1e-5
    # ... proportional to the ramp min(1, d/tau)
    np.testing.assert_allclose(s / s.max(), ramp, rtol=1e-6)
    assert s.shape[0] == n


def test_fused_scores_mix():
    rng = np.random.default_rng(6)
    L, S, W, tau, lam = 3000, 4, 64, 64, 0.1
    f = rng.random(L).astype(np.float32)
    f /= f.sum()
    s = oracle.fused_scores(L, S, W, tau, lam, f).astype(np.float64)
    n = L - W - S
    d = (L - W) - np.arange(S, L - W)
    r = np.minimum(1.0, d / tau)
    r /= r.sum()
    np.testing.assert_allclose(s, (1 - lam) * f[S:L - W] + lam * r, rtol=2e-7, atol=1e-12)


# ---------------------------------------------------------------------------------- top-K

def brute_topk(s, K):
    """Index i is chosen iff fewer than K indices come before it in the (score desc,
    index asc) order -- an O(n^2) restatement of the definition."""
    keys = [gen_key(x) for x in s]
    chosen = []
    for i in range(len(s)):
        before = sum(1 for j in range(len(s)) if keys[j] > keys[i] or (keys[j] == keys[i] and j < i))
        if before < K:
            chosen.append(i)
    return np.array(chosen, dtype=np.int32)


def gen_key(x):
    x = np.float32(x)
    if np.isnan(x):
        return 0
    u = int(np.array([x], np.float32).view(np.uint32)[0])
    return (~u & 0xFFFFFFFF) if u & 0x80000000 else (u | 0x80000000)


@pytest.mark.parametrize("kind", ["random", "equal", "two", "with_nan"])
def test_topk_brute_force(kind):
    rng = np.random.default_rng(7)
    for n in [1, 2, 5, 17, 64]:
        if kind == "random":
            s = rng.random(n).astype(np.float32)
        elif kind == "equal":
            s = np.full(n, 0.25, np.float32)
        elif kind == "two":
            s = rng.choice([0.5, 0.75], n).astype(np.float32)
        else:
            s = rng.random(n).astype(np.float32)
            s[rng.random(n) < 0.2] = np.nan
        for K in range(0, n + 2):
            got = oracle.topk(s, K)
            np.testing.assert_array_equal(got, brute_topk(s, K))


def test_topk_matches_library_lexsort():
    rng = np.random.default_rng(8)
    s = rng.choice(np.linspace(0, 1, 50), 4000).astype(np.float32)
    for K in [1, 10, 1980, 3999, 4000]:
        order = np.lexsort((np.arange(s.size), -s.astype(np.float64)))
        np.testing.assert_array_equal(oracle.topk(s, K), np.sort(order[:K]))


def test_select_lambda1_pins_tie_break():
    """lambda = 1: every candidate at distance >= tau ties at the top, so the lower-index
    tie-break must pick exactly [S, S+K) when n_C >= K + tau."""
    L, S, W, K, tau = 4096, 4, 64, 256, 64
    f = np.random.default_rng(9).random(L).astype(np.float32)
    sel = oracle.select(L, S, W, K, tau, 1.0, f)
    np.testing.assert_array_equal(sel, np.arange(S, S + K))


def test_select_lambda0_is_topk_of_evidence():
    L, S, W, K, tau = 5000, 4, 64, 300, 64
    f = np.random.default_rng(10).random(L).astype(np.float32)
    sel = oracle.select(L, S, W, K, tau, 0.0, f)
    cand = f[S:L - W]
    order = np.lexsort((np.arange(cand.size), -cand.astype(np.float64)))
    np.testing.assert_array_equal(sel, np.sort(order[:K]) + S)


def test_select_few_candidates_takes_all():
    f = np.ones(100, np.float32)
    np.testing.assert_array_equal(oracle.select(100, 4, 64, 256, 64, 0.1, f), np.arange(4, 36))
    assert oracle.select(60, 4, 64, 256, 64, 0.1, f).size == 0


# --------------------------------------------------------------------------- sparse state

def test_sparse_rows_hand_example():
    # S=2, W=3: slow step at L=10 selected {4, 2}; fast step at L=12
    rows = oracle.sparse_rows(10, 12, 2, 3, np.array([2, 4], np.int32))
    np.testing.assert_array_equal(rows, [0, 1, 2, 4, 9, 10, 11])
    # short context: window clipped at the sinks
    rows = oracle.sparse_rows(3, 4, 4, 64, np.array([], np.int32))
    np.testing.assert_array_equal(rows, [0, 1, 2, 3])


def test_budget_covering_context_equals_dense():
    """With K >= n_C the sparse state at the slow step is every position, so the fast step
    taken right after selection equals dense attention."""
    rng = np.random.default_rng(11)
    L, S, W, G = 700, 4, 64, 4
    q, k, v = rand_bf16(rng, G, D), rand_bf16(rng, L, D, scale=2.0), rand_bf16(rng, L, D)
    o_dense, p = oracle.attend(q, k, v, want_p=True)
    f = oracle.evidence(p).astype(np.float32)
    sel = oracle.select(L, S, W, 10_000, 64, 0.1, f)
    rows = oracle.sparse_rows(L, L, S, W, sel)
    assert sorted(rows.tolist()) == list(range(L))
    o_sparse, _ = oracle.attend(q, k, v, rows)
    np.testing.assert_allclose(o_sparse, o_dense, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------------------ scheduler

def test_schedule_periodic_mask():
    m = gen.boundary_mask(None, 32, "periodic", 16)
    slow = oracle.schedule(m, 64)
    assert np.flatnonzero(slow).tolist() == [0, 16]


def test_schedule_hand_example_and_tmax():
    m = np.array([0, 0, 1, 0, 0, 0, 0, 0, 1, 1, 0, 0], np.uint8)
    assert np.flatnonzero(oracle.schedule(m, 0)).tolist() == [0, 3, 9, 10]
    # T_max = 4 forces a refresh 4 steps after the last slow step
    assert np.flatnonzero(oracle.schedule(m, 4)).tolist() == [0, 3, 7, 9, 10]
    assert np.flatnonzero(oracle.schedule(np.zeros(9, np.uint8), 3)).tolist() == [0, 3, 6]


def test_geometric_mask_gap_mean():
    key = gen.key_from_seed(123)
    m = gen.boundary_mask(key, 200000, "geometric", 18)
    gaps = np.diff(np.flatnonzero(m))
    assert gaps.min() >= 1
    # mean 18, standard deviation sqrt(1 - 1/18) * 18; allow five standard errors
    assert abs(gaps.mean() - 18) < 5 * math.sqrt(1 - 1 / 18) * 18 / math.sqrt(gaps.size)


def test_token_schedule_hand_example_and_mask_equivalence():
    trig = np.array([13, 0], np.int32)
    toks = np.array([5, 13, 7, 7, 0, 9, 9, 9, 9], np.int32)
    assert np.flatnonzero(oracle.schedule_tokens(toks, trig, 0)).tolist() == [0, 2, 5]
    assert np.flatnonzero(oracle.schedule_tokens(toks, trig, 3)).tolist() == [0, 2, 5, 8]
    # a trigger token at step t is exactly a boundary mask bit at t
    key = gen.key_from_seed(7)
    toks = gen.token_stream(key, 3000)
    mask = np.isin(toks, np.array(gen.TRIGGER_TOKENS)).astype(np.uint8)
    for t_max in (0, 64):
        np.testing.assert_array_equal(oracle.schedule_tokens(toks, np.array(gen.TRIGGER_TOKENS), t_max),
                                      oracle.schedule(mask, t_max))
    gaps = np.diff(np.flatnonzero(mask))
    assert abs(gaps.mean() - 18) < 5 * 18 / math.sqrt(gaps.size)
