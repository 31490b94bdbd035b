"""Pins of the Selector refinements in the oracle (Soft-NMS within a head, cross-head
exclusivity, key-norm prior term, geometric mixture): a library routine, identities,
hand-checked examples and invariants. Source: the gist.science technical summary of
"Slow-Fast Inference", section 2B (Selector: fusion, Soft-NMS, cross-head exclusivity)."""
import numpy as np
import pytest

import oracle
from synth import gen

L, S, W, TAU = 700, 4, 64, 64


def evidence4():
    rng = np.random.default_rng(3)
    x = rng.random((4, L)).astype(np.float64) ** 4
    return (x / x.sum(axis=1, keepdims=True)).astype(np.float32)


def test_log2f_matches_library_log2():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.random(2000) * 10.0 ** rng.integers(-30, 30, 2000),
                        [1.0, 2.0, 0.5, 3.0, 1e-40, 3.4e38]]).astype(np.float32)
    got = np.array([oracle.log2f(float(v)) for v in x], np.float64)
    ref = np.log2(x.astype(np.float64))
    assert np.max(np.abs(got - ref) / np.maximum(1.0, np.abs(ref))) < 3e-7
    assert oracle.log2f(0.0) == -np.inf
    assert oracle.log2f(1.0) == 0.0 and oracle.log2f(8.0) == 3.0


def test_refine_off_is_the_plain_fusion():
    f = evidence4()
    for lam in (0.0, 0.1, 1.0):
        r = oracle.refine_scores(L, S, W, TAU, lam, f)
        for h in range(4):
            np.testing.assert_array_equal(r[h], oracle.fused_scores(L, S, W, TAU, lam, f[h]))


def test_soft_nms_hand_example():
    # one head, candidates 0..5 (S=0, W=1, L=7): scores are the fused scores with lambda=0
    s = np.array([[0.1, 0.5, 0.2, 0.2, 0.9, 0.05, 0.0]], np.float32)
    r = oracle.refine_scores(7, 0, 1, 1, 0.0, s, radius=1, gamma=0.5)[0]
    # 0.1 < 0.5 -> halved; 0.5 local max; 0.2 < 0.5 -> halved; 0.2 < 0.9 -> halved;
    # 0.9 local max; 0.05 < 0.9 -> halved (candidate 6 is the window, not a neighbour)
    np.testing.assert_array_equal(r, np.float32([0.05, 0.5, 0.1, 0.1, 0.9, 0.025]))
    r2 = oracle.refine_scores(7, 0, 1, 1, 0.0, s, radius=2, gamma=0.0)[0]
    np.testing.assert_array_equal(r2, np.float32([0, 0.5, 0, 0, 0.9, 0]))
    # a plateau is not dominated: equal neighbours suppress nobody
    p = np.array([[0.3, 0.3, 0.1, 0.0]], np.float32)
    np.testing.assert_array_equal(oracle.refine_scores(4, 0, 1, 1, 0.0, p, radius=1, gamma=0.5)[0],
                                  np.float32([0.3, 0.3, 0.05]))


def test_soft_nms_similarity_hand_example():
    # the damping acts only between close scores: with delta = 0.35 only a neighbour at
    # most 0.35 higher suppresses (same scores as the example above)
    s = np.array([[0.1, 0.5, 0.2, 0.2, 0.9, 0.05, 0.0]], np.float32)
    r = oracle.refine_scores(7, 0, 1, 1, 0.0, s, radius=1, gamma=0.5, delta=0.35)[0]
    # 0.1: 0.5 is 0.4 higher -> kept; 0.5 local max; 0.2: 0.5 is 0.3 higher -> halved;
    # 0.2: 0.9 is 0.7 higher, the other 0.2 not higher -> kept; 0.9 kept; 0.05: 0.85 -> kept
    np.testing.assert_array_equal(r, np.float32([0.1, 0.5, 0.1, 0.2, 0.9, 0.05]))
    # radius 2: 0.1 now sees 0.2 (0.1 higher) -> halved; the second 0.2 sees 0.5 (0.3
    # higher) -> halved; 0.05 sees 0.2 (0.15 higher) -> halved
    r2 = oracle.refine_scores(7, 0, 1, 1, 0.0, s, radius=2, gamma=0.5, delta=0.35)[0]
    np.testing.assert_array_equal(r2, np.float32([0.05, 0.5, 0.1, 0.1, 0.9, 0.025]))
    # a limit above every gap is the unlimited rule; one below every gap suppresses nobody
    for radius in (1, 2, 3):
        np.testing.assert_array_equal(
            oracle.refine_scores(7, 0, 1, 1, 0.0, s, radius=radius, gamma=0.5, delta=10.0),
            oracle.refine_scores(7, 0, 1, 1, 0.0, s, radius=radius, gamma=0.5))
        np.testing.assert_array_equal(
            oracle.refine_scores(7, 0, 1, 1, 0.0, s, radius=radius, gamma=0.5, delta=1e-3),
            s[:, :6])


def test_soft_nms_similarity_brute_force():
    # every candidate against the definition, evaluated here position by position: scaled
    # iff a neighbour within the radius is strictly higher by at most delta (fp32 difference)
    f = evidence4()
    n = L - W - S
    for radius, delta in ((1, 0.0), (3, 2e-4), (2, 5e-5)):
        plain = oracle.refine_scores(L, S, W, TAU, 0.1, f)
        r = oracle.refine_scores(L, S, W, TAU, 0.1, f, radius=radius, gamma=0.25, delta=delta)
        n_scaled = 0
        for h in range(4):
            for i in range(n):
                v = plain[h, i]
                nb = [plain[h, j] for j in range(max(0, i - radius), min(n, i + radius + 1))
                      if j != i]
                hit = any(w > v and (delta == 0.0 or np.float32(w - v) <= np.float32(delta))
                          for w in nb)
                n_scaled += hit
                assert r[h, i] == (np.float32(0.25) * v if hit else v)
        assert 0 < n_scaled < 4 * n


def test_exclusivity_identical_heads_keep_each_ranking():
    f = evidence4()
    same = np.repeat(f[:1], 4, axis=0)
    r = oracle.refine_scores(L, S, W, TAU, 0.0, same, mu=0.5)
    base = oracle.fused_scores(L, S, W, TAU, 0.0, f[0])
    # every head is scaled by the same (1 - mu): selections unchanged
    for h in range(4):
        np.testing.assert_allclose(r[h], 0.5 * base, rtol=3e-7)
        np.testing.assert_array_equal(oracle.topk(r[h], 100), oracle.topk(base, 100))


def test_exclusivity_penalises_shared_positions():
    f = evidence4()
    g = f.copy()
    g[:, 200] = g.max() * 2          # every head loves position 200
    g[0, 300] = g.max() * 2          # only head 0 loves position 300
    r = oracle.refine_scores(L, S, W, TAU, 0.0, g, mu=0.9)
    assert r[0, 300 - S] > r[0, 200 - S]   # the exclusive position now outranks the shared one


def test_key_norm_prior_term():
    f = evidence4()
    norms = np.full((4, L), 10.0, np.float32)
    r0 = oracle.refine_scores(L, S, W, TAU, 1.0, f)
    r1 = oracle.refine_scores(L, S, W, TAU, 1.0, f, nu=12.0, knorm=norms)   # all below nu
    np.testing.assert_array_equal(r0, r1)
    norms[:, 100] = 24.0                                                     # twice nu
    r2 = oracle.refine_scores(L, S, W, TAU, 1.0, f, nu=12.0, knorm=norms)
    np.testing.assert_array_equal(r2[:, 100 - S], np.float32(0.5) * r0[:, 100 - S])


def test_geometric_mixture_lambda0_ranks_by_evidence():
    f = evidence4()
    r = oracle.refine_scores(L, S, W, TAU, 0.0, f, geometric=True)
    for h in range(4):
        cand = f[h, S:L - W]
        np.testing.assert_allclose(r[h], np.log2(cand.astype(np.float64)), rtol=3e-7, atol=3e-7)
        # distinct evidence values keep their order
        order = np.argsort(-cand, kind="stable")[:50]
        assert np.all(np.diff(r[h][order]) <= 0)


def test_geometric_mixture_is_log_linear():
    f = evidence4()
    lam = 0.3
    r = oracle.refine_scores(L, S, W, TAU, lam, f, geometric=True)
    n = L - W - S
    d = (L - W) - np.arange(S, L - W)
    prior = np.minimum(1.0, d / TAU)
    prior /= prior.sum()
    ref = (1 - lam) * np.log2(f[:, S:L - W].astype(np.float64)) + lam * np.log2(prior)[None]
    np.testing.assert_allclose(r, ref, rtol=2e-6, atol=2e-5)
    assert r.shape == (4, n)


def test_key_norms_match_library_norm():
    rng = np.random.default_rng(4)
    k = gen.f32_to_bf16((rng.standard_normal((300, 128)) * 2).astype(np.float32))
    got = oracle.key_norms(k)
    ref = np.linalg.norm(gen.bf16_to_f32(k).astype(np.float64), axis=1)
    np.testing.assert_allclose(got, ref, rtol=1e-6)
