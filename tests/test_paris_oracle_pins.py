"""Pins for the ParisKV retrieval oracle (ParisKV notes, §2.2-§2.4): each function is tied
to a closed form, a library routine, brute force, or a hand-worked example."""

import math

import numpy as np
import pytest

from oracle import paris_oracle as po
from oracle import exact_topk


def test_lloyd_max_m3_is_the_uniform_quantiser():
    # m = 3: u_j^2 ~ Beta(1/2, 1), so |u_j| is uniform on [0, 1] and the 8-level
    # Lloyd-Max quantiser is the uniform one: levels (2i + 1) / 16, cuts i / 8
    lv, th = po.lloyd_max(3)
    np.testing.assert_allclose(lv, (2 * np.arange(8) + 1) / 16, atol=1e-9)
    np.testing.assert_allclose(th, np.arange(1, 8) / 8, atol=1e-9)


def test_magnitude_density_matches_the_beta_law():
    stats = pytest.importorskip("scipy.stats")
    integrate = pytest.importorskip("scipy.integrate")
    for m in (3, 5, 8, 16):
        z = integrate.quad(lambda x: po.magnitude_density(x, m), 0, 1)[0]
        for t in (0.1, 0.35, 0.7, 0.95):
            p = integrate.quad(lambda x: po.magnitude_density(x, m), 0, t)[0] / z
            # P(|u_j| <= t) = P(u_j^2 <= t^2) with u_j^2 ~ Beta(1/2, (m - 1)/2)
            assert p == pytest.approx(stats.beta.cdf(t * t, 0.5, (m - 1) / 2), abs=1e-9)


def test_lloyd_max_m8_satisfies_the_optimality_conditions():
    integrate = pytest.importorskip("scipy.integrate")
    m = 8
    lv, th = po.lloyd_max(m)
    f = lambda x: po.magnitude_density(x, m)  # noqa: E731
    edges = np.concatenate([[0.0], th, [1.0]])
    for i in range(8):
        a, b = edges[i], edges[i + 1]
        mass = integrate.quad(f, a, b, epsabs=1e-14)[0]
        mean = integrate.quad(lambda x: x * f(x), a, b, epsabs=1e-14)[0] / mass
        assert lv[i] == pytest.approx(mean, abs=1e-7)        # every level is its cell's mean
    np.testing.assert_allclose(th, 0.5 * (lv[1:] + lv[:-1]), atol=1e-15)  # every cut a midpoint
    assert np.all(np.diff(lv) > 0) and 0 < lv[0] and lv[-1] < 1

    def distortion(levels, cuts):
        e = np.concatenate([[0.0], cuts, [1.0]])
        return sum(integrate.quad(lambda x: (x - levels[i]) ** 2 * f(x), e[i], e[i + 1])[0] for i in range(8))

    uni = (2 * np.arange(8) + 1) / 16
    assert distortion(lv, th) < distortion(uni, np.arange(1, 8) / 8)


def test_srht_is_the_signed_hadamard_rotation():
    linalg = pytest.importorskip("scipy.linalg")
    rng = np.random.default_rng(5)
    for D in (8, 128):
        s = rng.choice([-1.0, 1.0], size=D)
        R = po.srht_matrix(s)
        np.testing.assert_array_equal(R * math.sqrt(D), linalg.hadamard(D) * s[None, :])
        np.testing.assert_allclose(R.T @ R, np.eye(D), atol=1e-12)
        x = rng.standard_normal((3, D))
        np.testing.assert_allclose(po.rotate(x, s), x @ R.T, atol=1e-12)
        # inner products survive the rotation
        np.testing.assert_allclose(po.rotate(x, s) @ po.rotate(x, s).T, x @ x.T, atol=1e-10)


def test_centroid_is_the_brute_force_argmax_and_the_pages_cube_example():
    rng = np.random.default_rng(9)
    for m in (4, 8):  # D = m, a power of two for the rotation
        om = po.centroid_vectors(m)
        assert om.shape == (1 << m, m)
        np.testing.assert_allclose(np.linalg.norm(om, axis=1), 1.0)
        keys = rng.standard_normal((200, m))
        meta = po.encode(keys, np.ones(m), m, *po.lloyd_max(3))
        # D = m: one subspace, identity-free check through the rotated direction u
        u = meta["u"][:, 0]
        np.testing.assert_array_equal(meta["cent"][:, 0], np.argmax(u @ om.T, axis=1))
    # the cube of m = 3: a direction with signs (+, +, -) falls on the centroid with bit 2 set
    u = np.array([0.5, 0.3, -0.8])
    assert int(np.argmax(po.centroid_vectors(3) @ u)) == 0b100


def test_unquantised_estimate_is_the_exact_inner_product():
    rng = np.random.default_rng(3)
    D, m = 128, 8
    s = rng.choice([-1.0, 1.0], size=D)
    keys = rng.standard_normal((64, D))
    q = rng.standard_normal((4, D))
    meta = po.encode(keys, s, m, *po.lloyd_max(m))
    qt, nq = po.retrieval_query(q, s)
    # with v = u (alpha = 1) the weights are |k| r and the estimate is <k, q_bar> exactly
    est = po.rerank_scores(qt, nq, meta["norm"][:, None] * meta["r"], meta["u"])
    np.testing.assert_allclose(est, keys @ q.mean(axis=0), rtol=1e-10, atol=1e-10)


def test_quantised_estimate_tracks_the_inner_product():
    rng = np.random.default_rng(4)
    D, m = 128, 8
    s = rng.choice([-1.0, 1.0], size=D)
    lv, th = po.lloyd_max(m)
    keys = rng.standard_normal((4000, D)) * rng.uniform(0.5, 2.0, size=(4000, 1))
    q = rng.standard_normal((8, D))
    meta = po.encode(keys, s, m, lv, th)
    np.testing.assert_allclose(po.decode_code(meta["code"], m, lv), meta["v"])
    assert np.all(meta["alpha"] > 0)
    # the centroid id is the code's sign bits
    signs = np.stack([(meta["code"] >> (4 * j + 3)) & 1 for j in range(m)], axis=-1)
    np.testing.assert_array_equal(meta["cent"], (signs << np.arange(m)).sum(axis=-1))
    qt, nq = po.retrieval_query(q, s)
    est = po.rerank_scores(qt, nq, meta["w"], meta["v"])
    exact = keys @ q.mean(axis=0)
    assert np.corrcoef(est, exact)[0, 1] > 0.97
    assert np.median(np.abs(est - exact)) < 0.2 * np.std(exact)


def test_collision_weights_hand_example():
    # one subspace of m = 3, q_tilde = (0.9, 0.3, 0.1): the centroids rank 0, 4, 2, 6, 1, 5, 3, 7
    sim = po.centroid_similarity(np.array([0.9, 0.3, 0.1]), 3)
    assert list(np.lexsort((np.arange(8), -sim[0]))) == [0, 4, 2, 6, 1, 5, 3, 7]
    counts = np.array([[3, 2, 4, 1, 5, 2, 2, 1]])  # n = 20 keys
    # rho = 50 %: N = 10 keys, cuts ceil(5 %, 15 %, 30 %, 50 %, 75 %, 100 % of 10) = 1, 2, 3, 5, 8, 10
    assert po.tier_cuts(20, 500) == (10, [1, 2, 3, 5, 8, 10])
    W = po.collision_weights(sim, counts, 20, 500)
    # centroid 0 starts at 0 (tier 1: weight 6); 4 at 3 (first cut above: 5, weight 3);
    # 2 at 8 (cut 10: weight 1); 6 starts at 12 >= N: nothing from there on
    np.testing.assert_array_equal(W[0], [6, 0, 1, 0, 3, 0, 0, 0])


def test_collision_scores_match_a_per_key_brute_force():
    rng = np.random.default_rng(11)
    m, B, n = 3, 2, 60
    cent = rng.integers(0, 8, size=(n, B))
    qt = rng.standard_normal(B * m)
    sim = po.centroid_similarity(qt, m)
    counts = np.stack([np.bincount(cent[:, b], minlength=8) for b in range(B)])
    for rho_pm in (100, 333, 1000):
        W = po.collision_weights(sim, counts, n, rho_pm)
        S = po.collision_scores(cent, W)
        N, cuts = po.tier_cuts(n, rho_pm)
        for i in range(n):
            want = 0
            for b in range(B):
                ci = cent[i, b]
                better = lambda c: sim[b, c] > sim[b, ci] or (sim[b, c] == sim[b, ci] and c < ci)  # noqa: E731
                start = sum(1 for j in range(n) if better(cent[j, b]))
                if start < N:
                    want += (6, 5, 4, 3, 2, 1)[next(t for t, e in enumerate(cuts) if start < e)]
            assert S[i] == want


def test_candidates_and_final_selection_follow_the_tie_rules():
    rng = np.random.default_rng(12)
    D, m = 128, 8
    s = rng.choice([-1.0, 1.0], size=D)
    lv, th = po.lloyd_max(m)
    keys = rng.standard_normal((3000, D))
    meta = po.encode(keys, s, m, lv, th)
    q = rng.standard_normal((2, D))
    qt, nq = po.retrieval_query(q, s)
    pos = np.arange(10, 2900)
    params = po.ParisParams(m=m, beta_pm=50, rho_pm=100)
    r = po.paris_select(meta, pos, qt, nq, 20, params, lv)
    n = len(pos)
    assert len(r["cand"]) == (50 * n + 999) // 1000
    S = dict(zip(pos.tolist(), r["S"].tolist()))
    order = sorted(pos.tolist(), key=lambda t: (-S[t], t))
    assert sorted(r["cand"].tolist()) == sorted(order[: len(r["cand"])])
    sh = dict(zip(r["cand"].tolist(), r["rerank"].tolist()))
    best = sorted(sh, key=lambda t: (-sh[t], t))[:20]
    assert r["idx"].tolist() == sorted(best)


def test_planted_keys_are_retrieved():
    rng = np.random.default_rng(13)
    D, m, n = 128, 8, 20000
    s = rng.choice([-1.0, 1.0], size=D)
    lv, th = po.lloyd_max(m)
    q = rng.standard_normal((4, D))
    qbar = q.mean(axis=0)
    keys = rng.standard_normal((n, D))
    planted = rng.choice(n, size=30, replace=False)
    keys[planted] = 0.3 * keys[planted] + 4.0 * qbar / np.linalg.norm(qbar)
    meta = po.encode(keys, s, m, lv, th)
    qt, nq = po.retrieval_query(q, s)
    r = po.paris_select(meta, np.arange(n), qt, nq, 100, po.ParisParams(m=m), lv)
    assert set(planted.tolist()) <= set(r["cand"].tolist())
    assert set(planted.tolist()) <= set(r["idx"].tolist())
    # and about half of the exact top-100 or more: the method is approximate (the notes
    # report a final Recall@100 near 64 % on a real decode trajectory, §4.4 / Fig. 10)
    exact = set(exact_topk(keys @ qbar, np.arange(n), 100).tolist())
    assert len(exact & set(r["idx"].tolist())) >= 50


def test_centroid_similarity_closed_forms():
    # ParisKV notes §2.2: the centroids are the sign patterns (+-1/sqrt m)^m.  The most
    # similar centroid of a subvector is its own sign pattern, with similarity |q_b|_1 / sqrt m;
    # antipodal centroids (all bits flipped) have opposite similarities; and a centroid
    # differing from the best one in bit j loses exactly 2 |q_bj| / sqrt m.
    rng = np.random.default_rng(14)
    m = 8
    qt = rng.standard_normal(128)
    sim = po.centroid_similarity(qt, m)
    qb = qt.reshape(16, m)
    for b in range(16):
        best = int(np.sum((qb[b] < 0) << np.arange(m)))
        assert int(np.argmax(sim[b])) == best
        assert sim[b, best] == pytest.approx(np.abs(qb[b]).sum() / np.sqrt(m), rel=1e-12)
        np.testing.assert_allclose(sim[b], -sim[b, np.arange(256) ^ 255], atol=1e-12)
        for j in range(m):
            assert sim[b, best ^ (1 << j)] == pytest.approx(sim[b, best] - 2 * abs(qb[b, j]) / np.sqrt(m), abs=1e-12)


def test_given_similarities_rank_the_tiers():
    # the integer stages take the similarities they are given and rank them with the same
    # lexsort: the fp64 values reproduce the plain call, and swapping the values of the two
    # best centroids of a subspace swaps their tier weights
    rng = np.random.default_rng(15)
    m, n = 8, 3000
    keys = rng.standard_normal((n, 128))
    s = np.where(rng.random(128) < 0.5, -1.0, 1.0)
    lv, th = po.lloyd_max(m)
    meta = po.encode(keys, s, m, lv, th)
    qt, nq = po.retrieval_query(rng.standard_normal((2, 128)), s)
    params = po.ParisParams(m=m, beta_pm=50, rho_pm=100)
    plain = po.paris_select(meta, np.arange(n), qt, nq, 50, params, lv)
    same = po.paris_select(meta, np.arange(n), qt, nq, 50, params, lv, given_sim=po.centroid_similarity(qt, m))
    for key in ("W", "S", "cand", "idx"):
        np.testing.assert_array_equal(plain[key], same[key])
    sim = po.centroid_similarity(qt, m)
    o = np.lexsort((np.arange(256), -sim[0]))
    c1, c2 = int(o[0]), int(o[1])
    swapped = sim.copy()
    swapped[0, c1], swapped[0, c2] = sim[0, c2], sim[0, c1]
    r = po.paris_select(meta, np.arange(n), qt, nq, 50, params, lv, given_sim=swapped)
    counts = plain["counts"][0]
    if counts[c1] > 0 and counts[c2] > 0:
        assert r["W"][0, c2] == plain["W"][0, c1]  # c2 now ranks first, so it takes the first tier
    np.testing.assert_array_equal(r["W"][1:], plain["W"][1:])
