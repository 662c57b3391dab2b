"""fp64 CPU oracle for ParisKV approximate retrieval (test infrastructure only).

TEST INFRASTRUCTURE ONLY, like the rest of this package: the test suite, the
package's smoke check and the benchmark's CPU legs may import it; the product path
never does.  It shares no code with the CUDA library.

ParisKV notes (cc.laoqi.cc, arXiv 2602.07721), §2 "method": the GPU keeps, per key,
a direction-centroid id, a 4-bit direction code and correction weights; a decode
step votes with the centroids (collision stage), keeps about beta * n candidates,
re-scores them from the codes (rerank) and fetches the full rows of the final
top-k.  Steps, in the pages' order:

  encode     k_hat = k / |k|, k_tilde = R k_hat with R an SRHT rotation shared with
             the query (§2.2); D splits into B subspaces of m dims; per subspace
             r = |k_tilde_b|, u = k_tilde_b / r; the fixed centroids are the 2^m
             sign patterns (+-1/sqrt m)^m and the key stores the one maximising
             <u, omega> (§2.2, Eqs. (5)-(6)); every coordinate of u is coded with
             1 sign bit and 3 magnitude bits from a Lloyd-Max quantiser designed for
             the magnitude of one coordinate of a random unit vector, whose square
             is Beta(1/2, (m-1)/2) (§2.4, Prop. 4.1); v = the decoded direction,
             alpha = <v, u>, w = |k| r / alpha (§2.4, Eqs. (7)-(12)).
  collision  per subspace the keys whose centroid is most similar to the query's
             subvector take integer weights 6..1 by tier, the tiers cutting the top
             rho fraction at 5/15/30/50/75/100 % (§2.3, Eq. (15)); S_i sums them.
  candidates the ceil(beta n) keys of largest S (§2.3, "bucket top-k").
  rerank     s_hat_i = |q| sum_b w_ib <v_ib, q_tilde_b> (§2.4).
  final      the exact top-k of s_hat over the candidates, then attention over
             sink U selected U local as in the exact path (§2.5).

Readings where the pages leave a step open (each also stated where it is used):
  - GQA: one retrieval query per KV head, the mean of the group's query heads (the
    exact path's reading); |q| is that mean's norm.
  - R = H_D diag(sigma) / sqrt(D): H_D the Sylvester Walsh-Hadamard matrix, sigma
    random signs passed in by the caller, no subsampling (D -> D).
  - centroid id: bit j set iff u_j < 0 (a zero coordinate counts as positive).
  - a tier is decided per centroid: the centroids of a subspace are ranked by
    similarity <q_tilde_b, omega> (ties: lower id); with N = ceil(rho n) and cuts
    e_l = ceil(P_l N / 100) for P = 5, 15, 30, 50, 75, 100, a centroid preceded by
    `start` keys (in better-ranked centroids) gets weight 6 - l for the first l with
    start < e_l, and 0 when start >= N: whole centroids, as a histogram and a
    prefix scan over centroids decide it.  n counts the row's candidate region.
  - beta and rho are given in per-mille; C = ceil(beta n / 1000), ties in S go to
    the lower position (the exact path's tie rule).
  - magnitude cell of |u_j|: the number of thresholds t_i <= |u_j| (a value on a
    threshold goes up).
  - zero vectors: |k| = 0 or r = 0 gives w = 0 (its code is all-positive, cell 0).
  - m = 8 and B = 16 for D = 128 (the notes flag the appendix's D = 256, B = 16,
    m = 8 as inconsistent; only D = B m is used).
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import numpy as np

from .skv_oracle import as_f64, attended_positions, attention, exact_topk, regions

TIER_PCT = (5, 15, 30, 50, 75, 100)
TIER_WEIGHTS = (6, 5, 4, 3, 2, 1)
N_LEVELS = 8  # 3 magnitude bits


@dataclass
class ParisParams:
    m: int = 8              # subspace dimension
    beta_pm: int = 50       # candidates: beta in per-mille of the candidate region
    rho_pm: int = 100       # collision: top rho (per-mille) per subspace; rho >= beta


# --------------------------------------------------------------------------------------
# Lloyd-Max magnitude quantiser (ParisKV notes §2.4, Prop. 4.1)
# --------------------------------------------------------------------------------------


def magnitude_density(x: np.ndarray, m: int) -> np.ndarray:
    """Unnormalised density of |u_j| for a uniformly random unit vector u in R^m.

    u_j^2 ~ Beta(1/2, (m-1)/2) gives, for x = |u_j| in [0, 1], a density proportional
    to (1 - x^2)^((m-3)/2)."""
    return np.power(np.clip(1.0 - np.asarray(x, dtype=np.float64) ** 2, 0.0, None), (m - 3) / 2.0)


def lloyd_max(m: int, n_levels: int = N_LEVELS, grid: int = 400001, tol: float = 1e-14, max_iter: int = 100000):
    """Lloyd-Max quantiser of |u_j| on [0, 1]: returns (levels [n_levels], thresholds [n_levels - 1]).

    Lloyd's iteration: every threshold is the midpoint of its two levels, every level
    the mean of the density over its cell.  The cell integrals come from cumulative
    trapezoid sums on a uniform grid, interpolated linearly.  Needs m >= 3 (for m = 2
    the density is unbounded at 1)."""
    if m < 3:
        raise ValueError("m >= 3")
    x = np.linspace(0.0, 1.0, grid)
    f = magnitude_density(x, m)
    dx = x[1] - x[0]
    c0 = np.concatenate([[0.0], np.cumsum((f[1:] + f[:-1]) * 0.5 * dx)])          # int f
    xf = x * f
    c1 = np.concatenate([[0.0], np.cumsum((xf[1:] + xf[:-1]) * 0.5 * dx)])        # int x f
    levels = (np.arange(n_levels) + 0.5) / n_levels
    for _ in range(max_iter):
        thr = 0.5 * (levels[1:] + levels[:-1])
        edges = np.concatenate([[0.0], thr, [1.0]])
        m0 = np.interp(edges, x, c0)
        m1 = np.interp(edges, x, c1)
        new = (m1[1:] - m1[:-1]) / (m0[1:] - m0[:-1])
        if np.max(np.abs(new - levels)) < tol:
            levels = new
            break
        levels = new
    return levels, 0.5 * (levels[1:] + levels[:-1])


# --------------------------------------------------------------------------------------
# SRHT rotation (ParisKV notes §2.2)
# --------------------------------------------------------------------------------------


def walsh_hadamard(D: int) -> np.ndarray:
    """Sylvester Walsh-Hadamard matrix of order D (a power of two), entries +-1."""
    if D < 1 or D & (D - 1):
        raise ValueError("D must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < D:
        h = np.block([[h, h], [h, -h]])
    return h


def srht_matrix(signs: np.ndarray) -> np.ndarray:
    """R = H_D diag(sigma) / sqrt(D) (orthogonal)."""
    s = np.asarray(signs, dtype=np.float64)
    D = s.shape[0]
    return walsh_hadamard(D) * s[None, :] / math.sqrt(D)


def rotate(x: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """R x for x [..., D]."""
    return as_f64(x) @ srht_matrix(signs).T


def unit(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """(x / |x|, |x|) along the last axis; a zero vector stays zero."""
    x = np.asarray(x, dtype=np.float64)
    n = np.sqrt(np.sum(x * x, axis=-1))
    safe = np.where(n > 0.0, n, 1.0)
    return np.where((n > 0.0)[..., None], x / safe[..., None], 0.0), n


# --------------------------------------------------------------------------------------
# encode (prefill side): centroid ids, 4-bit codes, weights (ParisKV notes §2.2, §2.4)
# --------------------------------------------------------------------------------------


def centroid_vectors(m: int) -> np.ndarray:
    """The 2^m fixed centroids, row c: coordinate j = -1/sqrt m if bit j of c is set, else +1/sqrt m."""
    c = np.arange(1 << m)[:, None]
    bits = (c >> np.arange(m)[None, :]) & 1
    return np.where(bits == 1, -1.0, 1.0) / math.sqrt(m)


def encode(keys: np.ndarray, signs: np.ndarray, m: int, levels: np.ndarray, thresholds: np.ndarray) -> dict:
    """Index metadata of keys [n, D]: cent [n, B] (uint8 when m <= 8), code [n, B] (uint32,
    nibble j = sign bit << 3 | magnitude cell of coordinate j), w [n, B], and the
    intermediates r [n, B], u [n, B, m], v [n, B, m], alpha [n, B], norm [n]."""
    k = as_f64(keys)
    n, D = k.shape
    if D % m:
        raise ValueError("m must divide D")
    B = D // m
    khat, kn = unit(k)
    kt = rotate(khat, signs).reshape(n, B, m)
    u, r = unit(kt)
    neg = u < 0.0
    cell = np.searchsorted(np.asarray(thresholds, dtype=np.float64), np.abs(u), side="right")
    v = np.where(neg, -1.0, 1.0) * np.asarray(levels, dtype=np.float64)[cell]
    alpha = np.sum(v * u, axis=-1)
    ok = (r > 0.0) & (kn[:, None] > 0.0)
    w = np.where(ok, kn[:, None] * r / np.where(ok, alpha, 1.0), 0.0)
    pw = 1 << np.arange(m)
    cent = (neg.astype(np.int64) * pw).sum(axis=-1)
    nib = (neg.astype(np.int64) << 3) | cell
    code = (nib << (4 * np.arange(m))).sum(axis=-1)
    return dict(cent=cent, code=code, w=w, r=r, u=u, v=v, alpha=alpha, norm=kn)


def decode_code(code: np.ndarray, m: int, levels: np.ndarray) -> np.ndarray:
    """The direction v [..., m] a code word [...] stands for."""
    c = np.asarray(code, dtype=np.int64)[..., None] >> (4 * np.arange(m))
    nib = c & 15
    return np.where(nib & 8, -1.0, 1.0) * np.asarray(levels, dtype=np.float64)[nib & 7]


# --------------------------------------------------------------------------------------
# decode step: query, collision, candidates, rerank (ParisKV notes §2.3, §2.4)
# --------------------------------------------------------------------------------------


def retrieval_query(q_group: np.ndarray, signs: np.ndarray) -> tuple[np.ndarray, float]:
    """(q_tilde [D], |q|) of a KV head's retrieval query, the mean of its group's heads."""
    qb = np.mean(as_f64(q_group), axis=0)
    qh, nq = unit(qb)
    return rotate(qh, signs), float(nq)


def centroid_similarity(q_tilde: np.ndarray, m: int) -> np.ndarray:
    """sim [B, 2^m]: <q_tilde_b, omega_c> for every subspace and centroid (fp64)."""
    qt = np.asarray(q_tilde, dtype=np.float64).reshape(-1, m)
    return qt @ centroid_vectors(m).T


def tier_cuts(n: int, rho_pm: int) -> tuple[int, list[int]]:
    """(N, cuts): N = ceil(rho n / 1000) keys in T_b(rho); cut l = ceil(P_l N / 100)."""
    N = (rho_pm * n + 999) // 1000
    return N, [(p * N + 99) // 100 for p in TIER_PCT]


def collision_weights(sim: np.ndarray, counts: np.ndarray, n: int, rho_pm: int) -> np.ndarray:
    """W [B, 2^m] (integers): the weight a key with centroid c earns in subspace b.

    Centroids are ranked by (similarity desc, id asc); `start` counts the keys in
    better-ranked centroids; the tier is the first cut above start (whole centroids)."""
    Bn, nc = sim.shape
    N, cuts = tier_cuts(n, rho_pm)
    W = np.zeros((Bn, nc), dtype=np.int64)
    for b in range(Bn):
        order = np.lexsort((np.arange(nc), -sim[b]))
        start = 0
        for c in order:
            if start < N:
                lvl = next(i for i, e in enumerate(cuts) if start < e)
                W[b, c] = TIER_WEIGHTS[lvl]
            start += int(counts[b, c])
    return W


def collision_scores(cent: np.ndarray, W: np.ndarray) -> np.ndarray:
    """S_i = sum_b W[b, cent[i, b]] (Eq. (15))."""
    cent = np.asarray(cent, dtype=np.int64)
    return W[np.arange(W.shape[0])[None, :], cent].sum(axis=1)


def rerank_scores(q_tilde: np.ndarray, nq: float, w: np.ndarray, v: np.ndarray) -> np.ndarray:
    """s_hat_i = |q| sum_b w_ib <v_ib, q_tilde_b> for w [n, B], v [n, B, m]."""
    B, m = v.shape[-2], v.shape[-1]
    qt = np.asarray(q_tilde, dtype=np.float64).reshape(B, m)
    return nq * np.sum(np.asarray(w, dtype=np.float64) * np.einsum("nbj,bj->nb", v, qt), axis=1)


def paris_select(meta: dict, positions: np.ndarray, q_tilde: np.ndarray, nq: float, k: int, params: ParisParams,
                 levels: np.ndarray, given_rerank: Optional[np.ndarray] = None,
                 given_sim: Optional[np.ndarray] = None) -> dict:
    """Collision, candidates, rerank and the final top-k over the candidate positions.

    meta: encode() output over the row's positions [0, L); positions: the candidate
    region.  given_rerank (indexed by position, optional): rerank scores used for
    the final top-k instead of the fp64 ones (the final selection's check on the
    GPU's own fp32 scores).  given_sim ([B, 2^m], optional): centroid similarities
    the tiers are ranked by instead of the fp64 ones (the integer stages' check on
    the GPU's own similarities); the ranking itself is the same lexsort either way."""
    m = params.m
    pos = np.asarray(positions, dtype=np.int64)
    n = len(pos)
    cent = np.asarray(meta["cent"])[pos]
    B = cent.shape[1]
    counts = np.zeros((B, 1 << m), dtype=np.int64)
    for b in range(B):
        counts[b] = np.bincount(cent[:, b], minlength=1 << m)
    sim = centroid_similarity(q_tilde, m) if given_sim is None else np.asarray(given_sim, dtype=np.float64)
    W = collision_weights(sim, counts, n, params.rho_pm)
    S = collision_scores(cent, W)
    C = (params.beta_pm * n + 999) // 1000
    cand = exact_topk(S.astype(np.float64), pos, C)
    v = decode_code(np.asarray(meta["code"])[cand], m, levels)
    sh = rerank_scores(q_tilde, nq, np.asarray(meta["w"])[cand], v)
    rank_on = sh if given_rerank is None else np.asarray(given_rerank, dtype=np.float64)[cand]
    idx = exact_topk(rank_on, cand, k)
    return dict(counts=counts, sim=sim, W=W, S=S, cand=cand, rerank=sh, idx=idx)


def paris_decode_unit(prob, b: int, h: int, q: np.ndarray, kpool, vpool, meta: dict, signs: np.ndarray,
                      params: ParisParams, levels: np.ndarray, given_q_tilde: Optional[np.ndarray] = None,
                      given_rerank: Optional[np.ndarray] = None, given_idx: Optional[np.ndarray] = None) -> dict:
    """All ParisKV steps for (request b, KV head h), then attention over sink U selected U local.

    q: [B, Hq, D] attention queries (the group mean is the retrieval query);
    meta: encode() of this row's keys over positions [0, L).  given_q_tilde /
    given_rerank / given_idx replace the fp64 rotated query, rerank scores or
    selection (the checks that take a decision in the GPU's precision)."""
    L = int(prob.seq_lens[b])
    G = prob.group
    s_end, l_start = regions(L, prob.n_sink, prob.n_local)
    cand_pos = np.arange(s_end, l_start, dtype=np.int64)
    qg = np.asarray(q)[b, h * G:(h + 1) * G]
    qt, nq = retrieval_query(qg, signs)
    if given_q_tilde is not None:
        qt = np.asarray(given_q_tilde, dtype=np.float64)
    res = paris_select(meta, cand_pos, qt, nq, prob.topk, params, levels, given_rerank)
    res["q_tilde"], res["nq"] = qt, nq
    sel = res["idx"] if given_idx is None else np.asarray(given_idx, dtype=np.int64)
    att = attended_positions(L, prob.n_sink, prob.n_local, sel)
    K = kpool.rows(b, h, att)[:, : prob.d_qk]
    V = K[:, : prob.d_v] if vpool is None else vpool.rows(b, h, att)[:, : prob.d_v]
    o, lse = attention(qg, K, V, prob.scale())
    res.update(out=o, lse=lse, attended=att)
    return res
