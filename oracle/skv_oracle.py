"""Plain fp64 CPU oracle for one sparse-decode step over an indirectly addressed KV pool.

TEST INFRASTRUCTURE ONLY. This module is the independent reference that the CUDA
path is checked against. Only the test suite, the package's smoke check and the
CPU-baseline leg of the benchmark may import it; the product path never does.
It shares no code with the CUDA library and imports nothing from it.

What it computes, per (request b, KV head h), in the pages' order:

  S0  group query   q_bar = mean of the scoring query heads of the group.
      (Per-KV-head ranking: OasisKV notes, §3.2 "compressed key summaries" --
      every KV head ranks the whole context on its own.  Reading: the G query
      heads of a GQA group are folded by their mean, which orders keys exactly
      like their sum.  A second reading, selectable per problem: each key
      scores its largest logit over the group's heads -- `group_scores`.  A
      third: every query head selects for itself -- `decode_head`.)
  S1  score         s_t = <q_bar, key_t> for every candidate position t
      (ParisKV notes, §1 "motivation and retrieval objective", Eqs. (1)-(3):
      s_i = <k_i, q>; ECHO-OSDI26 wiki, core method 3: the indexer scores every
      history key before the exact top-k.)
  S2  exact top-k   the k largest scores, ties to the lower position, reported
      in ascending position (ECHO-OSDI26 wiki, core method 3: the k-th score is
      a threshold; everything above it is in the top-k).
  S3  resolve       slot = table[t // bs]; >= 0 reads the GPU pool, < 0 reads
      host block (-slot - 1), row offset t % bs (vToken notes, §3.4 Eq. (2):
      slot = block_id * S + offset; UlaCache article §5: one logical address,
      the map says which tier holds it).
  S4  attention     softmax attention of every query head of the group over
      sink U selected U local (ParisKV notes, §2.5 "online window": Sink and
      Local are attended densely next to the retrieved set; §1 Eq. (1)-(3)).
  S5  merge         log-sum-exp merge of split partials (split-K decoding; the
      pages name FlashAttention as the dense baseline but print no merge rule --
      the merge here is the plain identity of the softmax normaliser).

Everything is float64.  Inputs stored as bf16 are passed either as float arrays
or as raw uint16 bit patterns (decoded by `bf16_bits_to_f64`).

Parity pins (tests/test_oracle_pins.py) tie every function here to something
other than itself: brute-force subset enumeration, closed forms, a library
attention routine, the pages' worked byte counts, and invariances the pages
state (physical placement does not change results).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import numpy as np

# --------------------------------------------------------------------------------------
# storage decoding
# --------------------------------------------------------------------------------------


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode bf16 bit patterns (uint16/int16) to float64.

    bf16 is the upper half of an IEEE-754 binary32: sign, 8 exponent bits, 7
    mantissa bits.  Shifting the 16 bits into the high half of a 32-bit word
    gives the binary32 with the same value, which widens exactly to binary64.
    """
    b = np.asarray(bits)
    if b.dtype == np.int16:
        b = b.view(np.uint16)
    if b.dtype != np.uint16:
        raise TypeError("bf16 bit patterns must be uint16 or int16")
    w = b.astype(np.uint32) << np.uint32(16)
    return w.view(np.float32).astype(np.float64)


def as_f64(x: np.ndarray) -> np.ndarray:
    """Float64 view of a stored tensor: uint16/int16 arrays are bf16 bit patterns."""
    x = np.asarray(x)
    if x.dtype in (np.uint16, np.int16):
        return bf16_bits_to_f64(x)
    return x.astype(np.float64)


# --------------------------------------------------------------------------------------
# regions of one request (sink / candidates / local)
# --------------------------------------------------------------------------------------


def regions(L: int, n_sink: int, n_local: int) -> tuple[int, int]:
    """Split positions [0, L) into sink [0, s_end), candidates [s_end, l_start), local [l_start, L).

    Sink and Local are attended densely; the retrieval (top-k) region is the rest
    (ParisKV notes, §2.5).  Reading for short histories (L < n_sink + n_local):
    the sink keeps its first min(n_sink, L) positions, the local window never
    reaches back into the sink, and the candidate region may be empty.  The three
    sets are disjoint and cover [0, L).
    """
    if L < 0 or n_sink < 0 or n_local < 0:
        raise ValueError("negative length")
    s_end = min(n_sink, L)
    l_start = max(s_end, L - n_local)
    return s_end, l_start


# --------------------------------------------------------------------------------------
# S0: group query
# --------------------------------------------------------------------------------------


def group_query(q_group: np.ndarray) -> np.ndarray:
    """Mean of the query heads that share one KV head: [G, d] -> [d] (float64)."""
    q = as_f64(q_group)
    if q.ndim != 2 or q.shape[0] < 1:
        raise ValueError("q_group must be [G, d] with G >= 1")
    return q.sum(axis=0) / q.shape[0]


# --------------------------------------------------------------------------------------
# S3: logical -> physical resolution
# --------------------------------------------------------------------------------------


@dataclass
class PagedPool:
    """KV rows addressed through a slot table (vToken notes §3.4 Eq. (2); UlaCache §5).

    gpu / host: arrays [n_blocks, H, block_size, d] (either may be None when that
    tier is unused).  A table entry e >= 0 names GPU block e; e < 0 names host
    block (-e - 1).  With block_size == 1 the table is a per-token map
    (ECHO-OSDI26 wiki, core method 2: HostTokenToGPU-style slot map).
    """

    gpu: Optional[np.ndarray]
    host: Optional[np.ndarray]
    table: np.ndarray  # [B, n_table_entries] int
    block_size: int

    def resolve(self, b: int, t: int) -> tuple[str, int, int]:
        """Return (tier, block, offset) of logical position t of request b."""
        bs = self.block_size
        e = int(self.table[b, t // bs])
        if e >= 0:
            if self.gpu is None or e >= self.gpu.shape[0]:
                raise IndexError(f"GPU block {e} out of range (b={b}, t={t})")
            return "gpu", e, t % bs
        hb = -e - 1
        if self.host is None or hb >= self.host.shape[0]:
            raise IndexError(f"host block {hb} out of range (b={b}, t={t})")
        return "host", hb, t % bs

    def row(self, b: int, h: int, t: int) -> np.ndarray:
        tier, blk, off = self.resolve(b, t)
        src = self.gpu if tier == "gpu" else self.host
        return as_f64(src[blk, h, off])

    def rows(self, b: int, h: int, positions: Sequence[int]) -> np.ndarray:
        """Rows of many positions (float64 [n, d]); the same rule as `resolve`, vectorised."""
        pos = np.asarray(positions, dtype=np.int64)
        d = (self.gpu if self.gpu is not None else self.host).shape[-1]
        out = np.zeros((len(pos), d))
        if len(pos) == 0:
            return out
        bs = self.block_size
        e = np.asarray(self.table[b])[pos // bs].astype(np.int64)
        off = pos % bs
        on_gpu = e >= 0
        if on_gpu.any():
            blk = e[on_gpu]
            if self.gpu is None or blk.max() >= self.gpu.shape[0]:
                raise IndexError(f"GPU block out of range (b={b})")
            out[on_gpu] = as_f64(self.gpu[blk, h, off[on_gpu]])
        on_host = ~on_gpu
        if on_host.any():
            blk = -e[on_host] - 1
            if self.host is None or blk.max() >= self.host.shape[0]:
                raise IndexError(f"host block out of range (b={b})")
            out[on_host] = as_f64(self.host[blk, h, off[on_host]])
        return out


@dataclass
class HeadTablePool:
    """KV rows addressed through one slot-table row per (request, KV head).

    Each KV head keeps its own map from logical blocks to where they live (OasisKV
    notes, §3.5, Fig. 9: a per-head logical-to-logical map, since different heads
    select different blocks).  table [B, H, n_table_entries]: an entry e >= 0 names
    GPU block e, which holds that one head's rows (gpu [n_blocks, block_size, d]);
    e < 0 names host block (-e - 1) of a pool that keeps every head
    (host [n_blocks, H, block_size, d]).
    """

    gpu: Optional[np.ndarray]
    host: Optional[np.ndarray]
    table: np.ndarray  # [B, H, n_table_entries] int
    block_size: int

    def resolve(self, b: int, h: int, t: int) -> tuple[str, int, int]:
        """Return (tier, block, offset) of logical position t of request b, KV head h."""
        bs = self.block_size
        e = int(self.table[b, h, t // bs])
        if e >= 0:
            if self.gpu is None or e >= self.gpu.shape[0]:
                raise IndexError(f"GPU block {e} out of range (b={b}, h={h}, t={t})")
            return "gpu", e, t % bs
        hb = -e - 1
        if self.host is None or hb >= self.host.shape[0]:
            raise IndexError(f"host block {hb} out of range (b={b}, h={h}, t={t})")
        return "host", hb, t % bs

    def row(self, b: int, h: int, t: int) -> np.ndarray:
        tier, blk, off = self.resolve(b, h, t)
        return as_f64(self.gpu[blk, off] if tier == "gpu" else self.host[blk, h, off])

    def rows(self, b: int, h: int, positions: Sequence[int]) -> np.ndarray:
        """Rows of many positions (float64 [n, d]), one `row` at a time."""
        pos = [int(t) for t in positions]
        d = (self.gpu if self.gpu is not None else self.host).shape[-1]
        if not pos:
            return np.zeros((0, d))
        return np.stack([self.row(b, h, t) for t in pos])


# --------------------------------------------------------------------------------------
# S1: scores
# --------------------------------------------------------------------------------------


def scores(q_bar: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """s_t = <q_bar, key_t> (ParisKV notes Eq. (1)); keys [n, d] -> [n] float64."""
    return as_f64(keys) @ as_f64(q_bar)


GROUP_AGGS = ("mean", "max")


def group_scores(q_group: np.ndarray, keys: np.ndarray, agg: str = "mean") -> np.ndarray:
    """S0 + S1 for one KV head: scores of keys [n, d] against the group's query heads [G, d].

    One ranking per KV head (OasisKV notes, §3.2: each KV head ranks the whole
    context on its own).  How the G heads of a group combine is left open by the
    pages; two readings:
      "mean": <q_bar, k_t> with q_bar the mean of the heads (orders keys like the
              sum of the heads' logits);
      "max":  max over the heads g of <q_g, k_t> (a key ranks by its largest logit
              in the group, so a key that any one head weighs heavily is kept).
    """
    if agg == "mean":
        return scores(group_query(q_group), keys)
    if agg == "max":
        q = as_f64(q_group)
        if q.ndim != 2 or q.shape[0] < 1:
            raise ValueError("q_group must be [G, d] with G >= 1")
        k = as_f64(keys)
        if len(k) == 0:
            return np.zeros(0)
        return (k @ q.T).max(axis=1)
    raise ValueError(f"unknown group aggregation {agg!r}")


# --------------------------------------------------------------------------------------
# S2: exact top-k
# --------------------------------------------------------------------------------------


def exact_topk(s: np.ndarray, positions: np.ndarray, k: int) -> np.ndarray:
    """The k largest scores by a full sort; ties go to the lower position.

    s[i] is the score of position positions[i].  The order is: larger score
    first, then lower position.  -0.0 and +0.0 compare equal; a NaN score ranks
    below every number.  Returns the chosen positions in ascending order;
    k >= len(s) returns all of them.
    """
    s = np.asarray(s, dtype=np.float64)
    positions = np.asarray(positions, dtype=np.int64)
    if s.shape != positions.shape:
        raise ValueError("scores and positions differ in shape")
    if k < 0:
        raise ValueError("k < 0")
    nan = np.isnan(s)
    neg = np.where(nan, 0.0, -s)
    # np.lexsort: the LAST key is the primary key.
    order = np.lexsort((positions, neg, nan))
    chosen = positions[order[: min(k, len(s))]]
    return np.sort(chosen)


# --------------------------------------------------------------------------------------
# S4 / S5: attention and the split merge
# --------------------------------------------------------------------------------------


def attention(q_heads: np.ndarray, K: np.ndarray, V: np.ndarray, sm_scale: float):
    """Softmax attention of each query row over the rows of K / V.

    z_{g,j} = sm_scale * <q_g, K_j>,  p = softmax_j(z),  o_g = sum_j p_{g,j} V_j,
    lse_g = log sum_j exp(z_{g,j})  (natural log).  Max-subtracted for range.
    An empty attended set gives o = 0 and lse = -inf.
    """
    q = as_f64(q_heads)
    K = as_f64(K)
    V = as_f64(V)
    G = q.shape[0]
    if K.shape[0] == 0:
        return np.zeros((G, V.shape[1])), np.full(G, -np.inf)
    z = sm_scale * (q @ K.T)  # [G, n]
    m = z.max(axis=1, keepdims=True)
    w = np.exp(z - m)
    l = w.sum(axis=1, keepdims=True)
    o = (w @ V) / l
    lse = (m + np.log(l))[:, 0]
    return o, lse


def attention_partial(q_heads, K, V, sm_scale: float):
    """One split of split-K decoding: (m, l, acc) with acc = sum_j exp(z_j - m) V_j."""
    q = as_f64(q_heads)
    K = as_f64(K)
    V = as_f64(V)
    G = q.shape[0]
    if K.shape[0] == 0:
        return np.full(G, -np.inf), np.zeros(G), np.zeros((G, V.shape[1]))
    z = sm_scale * (q @ K.T)
    m = z.max(axis=1)
    w = np.exp(z - m[:, None])
    return m, w.sum(axis=1), w @ V


def lse_merge(parts):
    """Merge split partials (m_s, l_s, acc_s) into (o, lse).

    lse = m* + log sum_s l_s exp(m_s - m*),  m* = max_s m_s,
    o   = sum_s exp(m_s - lse) acc_s.
    Splits with no rows (m = -inf, l = 0) contribute nothing.
    """
    ms = np.stack([p[0] for p in parts])  # [S, G]
    ls = np.stack([p[1] for p in parts])
    accs = np.stack([p[2] for p in parts])  # [S, G, dv]
    m_star = ms.max(axis=0)
    G = ms.shape[1]
    o = np.zeros((G, accs.shape[2]))
    lse = np.full(G, -np.inf)
    for g in range(G):
        if not np.isfinite(m_star[g]):
            continue
        live = np.isfinite(ms[:, g])
        tot = np.sum(ls[live, g] * np.exp(ms[live, g] - m_star[g]))
        lse[g] = m_star[g] + math.log(tot)
        o[g] = np.sum(np.exp(ms[live, g] - lse[g])[:, None] * accs[live, g], axis=0)
    return o, lse


# --------------------------------------------------------------------------------------
# one decode step
# --------------------------------------------------------------------------------------


@dataclass
class Problem:
    """Sizes of one decode step (mirrors the library's problem descriptor)."""

    batch: int
    n_kv_heads: int
    n_q_heads: int
    d_qk: int
    d_v: int
    topk: int
    n_sink: int
    n_local: int
    block_size: int
    seq_lens: Sequence[int]
    sm_scale: Optional[float] = None
    # scoring source: "paged" scores the K pool through the table with the mean
    # of the q heads; "contig" scores separate index keys [B, H, L, d_idx] with
    # the mean of the index query heads [B, H * G_idx, d_idx].
    index_layout: str = "paged"
    # how the scoring heads of a group combine into one score per key (group_scores)
    group_agg: str = "mean"
    extra: dict = field(default_factory=dict)

    @property
    def group(self) -> int:
        if self.n_q_heads % self.n_kv_heads:
            raise ValueError("n_q_heads must be a multiple of n_kv_heads")
        return self.n_q_heads // self.n_kv_heads

    def scale(self) -> float:
        return self.sm_scale if self.sm_scale is not None else 1.0 / math.sqrt(self.d_qk)


def attended_positions(L: int, n_sink: int, n_local: int, selected) -> np.ndarray:
    """Sink U selected U local, ascending (the three sets are disjoint)."""
    s_end, l_start = regions(L, n_sink, n_local)
    sel = np.asarray(selected, dtype=np.int64)
    return np.concatenate([np.arange(0, s_end), sel, np.arange(l_start, L)]).astype(np.int64)


def decode_unit(
    prob: Problem,
    b: int,
    h: int,
    q: np.ndarray,
    kpool: PagedPool,
    vpool: Optional[PagedPool],
    q_index: Optional[np.ndarray] = None,
    index_keys: Optional[np.ndarray] = None,
    given_scores: Optional[np.ndarray] = None,
    given_idx: Optional[np.ndarray] = None,
):
    """All steps for one (request b, KV head h).

    q:          [B, Hq, d_qk] query (bf16 bits or floats).
    kpool:      K rows through the slot table.
    vpool:      V rows through the slot table; None means the latent layout, where
                V is the first d_v dims of the K row (one shared latent row,
                UlaCache article §3 on MLA; ECHO-OSDI26 wiki, problem and motivation).
    q_index / index_keys: for index_layout == "contig", the scoring query
                [B, H * G_idx, d_idx] and the index keys [B, H, L, d_idx].
    given_scores: if set, float scores over [0, L) used instead of S0/S1 (the
                mode that checks the top-k on the GPU's own fp32 scores).
    given_idx:  if set, the selected positions used instead of S0-S2 (checks
                attention on the GPU's own selection).

    Returns dict(scores over C (positions, values), idx, out [G, d_v], lse [G]).
    """
    L = int(prob.seq_lens[b])
    G = prob.group
    s_end, l_start = regions(L, prob.n_sink, prob.n_local)
    cand = np.arange(s_end, l_start, dtype=np.int64)
    res = {"positions": cand}
    if given_idx is None:
        if given_scores is not None:
            s = np.asarray(given_scores, dtype=np.float64)[cand]
        elif prob.index_layout == "paged":
            s = group_scores(np.asarray(q)[b, h * G:(h + 1) * G], kpool.rows(b, h, cand), prob.group_agg)
        elif prob.index_layout == "contig":
            qi = np.asarray(q_index)[b]
            g_idx = qi.shape[0] // prob.n_kv_heads
            s = group_scores(qi[h * g_idx:(h + 1) * g_idx], np.asarray(index_keys)[b, h, s_end:l_start],
                             prob.group_agg)
        else:
            raise ValueError(prob.index_layout)
        res["scores"] = s
        sel = exact_topk(s, cand, prob.topk)
    else:
        sel = np.asarray(given_idx, dtype=np.int64)
    res["idx"] = sel
    att = attended_positions(L, prob.n_sink, prob.n_local, sel)
    K = kpool.rows(b, h, att)[:, : prob.d_qk]
    if vpool is None:
        V = K[:, : prob.d_v]
    else:
        V = vpool.rows(b, h, att)[:, : prob.d_v]
    qh = np.asarray(q)[b, h * G:(h + 1) * G]
    o, lse = attention(qh, K, V, prob.scale())
    res["out"] = o
    res["lse"] = lse
    res["attended"] = att
    return res


def decode_head(
    prob: Problem,
    b: int,
    j: int,
    q: np.ndarray,
    kpool: PagedPool,
    vpool: Optional[PagedPool],
    q_index: Optional[np.ndarray] = None,
    index_keys: Optional[np.ndarray] = None,
    given_scores: Optional[np.ndarray] = None,
    given_idx: Optional[np.ndarray] = None,
):
    """All steps for one (request b, query head j) under the per-query-head reading.

    Selection is per head (OasisKV notes, §3.5: different KV heads pick different
    blocks, so the map is kept per head); the pages do not say whether "head"
    means the KV head or each query head of its group.  This is the finest
    reading: query head j scores the keys of its KV head h = j // G with its own
    query, s_t = <q[b, j], key_t> (ParisKV notes Eq. (1)), keeps the exact
    top-k of those scores, and attends only its own list.  With G = 1 it is
    `decode_unit` of KV head j.

    Arguments as for `decode_unit`; for index_layout == "contig" q_index is
    [B, Hq, d_idx] (one scoring query per query head).  Returns the same dict,
    with out [1, d_v] and lse [1].
    """
    L = int(prob.seq_lens[b])
    h = j // prob.group
    s_end, l_start = regions(L, prob.n_sink, prob.n_local)
    cand = np.arange(s_end, l_start, dtype=np.int64)
    res = {"positions": cand}
    if given_idx is None:
        if given_scores is not None:
            s = np.asarray(given_scores, dtype=np.float64)[cand]
        elif prob.index_layout == "paged":
            s = scores(as_f64(np.asarray(q)[b, j]), kpool.rows(b, h, cand))
        elif prob.index_layout == "contig":
            s = scores(as_f64(np.asarray(q_index)[b, j]), np.asarray(index_keys)[b, h, s_end:l_start])
        else:
            raise ValueError(prob.index_layout)
        res["scores"] = s
        sel = exact_topk(s, cand, prob.topk)
    else:
        sel = np.asarray(given_idx, dtype=np.int64)
    res["idx"] = sel
    att = attended_positions(L, prob.n_sink, prob.n_local, sel)
    K = kpool.rows(b, h, att)[:, : prob.d_qk]
    V = K[:, : prob.d_v] if vpool is None else vpool.rows(b, h, att)[:, : prob.d_v]
    o, lse = attention(np.asarray(q)[b, j:j + 1], K, V, prob.scale())
    res["out"] = o
    res["lse"] = lse
    res["attended"] = att
    return res


# --------------------------------------------------------------------------------------
# threshold prediction for the prefetch of host rows (ECHO wiki, core method 3)
# --------------------------------------------------------------------------------------
#
# The exact k-th score of a step is a threshold: every key above it is selected.  The
# indexer predicts the next step's threshold with an exponential moving average of the
# k-th scores (the newest weighted alpha = 0.5), and while it scores, the rows of keys
# above the prediction start their host fetch early; a global cap bounds that work so
# the link cannot stall the indexer.  Readings: the prediction is per (request, KV
# head) and undefined (NaN) until a first step has selected; a step that selects
# nothing leaves it as it is; a key qualifies when its score is strictly above the
# prediction and its row lives in the host pool; the cap is per (request, KV head) and
# per step, and which qualifying rows fill it when more qualify is not fixed.


def prefetch_step(tau_prev: float, s: np.ndarray, positions: np.ndarray, on_host: np.ndarray, k: int,
                  alpha: float = 0.5, cap: Optional[int] = None) -> dict:
    """One step of the threshold prediction for one (request, KV head).

    tau_prev: the prediction this step uses (NaN: none yet).  s[i]: score of candidate
    position positions[i]; on_host[i]: its row is in the host pool.  Returns
      eligible  ascending positions of host-resident candidates scoring > tau_prev;
      n_staged  min(len(eligible), cap) (len(eligible) when cap is None);
      kth       the step's k-th largest candidate score under the exact top-k order
                (None when the selection is empty; -0 counts as +0);
      tau       the next prediction: kth when tau_prev is NaN, else
                alpha * kth + (1 - alpha) * tau_prev; tau_prev when nothing is selected.
    """
    s = np.asarray(s, dtype=np.float64)
    positions = np.asarray(positions, dtype=np.int64)
    on_host = np.asarray(on_host, dtype=bool)
    if s.shape != positions.shape or s.shape != on_host.shape:
        raise ValueError("scores, positions and residency differ in shape")
    if not 0.0 < alpha <= 1.0:
        raise ValueError("alpha must be in (0, 1]")
    tau_prev = float(tau_prev)
    if math.isnan(tau_prev):
        eligible = np.zeros(0, dtype=np.int64)
    else:
        eligible = np.sort(positions[on_host & (s > tau_prev)])
    n_staged = len(eligible) if cap is None else min(len(eligible), int(cap))
    sel = exact_topk(s, positions, k)
    if len(sel) == 0:
        return dict(eligible=eligible, n_staged=n_staged, kth=None, tau=tau_prev)
    chosen = s[np.isin(positions, sel)]
    nan = np.isnan(chosen)
    kth = float(np.nan) if nan.any() else float(np.min(chosen)) + 0.0  # + 0.0 turns -0 into +0
    tau = kth if math.isnan(tau_prev) else alpha * kth + (1.0 - alpha) * tau_prev
    return dict(eligible=eligible, n_staged=n_staged, kth=kth, tau=tau)


# --------------------------------------------------------------------------------------
# GPU slot cache over a host pool that backs every token (ECHO wiki, core method 2)
# --------------------------------------------------------------------------------------
#
# The host pool holds the row of token t of request b at b * max_len + t; the GPU
# pool's slots cache some of them.  A slot-table entry >= 0 names a GPU slot, < 0
# the host row -e - 1.  Per slot: its owner (b * max_len + t, or -1 when free) and
# its priority (the last step that used it).  After a step's attended sets are
# known the cache is updated (readings, the pages fixing only the ingredients --
# protect this step's tokens, then free the lowest-priority slots by argtopk):
#   1. every attended token that sits in a GPU slot marks the slot used this step;
#   2. the misses are the attended tokens read from the host, in (request, list
#      position) order;
#   3. the eviction candidates are ranked free first, then by age (step - priority)
#      descending, then by lower slot; the top `budget` of them are chosen (ties to
#      the lower slot), and those not used this step take the misses in ascending
#      slot order, one each, as long as both last;
#   4. a taken slot's old owner returns to its host row in the table; the slot's
#      owner, priority and the miss's table entry are set.


def cache_update(table: np.ndarray, owner: np.ndarray, prio: np.ndarray, step: int, attended, max_len: int,
                 budget: int):
    """One step of the slot cache.  table [B, >= max_len] int; owner, prio [n_slots] int;
    attended[b]: the positions request b attended, in list order.  Returns
    (table, owner, prio, promotions), promotions = [(slot, b, t, j)] with j the
    token's index in attended[b]; the inputs are not modified."""
    table = np.array(table, dtype=np.int64, copy=True)
    owner = np.array(owner, dtype=np.int64, copy=True)
    prio = np.array(prio, dtype=np.int64, copy=True)
    misses = []
    for b, toks in enumerate(attended):
        for j, t in enumerate(toks):
            e = int(table[b, int(t)])
            if e >= 0:
                prio[e] = step
            else:
                misses.append((b, int(t), j))
    n = len(owner)
    age = np.where(owner < 0, np.inf, (step - prio).astype(np.float64))
    score = np.where(prio == step, np.nan, age)
    chosen = exact_topk(score, np.arange(n), budget)
    free_to_take = [int(sl) for sl in chosen if prio[sl] != step]
    promotions = []
    for sl, (b, t, j) in zip(free_to_take, misses):
        old = int(owner[sl])
        if old >= 0:
            table[old // max_len, old % max_len] = -old - 1
        owner[sl] = b * max_len + t
        prio[sl] = step
        table[b, t] = sl
        promotions.append((sl, b, t, j))
    return table, owner, prio, promotions


def cache_update_heads(table: np.ndarray, owner: np.ndarray, prio: np.ndarray, step: int, attended,
                       block_size: int, budget: int):
    """One step of the slot cache over one table row per (request, KV head) (R20's rule on
    blocks, OasisKV notes §3.5: each head keeps its own blocks resident).

    table [B, H, stride] int: e >= 0 a GPU slot holding that head's block, e < 0 the host
    block (-e - 1); the host pool backs block j of request b at host block b * stride + j.
    owner, prio [n_slots] int: a slot's owner is (b * H + h) * stride + j, -1 when free;
    its priority the last step that used it.  attended[b][h]: the positions that (b, h)
    attended, ascending.  A (request, head) uses the distinct blocks of its positions; a
    used block in a slot protects the slot this step, the others are misses, taken in
    (request, head, block) order.  The `budget` best eviction candidates -- free slots,
    then the oldest last use, then the lower slot, as exact_topk ranks them -- in
    ascending slot order, skipping slots used this step, take the misses one each; an
    evicted owner's entry returns to its host block.  Returns (table, owner, prio,
    promotions) with promotions = [(slot, b, h, j)]; the inputs are not modified."""
    table = np.array(table, dtype=np.int64, copy=True)
    owner = np.array(owner, dtype=np.int64, copy=True)
    prio = np.array(prio, dtype=np.int64, copy=True)
    B, H, stride = table.shape
    misses = []
    for b in range(B):
        for h in range(H):
            for j in sorted({int(t) // block_size for t in attended[b][h]}):
                e = int(table[b, h, j])
                if e >= 0:
                    prio[e] = step
                else:
                    misses.append((b, h, j))
    n = len(owner)
    age = np.where(owner < 0, np.inf, (step - prio).astype(np.float64))
    score = np.where(prio == step, np.nan, age)
    chosen = exact_topk(score, np.arange(n), budget)
    free_to_take = [int(sl) for sl in chosen if prio[sl] != step]
    promotions = []
    for sl, (b, h, j) in zip(free_to_take, misses):
        old = int(owner[sl])
        if old >= 0:
            u, jo = divmod(old, stride)
            table[u // H, u % H, jo] = -((u // H) * stride + jo) - 1
        owner[sl] = (b * H + h) * stride + j
        prio[sl] = step
        table[b, h, j] = sl
        promotions.append((sl, b, h, j))
    return table, owner, prio, promotions


def cache_owner_from_table(table: np.ndarray, n_slots: int, max_len: int) -> np.ndarray:
    """The owner array a slot table implies (-1 for slots no token maps to)."""
    owner = np.full(n_slots, -1, dtype=np.int64)
    b, t = np.nonzero(np.asarray(table)[:, :max_len] >= 0)
    owner[np.asarray(table)[b, t]] = b * max_len + t
    return owner


# --------------------------------------------------------------------------------------
# Block selection from per-block key summaries (OasisKV notes, §3.2)
# --------------------------------------------------------------------------------------
#
# Every block of bs tokens keeps the per-coordinate minimum and maximum of its
# keys; a KV head ranks blocks from these two rows alone and attends the whole
# chosen blocks (OasisKV notes, §3.2 "compressed key summaries", after Quest).
# Readings: a block's score is the largest <q, k> any key inside its
# per-coordinate box can reach; the sink and local windows are rounded outward
# to whole blocks, and the candidates are the blocks between them.


def block_regions(L: int, n_sink: int, n_local: int, bs: int) -> tuple[int, int, int]:
    """(nb, s_blk, l_blk): nb blocks cover [0, L); blocks [0, s_blk) hold the sink,
    blocks [l_blk, nb) the local window, blocks [s_blk, l_blk) are candidates."""
    nb = -(-L // bs)
    s_blk = min(-(-n_sink // bs), nb)
    if n_local <= 0:
        l_blk = nb
    else:
        l_blk = max(s_blk, max(L - n_local, 0) // bs)
    return nb, s_blk, l_blk


def block_summary(rows: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Per-coordinate (min, max) of a block's keys [n, d] (n >= 1)."""
    r = as_f64(rows)
    return r.min(axis=0), r.max(axis=0)


def box_bound(q: np.ndarray, lo: np.ndarray, hi: np.ndarray) -> float:
    """max <q, k> over k with lo <= k <= hi coordinate-wise: each coordinate takes
    whichever end its query weight favours, sum_j max(q_j lo_j, q_j hi_j)."""
    q, lo, hi = as_f64(q), as_f64(lo), as_f64(hi)
    return float(np.maximum(q * lo, q * hi).sum())


def block_scores(q_group: np.ndarray, mins: np.ndarray, maxs: np.ndarray, agg: str = "mean") -> np.ndarray:
    """Scores of blocks [nb] from their summaries [nb, d] against a group's heads [G, d]:
    the box bound for the heads' mean ("mean"), or the largest head's bound ("max")."""
    if agg == "mean":
        heads = [group_query(q_group)]
    elif agg == "max":
        heads = list(as_f64(q_group))
    else:
        raise ValueError(f"unknown group aggregation {agg!r}")
    out = np.empty(len(mins))
    for i in range(len(mins)):
        out[i] = max(box_bound(qh, mins[i], maxs[i]) for qh in heads)
    return out


def block_attended_positions(L: int, bs: int, s_blk: int, l_blk: int, nb: int, selected_blocks) -> np.ndarray:
    """Tokens t < L of the sink blocks, the selected blocks and the local blocks, ascending."""
    blocks = sorted(set(range(s_blk)) | {int(x) for x in selected_blocks} | set(range(l_blk, nb)))
    toks = [t for blk in blocks for t in range(blk * bs, min(blk * bs + bs, L))]
    return np.asarray(toks, dtype=np.int64)


def decode_unit_blocks(prob: Problem, b: int, h: int, q: np.ndarray, kpool: PagedPool, vpool: PagedPool,
                       topk_blocks: int, given_block_scores: Optional[np.ndarray] = None,
                       given_blocks: Optional[np.ndarray] = None):
    """Block-selection decode for one (request b, KV head h), paged pool of block_size tokens.

    summaries of every block from its keys (tokens < L), block scores of the
    candidate blocks, the top topk_blocks of them (ties to the lower block, by the
    same full sort as the token top-k), attention of the group over every token of
    the sink, selected and local blocks.  given_block_scores replaces the scores
    (scores over blocks [0, nb)); given_blocks replaces the selection.
    """
    L = int(prob.seq_lens[b])
    G = prob.group
    bs = prob.block_size
    nb, s_blk, l_blk = block_regions(L, prob.n_sink, prob.n_local, bs)
    cand = np.arange(s_blk, l_blk, dtype=np.int64)
    res = {"block_positions": cand, "regions": (nb, s_blk, l_blk)}
    if given_blocks is None:
        if given_block_scores is not None:
            u = np.asarray(given_block_scores, dtype=np.float64)[cand]
        else:
            mins = np.empty((len(cand), prob.d_qk))
            maxs = np.empty((len(cand), prob.d_qk))
            for i, blk in enumerate(cand):
                toks = np.arange(blk * bs, min(blk * bs + bs, L))
                mins[i], maxs[i] = block_summary(kpool.rows(b, h, toks)[:, : prob.d_qk])
            u = block_scores(np.asarray(q)[b, h * G:(h + 1) * G], mins, maxs, prob.group_agg)
        res["block_scores"] = u
        sel = exact_topk(u, cand, topk_blocks)
    else:
        sel = np.asarray(given_blocks, dtype=np.int64)
    res["blocks"] = sel
    att = block_attended_positions(L, bs, s_blk, l_blk, nb, sel)
    res["attended"] = att
    K = kpool.rows(b, h, att)[:, : prob.d_qk]
    V = vpool.rows(b, h, att)[:, : prob.d_v]
    o, lse = attention(np.asarray(q)[b, h * G:(h + 1) * G], K, V, prob.scale())
    res["out"] = o
    res["lse"] = lse
    return res


# --------------------------------------------------------------------------------------
# byte models (UlaCache article §2 and §6.4-6.5; ECHO-OSDI26 wiki, core method 2)
# --------------------------------------------------------------------------------------


def step_read_bytes(k: int, s_kv: float, hit_rate: float = 0.0) -> float:
    """Bytes a step must fetch: V_step = (1 - h) * k * s_kv (UlaCache §6.4)."""
    return (1.0 - hit_rate) * k * s_kv


def fetch_time_s(v_bytes: float, link_bytes_per_s: float) -> float:
    """T_io = V_step / B_fetch (UlaCache §6.4)."""
    return v_bytes / link_bytes_per_s


def echo_metadata_bytes(n_host_tokens: int, n_gpu_tokens: int) -> int:
    """Per-layer slot-map metadata of the two-level pool: 4 N_H + 13 N_G bytes (ECHO core method 2)."""
    return 4 * n_host_tokens + 13 * n_gpu_tokens


def decode_step_hbm_bytes(B, H, Hq, d, L, k, ns, nl, elem=2, score_bytes=4, table_entry=4, block_size=16,
                          per_query_head=False):
    """Algorithmic HBM bytes of one decode step with keys scored in place (paged pool).

    keys of the candidate region read once, scores written once and read once,
    K and V rows of the attended set read once, queries read, output written.
    (Read volume R_step ~ k * s_kv of UlaCache §2 plus the indexer scan.)
    per_query_head: every query head keeps its own scores, selection and attended
    rows (`decode_head`); the candidate keys are still read once per KV head.
    """
    s_end, l_start = regions(L, ns, nl)
    n_c = l_start - s_end
    n_att = s_end + min(k, n_c) + (L - l_start)
    rows = Hq if per_query_head else H  # selection rows per request
    per_row = n_c * 2 * score_bytes + n_att * 2 * d * elem
    per_row += (-(-L // block_size)) * table_entry  # slot table, once per selection row
    keys = B * H * n_c * d * elem
    q_bytes = B * Hq * d * elem
    out_bytes = B * Hq * d * elem
    return keys + B * rows * per_row + q_bytes + out_bytes
