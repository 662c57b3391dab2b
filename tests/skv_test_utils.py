"""Helpers shared by the GPU parity tests: oracle inputs from a workload, tolerances."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

# attention tolerances (bf16 storage / fp32 storage), element-wise on the output
BF16_MAX_ABS, BF16_MEAN_ABS = 2e-2, 2e-3
F32_MAX_ABS = 1e-4
# selection band vs the fp64 oracle: a position may differ only if its fp64 score
# lies within this relative distance of the k-th score
BAND_REL = 1e-5

nv = workloads.numpy_view


class OracleView:
    """The workload's tensors as the oracle reads them (CPU numpy, bf16 as bit patterns)."""

    def __init__(self, wl, group_agg: str = "mean"):
        self.wl = wl
        self.prob = oracle.Problem(
            batch=wl.B, n_kv_heads=wl.H, n_q_heads=wl.Hq, d_qk=wl.d_qk, d_v=wl.d_v, topk=wl.k, n_sink=wl.ns,
            n_local=wl.nl, block_size=wl.bs, seq_lens=[int(x) for x in wl.seq_lens.cpu()], sm_scale=wl.sm_scale,
            index_layout=wl.index_layout, group_agg=group_agg)
        table = nv(wl.table)
        self.kpool = oracle.PagedPool(nv(wl.gpu_k), nv(wl.host_k), table, wl.bs)
        self.vpool = None if wl.gpu_v is None else oracle.PagedPool(nv(wl.gpu_v), nv(wl.host_v), table, wl.bs)
        self.q = nv(wl.q)
        self.q_idx = nv(wl.q_idx)
        self.index_keys = nv(wl.index_keys)

    def unit(self, b, h, **kw):
        return oracle.decode_unit(self.prob, b, h, self.q, self.kpool, self.vpool, q_index=self.q_idx,
                                  index_keys=self.index_keys, **kw)

    def head(self, b, j, **kw):
        """The per-query-head step of query head j (oracle.decode_head)."""
        return oracle.decode_head(self.prob, b, j, self.q, self.kpool, self.vpool, q_index=self.q_idx,
                                  index_keys=self.index_keys, **kw)

    def head_score_tolerance(self, b, j, positions):
        """fp32 accumulation bound for <q_j, k_t>: ~(d + 1) unit roundoffs of sum |q_j k_t|."""
        h = j // self.wl.G
        if self.prob.index_layout == "paged":
            qj = oracle.as_f64(self.q[b, j])
            keys = self.kpool.rows(b, h, positions)
        else:
            qj = oracle.as_f64(self.q_idx[b, j])
            keys = oracle.as_f64(self.index_keys[b, h, positions])
        return 4.0 * (keys.shape[1] + 1) * 2.0 ** -24 * (np.abs(keys) @ np.abs(qj)) + 1e-30


class UnitView:
    """One (request b, KV head h) of a paged K/V workload as the oracle reads it: only that
    unit's blocks are copied to the CPU (through its slot-table row, either tier), so
    full-size workloads whose pools are tens of GB can be checked unit by unit.  The
    unit becomes request 0, KV head 0 of a one-unit problem with an identity table."""

    def __init__(self, wl, b, h, group_agg: str = "mean"):
        assert wl.index_layout == "paged" and wl.gpu_v is not None
        L = int(wl.seq_lens[b])
        nblk = (L + wl.bs - 1) // wl.bs
        e = wl.table[b, :nblk].cpu().long()
        on_gpu = e >= 0

        def take(gpu_pool, host_pool):
            rows = torch.empty((nblk, 1, wl.bs, gpu_pool.shape[-1]), dtype=gpu_pool.dtype)
            if bool(on_gpu.any()):
                rows[on_gpu, 0] = gpu_pool[e[on_gpu].to(gpu_pool.device), h].cpu()
            if bool((~on_gpu).any()):
                rows[~on_gpu, 0] = host_pool[(-e[~on_gpu] - 1).to(host_pool.device), h].cpu()
            return nv(rows)

        G = wl.G
        table = np.arange(nblk, dtype=np.int64)[None, :]
        self.prob = oracle.Problem(
            batch=1, n_kv_heads=1, n_q_heads=G, d_qk=wl.d_qk, d_v=wl.d_v, topk=wl.k, n_sink=wl.ns,
            n_local=wl.nl, block_size=wl.bs, seq_lens=[L], sm_scale=wl.sm_scale, index_layout="paged",
            group_agg=group_agg)
        self.kpool = oracle.PagedPool(take(wl.gpu_k, wl.host_k), None, table, wl.bs)
        self.vpool = oracle.PagedPool(take(wl.gpu_v, wl.host_v), None, table, wl.bs)
        self.q = nv(wl.q[b:b + 1, h * G:(h + 1) * G])

    def unit(self, **kw):
        return oracle.decode_unit(self.prob, 0, 0, self.q, self.kpool, self.vpool, **kw)


def score_tolerance(view: OracleView, b: int, h: int, positions: np.ndarray) -> np.ndarray:
    """fp32 accumulation bound for a group score: ~(d + G) unit roundoffs of sum_j |q_j k_tj| (q the
    heads' mean for the mean reading; the largest head's bound for the max reading)."""
    wl = view.wl
    if view.prob.index_layout == "paged":
        G = wl.G
        qg = oracle.as_f64(view.q[b, h * G:(h + 1) * G])
        keys = view.kpool.rows(b, h, positions)
    else:
        gi = view.q_idx.shape[1] // wl.H
        qg = oracle.as_f64(view.q_idx[b, h * gi:(h + 1) * gi])
        keys = oracle.as_f64(view.index_keys[b, h, positions])
        G = gi
    if view.prob.group_agg == "max":  # the largest of the heads' own bounds
        mag = (np.abs(keys) @ np.abs(qg).T).max(axis=1)
    else:
        mag = np.abs(keys) @ np.abs(qg).mean(axis=0)
    return 4.0 * (keys.shape[1] + G) * 2.0 ** -24 * mag + 1e-30


def check_band(gpu_idx: np.ndarray, ref: dict, k: int):
    """The GPU's selection equals the fp64 oracle's except for positions whose fp64
    score lies within BAND_REL (relative) of the oracle's k-th score."""
    want = set(int(t) for t in ref["idx"])
    got = set(int(t) for t in gpu_idx if t >= 0)
    assert len(got) == len(want) == min(k, len(ref["positions"]))
    diff = want ^ got
    if not diff:
        return 0
    s = ref["scores"]
    pos = ref["positions"]
    score_of = dict(zip(pos.tolist(), s.tolist()))
    tau = min(score_of[t] for t in want)
    scale = max(abs(tau), float(np.sqrt(np.mean(s ** 2))))
    for t in diff:
        assert abs(score_of[t] - tau) <= BAND_REL * scale, (t, score_of[t], tau)
    return len(diff)


def assert_attention_close(got: torch.Tensor, want: np.ndarray, dtype: torch.dtype):
    g = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - want)
    if dtype == torch.float32:
        assert err.max() <= F32_MAX_ABS, err.max()
    else:
        assert err.max() <= BF16_MAX_ABS and err.mean() <= BF16_MEAN_ABS, (err.max(), err.mean())
    return float(err.max())
