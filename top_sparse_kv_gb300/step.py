"""DecodeStep: owns the output and workspace tensors of one decode step and calls the C ABI.

A thin convenience over the binding: it allocates (with torch) the scores,
index, output, lse, workspace and status buffers once, then every `run()` is a
single skv_decode_step call enqueued on the current stream.
"""

from __future__ import annotations

from typing import Optional

import torch

from . import binding as B


class DecodeStep:
    def __init__(self, problem: B.Problem, pool: B.Pool, q: torch.Tensor, index: B.IndexSrc,
                 q_score: Optional[torch.Tensor] = None, out_dtype: Optional[torch.dtype] = None):
        self.p = problem
        self.pool = pool
        self.q = q
        self.q_score = q_score
        self.index = index
        dev = q.device
        # one selection row per KV head, or per query head under the per-head reading
        sel_heads = problem.n_q_heads if problem.group_agg == B.SKV_AGG_HEAD else problem.n_kv_heads
        rows = problem.batch * sel_heads
        self.scores = torch.empty((problem.batch, sel_heads, problem.max_len), dtype=torch.float32, device=dev)
        self.idx = torch.empty((problem.batch, sel_heads, max(problem.topk, 1)), dtype=torch.int32, device=dev)
        self.out = torch.empty((problem.batch, problem.n_q_heads, problem.d_v), dtype=out_dtype or q.dtype,
                               device=dev)
        self.lse = torch.empty((problem.batch, problem.n_q_heads), dtype=torch.float32, device=dev)
        ws_bytes = B.skv_workspace_size(problem)
        self.ws = torch.empty((max(ws_bytes, 16),), dtype=torch.uint8, device=dev)
        self.status = torch.zeros((1,), dtype=torch.int32, device=dev)
        assert rows > 0

    def run(self, stream=None):
        B.skv_decode_step(self.p, self.q, self.q_score, self.index, self.pool, self.scores, self.idx, self.out,
                          self.lse, self.ws, self.status, stream)

    def enable_prefetch(self, cap: int, alpha: float = 0.5):
        """Fresh threshold-prefetch state for run_prefetch() (latent layout, or a paged pool with
        contiguous index keys)."""
        self.pf = B.Prefetch.new(self.p, cap, self.pool.gpu_k.dtype, self.q.device, alpha,
                                 paged=self.pool.gpu_v is not None)
        return self.pf

    def run_prefetch(self, stream=None, stats: bool = True):
        """One step with threshold prefetch; stats=False leaves the staged/read counters untouched."""
        B.skv_decode_step_prefetch(self.p, self.q, self.q_score, self.index, self.pool, self.scores, self.idx,
                                   self.out, self.lse, self.ws, self.pf, self.status, stream, stats=stats)

    def enable_cache(self, budget: int):
        """Switch to skv_decode_step_cached: the GPU slot pool becomes a managed cache (the latent
        layout, or K/V pools with one table row per (request, KV head))."""
        self.cache = B.SlotCache.from_table(self.p, self.pool, budget)
        return self.cache

    def run_cached(self, stream=None):
        B.skv_decode_step_cached(self.p, self.q, self.q_score, self.index, self.pool, self.scores, self.idx, self.out,
                                 self.lse, self.ws, self.cache, self.status, stream)

    def cache_update(self, stream=None):
        """The slot-cache update alone, for the step run() just enqueued."""
        B.skv_cache_update(self.p, self.pool, self.idx, self.ws, self.cache, self.status, stream)

    def score(self, stream=None):
        B.skv_score(self.p, self.q_score if self.q_score is not None else self.q, self.index, self.pool,
                    self.scores, self.status, stream)

    def topk(self, stream=None):
        B.skv_topk(self.p, self.scores, self.idx, self.ws, self.status, stream)

    def attend(self, stream=None):
        B.skv_sparse_attn(self.p, self.q, self.pool, self.idx, self.out, self.lse, self.ws, self.status, stream)

    @classmethod
    def from_workload(cls, wl, n_splits: int = 0, sm_scale: Optional[float] = None, group_agg: int = B.SKV_AGG_MEAN):
        """Build from an object with the seeded generator's attribute names (duck-typed)."""
        dtype = B.SKV_DTYPE_F32 if wl.dtype == torch.float32 else B.SKV_DTYPE_BF16
        contig = getattr(wl, "index_keys", None) is not None
        q_score = wl.q_idx if contig else None
        p = B.Problem(batch=wl.B, n_kv_heads=wl.H, n_q_heads=wl.Hq, d_qk=wl.d_qk, d_v=wl.d_v, max_len=wl.L,
                      topk=wl.k, n_sink=wl.ns, n_local=wl.nl, block_size=wl.bs, seq_lens=wl.seq_lens,
                      d_idx=wl.d_idx, n_idx_q_heads=(q_score.shape[1] if contig else wl.Hq), dtype=dtype,
                      sm_scale=float(sm_scale if sm_scale is not None else wl.sm_scale), n_splits=n_splits,
                      group_agg=group_agg)
        pool = B.Pool(wl.gpu_k, wl.gpu_v, wl.table, wl.host_k, wl.host_v)
        index = B.IndexSrc(B.SKV_INDEX_CONTIG, wl.index_keys) if contig else B.IndexSrc(B.SKV_INDEX_PAGED)
        return cls(p, pool, wl.q, index, q_score=q_score)


class BlockStep:
    """Block-selection decode (per-block key summaries): owns the summaries, the
    chosen blocks, the attended list, the output and the workspace; `summarize()`
    is the maintenance call, `run()` one skv_block_decode_step."""

    def __init__(self, problem: B.Problem, pool: B.Pool, q: torch.Tensor, topk_blocks: int):
        self.p = problem
        self.pool = pool
        self.q = q
        self.K = int(topk_blocks)
        dev = q.device
        nb = (problem.max_len + 15) // 16
        self.summaries = torch.empty((problem.batch, problem.n_kv_heads, nb, 2, problem.d_qk),
                                     dtype=pool.gpu_k.dtype, device=dev)
        ws_bytes, self.list_len = B.skv_block_workspace_size(problem, self.K)
        self.block_idx = torch.empty((problem.batch, problem.n_kv_heads, max(self.K, 1)), dtype=torch.int32,
                                     device=dev)
        self.att_idx = torch.empty((problem.batch, problem.n_kv_heads, max(self.list_len, 1)), dtype=torch.int32,
                                   device=dev)
        self.out = torch.empty((problem.batch, problem.n_q_heads, problem.d_v), dtype=q.dtype, device=dev)
        self.lse = torch.empty((problem.batch, problem.n_q_heads), dtype=torch.float32, device=dev)
        self.ws = torch.empty((max(ws_bytes, 16),), dtype=torch.uint8, device=dev)
        self.status = torch.zeros((1,), dtype=torch.int32, device=dev)

    def summarize(self, stream=None):
        B.skv_block_summaries(self.p, self.pool, self.summaries, self.status, stream)

    def select(self, stream=None):
        B.skv_block_select(self.p, self.K, self.q, self.summaries, self.block_idx, self.att_idx, self.ws,
                           self.status, stream)

    def run(self, stream=None):
        B.skv_block_decode_step(self.p, self.K, self.q, self.summaries, self.pool, self.block_idx, self.att_idx,
                                self.out, self.lse, self.ws, self.status, stream)

    @classmethod
    def from_workload(cls, wl, topk_blocks: int, group_agg: int = B.SKV_AGG_MEAN, n_splits: int = 0):
        """Build from a paged workload of the seeded generator (duck-typed attribute names)."""
        dtype = B.SKV_DTYPE_F32 if wl.dtype == torch.float32 else B.SKV_DTYPE_BF16
        p = B.Problem(batch=wl.B, n_kv_heads=wl.H, n_q_heads=wl.Hq, d_qk=wl.d_qk, d_v=wl.d_v, max_len=wl.L,
                      topk=topk_blocks, n_sink=wl.ns, n_local=wl.nl, block_size=wl.bs, seq_lens=wl.seq_lens,
                      d_idx=wl.d_qk, n_idx_q_heads=wl.Hq, dtype=dtype, sm_scale=float(wl.sm_scale),
                      n_splits=n_splits, group_agg=group_agg)
        pool = B.Pool(wl.gpu_k, wl.gpu_v, wl.table, wl.host_k, wl.host_v)
        return cls(p, pool, wl.q, topk_blocks)


class ParisStep:
    """ParisKV retrieval decode (skv_paris_decode_step): owns the index, the selection, the
    output and the workspace; `encode()` builds the index from the keys (maintenance),
    `run()` is one step."""

    def __init__(self, step: DecodeStep, signs: torch.Tensor, beta_pm: int = 50, rho_pm: int = 100):
        self.p, self.pool, self.q, self.q_score, self.index = step.p, step.pool, step.q, step.q_score, step.index
        self.paris = B.Paris.new(self.p, signs, beta_pm, rho_pm)
        self.idx, self.out, self.lse, self.status = step.idx, step.out, step.lse, step.status
        n = B.skv_paris_workspace_size(self.p, self.paris)
        self.ws = torch.empty((max(n, 16),), dtype=torch.uint8, device=signs.device)
        self.offsets = B.skv_paris_workspace_offsets(self.p, self.paris)

    @classmethod
    def from_workload(cls, wl, signs: torch.Tensor, beta_pm: int = 50, rho_pm: int = 100, n_splits: int = 0):
        return cls(DecodeStep.from_workload(wl, n_splits=n_splits), signs, beta_pm, rho_pm)

    def encode(self, stream=None):
        B.skv_paris_encode(self.p, self.paris, self.index, self.pool, self.status, stream)

    def run(self, stream=None):
        B.skv_paris_decode_step(self.p, self.paris, self.q, self.q_score, self.index, self.pool, self.idx,
                                self.out, self.lse, self.ws, self.status, stream)

    def select(self, stream=None):
        """The retrieval alone: the selection into idx."""
        B.skv_paris_select(self.p, self.paris, self.q_score if self.q_score is not None else self.q, self.index,
                           self.pool, self.idx, self.ws, self.status, stream)

    def attend(self, stream=None):
        """The attention alone over the current selection (same workspace)."""
        B.skv_sparse_attn(self.p, self.q, self.pool, self.idx, self.out, self.lse, self.ws, self.status, stream)

    def view(self, name: str) -> torch.Tensor:
        """A workspace intermediate: qt, nq, W, S, cand_len, cand, cand_score, sim."""
        rows, c_cap, L = self.p.batch * self.p.n_kv_heads, self.offsets[7], self.p.max_len
        k = ("qt", "nq", "W", "S", "cand_len", "cand", "cand_score", None, "sim").index(name)
        shape, dt = {"qt": ((rows, 128), torch.float32), "nq": ((rows,), torch.float32),
                     "W": ((rows, 16, 256), torch.uint8), "S": ((rows, L), torch.uint8),
                     "sim": ((rows, 16, 256), torch.float32),
                     "cand_len": ((self.p.batch,), torch.int32), "cand": ((rows, c_cap), torch.int32),
                     "cand_score": ((rows, c_cap), torch.float32)}[name]
        n = int(torch.tensor(shape).prod().item()) * torch.tensor([], dtype=dt).element_size()
        return self.ws[self.offsets[k]: self.offsets[k] + n].view(dt).view(shape)
