"""ctypes binding of libskv.so: the C ABI's names, argument marshalling only.

Every function takes torch tensors (device memory, or pinned host memory for
host pools), passes their raw pointers to the C entry point of the same name
and raises SkvError on a non-OK status.  No arithmetic of the step happens
here; if the library is missing the import fails loudly -- there is no
fallback path.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libskv.so")

SKV_OK = 0
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "CUDA error",
                4: "workspace too small", 5: "device fault", 6: "timeout"}
SKV_DEV_BAD_SLOT, SKV_DEV_BAD_INDEX, SKV_DEV_BAD_LENGTH, SKV_DEV_TIMEOUT = 1, 2, 4, 8
SKV_DTYPE_BF16, SKV_DTYPE_F32 = 0, 1
SKV_AGG_MEAN = 0
SKV_AGG_MAX = 1
SKV_AGG_HEAD = 2  # every query head selects its own top-k
SKV_INDEX_PAGED, SKV_INDEX_CONTIG = 0, 1


class SkvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)} (status {status})")
        self.status = status


class CProblem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "n_kv_heads", "n_q_heads", "d_qk", "d_v", "d_idx", "n_idx_q_heads", "max_len",
        "topk", "n_sink", "n_local", "block_size", "dtype", "group_agg")] + [
        ("sm_scale", ctypes.c_float), ("n_splits", ctypes.c_int32), ("seq_lens", ctypes.c_void_p)]


class CPool(ctypes.Structure):
    _fields_ = [("gpu_k", ctypes.c_void_p), ("gpu_v", ctypes.c_void_p), ("n_gpu_blocks", ctypes.c_int64),
                ("host_k", ctypes.c_void_p), ("host_v", ctypes.c_void_p), ("n_host_blocks", ctypes.c_int64),
                ("slot_table", ctypes.c_void_p), ("table_stride", ctypes.c_int32), ("table_heads", ctypes.c_int32)]


class CIndex(ctypes.Structure):
    _fields_ = [("layout", ctypes.c_int32), ("keys", ctypes.c_void_p)]


class CSlotCache(ctypes.Structure):
    _fields_ = [("owner", ctypes.c_void_p), ("prio", ctypes.c_void_p), ("step", ctypes.c_void_p),
                ("budget", ctypes.c_int32), ("stats", ctypes.c_void_p)]


class CParis(ctypes.Structure):
    _fields_ = [("m", ctypes.c_int32), ("beta_pm", ctypes.c_int32), ("rho_pm", ctypes.c_int32),
                ("signs", ctypes.c_void_p)]


class CParisIndex(ctypes.Structure):
    _fields_ = [("cent", ctypes.c_void_p), ("rec", ctypes.c_void_p), ("hist", ctypes.c_void_p)]


class CPrefetch(ctypes.Structure):
    _fields_ = [("tau_ema", ctypes.c_void_p), ("epoch", ctypes.c_void_p), ("map", ctypes.c_void_p),
                ("staging", ctypes.c_void_p), ("count", ctypes.c_void_p), ("stats", ctypes.c_void_p),
                ("cap", ctypes.c_int32), ("alpha", ctypes.c_float)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libskv.so is not built ({LIB_PATH}); run __graft_entry__.build() "
                          "or python -m top_sparse_kv_gb300.build_lib")
    lib = ctypes.CDLL(LIB_PATH)
    P, VP, SZ = ctypes.POINTER(CProblem), ctypes.c_void_p, ctypes.c_size_t
    sig = {
        "skv_workspace_size": [P, ctypes.POINTER(ctypes.c_size_t)],
        "skv_score": [P, VP, ctypes.POINTER(CIndex), ctypes.POINTER(CPool), VP, VP, VP],
        "skv_topk": [P, VP, VP, VP, SZ, VP, VP],
        "skv_gather": [P, ctypes.POINTER(CPool), VP, VP, VP, VP, VP],
        "skv_sparse_attn": [P, VP, ctypes.POINTER(CPool), VP, VP, VP, VP, SZ, VP, VP],
        "skv_decode_step": [P, VP, VP, ctypes.POINTER(CIndex), ctypes.POINTER(CPool), VP, VP, VP, VP, VP, SZ,
                            VP, VP],
        "skv_decode_step_prefetch": [P, VP, VP, ctypes.POINTER(CIndex), ctypes.POINTER(CPool), VP, VP, VP, VP,
                                     VP, SZ, ctypes.POINTER(CPrefetch), VP, VP],
        "skv_cache_workspace_size": [P, ctypes.POINTER(CPool), ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)],
        "skv_decode_step_cached": [P, VP, VP, ctypes.POINTER(CIndex), ctypes.POINTER(CPool), VP, VP, VP, VP, VP,
                                   SZ, ctypes.POINTER(CSlotCache), VP, SZ, VP, VP],
        "skv_cache_prepare": [],
        "skv_cache_update": [P, ctypes.POINTER(CPool), VP, VP, SZ, ctypes.POINTER(CSlotCache), VP, SZ, VP, VP],
        "skv_paris_quantizer": [ctypes.c_int32, VP, VP],
        "skv_paris_encode": [P, ctypes.POINTER(CParis), ctypes.POINTER(CIndex), ctypes.POINTER(CPool),
                             ctypes.POINTER(CParisIndex), VP, VP],
        "skv_paris_workspace_size": [P, ctypes.POINTER(CParis), ctypes.POINTER(ctypes.c_size_t)],
        "skv_paris_workspace_offsets": [P, ctypes.POINTER(CParis), VP],
        "skv_paris_select": [P, ctypes.POINTER(CParis), VP, ctypes.POINTER(CIndex), ctypes.POINTER(CParisIndex),
                             ctypes.POINTER(CPool), VP, VP, SZ, VP, VP],
        "skv_paris_decode_step": [P, ctypes.POINTER(CParis), VP, VP, ctypes.POINTER(CIndex),
                                  ctypes.POINTER(CParisIndex), ctypes.POINTER(CPool), VP, VP, VP, VP, SZ, VP, VP],
        "skv_block_workspace_size": [P, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t),
                                     ctypes.POINTER(ctypes.c_int32)],
        "skv_block_summaries": [P, ctypes.POINTER(CPool), VP, VP, VP],
        "skv_block_select": [P, ctypes.c_int32, VP, VP, VP, VP, VP, SZ, VP, VP],
        "skv_block_decode_step": [P, ctypes.c_int32, VP, VP, ctypes.POINTER(CPool), VP, VP, VP, VP, VP, SZ, VP,
                                  VP],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int32
    lib.skv_status_string.argtypes = [ctypes.c_int32]
    lib.skv_status_string.restype = ctypes.c_char_p
    lib.skv_launch_count.argtypes = []
    lib.skv_launch_count.restype = ctypes.c_uint64
    lib.skv_check_wait_timeout.argtypes = [ctypes.c_int64, ctypes.c_int32, VP, VP]
    lib.skv_check_wait_timeout.restype = ctypes.c_int32
    return lib


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libskv must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, st: int):
    if st != SKV_OK:
        raise SkvError(fn, st)


@dataclass
class Problem:
    """Python mirror of skv_problem (see include/skv.h for every field's meaning)."""

    batch: int
    n_kv_heads: int
    n_q_heads: int
    d_qk: int
    d_v: int
    max_len: int
    topk: int
    n_sink: int
    n_local: int
    block_size: int
    seq_lens: torch.Tensor  # device int32 [batch]
    d_idx: int = 0  # 0 -> d_qk
    n_idx_q_heads: int = 0  # 0 -> n_q_heads
    dtype: int = SKV_DTYPE_BF16
    group_agg: int = SKV_AGG_MEAN
    sm_scale: float = 0.0
    n_splits: int = 0

    def c(self) -> CProblem:
        return CProblem(self.batch, self.n_kv_heads, self.n_q_heads, self.d_qk, self.d_v,
                        self.d_idx or self.d_qk, self.n_idx_q_heads or self.n_q_heads, self.max_len,
                        self.topk, self.n_sink, self.n_local, self.block_size, self.dtype, self.group_agg,
                        float(self.sm_scale), self.n_splits,
                        None if self.seq_lens is None else self.seq_lens.data_ptr())


@dataclass
class Pool:
    """Python mirror of skv_kv_pool; tensors are [n_blocks, H, block_size, d].  With
    table_heads = 1 the table is [batch, H, stride] and the GPU pools [n_blocks, block_size, d]."""

    gpu_k: torch.Tensor
    gpu_v: Optional[torch.Tensor]
    slot_table: torch.Tensor  # device int32 [batch, stride], or [batch, H, stride] with table_heads = 1
    host_k: Optional[torch.Tensor] = None
    host_v: Optional[torch.Tensor] = None
    table_heads: int = 0

    def c(self) -> CPool:
        return CPool(self.gpu_k.data_ptr(), None if self.gpu_v is None else self.gpu_v.data_ptr(),
                     self.gpu_k.shape[0],
                     None if self.host_k is None else self.host_k.data_ptr(),
                     None if self.host_v is None else self.host_v.data_ptr(),
                     0 if self.host_k is None else self.host_k.shape[0],
                     self.slot_table.data_ptr(), self.slot_table.shape[-1], self.table_heads)


@dataclass
class IndexSrc:
    layout: int = SKV_INDEX_PAGED
    keys: Optional[torch.Tensor] = None

    def c(self) -> CIndex:
        return CIndex(self.layout, None if self.keys is None else self.keys.data_ptr())


def skv_workspace_size(p: Problem) -> int:
    n = ctypes.c_size_t(0)
    cp = p.c()
    _check("skv_workspace_size", lib().skv_workspace_size(ctypes.byref(cp), ctypes.byref(n)))
    return n.value


def skv_score(p: Problem, q_score, index: IndexSrc, pool: Optional[Pool], scores, dev_status=None, stream=None):
    cp, ci = p.c(), index.c()
    cpool = pool.c() if pool is not None else None
    _check("skv_score", lib().skv_score(ctypes.byref(cp), _ptr(q_score), ctypes.byref(ci),
                                        ctypes.byref(cpool) if cpool is not None else None, _ptr(scores),
                                        _ptr(dev_status), _stream(stream)))


def skv_topk(p: Problem, scores, idx, ws, dev_status=None, stream=None):
    cp = p.c()
    _check("skv_topk", lib().skv_topk(ctypes.byref(cp), _ptr(scores), _ptr(idx), _ptr(ws),
                                      ws.numel() * ws.element_size(), _ptr(dev_status), _stream(stream)))


def skv_gather(p: Problem, pool: Pool, idx, k_out, v_out=None, dev_status=None, stream=None):
    cp, cpool = p.c(), pool.c()
    _check("skv_gather", lib().skv_gather(ctypes.byref(cp), ctypes.byref(cpool), _ptr(idx), _ptr(k_out),
                                          _ptr(v_out), _ptr(dev_status), _stream(stream)))


def skv_sparse_attn(p: Problem, q, pool: Pool, idx, out, lse, ws, dev_status=None, stream=None):
    cp, cpool = p.c(), pool.c()
    _check("skv_sparse_attn", lib().skv_sparse_attn(
        ctypes.byref(cp), _ptr(q), ctypes.byref(cpool), _ptr(idx), _ptr(out), _ptr(lse), _ptr(ws),
        ws.numel() * ws.element_size(), _ptr(dev_status), _stream(stream)))


def skv_decode_step(p: Problem, q, q_score, index: IndexSrc, pool: Pool, scores, idx, out, lse, ws,
                    dev_status=None, stream=None):
    cp, ci, cpool = p.c(), index.c(), pool.c()
    _check("skv_decode_step", lib().skv_decode_step(
        ctypes.byref(cp), _ptr(q), _ptr(q_score), ctypes.byref(ci), ctypes.byref(cpool), _ptr(scores),
        _ptr(idx), _ptr(out), _ptr(lse), _ptr(ws), ws.numel() * ws.element_size(), _ptr(dev_status),
        _stream(stream)))


def skv_block_workspace_size(p: Problem, topk_blocks: int) -> tuple[int, int]:
    """(workspace bytes, attended-list length) of the block-selection calls."""
    n, ln = ctypes.c_size_t(0), ctypes.c_int32(0)
    cp = p.c()
    _check("skv_block_workspace_size", lib().skv_block_workspace_size(ctypes.byref(cp), int(topk_blocks),
                                                                      ctypes.byref(n), ctypes.byref(ln)))
    return n.value, ln.value


def skv_block_summaries(p: Problem, pool: Pool, summaries, dev_status=None, stream=None):
    cp, cpool = p.c(), pool.c()
    _check("skv_block_summaries", lib().skv_block_summaries(ctypes.byref(cp), ctypes.byref(cpool), _ptr(summaries),
                                                            _ptr(dev_status), _stream(stream)))


def skv_block_select(p: Problem, topk_blocks: int, q, summaries, block_idx, att_idx, ws, dev_status=None,
                     stream=None):
    cp = p.c()
    _check("skv_block_select", lib().skv_block_select(
        ctypes.byref(cp), int(topk_blocks), _ptr(q), _ptr(summaries), _ptr(block_idx), _ptr(att_idx), _ptr(ws),
        ws.numel() * ws.element_size(), _ptr(dev_status), _stream(stream)))


def skv_block_decode_step(p: Problem, topk_blocks: int, q, summaries, pool: Pool, block_idx, att_idx, out, lse,
                          ws, dev_status=None, stream=None):
    cp, cpool = p.c(), pool.c()
    _check("skv_block_decode_step", lib().skv_block_decode_step(
        ctypes.byref(cp), int(topk_blocks), _ptr(q), _ptr(summaries), ctypes.byref(cpool), _ptr(block_idx),
        _ptr(att_idx), _ptr(out), _ptr(lse), _ptr(ws), ws.numel() * ws.element_size(), _ptr(dev_status),
        _stream(stream)))


@dataclass
class Prefetch:
    """Threshold-prefetch state (persistent across steps); see skv_prefetch in include/skv.h."""

    tau_ema: torch.Tensor   # float32 [rows], NaN to start
    epoch: torch.Tensor     # int32 [1] (uint32 on the device), 0 to start
    map: torch.Tensor       # int64 [rows * max_len], 0 to start
    staging: torch.Tensor   # [rows, cap, d_qk] of the pool's dtype
    count: torch.Tensor     # int32 [rows], 0 to start
    stats: Optional[torch.Tensor] = None  # int32 [2]
    alpha: float = 0.5

    @classmethod
    def new(cls, p: "Problem", cap: int, dtype: torch.dtype, device, alpha: float = 0.5,
            paged: bool = False) -> "Prefetch":
        """paged: a pool with separate V rows, whose staging holds the K rows, then the V rows."""
        rows = p.batch * p.n_kv_heads
        shape = (2, rows, max(cap, 1), p.d_qk) if paged else (rows, max(cap, 1), p.d_qk)
        return cls(tau_ema=torch.full((rows,), float("nan"), dtype=torch.float32, device=device),
                   epoch=torch.zeros((1,), dtype=torch.int32, device=device),
                   map=torch.zeros((rows * p.max_len,), dtype=torch.int64, device=device),
                   staging=torch.empty(shape, dtype=dtype, device=device),
                   count=torch.zeros((rows,), dtype=torch.int32, device=device),
                   stats=torch.zeros((2,), dtype=torch.int32, device=device), alpha=alpha)

    def c(self, cap: int, stats: bool = True) -> CPrefetch:
        st = self.stats.data_ptr() if (stats and self.stats is not None) else None
        return CPrefetch(self.tau_ema.data_ptr(), self.epoch.data_ptr(), self.map.data_ptr(), self.staging.data_ptr(),
                         self.count.data_ptr(), st, int(cap), float(self.alpha))


def skv_decode_step_prefetch(p: Problem, q, q_score, index: IndexSrc, pool: Pool, scores, idx, out, lse, ws,
                             pf: Prefetch, dev_status=None, stream=None, stats: bool = True):
    cp, ci, cpool, cpf = p.c(), index.c(), pool.c(), pf.c(pf.staging.shape[-2], stats)  # [..., cap, d]
    _check("skv_decode_step_prefetch", lib().skv_decode_step_prefetch(
        ctypes.byref(cp), _ptr(q), _ptr(q_score), ctypes.byref(ci), ctypes.byref(cpool), _ptr(scores), _ptr(idx),
        _ptr(out), _ptr(lse), _ptr(ws), ws.numel() * ws.element_size(), ctypes.byref(cpf), _ptr(dev_status),
        _stream(stream)))


@dataclass
class SlotCache:
    """GPU slot-cache state (persistent across steps); see skv_slot_cache in include/skv.h."""

    owner: torch.Tensor   # int32 [n_gpu]
    prio: torch.Tensor    # int32 [n_gpu]
    step: torch.Tensor    # int32 [1]
    budget: int
    ws: torch.Tensor      # uint8: the update's own workspace
    stats: torch.Tensor   # int64 [3]: hits, misses, promotions summed over steps
    count: bool = True    # False: the update leaves stats untouched

    @classmethod
    def from_table(cls, p: "Problem", pool: "Pool", budget: int) -> "SlotCache":
        """Owners as the slot table names them, every slot unused so far."""
        n = pool.gpu_k.shape[0]
        dev = pool.gpu_k.device
        owner = torch.full((n,), -1, dtype=torch.int64, device=dev)
        if pool.table_heads:  # one row per (request, KV head): owners (b * H + h) * stride + block
            t = pool.slot_table.reshape(-1).to(torch.int64)
            m = t >= 0
            owner[t[m]] = torch.arange(t.numel(), device=dev)[m]
        else:  # the latent layout's per-token map: owners b * max_len + position
            t = pool.slot_table[:, : p.max_len].to(torch.int64)
            b = torch.arange(t.shape[0], device=dev)[:, None].expand_as(t)
            pos = torch.arange(p.max_len, device=dev)[None, :].expand_as(t)
            m = t >= 0
            owner[t[m]] = (b[m] * p.max_len + pos[m])
        nb = ctypes.c_size_t(0)
        cp, cpool = p.c(), pool.c()
        _check("skv_cache_prepare", lib().skv_cache_prepare())
        _check("skv_cache_workspace_size", lib().skv_cache_workspace_size(ctypes.byref(cp), ctypes.byref(cpool),
                                                                          int(budget), ctypes.byref(nb)))
        return cls(owner=owner.to(torch.int32), prio=torch.full((n,), -1, dtype=torch.int32, device=dev),
                   step=torch.zeros((1,), dtype=torch.int32, device=dev), budget=int(budget),
                   ws=torch.empty((max(nb.value, 16),), dtype=torch.uint8, device=dev),
                   stats=torch.zeros((3,), dtype=torch.int64, device=dev))

    def c(self) -> CSlotCache:
        return CSlotCache(self.owner.data_ptr(), self.prio.data_ptr(), self.step.data_ptr(), self.budget,
                          self.stats.data_ptr() if self.count else None)


def skv_decode_step_cached(p: Problem, q, q_score, index: IndexSrc, pool: Pool, scores, idx, out, lse, ws,
                           cache: SlotCache, dev_status=None, stream=None):
    cp, ci, cpool, cc = p.c(), index.c(), pool.c(), cache.c()
    _check("skv_decode_step_cached", lib().skv_decode_step_cached(
        ctypes.byref(cp), _ptr(q), _ptr(q_score), ctypes.byref(ci), ctypes.byref(cpool), _ptr(scores), _ptr(idx),
        _ptr(out), _ptr(lse), _ptr(ws), ws.numel() * ws.element_size(), ctypes.byref(cc), _ptr(cache.ws),
        cache.ws.numel(), _ptr(dev_status), _stream(stream)))


def skv_cache_update(p: Problem, pool: Pool, idx, ws, cache: SlotCache, dev_status=None, stream=None):
    cp, cpool, cc = p.c(), pool.c(), cache.c()
    _check("skv_cache_update", lib().skv_cache_update(
        ctypes.byref(cp), ctypes.byref(cpool), _ptr(idx), _ptr(ws), ws.numel() * ws.element_size(), ctypes.byref(cc),
        _ptr(cache.ws), cache.ws.numel(), _ptr(dev_status), _stream(stream)))


@dataclass
class Paris:
    """ParisKV retrieval parameters (skv_paris) and the per-row index it reads (skv_paris_index)."""

    signs: torch.Tensor          # device int8 [128]
    cent: torch.Tensor           # device uint8 [rows, max_len, 16]
    rec: torch.Tensor            # device int32 [rows, max_len, 32]: 16 code words, 16 fp32 weights
    hist: torch.Tensor           # device int32 [rows, 16, 256]
    beta_pm: int = 50
    rho_pm: int = 100
    m: int = 8

    @classmethod
    def new(cls, p: "Problem", signs: torch.Tensor, beta_pm: int = 50, rho_pm: int = 100) -> "Paris":
        rows, dev = p.batch * p.n_kv_heads, signs.device
        return cls(signs=signs, beta_pm=beta_pm, rho_pm=rho_pm,
                   cent=torch.zeros((rows, p.max_len, 16), dtype=torch.uint8, device=dev),
                   rec=torch.zeros((rows, p.max_len, 32), dtype=torch.int32, device=dev),
                   hist=torch.empty((rows, 16, 256), dtype=torch.int32, device=dev))

    @property
    def code(self) -> torch.Tensor:
        """[rows, max_len, 16] code words (a view of the records)."""
        return self.rec[..., :16]

    @property
    def w(self) -> torch.Tensor:
        """[rows, max_len, 16] fp32 weights (a view of the records)."""
        return self.rec[..., 16:].view(torch.float32)

    def c(self) -> CParis:
        return CParis(self.m, self.beta_pm, self.rho_pm, self.signs.data_ptr())

    def c_index(self) -> CParisIndex:
        return CParisIndex(self.cent.data_ptr(), self.rec.data_ptr(), self.hist.data_ptr())


def skv_paris_quantizer(m: int = 8):
    lv, th = (ctypes.c_float * 8)(), (ctypes.c_float * 7)()
    _check("skv_paris_quantizer", lib().skv_paris_quantizer(int(m), ctypes.cast(lv, ctypes.c_void_p),
                                                            ctypes.cast(th, ctypes.c_void_p)))
    return list(lv), list(th)


def skv_paris_encode(p: Problem, paris: Paris, index: IndexSrc, pool: Pool, dev_status=None, stream=None):
    cp, cpr, ci, cpool, cix = p.c(), paris.c(), index.c(), pool.c(), paris.c_index()
    _check("skv_paris_encode", lib().skv_paris_encode(ctypes.byref(cp), ctypes.byref(cpr), ctypes.byref(ci),
                                                      ctypes.byref(cpool), ctypes.byref(cix), _ptr(dev_status),
                                                      _stream(stream)))


def skv_paris_workspace_size(p: Problem, paris: Paris) -> int:
    n = ctypes.c_size_t(0)
    cp, cpr = p.c(), paris.c()
    _check("skv_paris_workspace_size", lib().skv_paris_workspace_size(ctypes.byref(cp), ctypes.byref(cpr),
                                                                      ctypes.byref(n)))
    return n.value


def skv_paris_workspace_offsets(p: Problem, paris: Paris) -> list:
    out = (ctypes.c_int64 * 9)()
    cp, cpr = p.c(), paris.c()
    _check("skv_paris_workspace_offsets", lib().skv_paris_workspace_offsets(
        ctypes.byref(cp), ctypes.byref(cpr), ctypes.cast(out, ctypes.c_void_p)))
    return list(out)


def skv_paris_select(p: Problem, paris: Paris, q_score, index: IndexSrc, pool: Pool, idx, ws, dev_status=None,
                     stream=None):
    cp, cpr, ci, cpool, cix = p.c(), paris.c(), index.c(), pool.c(), paris.c_index()
    _check("skv_paris_select", lib().skv_paris_select(
        ctypes.byref(cp), ctypes.byref(cpr), _ptr(q_score), ctypes.byref(ci), ctypes.byref(cix), ctypes.byref(cpool),
        _ptr(idx), _ptr(ws), ws.numel() * ws.element_size(), _ptr(dev_status), _stream(stream)))


def skv_paris_decode_step(p: Problem, paris: Paris, q, q_score, index: IndexSrc, pool: Pool, idx, out, lse, ws,
                          dev_status=None, stream=None):
    cp, cpr, ci, cpool, cix = p.c(), paris.c(), index.c(), pool.c(), paris.c_index()
    _check("skv_paris_decode_step", lib().skv_paris_decode_step(
        ctypes.byref(cp), ctypes.byref(cpr), _ptr(q), _ptr(q_score), ctypes.byref(ci), ctypes.byref(cix),
        ctypes.byref(cpool), _ptr(idx), _ptr(out), _ptr(lse), _ptr(ws), ws.numel() * ws.element_size(),
        _ptr(dev_status), _stream(stream)))


def skv_status_string(status: int) -> str:
    return lib().skv_status_string(status).decode()


def skv_launch_count() -> int:
    return int(lib().skv_launch_count())


def skv_check_wait_timeout(limit_cycles: int, arrive: int, dev_status, stream=None):
    _check("skv_check_wait_timeout", lib().skv_check_wait_timeout(int(limit_cycles), int(arrive), _ptr(dev_status),
                                                                  _stream(stream)))
