"""Seeded synthetic inputs for the sparse-decode step.

This module only draws inputs.  It holds none of the step's arithmetic (no scores,
no selection, no attention) and imports neither the CUDA library nor the oracle;
both sides are fed from here.

Workloads (sizes follow the pages' model classes; the data is synthetic because
the pages' datasets and models are not available):

  tiny     B1, 1 KV x 8 q heads, d128, L4096, k256 + 4 sink + 64 local; identity
           16-token blocks; q,k,v ~ N(0,1); 1% planted heavy keys.
  gqa32b   B8, 8 KV x 64 q heads, d128, L32768, k3277 (10%) + 4 sink + 128 local;
           paged GPU pool of 16-token blocks with a seeded random physical block
           permutation; q,k,v ~ N(0,1); 1% heavy keys per head.
  host1m   B1, 8 KV x 32 q heads, d128, L1048576, k100 + 16 sink + 512 local; the
           blocks holding sink/local positions sit in the GPU pool, every block is
           backed in pinned host memory and the table sends the rest there; keys
           from a 64-component Gaussian mixture whose means drift linearly with
           position; a GPU-resident contiguous copy of the keys is the index.
  mla      B16, L131072, one shared 576-wide latent row per token (512 latent + 64
           rope), 128 absorbed q heads, a single-head d128 indexer, k2048, no
           sink/local; latent rows in pinned host memory, a GPU slot cache holds
           25% of each request's tokens via a seeded random token -> slot map.
  sweep    B in {1,4,16,64} x L in {8K,32K,128K} x k in {256,1024,4096}; 8 KV x 64 q
           heads, d128, 4 sink + 128 local, random block permutation.

Heavy keys: k_t += 3 * u at 1% of positions (uniform without replacement), where u
is the unit direction of the group's mean query; values are drawn after rounding q
to the storage type so the direction is that of the stored query.
"""

from __future__ import annotations

import itertools
import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch

CONFIG_NAMES = ("tiny", "gqa32b", "host1m", "mla", "sweep")

BASE = {
    "tiny": dict(B=1, H=1, Hq=8, d_qk=128, d_v=128, L=4096, k=256, ns=4, nl=64, bs=16,
                 layout="paged", permute=False, heavy=0.01, keys="normal"),
    "gqa32b": dict(B=8, H=8, Hq=64, d_qk=128, d_v=128, L=32768, k=3277, ns=4, nl=128, bs=16,
                   layout="paged", permute=True, heavy=0.01, keys="normal"),
    "host1m": dict(B=1, H=8, Hq=32, d_qk=128, d_v=128, L=1048576, k=100, ns=16, nl=512, bs=16,
                   layout="host_paged", permute=False, heavy=0.0, keys="mixture"),
    "mla": dict(B=16, H=1, Hq=128, d_qk=576, d_v=512, d_idx=128, L=131072, k=2048, ns=0, nl=0,
                bs=1, layout="latent", gpu_cache_frac=0.25, keys="normal", heavy=0.0),
    "sweep": dict(B=1, H=8, Hq=64, d_qk=128, d_v=128, L=8192, k=256, ns=4, nl=128, bs=16,
                  layout="paged", permute=True, heavy=0.01, keys="normal"),
}

SWEEP_POINTS = list(itertools.product((1, 4, 16, 64), (8192, 32768, 131072), (256, 1024, 4096)))


def seed_for(name: str, point: Optional[int] = None) -> int:
    if name == "sweep" and point is not None:
        return 2000 + point
    return 1000 + CONFIG_NAMES.index(name)


@dataclass
class Workload:
    """Tensors of one decode step plus their sizes.

    Device tensors live on `device`; host pools are pinned CPU tensors when the
    target device is CUDA (plain CPU tensors otherwise).
    """

    name: str
    B: int
    H: int
    Hq: int
    d_qk: int
    d_v: int
    d_idx: int
    L: int  # max history length (table capacity)
    k: int
    ns: int
    nl: int
    bs: int
    layout: str  # "paged" | "host_paged" | "latent"
    dtype: torch.dtype
    seq_lens: torch.Tensor  # int32 [B]
    q: torch.Tensor  # [B, Hq, d_qk]
    table: torch.Tensor  # int32 [B, n_entries]
    gpu_k: torch.Tensor  # [NBg, H, bs, d_qk]
    gpu_v: Optional[torch.Tensor]  # [NBg, H, bs, d_v] (None: V = leading dims of the K row)
    host_k: Optional[torch.Tensor] = None
    host_v: Optional[torch.Tensor] = None
    q_idx: Optional[torch.Tensor] = None  # [B, H * G_idx, d_idx]
    index_keys: Optional[torch.Tensor] = None  # [B, H, L, d_idx]
    sm_scale: float = 0.0
    meta: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return self.Hq // self.H

    @property
    def index_layout(self) -> str:
        return "contig" if self.index_keys is not None else "paged"

    def tensors(self):
        out = {}
        for k_, v_ in self.__dict__.items():
            if isinstance(v_, torch.Tensor):
                out[k_] = v_
        return out


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def _pin(t: torch.Tensor, device) -> torch.Tensor:
    t = t.to("cpu")
    if torch.device(device).type == "cuda":
        t = t.pin_memory()
    return t


def _heavy_positions(B, H, L, frac, g, device):
    n = int(round(frac * L))
    if n == 0:
        return None
    r = torch.rand((B, H, L), generator=g, device=device)
    return r.argsort(dim=-1)[..., :n]


def _plant_heavy(keys, q_store, H, pos):
    """keys [B,H,L,d] fp32 += 3 * unit(mean of the group's stored queries) at pos."""
    B, Hq, d = q_store.shape
    G = Hq // H
    direction = q_store.float().view(B, H, G, d).mean(dim=2)
    direction = direction / direction.norm(dim=-1, keepdim=True)
    add = (3.0 * direction)[:, :, None, :].expand(B, H, pos.shape[-1], d)
    keys.scatter_add_(2, pos[..., None].expand(B, H, pos.shape[-1], d), add)


def _to_paged(logical, table_np_blocks, n_blocks, bs):
    """logical [B, H, L, d] -> pool [n_blocks, H, bs, d] using phys = table[b, j]."""
    B, H, L, d = logical.shape
    nblk = -(-L // bs)
    pad = nblk * bs - L
    if pad:
        logical = torch.nn.functional.pad(logical, (0, 0, 0, pad))
    blocks = logical.view(B, H, nblk, bs, d).permute(0, 2, 1, 3, 4).reshape(B * nblk, H, bs, d)
    pool = torch.zeros((n_blocks, H, bs, d), dtype=logical.dtype, device=logical.device)
    pool[table_np_blocks.reshape(-1).long()] = blocks
    return pool


def make_workload(
    name: str,
    device="cpu",
    gen_device=None,
    dtype: torch.dtype = torch.bfloat16,
    seed: Optional[int] = None,
    seq_lens: Optional[Sequence[int]] = None,
    host_frac: float = 0.0,
    keep_logical: bool = False,
    **over,
) -> Workload:
    """Draw one workload.  `over` overrides sizes (B, H, Hq, L, k, ns, nl, ...).

    seq_lens:  per-request history lengths (<= L); default all L.
    host_frac: for paged layouts, the fraction of blocks placed in the host pool
               instead of the GPU pool (seeded choice), to exercise the host tier.
    keep_logical: keep the logical [B, H, L, d] keys/values (or [B, L, d] latent
               rows) in `meta` so tests can check addressing against them.
    """
    logical = {}
    if name not in BASE:
        raise KeyError(name)
    cfg = dict(BASE[name])
    cfg.update(over)
    seed = seed_for(name) if seed is None else seed
    gdev = torch.device(gen_device if gen_device is not None else device)
    g = _gen(seed, gdev)
    B, H, Hq, L = cfg["B"], cfg["H"], cfg["Hq"], cfg["L"]
    d_qk, d_v, bs = cfg["d_qk"], cfg["d_v"], cfg["bs"]
    if Hq % H:
        raise ValueError("Hq must be a multiple of H")
    lens = [L] * B if seq_lens is None else [int(x) for x in seq_lens]
    if len(lens) != B or max(lens) > L or min(lens) < 0:
        raise ValueError("bad seq_lens")
    layout = cfg["layout"]
    dev = torch.device(device)

    q = _randn((B, Hq, d_qk), g, gdev).to(dtype)

    if layout == "paged":
        # drawn one request at a time, so peak memory stays a few times one request's KV
        nblk = -(-L // bs)
        total = B * nblk
        perm = torch.randperm(total, generator=g, device=gdev) if cfg.get("permute") else \
            torch.arange(total, device=gdev)
        phys = perm.view(B, nblk).to(torch.int32)
        pool_k = torch.zeros((total, H, bs, d_qk), dtype=dtype, device=gdev)
        pool_v = torch.zeros((total, H, bs, d_v), dtype=dtype, device=gdev)
        lk, lv = [], []
        for b in range(B):
            kb = _randn((1, H, L, d_qk), g, gdev)
            pos = _heavy_positions(1, H, L, cfg.get("heavy", 0.0), g, gdev)
            if pos is not None:
                _plant_heavy(kb, q[b:b + 1], H, pos)
            kb = kb.to(dtype)
            vb = _randn((1, H, L, d_v), g, gdev).to(dtype)
            pool_k[phys[b].long()] = _to_paged(kb, torch.arange(nblk, device=gdev, dtype=torch.int32), nblk, bs)
            pool_v[phys[b].long()] = _to_paged(vb, torch.arange(nblk, device=gdev, dtype=torch.int32), nblk, bs)
            if keep_logical:
                lk.append(kb)
                lv.append(vb)
            del kb, vb
        if keep_logical:
            logical = dict(logical_k=torch.cat(lk), logical_v=torch.cat(lv))
        table = phys.clone()
        host_k = host_v = None
        if host_frac > 0.0:
            table, pool_k, pool_v, host_k, host_v = _split_tiers(
                table, pool_k, pool_v, host_frac, g, gdev)
        wl = Workload(name, B, H, Hq, d_qk, d_v, d_qk, L, cfg["k"], cfg["ns"], cfg["nl"], bs,
                      layout, dtype, torch.tensor(lens, dtype=torch.int32), q, table,
                      pool_k, pool_v, host_k, host_v)
    elif layout == "host_paged":  # every block backed on the host, sink/local blocks in the GPU pool
        if cfg["keys"] == "mixture":
            keys = _mixture_keys(B, H, L, d_qk, g, gdev)
        else:
            keys = _randn((B, H, L, d_qk), g, gdev)
        pos = _heavy_positions(B, H, L, cfg.get("heavy", 0.0), g, gdev)
        if pos is not None:
            _plant_heavy(keys, q, H, pos)
        keys = keys.to(dtype)
        values = _randn((B, H, L, d_v), g, gdev).to(dtype)
        if keep_logical:
            logical = dict(logical_k=keys, logical_v=values)
        nblk = -(-L // bs)
        total = B * nblk
        ident = torch.arange(total, device=gdev, dtype=torch.int32).view(B, nblk)
        host_k_full = _to_paged(keys, ident, total, bs)
        host_v_full = _to_paged(values, ident, total, bs)
        resident = torch.zeros((B, nblk), dtype=torch.bool, device=gdev)
        for b in range(B):
            Lb = lens[b]
            s_end = min(cfg["ns"], Lb)
            l_start = max(s_end, Lb - cfg["nl"])
            if s_end > 0:
                resident[b, 0:-(-s_end // bs)] = True
            if Lb > l_start:
                resident[b, l_start // bs: -(-Lb // bs)] = True
        flat = resident.view(-1).nonzero().view(-1)
        gpu_slots = torch.full((total,), -1, dtype=torch.int64, device=gdev)
        gpu_slots[flat] = torch.arange(flat.numel(), device=gdev)
        table = torch.where(gpu_slots >= 0, gpu_slots,
                            -torch.arange(total, device=gdev) - 1).view(B, nblk).to(torch.int32)
        gpu_k = host_k_full[flat].clone()
        gpu_v = host_v_full[flat].clone()
        wl = Workload(name, B, H, Hq, d_qk, d_v, d_qk, L, cfg["k"], cfg["ns"], cfg["nl"], bs,
                      layout, dtype, torch.tensor(lens, dtype=torch.int32), q, table,
                      gpu_k, gpu_v, host_k_full, host_v_full)
        # GPU-resident contiguous copy of the keys is the index (scored in place of the pool)
        wl.index_keys = keys
        wl.q_idx = q
    elif layout == "latent":
        d_idx = cfg["d_idx"]
        latent = _randn((B * L, d_qk), g, gdev).to(dtype)
        if keep_logical:
            logical = dict(logical_latent=latent.view(B, L, d_qk))
        index_keys = _randn((B, H, L, d_idx), g, gdev).to(dtype)
        q_idx = _randn((B, H, d_idx), g, gdev).to(dtype)
        per_req = int(round(cfg["gpu_cache_frac"] * L))
        n_cache = per_req * B
        cached = torch.rand((B, L), generator=g, device=gdev).argsort(dim=-1)[:, :per_req]
        slots = torch.randperm(n_cache, generator=g, device=gdev).view(B, per_req)
        tok = torch.arange(L, device=gdev)
        table = (-(torch.arange(B, device=gdev)[:, None] * L + tok[None, :]) - 1).to(torch.int64)
        table.scatter_(1, cached, slots)
        table = table.to(torch.int32)
        gpu_cache = torch.zeros((max(n_cache, 1), d_qk), dtype=dtype, device=gdev)
        src_rows = (torch.arange(B, device=gdev)[:, None] * L + cached).view(-1)
        gpu_cache[slots.view(-1)] = latent[src_rows]
        wl = Workload(name, B, H, Hq, d_qk, d_v, d_idx, L, cfg["k"], cfg["ns"], cfg["nl"], 1,
                      layout, dtype, torch.tensor(lens, dtype=torch.int32), q, table,
                      gpu_cache.view(-1, 1, 1, d_qk), None,
                      latent.view(-1, 1, 1, d_qk), None, q_idx, index_keys)
    else:
        raise ValueError(layout)

    wl.sm_scale = 1.0 / math.sqrt(d_qk)
    wl.meta = dict(seed=seed, config=cfg, host_frac=host_frac, **logical)
    return _place(wl, dev)


def head_table_layout(wl: Workload, gpu_frac: float = 1.0, seed: int = 0) -> dict:
    """The same logical K/V as the paged workload `wl`, laid out for one slot-table row
    per (request, KV head): every (request, head, block) is resident on the GPU with
    probability gpu_frac (seeded), at a seeded random slot of a pool whose blocks hold
    one head's rows ([n_slots, bs, d]); every block is backed by a host pool that keeps
    all heads ([B * stride, H, bs, d], block j of request b at host block b * stride + j).
    Returns gpu_k, gpu_v, host_k, host_v and table ([B, H, stride] int32) on wl's device
    (host pools pinned when that is a CUDA device)."""
    if wl.layout not in ("paged", "host_paged") or wl.gpu_v is None:
        raise ValueError("a paged K/V workload")
    dev = wl.q.device
    B, H, bs = wl.B, wl.H, wl.bs
    stride = wl.table.shape[1]
    t = wl.table.to(dev).long()

    def logical_blocks(gpu, host):  # [B, stride, H, bs, d] through the shared table
        out = torch.empty((B, stride) + tuple(gpu.shape[1:]), dtype=gpu.dtype, device=dev)
        on_gpu = t >= 0
        out[on_gpu] = gpu.to(dev)[t[on_gpu]]
        if bool((~on_gpu).any()):
            out[~on_gpu] = host.to(dev)[-t[~on_gpu] - 1]
        return out

    lk = logical_blocks(wl.gpu_k, wl.host_k)
    lv = logical_blocks(wl.gpu_v, wl.host_v)
    g = _gen(seed, "cpu")
    n = B * H * stride
    resident = torch.rand(n, generator=g) < gpu_frac
    n_res = int(resident.sum())
    slot = torch.full((n,), -1, dtype=torch.int64)
    slot[resident] = torch.randperm(n_res, generator=g)
    bb = torch.arange(B).view(B, 1, 1).expand(B, H, stride).reshape(-1)
    jj = torch.arange(stride).view(1, 1, stride).expand(B, H, stride).reshape(-1)
    table = torch.where(slot >= 0, slot, -(bb * stride + jj) - 1).view(B, H, stride).to(torch.int32)
    per_head_k = lk.permute(0, 2, 1, 3, 4).reshape(n, bs, -1)  # (b, h, j) blocks of one head
    per_head_v = lv.permute(0, 2, 1, 3, 4).reshape(n, bs, -1)
    res = resident.to(dev)
    dst = slot[resident].to(dev)
    gpu_k = torch.zeros((max(n_res, 1), bs, per_head_k.shape[-1]), dtype=lk.dtype, device=dev)
    gpu_v = torch.zeros((max(n_res, 1), bs, per_head_v.shape[-1]), dtype=lv.dtype, device=dev)
    gpu_k[dst] = per_head_k[res]
    gpu_v[dst] = per_head_v[res]
    return dict(gpu_k=gpu_k, gpu_v=gpu_v, host_k=_pin(lk.reshape(B * stride, H, bs, -1), dev),
                host_v=_pin(lv.reshape(B * stride, H, bs, -1), dev), table=table.to(dev))


def _split_tiers(table, pool_k, pool_v, host_frac, g, gdev):
    """Move a seeded fraction of the physical blocks to a host pool; rewrite the table."""
    total = pool_k.shape[0]
    n_host = int(round(host_frac * total))
    order = torch.randperm(total, generator=g, device=gdev)
    host_blocks = order[:n_host]
    gpu_blocks = order[n_host:].sort().values
    new_gpu = torch.full((total,), -1, dtype=torch.int64, device=gdev)
    new_gpu[gpu_blocks] = torch.arange(gpu_blocks.numel(), device=gdev)
    new_host = torch.full((total,), -1, dtype=torch.int64, device=gdev)
    new_host[host_blocks] = torch.arange(n_host, device=gdev)
    t = table.long()
    remapped = torch.where(new_gpu[t] >= 0, new_gpu[t], -new_host[t] - 1)
    host_k = pool_k[host_blocks].clone()
    host_v = pool_v[host_blocks].clone()
    return (remapped.to(torch.int32), pool_k[gpu_blocks].clone(), pool_v[gpu_blocks].clone(),
            host_k, host_v)


def _mixture_keys(B, H, L, d, g, gdev, n_comp=64, sigma=0.5, chunk=1 << 18):
    """Keys per KV head from a 64-component mixture; component means drift linearly
    with position: mu_c(t) = mu_c + (t / L) * delta_c; within-component sd 0.5."""
    mu = _randn((H, n_comp, d), g, gdev)
    delta = _randn((H, n_comp, d), g, gdev)
    keys = torch.empty((B, H, L, d), dtype=torch.float32, device=gdev)
    for b in range(B):
        for t0 in range(0, L, chunk):
            t1 = min(L, t0 + chunk)
            n = t1 - t0
            comp = torch.randint(0, n_comp, (H, n), generator=g, device=gdev)
            frac = (torch.arange(t0, t1, device=gdev, dtype=torch.float32) / L)[None, :, None]
            hidx = torch.arange(H, device=gdev)[:, None]
            keys[b, :, t0:t1] = mu[hidx, comp] + frac * delta[hidx, comp] + \
                sigma * _randn((H, n, d), g, gdev)
    return keys


def _place(wl: Workload, dev: torch.device) -> Workload:
    for name in ("seq_lens", "q", "table", "gpu_k", "gpu_v", "q_idx", "index_keys"):
        t = getattr(wl, name)
        if t is not None:
            setattr(wl, name, t.to(dev).contiguous())
    for name in ("host_k", "host_v"):
        t = getattr(wl, name)
        if t is not None:
            setattr(wl, name, _pin(t.contiguous(), dev))
    return wl


def permute_blocks(wl: Workload, seed: int) -> Workload:
    """The same logical KV with the GPU pool's physical blocks shuffled (table rewritten).

    The pages state that moving a token's physical slot never changes its logical
    identity or contents (vToken notes §3.5, invariants I1/I2); results must not change.
    """
    g = _gen(seed, "cpu")
    n = wl.gpu_k.shape[0]
    perm = torch.randperm(n, generator=g).to(wl.gpu_k.device)  # new position of old block i
    new_k = torch.empty_like(wl.gpu_k)
    new_k[perm] = wl.gpu_k
    new_v = None
    if wl.gpu_v is not None:
        new_v = torch.empty_like(wl.gpu_v)
        new_v[perm] = wl.gpu_v
    t = wl.table.long()
    remap = torch.where(t >= 0, perm.to(t.device)[t.clamp(min=0)], t)
    out = Workload(**{**wl.__dict__})
    out.gpu_k, out.gpu_v, out.table = new_k, new_v, remap.to(torch.int32).contiguous()
    return out


def numpy_view(t: Optional[torch.Tensor]):
    """CPU numpy array of a tensor; bf16 tensors become uint16 bit patterns."""
    if t is None:
        return None
    t = t.detach().to("cpu")
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()


def srht_signs(D: int = 128, seed: int = 4711, device="cpu") -> torch.Tensor:
    """The random signs (+1 / -1, int8 [D]) a randomised Hadamard rotation draws: seeded
    input for ParisKV retrieval, generated here so that both sides receive the same."""
    g = torch.Generator().manual_seed(seed)
    s = torch.randint(0, 2, (D,), generator=g, dtype=torch.int8) * 2 - 1
    return s.to(device)
