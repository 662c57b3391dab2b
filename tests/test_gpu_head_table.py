"""One slot-table row per (request, KV head) (skv_kv_pool.table_heads = 1) on the GPU.

The same logical K/V laid out per head (each (request, head, block) at its own GPU slot
of a one-head block pool, or in the host pool) must give the shared-table step bit for
bit: placement never changes results.  Also checked against the oracle's per-head pool,
and the gather's rows against the generator's logical rows.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from skv_test_utils import OracleView, assert_attention_close, nv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def skv():
    import __graft_entry__

    __graft_entry__.build()
    import top_sparse_kv_gb300 as m

    return m


def _head_table_step(skv, wl, lay, agg=0, n_splits=0):
    base = skv.DecodeStep.from_workload(wl, n_splits=n_splits, group_agg=agg)
    pool = skv.Pool(lay["gpu_k"], lay["gpu_v"], lay["table"], lay["host_k"], lay["host_v"], table_heads=1)
    return base, skv.DecodeStep(base.p, pool, base.q, base.index, q_score=base.q_score)


def _run(step):
    step.scores.fill_(float("nan"))
    step.run()
    torch.cuda.synchronize()
    return int(step.status.item())


CASES = [
    ("gqa32b", dict(B=3, H=2, Hq=16, L=2000, k=150), [2000, 1377, 140], 0.0, 1.0, torch.bfloat16, "mean"),
    ("gqa32b", dict(B=2, H=2, Hq=8, L=1500, k=90), [1500, 999], 0.3, 0.5, torch.bfloat16, "mean"),
    ("gqa32b", dict(B=2, H=2, Hq=8, L=1500, k=90), [1500, 999], 0.0, 0.0, torch.bfloat16, "mean"),  # all host
    ("gqa32b", dict(B=2, H=2, Hq=8, L=1000, k=60), [1000, 700], 0.2, 0.7, torch.float32, "mean"),
    ("gqa32b", dict(B=2, H=2, Hq=16, L=1500, k=90), None, 0.0, 0.8, torch.bfloat16, "max"),
    ("gqa32b", dict(B=2, H=2, Hq=16, L=1500, k=90), [1500, 1200], 0.0, 0.8, torch.bfloat16, "head"),
    ("host1m", dict(L=20000, k=100), None, 0.0, 0.25, torch.bfloat16, "mean"),  # contiguous index keys
]


@pytest.mark.parametrize("name,over,lens,host_frac,gpu_frac,dtype,agg", CASES)
def test_head_table_step_equals_the_shared_table_step(skv, name, over, lens, host_frac, gpu_frac, dtype, agg):
    wl = workloads.make_workload(name, device="cuda", gen_device="cpu", seq_lens=lens, host_frac=host_frac,
                                 dtype=dtype, **over)
    code = {"mean": skv.SKV_AGG_MEAN, "max": skv.SKV_AGG_MAX, "head": skv.SKV_AGG_HEAD}[agg]
    lay = workloads.head_table_layout(wl, gpu_frac=gpu_frac, seed=7)
    base, per_head = _head_table_step(skv, wl, lay, code)
    assert _run(base) == 0
    assert _run(per_head) == 0
    for b in range(wl.B):
        L = int(wl.seq_lens[b])
        s_end, l_start = oracle.regions(L, wl.ns, wl.nl)
        assert torch.equal(per_head.scores[b, :, s_end:l_start], base.scores[b, :, s_end:l_start])
    assert torch.equal(per_head.idx, base.idx)
    assert torch.equal(per_head.out, base.out)
    assert torch.equal(per_head.lse, base.lse)


def test_head_table_step_matches_the_oracle(skv):
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=2, H=2, Hq=8, L=1200, k=80,
                                 seq_lens=[1200, 801], host_frac=0.2)
    lay = workloads.head_table_layout(wl, gpu_frac=0.5, seed=11)
    _, step = _head_table_step(skv, wl, lay)
    assert _run(step) == 0
    view = OracleView(wl)
    tbl = nv(lay["table"])
    kp = oracle.HeadTablePool(nv(lay["gpu_k"]), nv(lay["host_k"]), tbl, wl.bs)
    vp = oracle.HeadTablePool(nv(lay["gpu_v"]), nv(lay["host_v"]), tbl, wl.bs)
    scores = step.scores.cpu().numpy()
    idx = step.idx.cpu().numpy()
    G = wl.G
    for b in range(wl.B):
        for h in range(wl.H):
            ref = oracle.decode_unit(view.prob, b, h, view.q, kp, vp, given_scores=scores[b, h])
            np.testing.assert_array_equal(idx[b, h][: len(ref["idx"])], ref["idx"])
            assert_attention_close(step.out[b, h * G:(h + 1) * G], ref["out"], torch.bfloat16)
            np.testing.assert_allclose(step.lse[b, h * G:(h + 1) * G].cpu().numpy(), ref["lse"], rtol=1e-5,
                                       atol=1e-5)


def test_head_table_gather_gives_each_heads_rows(skv):
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=2, H=3, Hq=6, L=900, k=50,
                                 seq_lens=[900, 433], host_frac=0.3, keep_logical=True)
    lay = workloads.head_table_layout(wl, gpu_frac=0.5, seed=13)
    _, step = _head_table_step(skv, wl, lay)
    assert _run(step) == 0
    n_att = wl.ns + wl.k + wl.nl
    k_out = torch.empty((wl.B, wl.H, n_att, wl.d_qk), dtype=wl.q.dtype, device="cuda")
    v_out = torch.empty_like(k_out)
    skv.skv_gather(step.p, step.pool, step.idx, k_out, v_out, step.status)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    lk = wl.meta["logical_k"].to("cuda")
    lv = wl.meta["logical_v"].to("cuda")
    idx = step.idx.cpu()
    for b, L in enumerate((900, 433)):
        s_end, l_start = oracle.regions(L, wl.ns, wl.nl)
        for h in range(wl.H):
            listing = list(range(s_end)) + idx[b, h].tolist() + list(range(l_start, L))
            listing += [-1] * (n_att - len(listing))
            t = torch.tensor(listing, device="cuda")
            ok = t >= 0
            assert torch.equal(k_out[b, h, ok], lk[b, h, t[ok]])
            assert torch.equal(v_out[b, h, ok], lv[b, h, t[ok]])
            assert not k_out[b, h, ~ok].any() and not v_out[b, h, ~ok].any()


def test_head_table_bad_entry_is_flagged(skv):
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=1, H=2, Hq=8, L=800, k=40)
    lay = workloads.head_table_layout(wl, gpu_frac=1.0, seed=1)
    lay["table"][0, 1, 5] = 10 ** 6  # past the GPU pool, in head 1's row only
    _, step = _head_table_step(skv, wl, lay)
    assert _run(step) == skv.SKV_DEV_BAD_SLOT


def test_head_table_full_size_gqa32b_equals_the_shared_table(skv):
    """gqa32b at its full size (B8, 8 KV x 64 q heads, L32768, k3277), every block resident
    at its own per-head slot: the same step as the shared table, bit for bit."""
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cuda")
    lay = workloads.head_table_layout(wl, gpu_frac=1.0, seed=2)
    base, per_head = _head_table_step(skv, wl, lay)
    assert _run(base) == 0
    assert _run(per_head) == 0
    assert torch.equal(per_head.idx, base.idx)
    assert torch.equal(per_head.out, base.out)
    assert torch.equal(per_head.lse, base.lse)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_head_table_slot_cache_matches_the_oracle_over_steps(skv, dtype):
    """The slot cache over per-head tables (f4 on K/V pools): after every step of a drifting
    query, table, owners and priorities equal oracle.cache_update_heads bit for bit, the
    promoted slots hold their host rows, and idx, out and lse equal the step without a cache."""
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=2, H=2, Hq=8, L=1200, k=60,
                                 seq_lens=[1200, 900], dtype=dtype)
    lay = workloads.head_table_layout(wl, gpu_frac=0.3, seed=17)
    spare = 24  # free slots besides the resident blocks
    gpu_k = torch.cat([lay["gpu_k"], torch.zeros((spare,) + tuple(lay["gpu_k"].shape[1:]), dtype=wl.dtype,
                                                 device="cuda")])
    gpu_v = torch.cat([lay["gpu_v"], torch.zeros((spare,) + tuple(lay["gpu_v"].shape[1:]), dtype=wl.dtype,
                                                 device="cuda")])
    base = skv.DecodeStep.from_workload(wl)
    pool = skv.Pool(gpu_k, gpu_v, lay["table"].clone(), lay["host_k"], lay["host_v"], table_heads=1)
    step = skv.DecodeStep(base.p, pool, base.q.clone(), base.index, q_score=base.q_score)
    budget = 16
    cache = step.enable_cache(budget)
    rng = np.random.default_rng(19)
    q0 = wl.q.float().cpu().numpy()
    qn = q0.copy()
    host_k, host_v = lay["host_k"], lay["host_v"]
    H, stride, bs = wl.H, lay["table"].shape[2], wl.bs
    totals = np.zeros(3, dtype=np.int64)
    for it in range(6):
        qn = 0.8 * qn + 0.6 * rng.standard_normal(qn.shape)
        qt = torch.from_numpy(qn.astype(np.float32)).to(dtype).cuda()
        step.q.copy_(qt)
        base.q.copy_(qt)
        table0 = nv(pool.slot_table).copy()
        owner0 = cache.owner.cpu().numpy().astype(np.int64)
        prio0 = cache.prio.cpu().numpy().astype(np.int64)
        stp = int(cache.step.item())
        step.run_cached()
        base.run()
        torch.cuda.synchronize()
        assert int(step.status.item()) == 0 and int(base.status.item()) == 0
        assert torch.equal(step.idx, base.idx) and torch.equal(step.out, base.out) and torch.equal(step.lse, base.lse)
        idx = step.idx.cpu().numpy()
        attended = []
        for b in range(wl.B):
            L = int(wl.seq_lens[b])
            attended.append([oracle.attended_positions(L, wl.ns, wl.nl, [t for t in idx[b, h] if t >= 0])
                             for h in range(H)])
        t2, o2, p2, promo = oracle.cache_update_heads(table0, owner0, prio0, stp, attended, bs, budget)
        np.testing.assert_array_equal(nv(pool.slot_table), t2)
        np.testing.assert_array_equal(cache.owner.cpu().numpy(), o2)
        np.testing.assert_array_equal(cache.prio.cpu().numpy(), p2)
        assert int(cache.step.item()) == stp + 1
        for sl, b, h, j in promo:
            hb = b * stride + j
            assert torch.equal(gpu_k[sl].cpu(), host_k[hb, h])
            assert torch.equal(gpu_v[sl].cpu(), host_v[hb, h])
        used = [(b, h, jb) for b in range(wl.B) for h in range(H) for jb in {t // bs for t in attended[b][h]}]
        hits = sum(1 for b, h, jb in used if table0[b, h, jb] >= 0)
        totals += np.array([hits, len(used) - hits, len(promo)])
    # the counters: blocks found in slots, blocks missed, promotions, over the six steps
    np.testing.assert_array_equal(cache.stats.cpu().numpy(), totals)
    assert totals[0] > 0 and totals[2] > 0
