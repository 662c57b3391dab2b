"""The per-query-head reading (SKV_AGG_HEAD) on the GPU against the fp64 oracle.

Every query head j scores the keys of its KV head j // G with its own query, keeps its
own exact top-k and attends its own list (oracle.decode_head).  Checked per head: the
scores within the fp32 accumulation bound, the selection bit for bit against the
oracle's exact top-k of the GPU's own scores (and within the tie band of the fp64
scores), and the attention output and lse on the GPU's selection.
"""

import numpy as np
import pytest
import torch

import workloads
from skv_test_utils import OracleView, assert_attention_close, check_band

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def skv():
    import __graft_entry__

    __graft_entry__.build()
    import top_sparse_kv_gb300 as m

    return m


HEAD_CASES = [
    ("gqa32b", dict(B=3, H=2, Hq=16, L=2000, k=150), [2000, 1377, 140], 0.0),   # G = 8, ragged, short row
    ("gqa32b", dict(B=2, H=2, Hq=32, L=1500, k=90), [1500, 1001], 0.0),         # G = 16: two 8-head tiles
    ("gqa32b", dict(B=1, H=2, Hq=14, L=1500, k=90), None, 0.0),                 # G = 7: a masked head
    ("gqa32b", dict(B=2, H=4, Hq=4, L=1000, k=60), [1000, 517], 0.0),           # G = 1
    ("gqa32b", dict(B=2, H=2, Hq=8, L=777, k=40), [777, 300], 0.4),             # host tier over UVA
    ("host1m", dict(L=20000, k=100), None, 0.0),                                # contiguous index keys
    ("tiny", dict(L=1000, k=2000), None, 0.0),                                  # k >= |C|: dense
]


def _head_step(skv, wl, n_splits=0):
    step = skv.DecodeStep.from_workload(wl, n_splits=n_splits, group_agg=skv.SKV_AGG_HEAD)
    assert tuple(step.scores.shape) == (wl.B, wl.Hq, wl.L) and step.idx.shape[1] == wl.Hq
    step.scores.fill_(float("nan"))
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    return step


@pytest.mark.parametrize("name,over,lens,host_frac", HEAD_CASES)
def test_per_head_step_matches_oracle(skv, name, over, lens, host_frac):
    wl = workloads.make_workload(name, device="cuda", gen_device="cpu", seq_lens=lens, host_frac=host_frac, **over)
    step = _head_step(skv, wl)
    view = OracleView(wl)
    scores = step.scores.cpu().numpy()
    idx = step.idx.cpu().numpy()
    out = step.out.float().cpu().numpy()
    lse = step.lse.cpu().numpy()
    for b in range(wl.B):
        for j in range(wl.Hq):
            ref = view.head(b, j)
            pos = ref["positions"]
            tol = view.head_score_tolerance(b, j, pos)
            got = scores[b, j, pos].astype(np.float64)
            assert np.all(np.abs(got - ref["scores"]) <= tol), (b, j, np.max(np.abs(got - ref["scores"]) / tol))
            mine = view.head(b, j, given_scores=scores[b, j])
            n = len(mine["idx"])
            np.testing.assert_array_equal(idx[b, j][:n], mine["idx"])
            assert np.all(idx[b, j][n:wl.k] < 0)
            check_band(idx[b, j], ref, wl.k)
            assert_attention_close(torch.from_numpy(out[b, j:j + 1]), mine["out"], torch.bfloat16)
            np.testing.assert_allclose(lse[b, j], mine["lse"][0], rtol=1e-5, atol=1e-5)


def test_per_head_split_counts_agree(skv):
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=2, H=2, Hq=16, L=3000, k=300)
    base = _head_step(skv, wl, n_splits=1)
    for s in (2, 7, 16):
        other = _head_step(skv, wl, n_splits=s)
        assert torch.equal(base.idx, other.idx)
        assert torch.allclose(base.out.float(), other.out.float(), atol=1e-2, rtol=0)
        assert torch.allclose(base.lse, other.lse, atol=1e-5, rtol=1e-5)


def test_per_head_gather_and_entry_points_compose(skv):
    """skv_score, skv_topk, skv_gather and skv_sparse_attn called one by one give the step's
    own results, and the gathered rows of query head j are the rows of KV head j // G."""
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=2, H=2, Hq=8, L=900, k=50,
                                 seq_lens=[900, 611], host_frac=0.3, keep_logical=True)
    step = _head_step(skv, wl)
    scores, idx, out, lse = (step.scores.clone(), step.idx.clone(), step.out.clone(), step.lse.clone())
    step.scores.fill_(float("nan"))
    step.idx.fill_(-7)
    step.score()
    step.topk()
    step.attend()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    for b, L in enumerate((900, 611)):
        s_end, l_start = wl.ns, L - wl.nl
        assert torch.equal(step.scores[b, :, s_end:l_start], scores[b, :, s_end:l_start])
    assert torch.equal(step.idx, idx)
    assert torch.equal(step.out, out) and torch.equal(step.lse, lse)

    n_att = wl.ns + wl.k + wl.nl
    k_out = torch.empty((wl.B, wl.Hq, n_att, wl.d_qk), dtype=wl.q.dtype, device="cuda")
    v_out = torch.empty((wl.B, wl.Hq, n_att, wl.d_v), dtype=wl.q.dtype, device="cuda")
    skv.skv_gather(step.p, step.pool, step.idx, k_out, v_out, step.status)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    lk = wl.meta["logical_k"].to("cuda")
    lv = wl.meta["logical_v"].to("cuda")
    G = wl.G
    for b, L in enumerate((900, 611)):
        s_end, l_start = wl.ns, L - wl.nl
        for j in range(wl.Hq):
            # sink, then the head's idx entries (empty ones give zero rows), then local
            listing = list(range(s_end)) + idx[b, j].cpu().tolist() + list(range(l_start, L))
            listing += [-1] * (n_att - len(listing))
            t = torch.tensor(listing, device="cuda")
            ok = t >= 0
            assert torch.equal(k_out[b, j, ok], lk[b, j // G, t[ok]])
            assert torch.equal(v_out[b, j, ok], lv[b, j // G, t[ok]])
            assert not k_out[b, j, ~ok].any() and not v_out[b, j, ~ok].any()


def test_per_head_differs_from_the_group_readings(skv):
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=1, H=2, Hq=16, L=3000, k=300)
    head = _head_step(skv, wl).idx.cpu().numpy()
    for agg in (skv.SKV_AGG_MEAN, skv.SKV_AGG_MAX):
        grp = skv.DecodeStep.from_workload(wl, group_agg=agg)
        grp.run()
        torch.cuda.synchronize()
        g = grp.idx.cpu().numpy()
        # the group's one list against each of its heads' own lists
        assert any(not np.array_equal(head[0, j], g[0, j // 8]) for j in range(16))


def test_per_head_full_size_gqa32b_sampled(skv):
    """The bench's workload (B8, 8 KV x 64 q heads, L32768, k3277) in the launch shape the
    bench times: sampled query heads against the oracle on the GPU's own scores."""
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cuda")
    step = _head_step(skv, wl)
    view = OracleView(wl)
    for b, j in ((0, 0), (3, 17), (7, 63)):
        scores = step.scores[b, j].cpu().numpy()
        ref = view.head(b, j)
        pos = ref["positions"]
        tol = view.head_score_tolerance(b, j, pos)
        assert np.all(np.abs(scores[pos].astype(np.float64) - ref["scores"]) <= tol)
        check_band(step.idx[b, j].cpu().numpy(), ref, wl.k)
        mine = view.head(b, j, given_scores=scores)
        np.testing.assert_array_equal(step.idx[b, j].cpu().numpy(), mine["idx"])
        assert_attention_close(step.out[b, j:j + 1], mine["out"], torch.bfloat16)
        np.testing.assert_allclose(step.lse[b, j].item(), mine["lse"][0], rtol=1e-5, atol=1e-5)
