"""Threshold prefetch of host rows (ECHO-OSDI26 wiki, core methods 3 and 5): the
results are the same bits with and without it, the staged rows are the host rows, and
on a drifting query the prediction, the staged positions, the selection and the
attention follow the fp64 oracle step by step."""

import math

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


def _plain(skv, wl):
    step = skv.DecodeStep.from_workload(wl)
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    return step


@pytest.mark.parametrize("cap", [4096, 8])
def test_prefetch_is_lossless_and_stages_host_rows(skv, cap):
    wl = workloads.make_workload("mla", device="cuda", gen_device="cpu", B=2, L=3000, k=256, seq_lens=[3000, 2500])
    ref = _plain(skv, wl)
    step = skv.DecodeStep.from_workload(wl)
    pf = step.enable_prefetch(cap)
    host_rows = nv(wl.host_k).reshape(wl.host_k.shape[0], -1)
    table = wl.table.cpu().numpy()
    for s in range(4):
        step.status.zero_()
        step.run_prefetch()
        torch.cuda.synchronize()
        assert int(step.status.item()) == 0
        assert torch.equal(step.idx, ref.idx) and torch.equal(step.out, ref.out) and torch.equal(step.lse, ref.lse)
        assert int(pf.epoch.item()) == s + 1 and int(pf.count.sum().item()) == 0  # the step's end reset them
        hits, misses = (int(x) for x in pf.stats.cpu())
        if s == 0:
            # no prediction yet: nothing staged; the EMA starts at the step's k-th score
            assert hits == 0 and misses > 0
            scores = ref.scores.cpu().numpy()
            for b in range(wl.B):
                s_end, l_start = oracle.regions(int(wl.seq_lens[b]), wl.ns, wl.nl)
                pos = np.arange(s_end, l_start)
                want = oracle.prefetch_step(float("nan"), scores[b, 0, pos], pos, table[b, pos] < 0, wl.k)
                assert float(pf.tau_ema[b]) == want["tau"] == want["kth"]
        else:
            assert hits > 0
        # every map entry tagged by this step names a staging slot holding that position's host row
        tag = s + 1
        m = pf.map.view(wl.B, -1).cpu().numpy()
        for b in range(wl.B):
            tagged = np.nonzero((m[b] >> 32) == tag)[0]
            if s > 0:
                assert len(tagged) > 0
            for t in tagged[:50]:
                slot = int(m[b, t] & 0xFFFFFFFF)
                assert slot < cap and table[b, t] < 0
                np.testing.assert_array_equal(nv(pf.staging[b, slot]).reshape(-1), host_rows[-table[b, t] - 1])


def test_prefetch_with_a_prediction_below_every_score_is_lossless(skv):
    wl = workloads.make_workload("mla", device="cuda", gen_device="cpu", B=2, L=2000, k=128)
    ref = _plain(skv, wl)
    step = skv.DecodeStep.from_workload(wl)
    pf = step.enable_prefetch(64)
    pf.tau_ema.fill_(-float("inf"))  # every host key qualifies: the cap decides what is staged
    step.run_prefetch()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    assert torch.equal(step.out, ref.out) and torch.equal(step.idx, ref.idx)


def test_prefetch_full_size_mla(skv):
    wl = workloads.make_workload("mla", device="cuda", gen_device="cuda")
    ref = _plain(skv, wl)
    out0, idx0 = ref.out.clone(), ref.idx.clone()
    del ref
    step = skv.DecodeStep.from_workload(wl)
    pf = step.enable_prefetch(4096)
    for _ in range(3):
        step.run_prefetch()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    assert torch.equal(step.idx, idx0) and torch.equal(step.out, out0)
    hits, misses = (int(x) for x in pf.stats.cpu())
    assert hits > misses  # after the first step the prediction stages most selected host rows


def test_prefetch_full_size_host1m(skv):
    # the paged host pool at the benchmarked size (8 KV heads x 1M tokens, 0.41 MB of host
    # K and V rows a step): three steps with prefetch equal the plain step bit for bit, and
    # from the second step on the staging serves most of the attended host rows
    wl = workloads.make_workload("host1m", device="cuda", gen_device="cuda")
    ref = _plain(skv, wl)
    out0, idx0, lse0 = ref.out.clone(), ref.idx.clone(), ref.lse.clone()
    del ref
    step = skv.DecodeStep.from_workload(wl)
    pf = step.enable_prefetch(4096)
    for _ in range(3):
        step.run_prefetch()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    assert torch.equal(step.idx, idx0) and torch.equal(step.out, out0) and torch.equal(step.lse, lse0)
    hits, misses = (int(x) for x in pf.stats.cpu())
    assert hits > misses


DRIFT_CASES = [
    ("mla", dict(B=2, L=3000, k=256), [3000, 2500], 4096),
    ("mla", dict(B=2, L=3000, k=256), [3000, 2500], 8),
    # a paged pool of 16-token blocks whose non-window blocks live on the host (K and V rows staged)
    ("host1m", dict(H=2, Hq=8, L=12000, k=100), None, 4096),
    ("host1m", dict(B=2, H=2, Hq=8, L=12000, k=100), [12000, 9001], 6),
]


@pytest.mark.parametrize("name,over,lens,cap", DRIFT_CASES)
def test_prefetch_follows_the_oracle_on_a_drifting_query(skv, name, over, lens, cap):
    # every step: q <- r q + sqrt(1 - r^2) n (attention and indexer queries alike), so the
    # k-th score moves and the EMA (alpha = 0.5) is exercised past its first value
    wl = workloads.make_workload(name, device="cuda", gen_device="cpu", seq_lens=lens, **over)
    step = skv.DecodeStep.from_workload(wl)
    pf = step.enable_prefetch(cap)
    view = OracleView(wl)
    table = nv(wl.table)
    r = math.cos(2 * math.pi / 16)
    gen = torch.Generator().manual_seed(77)
    shared_q = step.q_score.data_ptr() == step.q.data_ptr()  # the host-pool workload scores with q itself
    q, qi = step.q.float().cpu(), step.q_score.float().cpu()
    rows = wl.B * wl.H
    chain = [float("nan")] * rows  # the oracle's own prediction, chained in fp64
    for s in range(5):
        tau_prev = pf.tau_ema.cpu().numpy().astype(np.float64)
        step.status.zero_()
        step.run_prefetch()
        torch.cuda.synchronize()
        assert int(step.status.item()) == 0
        scores = step.scores.cpu().numpy()
        tau_gpu = pf.tau_ema.cpu().numpy().astype(np.float64)
        m = pf.map.view(rows, -1).cpu().numpy()
        view.q, view.q_idx = nv(step.q), nv(step.q_score)
        for b in range(wl.B):
            s_end, l_start = oracle.regions(int(wl.seq_lens[b]), wl.ns, wl.nl)
            pos = np.arange(s_end, l_start)
            on_host = table[b, pos // wl.bs] < 0
            for h in range(wl.H):
                row = b * wl.H + h
                # the decisions in the kernel's precision: its fp32 scores against its fp32 prediction
                want = oracle.prefetch_step(tau_prev[row], scores[b, h, pos], pos, on_host, wl.k, alpha=0.5,
                                            cap=cap)
                ulp = float(np.spacing(np.float32(abs(want["tau"]))))
                assert abs(tau_gpu[row] - want["tau"]) <= ulp, (s, row, tau_gpu[row], want["tau"])
                own = oracle.prefetch_step(chain[row], scores[b, h, pos], pos, on_host, wl.k, alpha=0.5)
                chain[row] = own["tau"]
                assert abs(tau_gpu[row] - chain[row]) <= 2 * ulp, (s, row, tau_gpu[row], chain[row])
                staged = np.nonzero((m[row] >> 32) == s + 1)[0]
                if s == 0:
                    assert len(want["eligible"]) == 0 and len(staged) == 0
                if len(want["eligible"]) <= cap:
                    np.testing.assert_array_equal(staged, want["eligible"])
                else:  # past the cap, which qualifying rows were staged first is not fixed
                    assert set(staged.tolist()) <= set(want["eligible"].tolist()) and len(staged) == cap
                if s > 0:
                    assert len(want["eligible"]) > 0
                # the step's selection and attention against the oracle directly
                ref = view.unit(b, h, given_scores=scores[b, h])
                got = step.idx[b, h].cpu().numpy()
                np.testing.assert_array_equal(got[: len(ref["idx"])], ref["idx"])
                assert_attention_close(step.out[b, h * wl.G:(h + 1) * wl.G], ref["out"], wl.dtype)
        q = r * q + math.sqrt(1 - r * r) * torch.randn(q.shape, generator=gen)
        step.q.copy_(q.to(step.q.dtype))
        if not shared_q:
            qi = r * qi + math.sqrt(1 - r * r) * torch.randn(qi.shape, generator=gen)
            step.q_score.copy_(qi.to(step.q_score.dtype))


@pytest.mark.parametrize("cap", [4096, 4])
def test_paged_prefetch_is_lossless_and_stages_k_and_v_rows(skv, cap):
    wl = workloads.make_workload("host1m", device="cuda", gen_device="cpu", B=2, H=2, Hq=8, L=20000, k=100,
                                 seq_lens=[20000, 15003])
    ref = _plain(skv, wl)
    step = skv.DecodeStep.from_workload(wl)
    pf = step.enable_prefetch(cap)
    table = wl.table.cpu().numpy()
    hk, hv = wl.host_k.cpu(), wl.host_v.cpu()
    rows = wl.B * wl.H
    for s in range(3):
        step.status.zero_()
        step.run_prefetch()
        torch.cuda.synchronize()
        assert int(step.status.item()) == 0
        assert torch.equal(step.idx, ref.idx) and torch.equal(step.out, ref.out) and torch.equal(step.lse, ref.lse)
        assert int(pf.epoch.item()) == s + 1 and int(pf.count.sum().item()) == 0  # the step's end reset them
        hits, misses = (int(x) for x in pf.stats.cpu())
        if s == 0:
            assert hits == 0 and misses > 0
        else:
            assert hits > 0
        m = pf.map.view(rows, -1).cpu().numpy()
        stg = pf.staging.cpu()
        for row in range(rows):
            b, h = divmod(row, wl.H)
            tagged = np.nonzero((m[row] >> 32) == s + 1)[0]
            if s > 0:
                assert len(tagged) > 0
            assert len(tagged) <= cap
            for t in tagged[:40]:
                slot = int(m[row, t] & 0xFFFFFFFF)
                e = int(table[b, t // 16])
                assert slot < cap and e < 0
                assert torch.equal(stg[0, row, slot], hk[-e - 1, h, t % 16])
                assert torch.equal(stg[1, row, slot], hv[-e - 1, h, t % 16])


@pytest.mark.parametrize("name,over", [("mla", dict(B=2, L=3000, k=256)),
                                        ("host1m", dict(H=2, Hq=8, L=12000, k=100))])
def test_prefetch_step_replays_from_a_cuda_graph(skv, name, over):
    # the prefetch state moves every step (EMA, tag, staging counts): a captured step
    # replayed three times gives the same bits as three eager steps from the same start
    wl = workloads.make_workload(name, device="cuda", gen_device="cpu", **over)
    eager = skv.DecodeStep.from_workload(wl)
    pe = eager.enable_prefetch(64)
    graphed = skv.DecodeStep.from_workload(wl)
    pg = graphed.enable_prefetch(64)
    graphed.run_prefetch()  # step 0 outside the graph, as eager step 0 below
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            graphed.run_prefetch()
    torch.cuda.current_stream().wait_stream(side)
    # capture recorded the step without running it: rewind the graphed state to after step 0
    eager.run_prefetch()
    torch.cuda.synchronize()
    for s in range(3):
        g.replay()
        eager.run_prefetch()
        torch.cuda.synchronize()
        assert int(graphed.status.item()) == 0 and int(eager.status.item()) == 0
        assert torch.equal(graphed.idx, eager.idx) and torch.equal(graphed.out, eager.out)
        assert torch.equal(pg.tau_ema, pe.tau_ema) and int(pg.epoch.item()) == int(pe.epoch.item())


def test_paged_prefetch_flags_bad_slots_and_stays_lossless_elsewhere(skv):
    wl = workloads.make_workload("host1m", device="cuda", gen_device="cpu", H=2, Hq=8, L=12000, k=100)
    wl.table[0, -1] = -(10 ** 7)  # the last local-window block points past the host pool
    ref = skv.DecodeStep.from_workload(wl)
    ref.run()
    step = skv.DecodeStep.from_workload(wl)
    step.enable_prefetch(4096)
    for _ in range(3):
        step.status.zero_()
        step.run_prefetch()
        torch.cuda.synchronize()
        assert int(step.status.item()) & skv.SKV_DEV_BAD_SLOT
        assert torch.equal(step.idx, ref.idx) and torch.equal(step.out, ref.out)
