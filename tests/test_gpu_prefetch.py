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


@pytest.mark.parametrize("cap", [4096, 8])
def test_prefetch_follows_the_oracle_on_a_drifting_query(skv, cap):
    # every step: q <- r q + sqrt(1 - r^2) n (attention and indexer queries alike), so the
    # k-th score moves and the EMA (alpha = 0.5) is exercised past its first value
    wl = workloads.make_workload("mla", device="cuda", gen_device="cpu", B=2, L=3000, k=256,
                                 seq_lens=[3000, 2500])
    step = skv.DecodeStep.from_workload(wl)
    pf = step.enable_prefetch(cap)
    view = OracleView(wl)
    table = nv(wl.table)
    r = math.cos(2 * math.pi / 16)
    gen = torch.Generator().manual_seed(77)
    q, qi = step.q.float().cpu(), step.q_score.float().cpu()
    chain = [float("nan")] * wl.B  # the oracle's own prediction, chained in fp64
    for s in range(5):
        tau_prev = pf.tau_ema.cpu().numpy().astype(np.float64)
        step.status.zero_()
        step.run_prefetch()
        torch.cuda.synchronize()
        assert int(step.status.item()) == 0
        scores = step.scores.cpu().numpy()
        tau_gpu = pf.tau_ema.cpu().numpy().astype(np.float64)
        m = pf.map.view(wl.B, -1).cpu().numpy()
        view.q, view.q_idx = nv(step.q), nv(step.q_score)
        for b in range(wl.B):
            s_end, l_start = oracle.regions(int(wl.seq_lens[b]), wl.ns, wl.nl)
            pos = np.arange(s_end, l_start)
            on_host = table[b, pos] < 0
            # the decisions in the kernel's precision: its fp32 scores against its fp32 prediction
            want = oracle.prefetch_step(tau_prev[b], scores[b, 0, pos], pos, on_host, wl.k, alpha=0.5, cap=cap)
            ulp = float(np.spacing(np.float32(abs(want["tau"]))))
            assert abs(tau_gpu[b] - want["tau"]) <= ulp, (s, b, tau_gpu[b], want["tau"])
            own = oracle.prefetch_step(chain[b], scores[b, 0, pos], pos, on_host, wl.k, alpha=0.5)
            chain[b] = own["tau"]
            assert abs(tau_gpu[b] - chain[b]) <= 2 * ulp, (s, b, tau_gpu[b], chain[b])
            staged = np.nonzero((m[b] >> 32) == s + 1)[0]
            if s == 0:
                assert len(want["eligible"]) == 0 and len(staged) == 0
            if len(want["eligible"]) <= cap:
                np.testing.assert_array_equal(staged, want["eligible"])
            else:  # past the cap, which qualifying rows were staged first is not fixed
                assert set(staged.tolist()) <= set(want["eligible"].tolist()) and len(staged) == cap
            if s > 0:
                assert len(want["eligible"]) > 0
            # the step's selection and attention against the oracle directly
            ref = view.unit(b, 0, given_scores=scores[b, 0])
            got = step.idx[b, 0].cpu().numpy()
            np.testing.assert_array_equal(got[: len(ref["idx"])], ref["idx"])
            assert_attention_close(step.out[b], ref["out"], wl.dtype)
        n = torch.randn(q.shape, generator=gen)
        q = r * q + math.sqrt(1 - r * r) * n
        qi = r * qi + math.sqrt(1 - r * r) * torch.randn(qi.shape, generator=gen)
        step.q.copy_(q.to(step.q.dtype))
        step.q_score.copy_(qi.to(step.q_score.dtype))
