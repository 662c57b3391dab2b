"""Threshold prefetch of host rows (ECHO-OSDI26 wiki, core methods 3 and 5): the
results are the same bits with and without it, and the staged rows are the host rows."""

import numpy as np
import pytest
import torch

import workloads
from skv_test_utils import nv

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
            for b in range(wl.B):
                kth = np.sort(ref.scores[b, 0].cpu().numpy()[: int(wl.seq_lens[b])])[::-1][wl.k - 1]
                assert float(pf.tau_ema[b]) == kth
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
