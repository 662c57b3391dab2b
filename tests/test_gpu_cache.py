"""GPU slot cache over a host pool that backs every token (ECHO-OSDI26 wiki, core
method 2): the table, owners and priorities after each step equal the oracle's
update bit for bit, promoted slots hold their tokens' host rows, and the step's
results are those of the uncached step."""

import copy

import numpy as np
import pytest
import torch

import oracle
import workloads
from skv_test_utils import OracleView, check_band, nv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def skv():
    import __graft_entry__

    __graft_entry__.build()
    import top_sparse_kv_gb300 as m

    return m


def _twin(wl):
    """A copy of the workload with its own slot table and GPU pool (the uncached reference)."""
    t = copy.copy(wl)
    t.table = wl.table.clone()
    t.gpu_k = wl.gpu_k.clone()
    return t


def _attended(wl, step, view=None):
    """Per request, the attended positions in list order.  With `view`, the selection is
    first checked against the fp64 oracle's (equal up to positions within the fp32 band)."""
    idx = step.idx.cpu().numpy()
    att = []
    for b in range(wl.B):
        L = int(wl.seq_lens[b])
        sel = idx[b, 0][idx[b, 0] >= 0]
        if view is not None:
            check_band(idx[b, 0], view.unit(b, 0), wl.k)
        else:  # validity only: ascending, unique, inside the candidates
            s_end, l_start = oracle.regions(L, wl.ns, wl.nl)
            assert np.all(np.diff(sel) > 0) and (len(sel) == 0 or (sel[0] >= s_end and sel[-1] < l_start))
        att.append(oracle.attended_positions(L, wl.ns, wl.nl, sel))
    return att


def _state(wl, cache):
    return (wl.table.cpu().numpy().astype(np.int64), cache.owner.cpu().numpy().astype(np.int64),
            cache.prio.cpu().numpy().astype(np.int64))


def _check_step(wl, step, cache, before, s, attended, budget, host_rows):
    t0, o0, p0 = before
    want_t, want_o, want_p, promos = oracle.cache_update(t0, o0, p0, s, attended, wl.L, budget)
    got_t, got_o, got_p = _state(wl, cache)
    np.testing.assert_array_equal(got_t, want_t)
    np.testing.assert_array_equal(got_o, want_o)
    np.testing.assert_array_equal(got_p, want_p)
    assert int(cache.step.item()) == s + 1
    if promos:
        slots = torch.tensor([p[0] for p in promos], dtype=torch.long, device=wl.gpu_k.device)
        got = nv(wl.gpu_k.view(wl.gpu_k.shape[0], -1)[slots].cpu())
        rows = np.array([p[1] * wl.L + p[2] for p in promos])
        np.testing.assert_array_equal(got, host_rows[rows])
    return promos


def _fresh_queries(wl, twin, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(wl.q.shape, generator=g).to(wl.q.dtype)
    qi = torch.randn(wl.q_idx.shape, generator=g).to(wl.q_idx.dtype)
    for w in (wl, twin):
        w.q.copy_(q)
        w.q_idx.copy_(qi)


CASES = [
    # name, overrides, seq_lens, budget, steps
    (dict(B=3, L=3000, k=256), [3000, 2500, 1800], 512, 4),
    (dict(B=2, L=2000, k=300, ns=4, nl=64), [2000, 1500], 200, 3),   # sink and local windows in the list
    (dict(B=2, L=1500, k=128), None, 0, 2),                          # no promotions: priorities only
    (dict(B=2, L=1200, k=200), [1200, 900], 100000, 3),              # budget above the slot count
    (dict(B=3, L=1500, k=128, ns=4, nl=16), [1500, 0, 10], 300, 3),  # an empty history, one inside the windows
]


@pytest.mark.parametrize("over,lens,budget,steps", CASES)
def test_cache_update_matches_oracle(skv, over, lens, budget, steps):
    wl = workloads.make_workload("mla", device="cuda", gen_device="cpu", seq_lens=lens, **over)
    twin = _twin(wl)
    step = skv.DecodeStep.from_workload(wl)
    ref = skv.DecodeStep.from_workload(twin)
    cache = step.enable_cache(budget)
    n_slots = wl.gpu_k.shape[0]
    np.testing.assert_array_equal(cache.owner.cpu().numpy(),
                                  oracle.cache_owner_from_table(nv(wl.table), n_slots, wl.L))
    host_rows = nv(wl.host_k).reshape(wl.host_k.shape[0], -1)
    hits = []
    want_stats = np.zeros(3, dtype=np.int64)
    for s in range(steps):
        if s % 2 == 0:
            _fresh_queries(wl, twin, 77 + s)  # odd steps repeat the query: the promoted tokens hit
        before = _state(wl, cache)
        step.status.zero_()
        step.run_cached()
        ref.run()
        torch.cuda.synchronize()
        assert int(step.status.item()) == 0 and int(ref.status.item()) == 0
        assert torch.equal(step.idx, ref.idx) and torch.equal(step.out, ref.out) and torch.equal(step.lse, ref.lse)
        att = _attended(wl, step, OracleView(wl))
        in_gpu = sum(int((before[0][b, a] >= 0).sum()) for b, a in enumerate(att))
        hits.append(in_gpu)
        promos = _check_step(wl, step, cache, before, s, att, budget, host_rows)
        assert len(promos) <= budget
        want_stats += (in_gpu, sum(len(a) for a in att) - in_gpu, len(promos))
        np.testing.assert_array_equal(cache.stats.cpu().numpy(), want_stats)
    if budget > 0 and steps >= 2:
        assert hits[1] > hits[0]  # the repeated query finds what the first step promoted


def test_free_slots_are_taken_first(skv):
    wl = workloads.make_workload("mla", device="cuda", gen_device="cpu", B=2, L=1000, k=100)
    step = skv.DecodeStep.from_workload(wl)
    cache = step.enable_cache(16)
    # free eight slots: their tokens return to the host rows
    owner = cache.owner.cpu().numpy()
    freed = np.nonzero(owner >= 0)[0][[3, 50, 90, 100, 140, 200, 300, 400]]
    for sl in freed:
        o = int(owner[sl])
        wl.table[o // wl.L, o % wl.L] = -o - 1
        cache.owner[int(sl)] = -1
    before = _state(wl, cache)
    step.run_cached()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    att = _attended(wl, step, OracleView(wl))
    promos = _check_step(wl, step, cache, before, 0, att, 16, nv(wl.host_k).reshape(wl.host_k.shape[0], -1))
    assert len(promos) == 16
    taken = {p[0] for p in promos}
    assert {int(x) for x in freed} <= taken  # free slots rank first; the pairing itself runs in slot order
    used = {int(before[0][b, t]) for b, a in enumerate(att) for t in a if before[0][b, t] >= 0}
    rest = [sl for sl in range(len(owner)) if sl not in used and sl not in set(freed.tolist())]
    assert taken - {int(x) for x in freed} == set(rest[:8])  # equal ages: the lower slots


def test_separate_update_equals_the_fused_call(skv):
    wl = workloads.make_workload("mla", device="cuda", gen_device="cpu", B=2, L=2500, k=256, seq_lens=[2500, 2000])
    twin = _twin(wl)
    fused = skv.DecodeStep.from_workload(wl)
    split = skv.DecodeStep.from_workload(twin)
    a, b = fused.enable_cache(64), split.enable_cache(64)
    b.count = False  # counters off: the update leaves them alone
    for s in range(3):
        if s != 1:
            _fresh_queries(wl, twin, 300 + s)
        fused.run_cached()
        split.run()
        split.cache_update()
        torch.cuda.synchronize()
        assert int(fused.status.item()) == 0 and int(split.status.item()) == 0
        assert torch.equal(fused.out, split.out) and torch.equal(wl.table, twin.table)
        assert torch.equal(a.owner, b.owner) and torch.equal(a.prio, b.prio) and torch.equal(wl.gpu_k, twin.gpu_k)
    assert int(b.stats.abs().sum().item()) == 0 and int(a.stats[2].item()) > 0


def test_cache_full_size_mla(skv):
    wl = workloads.make_workload("mla", device="cuda", gen_device="cuda")
    plain = skv.DecodeStep.from_workload(wl)
    plain.run()
    torch.cuda.synchronize()
    assert int(plain.status.item()) == 0
    want_idx, want_out, want_lse = plain.idx.clone(), plain.out.clone(), plain.lse.clone()
    step = skv.DecodeStep.from_workload(wl)
    budget = 4096
    cache = step.enable_cache(budget)
    host_k = wl.host_k.view(wl.host_k.shape[0], -1)
    for s in range(2):
        before = _state(wl, cache)
        step.run_cached()
        torch.cuda.synchronize()
        assert int(step.status.item()) == 0
        assert torch.equal(step.idx, want_idx) and torch.equal(step.out, want_out) and torch.equal(step.lse, want_lse)
        att = _attended(wl, step)
        want_t, want_o, want_p, promos = oracle.cache_update(*before, s, att, wl.L, budget)
        got_t, got_o, got_p = _state(wl, cache)
        np.testing.assert_array_equal(got_t, want_t)
        np.testing.assert_array_equal(got_o, want_o)
        np.testing.assert_array_equal(got_p, want_p)
        assert len(promos) == budget
        pick = promos[:: max(1, len(promos) // 256)]
        slots = torch.tensor([p[0] for p in pick], dtype=torch.long, device="cuda")
        rows = torch.tensor([p[1] * wl.L + p[2] for p in pick], dtype=torch.long)
        assert torch.equal(wl.gpu_k.view(wl.gpu_k.shape[0], -1)[slots].cpu(), host_k[rows])


def test_bad_owner_is_flagged_and_left_out_of_the_table(skv):
    wl = workloads.make_workload("mla", device="cuda", gen_device="cpu", B=1, L=800, k=64)
    step = skv.DecodeStep.from_workload(wl)
    cache = step.enable_cache(4)
    cache.prio.fill_(5)        # every slot recently used: age ranks slot 0 first among the unused
    cache.step.fill_(10)
    victim = 0
    o = int(cache.owner[victim].item())
    wl.table[o // wl.L, o % wl.L] = -o - 1   # its token goes back to the host...
    cache.owner[victim] = 7 * wl.L           # ... and the slot names a request that does not exist
    table_before = wl.table.clone()
    step.run_cached()
    torch.cuda.synchronize()
    assert int(step.status.item()) & skv.SKV_DEV_BAD_SLOT
    changed = (wl.table != table_before).nonzero()
    assert changed.shape[0] >= 1 and int(wl.table[0].max()) < wl.gpu_k.shape[0]


def test_cached_step_replays_in_a_cuda_graph_like_eager_steps(skv):
    # the ranking forks onto the library's side stream and joins back: a capture of the
    # caller's stream must hold both branches, and replays must advance the cache state
    wl = workloads.make_workload("mla", device="cuda", gen_device="cpu", B=2, L=2500, k=256, seq_lens=[2500, 2000])
    twin = _twin(wl)
    eager = skv.DecodeStep.from_workload(wl)
    graphed = skv.DecodeStep.from_workload(twin)
    ce, cg = eager.enable_cache(128), graphed.enable_cache(128)
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        graphed.run_cached()
    for s in range(3):
        if s == 1:
            _fresh_queries(wl, twin, 900)
        eager.run_cached()
        g.replay()
        torch.cuda.synchronize()
        assert int(eager.status.item()) == 0 and int(graphed.status.item()) == 0
        assert torch.equal(eager.idx, graphed.idx) and torch.equal(eager.out, graphed.out)
        assert torch.equal(wl.table, twin.table) and torch.equal(wl.gpu_k, twin.gpu_k)
        assert torch.equal(ce.owner, cg.owner) and torch.equal(ce.prio, cg.prio) and torch.equal(ce.step, cg.step)
        assert torch.equal(ce.stats, cg.stats)
    assert int(cg.step.item()) == 3 and int(cg.stats[2].item()) > 0
