"""S1 scoring and S2 exact top-k on the GPU against the fp64 oracle."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from skv_test_utils import OracleView, check_band, nv, score_tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def skv():
    import __graft_entry__

    __graft_entry__.build()
    import top_sparse_kv_gb300 as m

    return m


SCORE_CASES = [
    ("tiny", dict(), None, 0.0, torch.bfloat16),
    ("tiny", dict(L=1000, k=17), [1000], 0.0, torch.float32),
    ("gqa32b", dict(B=3, H=2, Hq=16, L=2000, k=150), [2000, 1377, 140], 0.0, torch.bfloat16),
    ("gqa32b", dict(B=2, H=2, Hq=8, L=777, k=40), [777, 300], 0.4, torch.bfloat16),  # host tier
    ("host1m", dict(L=20000, k=100), None, 0.0, torch.bfloat16),
    ("mla", dict(B=2, L=3000, k=256), [3000, 2500], 0.0, torch.bfloat16),
]


@pytest.mark.parametrize("name,over,lens,host_frac,dtype", SCORE_CASES)
def test_scores_match_oracle(skv, name, over, lens, host_frac, dtype):
    wl = workloads.make_workload(name, device="cuda", gen_device="cpu", seq_lens=lens, host_frac=host_frac,
                                 dtype=dtype, **over)
    step = skv.DecodeStep.from_workload(wl)
    step.scores.fill_(float("nan"))
    step.score()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    view = OracleView(wl)
    scores = step.scores.cpu().numpy()
    for b in range(wl.B):
        for h in range(wl.H):
            ref = view.unit(b, h)
            pos = ref["positions"]
            got = scores[b, h, pos].astype(np.float64)
            tol = score_tolerance(view, b, h, pos)
            assert np.all(np.abs(got - ref["scores"]) <= tol), (b, h, np.max(np.abs(got - ref["scores"]) / tol))


def _topk_on(skv, scores_np, lens, k, ns, nl, H=1):
    """Run skv_topk on a given score tensor [B, H, L]; returns idx [B, H, k] (numpy)."""
    B, _, L = scores_np.shape
    dev = "cuda"
    p = skv.Problem(batch=B, n_kv_heads=H, n_q_heads=H, d_qk=128, d_v=128, max_len=L, topk=k, n_sink=ns,
                    n_local=nl, block_size=16, seq_lens=torch.tensor(lens, dtype=torch.int32, device=dev))
    scores = torch.from_numpy(np.ascontiguousarray(scores_np, dtype=np.float32)).to(dev)
    idx = torch.full((B, H, max(k, 1)), -7, dtype=torch.int32, device=dev)
    ws = torch.empty((skv.skv_workspace_size(p),), dtype=torch.uint8, device=dev)
    status = torch.zeros((1,), dtype=torch.int32, device=dev)
    skv.skv_topk(p, scores, idx, ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return idx.cpu().numpy()[..., :k]


def _expect(scores_row, L, k, ns, nl):
    s_end, l_start = oracle.regions(L, ns, nl)
    pos = np.arange(s_end, l_start)
    sel = oracle.exact_topk(scores_row[pos].astype(np.float64), pos, k)
    out = np.full(k, -1, dtype=np.int64)
    out[: len(sel)] = sel
    return out


TOPK_CASES = [
    # (B, H, L, lens, k, ns, nl, kind)
    (1, 1, 4096, [4096], 256, 4, 64, "normal"),
    (2, 3, 5000, [5000, 4321], 1, 4, 64, "normal"),           # argmax
    (1, 2, 3000, [3000], 5000, 4, 64, "normal"),              # k >= |C|: all candidates
    (2, 1, 100, [60, 3], 10, 4, 64, "normal"),                # tiny / empty candidate regions
    (1, 1, 20000, [20000], 700, 0, 0, "ties"),                # heavy ties across segments
    (1, 1, 20000, [20000], 333, 16, 16, "allequal"),          # one value everywhere
    (1, 1, 9000, [9000], 500, 4, 8, "specials"),              # -0/+0, inf, NaN
    (1, 2, 300000, [300000], 3000, 4, 128, "normal"),         # long rows: many CTAs per row
    (1, 2, 300000, [300000], 30000, 4, 128, "normal"),        # long rows, large k: multi-CTA passes
    (2, 2, 100000, [100000, 77777], 2048, 0, 0, "ties"),      # two stages: segment winners, then the row
    (3, 1, 40960, [40960, 40000, 5], 4096, 4, 128, "normal"),  # two stages, a row shorter than one segment
    (2, 1, 60000, [60000, 41000], 3000, 4, 128, "normal"),    # two stages
    (3, 1, 50000, [50000, 20000, 700], 2000, 4, 128, "coarse"),  # two stages, ragged rows, heavy ties
    (1, 2, 1048576, [1048576], 100, 16, 512, "normal"),        # two stages, 64 segments
    (1, 1, 60000, [60000], 12000, 4, 128, "normal"),          # winners too many for one CTA: 4-CTA clusters
    (1, 1, 100000, [100000], 9000, 0, 0, "ties"),             # 8-CTA clusters
    (1, 2, 30000, [30000], 1500, 4, 64, "coarse"),            # a tie group far larger than the bucket list
    (4, 2, 8192, [8192, 7000, 10, 8192], 0, 4, 128, "normal"),  # k = 0
    # short rows (one CTA of 256 or 512 threads)
    (1, 1, 4000, [4000], 300, 4, 8, "specials"),              # -0/+0, inf, NaN in a short row
    (2, 2, 8000, [8000, 6000], 1000, 4, 64, "ties"),          # 512 threads, ragged rows
    (1, 1, 8192, [8192], 100, 0, 0, "allequal"),              # one value everywhere, at capacity
    (3, 1, 4096, [4096, 4095, 33], 2000, 0, 0, "coarse"),     # 256 threads at capacity
    # two stages over 32K-key segments (fewer first-stage waves than 16K segments)
    (3, 1, 1048576, [1048576, 1000000, 40000], 100, 16, 512, "normal"),
    (8, 4, 131072, [131072] * 7 + [70000], 1000, 4, 128, "coarse"),
    # path boundaries at their largest rows
    (2, 1, 32768, [32768, 32767], 3000, 0, 0, "normal"),      # one CTA at its 32K capacity
    (1, 1, 32769, [32769], 3000, 0, 0, "ties"),               # one past it: two stages (three segments)
    (1, 1, 131072, [131072], 20000, 0, 0, "normal"),          # 8-CTA clusters at their 128K capacity
    (1, 1, 131073, [131073], 20000, 0, 0, "coarse"),          # one past it: multi-CTA passes
    (1, 1, 131073, [131073], 30000, 0, 0, "ties"),            # the same with heavier ties
    (1, 1, 524288, [524288], 4096, 0, 0, "coarse"),           # a slot-cache ranking's shape, multi-CTA
    (2, 2, 300000, [300000, 150001], 8000, 4, 128, "normal"),  # multi-CTA, ragged rows
    # more rows than SMs of up to 8K keys: the lean kernel (three 512-thread rows an SM)
    (40, 8, 5000, [5000 - 97 * i for i in range(40)], 300, 4, 64, "normal"),     # ragged rows
    (20, 8, 8192, [8192] * 19 + [17], 819, 4, 128, "ties"),                     # 16 keys a thread
    (32, 8, 8192, [8192] * 32, 500, 4, 8, "specials"),                          # -0/+0, inf, NaN
    (160, 1, 2000, [2000 - 12 * i for i in range(160)], 1500, 4, 64, "coarse"),  # k >= |C| in some rows
    (40, 4, 8000, [8000] * 40, 333, 16, 16, "allequal"),                        # one value everywhere
    (200, 1, 1000, [1000] * 200, 0, 4, 64, "normal"),                           # k = 0
    (20, 8, 8191, [8191 - i for i in range(20)], 1, 0, 0, "normal"),            # argmax, unaligned rows
    # more rows than SMs of longer rows: the one-CTA kernel, in waves
    (20, 8, 32768, [32768] * 19 + [17], 3277, 4, 128, "ties"),
    (20, 8, 32767, [32767 - i for i in range(20)], 1, 0, 0, "normal"),
]


@pytest.mark.parametrize("B,H,L,lens,k,ns,nl,kind", TOPK_CASES)
def test_topk_bit_exact_on_given_scores(skv, B, H, L, lens, k, ns, nl, kind):
    rng = np.random.default_rng(L + k)
    s = rng.standard_normal((B, H, L)).astype(np.float32)
    if kind == "ties":
        s = np.round(s * 2) / 2
    elif kind == "coarse":
        s = np.round(s)
    elif kind == "allequal":
        s[:] = 0.75
    elif kind == "specials":
        s = np.round(s * 4) / 4
        flat = s.reshape(-1)
        flat[rng.choice(flat.size, 300, replace=False)] = -0.0
        flat[rng.choice(flat.size, 5, replace=False)] = np.inf
        flat[rng.choice(flat.size, 5, replace=False)] = -np.inf
        flat[rng.choice(flat.size, 50, replace=False)] = np.nan
    got = _topk_on(skv, s, lens, k, ns, nl, H)
    for b in range(B):
        for h in range(H):
            want = _expect(s[b, h], lens[b], k, ns, nl)
            np.testing.assert_array_equal(got[b, h], want)


def test_topk_on_gpu_scores_matches_oracle_and_fp64_band(skv):
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=2, H=4, Hq=32, L=6000, k=600,
                                 seq_lens=[6000, 4097])
    step = skv.DecodeStep.from_workload(wl)
    step.score()
    step.topk()
    torch.cuda.synchronize()
    view = OracleView(wl)
    scores = step.scores.cpu().numpy()
    idx = step.idx.cpu().numpy()
    for b in range(wl.B):
        for h in range(wl.H):
            on_gpu_scores = view.unit(b, h, given_scores=scores[b, h])
            np.testing.assert_array_equal(idx[b, h][: len(on_gpu_scores["idx"])], on_gpu_scores["idx"])
            check_band(idx[b, h], view.unit(b, h), wl.k)


def test_topk_deterministic(skv):
    rng = np.random.default_rng(11)
    s = (np.round(rng.standard_normal((2, 2, 50000)) * 3) / 3).astype(np.float32)
    a = _topk_on(skv, s, [50000, 40000], 4000, 4, 128, 2)
    b = _topk_on(skv, s, [50000, 40000], 4000, 4, 128, 2)
    np.testing.assert_array_equal(a, b)


MAX_CASES = [
    ("gqa32b", dict(B=3, H=2, Hq=16, L=2000, k=150), [2000, 1377, 140], 0.0),   # G = 8
    ("gqa32b", dict(B=2, H=2, Hq=8, L=777, k=40), [777, 300], 0.4),             # G = 4, host tier read in place
    ("gqa32b", dict(B=1, H=2, Hq=14, L=1500, k=90), None, 0.0),                 # G = 7: a masked head
    ("host1m", dict(L=20000, k=100), None, 0.0),                                # contiguous index keys, G = 4
    ("mla", dict(B=2, L=3000, k=256), [3000, 2500], 0.0),                       # one indexer head
]


@pytest.mark.parametrize("name,over,lens,host_frac", MAX_CASES)
def test_max_aggregation_scores_and_selection(skv, name, over, lens, host_frac):
    wl = workloads.make_workload(name, device="cuda", gen_device="cpu", seq_lens=lens, host_frac=host_frac, **over)
    step = skv.DecodeStep.from_workload(wl, group_agg=skv.SKV_AGG_MAX)
    step.scores.fill_(float("nan"))
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    view = OracleView(wl, group_agg="max")
    scores = step.scores.cpu().numpy()
    idx = step.idx.cpu().numpy()
    for b in range(wl.B):
        for h in range(wl.H):
            ref = view.unit(b, h)
            pos = ref["positions"]
            tol = score_tolerance(view, b, h, pos)
            got = scores[b, h, pos].astype(np.float64)
            assert np.all(np.abs(got - ref["scores"]) <= tol), (b, h, np.max(np.abs(got - ref["scores"]) / tol))
            mine = view.unit(b, h, given_scores=scores[b, h])
            np.testing.assert_array_equal(idx[b, h][: len(mine["idx"])], mine["idx"])
            check_band(idx[b, h], ref, wl.k)


def test_max_and_mean_select_differently_on_the_gpu(skv):
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=1, H=2, Hq=16, L=3000, k=300)
    sel = {}
    for agg in (skv.SKV_AGG_MEAN, skv.SKV_AGG_MAX):
        step = skv.DecodeStep.from_workload(wl, group_agg=agg)
        step.run()
        torch.cuda.synchronize()
        sel[agg] = step.idx.cpu().numpy()
    assert not np.array_equal(sel[skv.SKV_AGG_MEAN], sel[skv.SKV_AGG_MAX])


def test_max_aggregation_full_size_gqa32b_sampled(skv):
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cuda")
    step = skv.DecodeStep.from_workload(wl, group_agg=skv.SKV_AGG_MAX)
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    view = OracleView(wl, group_agg="max")
    idx = step.idx.cpu().numpy()
    for b, h in ((0, 0), (5, 3), (7, 7)):
        scores = step.scores[b, h].cpu().numpy()
        ref = view.unit(b, h)
        check_band(idx[b, h], ref, wl.k)
        mine = view.unit(b, h, given_scores=scores)
        np.testing.assert_array_equal(idx[b, h], mine["idx"])


STEP_SELECTION_CASES = [
    ("tiny", dict(), None, "plain"),
    ("gqa32b", dict(B=3, H=2, Hq=16, L=2000, k=150), [2000, 1377, 140], "plain"),  # ragged, one row empty
    ("gqa32b", dict(B=2, H=2, Hq=8, L=32768, k=3277), [32768, 30000], "plain"),    # the one-CTA capacity
    ("tiny", dict(L=3000, k=100), None, "zero_keys"),                              # every score ties
    ("gqa32b", dict(B=2, H=2, Hq=8, L=5000, k=300), [5000, 4000], "bad_slot"),     # NaN scores in a block
    ("mla", dict(B=2, L=3000, k=256), [3000, 2500], "plain"),                      # contiguous index keys
    ("tiny", dict(L=1000, k=2000), None, "plain"),                                 # k >= |C|
    ("gqa32b", dict(B=24, H=8, Hq=64, L=3000, k=200), [3000 - 50 * i for i in range(24)], "plain"),  # 192 rows
]


@pytest.mark.parametrize("name,over,lens,kind", STEP_SELECTION_CASES)
def test_step_selection_equals_the_selection_on_its_scores(skv, name, over, lens, kind):
    """The selection inside skv_decode_step is the same bits as skv_topk on the step's own
    scores, and as the oracle's exact top-k on them: ties everywhere, NaN scores from a
    bad slot, ragged and empty rows, the one-CTA capacity, k >= |C|."""
    wl = workloads.make_workload(name, device="cuda", gen_device="cpu", seq_lens=lens, **over)
    if kind == "zero_keys":
        (wl.gpu_k if wl.index_keys is None else wl.index_keys).zero_()
    if kind == "bad_slot":
        wl.table[0, 7] = 10 ** 6
    step = skv.DecodeStep.from_workload(wl)
    step.run()
    torch.cuda.synchronize()
    st = int(step.status.item())
    assert st == (skv.SKV_DEV_BAD_SLOT if kind == "bad_slot" else 0)
    scores = step.scores.cpu().numpy()
    got = step.idx.cpu().numpy()
    plain = _topk_on(skv, scores, [int(x) for x in wl.seq_lens.cpu()], wl.k, wl.ns, wl.nl, wl.H)
    np.testing.assert_array_equal(got[..., :wl.k], plain)
    for b in range(wl.B):
        for h in range(wl.H):
            want = _expect(scores[b, h], int(wl.seq_lens[b]), wl.k, wl.ns, wl.nl)
            np.testing.assert_array_equal(got[b, h, :wl.k], want)
