"""S3 gather, S4/S5 attention and the whole decode step on the GPU against the fp64 oracle."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from skv_test_utils import OracleView, UnitView, assert_attention_close, check_band, nv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def skv():
    import __graft_entry__

    __graft_entry__.build()
    import top_sparse_kv_gb300 as m

    return m


def _gpu_step(skv, wl, n_splits=0):
    step = skv.DecodeStep.from_workload(wl, n_splits=n_splits)
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0, int(step.status.item())
    return step


DECODE_CASES = [
    ("tiny", dict(), None, 0.0, torch.bfloat16),
    ("tiny", dict(L=2000, k=100), [1999], 0.0, torch.float32),
    ("gqa32b", dict(B=3, H=2, Hq=16, L=3000, k=300), [3000, 2222, 100], 0.0, torch.bfloat16),
    ("gqa32b", dict(B=2, H=2, Hq=8, L=1500, k=150), [1500, 1001], 0.5, torch.bfloat16),
    ("gqa32b", dict(B=2, H=4, Hq=8, L=1500, k=150), None, 0.5, torch.float32),  # G = 2
    ("host1m", dict(L=30000, k=100), None, 0.0, torch.bfloat16),
    ("sweep", dict(B=2, L=8192, k=256), None, 0.0, torch.bfloat16),
    ("mla", dict(B=2, L=3000, k=256), [3000, 2500], 0.0, torch.bfloat16),
    ("mla", dict(B=1, L=700, k=1000), None, 0.0, torch.bfloat16),  # k >= |C|: every row attended
    ("mla", dict(B=3, L=5000, k=2048), [5000, 4999, 2100], 0.0, torch.bfloat16),
    # lists longer than one 512-entry CTA on few units: the three-stage gather ring with up
    # to 1,024 entries a CTA (a host tier and ragged rows; a list of four such chunks)
    ("gqa32b", dict(B=2, H=2, Hq=16, L=8000, k=1500), [8000, 5000], 0.3, torch.bfloat16),
    ("gqa32b", dict(B=1, H=2, Hq=16, L=12000, k=3000), None, 0.0, torch.bfloat16),
]


@pytest.mark.parametrize("name,over,lens,host_frac,dtype", DECODE_CASES)
def test_decode_step_matches_oracle(skv, name, over, lens, host_frac, dtype):
    wl = workloads.make_workload(name, device="cuda", gen_device="cpu", seq_lens=lens, host_frac=host_frac,
                                 dtype=dtype, **over)
    step = _gpu_step(skv, wl)
    view = OracleView(wl)
    scores = step.scores.cpu().numpy()
    idx = step.idx.cpu().numpy()
    lse = step.lse.cpu().numpy()
    G = wl.G
    for b in range(wl.B):
        for h in range(wl.H):
            full = view.unit(b, h)
            check_band(idx[b, h], full, wl.k)
            # exact on the GPU's own scores
            mine = view.unit(b, h, given_scores=scores[b, h])
            np.testing.assert_array_equal(idx[b, h][: len(mine["idx"])], mine["idx"])
            # attention on the GPU's selection
            att = view.unit(b, h, given_idx=mine["idx"])
            assert_attention_close(step.out[b, h * G:(h + 1) * G], att["out"], dtype)
            np.testing.assert_allclose(lse[b, h * G:(h + 1) * G], att["lse"], rtol=1e-5, atol=1e-5)


EDGE_CASES = [
    # an empty history, one token, a history inside the sink, one that ends where the
    # local window begins (no candidates), exactly one candidate, k candidates, full
    ("gqa32b", dict(B=7, H=2, Hq=16, L=600, k=40), [0, 1, 4, 132, 133, 173, 600], torch.bfloat16),
    ("gqa32b", dict(B=7, H=2, Hq=16, L=600, k=40), [0, 1, 4, 132, 133, 173, 600], torch.float32),
    ("mla", dict(B=4, L=900, k=300), [0, 1, 2, 900], torch.bfloat16),  # no sink or local window
]


@pytest.mark.parametrize("name,over,lens,dtype", EDGE_CASES)
def test_degenerate_lengths_match_oracle(skv, name, over, lens, dtype):
    """Regions clipped to short histories: an empty attended set gives o = 0 and lse = -inf."""
    wl = workloads.make_workload(name, device="cuda", gen_device="cpu", seq_lens=lens, dtype=dtype, **over)
    step = _gpu_step(skv, wl)
    view = OracleView(wl)
    scores = step.scores.cpu().numpy()
    idx = step.idx.cpu().numpy()
    lse = step.lse.cpu().numpy()
    G = wl.G
    for b in range(wl.B):
        for h in range(wl.H):
            full = view.unit(b, h)
            check_band(idx[b, h], full, wl.k)
            mine = view.unit(b, h, given_scores=scores[b, h])
            n = len(mine["idx"])
            assert n == len(full["idx"]) == min(wl.k, max(0, lens[b] - wl.ns - wl.nl))
            np.testing.assert_array_equal(idx[b, h][:n], mine["idx"])
            assert np.all(idx[b, h][n:] == -1)
            att = view.unit(b, h, given_idx=mine["idx"])
            if lens[b] == 0:
                assert torch.count_nonzero(step.out[b, h * G:(h + 1) * G]).item() == 0
                assert np.all(np.isneginf(lse[b, h * G:(h + 1) * G]))
                continue
            assert_attention_close(step.out[b, h * G:(h + 1) * G], att["out"], dtype)
            np.testing.assert_allclose(lse[b, h * G:(h + 1) * G], att["lse"], rtol=1e-5, atol=1e-5)


def test_lengths_outside_capacity_are_flagged_and_clamped(skv):
    """seq_lens[b] above max_len or below 0 sets SKV_DEV_BAD_LENGTH; the step then runs on
    the length clamped to [0, max_len]."""
    over = dict(B=3, H=2, Hq=16, L=700, k=50)
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", seq_lens=[700, 0, 300], **over)
    good = _gpu_step(skv, wl)
    ref = (good.idx.clone(), good.out.clone(), good.lse.clone())
    wl.seq_lens.copy_(torch.tensor([700 + 9, -5, 300], dtype=torch.int32))
    bad = skv.DecodeStep.from_workload(wl)
    bad.run()
    torch.cuda.synchronize()
    assert int(bad.status.item()) == skv.SKV_DEV_BAD_LENGTH
    assert torch.equal(bad.idx, ref[0]) and torch.equal(bad.out, ref[1]) and torch.equal(bad.lse, ref[2])


@pytest.mark.parametrize("n_splits", [1, 2, 7, 10 ** 6])
def test_split_count_does_not_change_results(skv, n_splits):
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=2, H=2, Hq=16, L=2500, k=200,
                                 dtype=torch.float32)
    base = _gpu_step(skv, wl, n_splits=3)
    other = _gpu_step(skv, wl, n_splits=n_splits)
    np.testing.assert_array_equal(base.idx.cpu().numpy(), other.idx.cpu().numpy())
    assert torch.allclose(base.out, other.out, atol=1e-5, rtol=1e-5)
    view = OracleView(wl)
    for b in range(2):
        for h in range(2):
            att = view.unit(b, h, given_idx=[t for t in other.idx[b, h].cpu().tolist() if t >= 0])
            assert_attention_close(other.out[b, h * 8:(h + 1) * 8], att["out"], torch.float32)


@pytest.mark.parametrize("n_splits", [1, 2, 4, 7, 8, 9, 16, 10 ** 6])
@pytest.mark.parametrize("H,Hq", [(2, 16), (1, 16), (4, 4), (2, 6)])
def test_tensor_core_split_merge_paths(skv, n_splits, H, Hq):
    """bf16 splits of a unit merge inside one thread-block cluster up to 8 splits and through
    the workspace beyond; G = 8, 1 and 3 (keys-on-M tiles, heads padded to 8) and G = 16
    (heads-on-M tiles; a CTA of the cluster merges several heads), one ragged row, every
    split count against the oracle on the step's own selection."""
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=2, H=H, Hq=Hq, L=2500, k=200,
                                 seq_lens=[2500, 1777], dtype=torch.bfloat16)
    step = _gpu_step(skv, wl, n_splits=n_splits)
    view = OracleView(wl)
    G = wl.G
    lse = step.lse.cpu().numpy()
    for b in range(wl.B):
        for h in range(wl.H):
            att = view.unit(b, h, given_idx=[t for t in step.idx[b, h].cpu().tolist() if t >= 0])
            assert_attention_close(step.out[b, h * G:(h + 1) * G], att["out"], torch.bfloat16)
            np.testing.assert_allclose(lse[b, h * G:(h + 1) * G], att["lse"], rtol=1e-5, atol=1e-5)


def test_sparse_attn_with_empty_slots_and_dense_reduction(skv):
    # k >= |C|, no sink/local: the step is dense attention over all L rows
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=1, H=2, Hq=16, L=700, k=2000, ns=0,
                                 nl=0, dtype=torch.float32, keep_logical=True)
    step = _gpu_step(skv, wl)
    idx = step.idx.cpu().numpy()
    assert np.array_equal(idx[0, 0, :700], np.arange(700)) and np.all(idx[0, 0, 700:] == -1)
    lk = wl.meta["logical_k"].double()
    lv = wl.meta["logical_v"].double()
    for h in range(2):
        ref = torch.nn.functional.scaled_dot_product_attention(
            wl.q[0, 8 * h:8 * h + 8].double().cpu()[None], lk[0, h].cpu()[None], lv[0, h].cpu()[None],
            scale=wl.sm_scale)[0]
        assert (step.out[0, 8 * h:8 * h + 8].double().cpu() - ref).abs().max().item() <= 1e-4


def test_gather_is_bit_exact(skv):
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=2, H=2, Hq=8, L=900, k=50,
                                 seq_lens=[900, 333], host_frac=0.3)
    step = _gpu_step(skv, wl)
    n_att = wl.ns + wl.k + wl.nl
    k_out = torch.empty((wl.B, wl.H, n_att, 128), dtype=wl.dtype, device="cuda")
    v_out = torch.empty_like(k_out)
    skv.skv_gather(step.p, step.pool, step.idx, k_out, v_out, step.status)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    view = OracleView(wl)
    ko, vo = nv(k_out), nv(v_out)
    for b in range(wl.B):
        for h in range(wl.H):
            att = view.unit(b, h, given_idx=[t for t in step.idx[b, h].cpu().tolist() if t >= 0])["attended"]
            L = int(wl.seq_lens[b])
            s_end, l_start = oracle.regions(L, wl.ns, wl.nl)
            sel = [t for t in step.idx[b, h].cpu().tolist()]
            listing = list(range(s_end)) + sel + list(range(l_start, L))
            listing += [-1] * (n_att - len(listing))
            for j, t in enumerate(listing):
                if t < 0:
                    assert not ko[b, h, j].any() and not vo[b, h, j].any()
                else:
                    np.testing.assert_array_equal(oracle.as_f64(ko[b, h, j]), view.kpool.row(b, h, t))
                    np.testing.assert_array_equal(oracle.as_f64(vo[b, h, j]), view.vpool.row(b, h, t))
            assert sorted(t for t in listing if t >= 0) == list(att)


def test_placement_invariance_bitwise(skv):
    # permuted physical blocks and blocks moved to the host pool give identical bits
    base = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=2, H=2, Hq=16, L=3000, k=300)
    moved = workloads.permute_blocks(base, seed=3)
    tiered = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=2, H=2, Hq=16, L=3000, k=300,
                                     host_frac=0.6)
    r0 = _gpu_step(skv, base)
    for other in (moved, tiered):
        r1 = _gpu_step(skv, other)
        assert torch.equal(r0.idx, r1.idx)
        assert torch.equal(r0.out, r1.out)
        assert torch.equal(r0.lse, r1.lse)
        s_end, l_start = oracle.regions(3000, 4, 128)
        assert torch.equal(r0.scores[..., s_end:l_start], r1.scores[..., s_end:l_start])


def test_deterministic_runs(skv):
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=2, H=2, Hq=16, L=4000, k=400)
    a = _gpu_step(skv, wl)
    outs = (a.idx.clone(), a.out.clone(), a.lse.clone())
    a.run()
    torch.cuda.synchronize()
    assert torch.equal(outs[0], a.idx) and torch.equal(outs[1], a.out) and torch.equal(outs[2], a.lse)


def test_bad_slot_entries_are_flagged_not_faulted(skv):
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=1, H=2, Hq=8, L=800, k=40)
    step = skv.DecodeStep.from_workload(wl)
    wl.table[0, 5] = 10 ** 6          # GPU block out of range
    wl.table[0, 20] = -(10 ** 6)      # host block with no host pool
    step.run()
    torch.cuda.synchronize()
    st = int(step.status.item())
    assert st & skv.SKV_DEV_BAD_SLOT
    assert torch.isfinite(step.out.float()).all()
    idx = step.idx.cpu().numpy()
    bad = set(range(80, 96)) | set(range(320, 336))
    assert not (set(idx.reshape(-1).tolist()) & bad)  # NaN-scored keys are never selected


def test_bad_selected_positions_are_flagged(skv):
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=1, H=1, Hq=8, L=800, k=8)
    step = _gpu_step(skv, wl)
    idx = step.idx.clone()
    idx[0, 0, 0] = 2           # inside the sink: not a candidate
    idx[0, 0, 1] = 10 ** 7     # past the history
    step.status.zero_()
    skv.skv_sparse_attn(step.p, step.q, step.pool, idx, step.out, step.lse, step.ws, step.status)
    torch.cuda.synchronize()
    assert int(step.status.item()) & skv.SKV_DEV_BAD_INDEX
    assert torch.isfinite(step.out.float()).all()


def test_full_size_gqa32b_sampled(skv):
    # the benchmarked workload at full size, checked on sampled (request, head) units
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cuda")
    step = _gpu_step(skv, wl)
    view = OracleView(wl)
    scores = step.scores.cpu().numpy()
    idx = step.idx.cpu().numpy()
    for b, h in ((0, 0), (3, 5), (7, 7)):
        full = view.unit(b, h)
        check_band(idx[b, h], full, wl.k)
        mine = view.unit(b, h, given_scores=scores[b, h])
        np.testing.assert_array_equal(idx[b, h], mine["idx"])
        att = view.unit(b, h, given_idx=mine["idx"])
        assert_attention_close(step.out[b, h * 8:(h + 1) * 8], att["out"], torch.bfloat16)


def _sampled_check(skv, wl, units):
    step = _gpu_step(skv, wl)
    view = OracleView(wl)
    idx = step.idx.cpu().numpy()
    G = wl.G
    for b, h in units:
        scores = step.scores[b, h].cpu().numpy()
        full = view.unit(b, h)
        check_band(idx[b, h], full, wl.k)
        mine = view.unit(b, h, given_scores=scores)
        np.testing.assert_array_equal(idx[b, h][: len(mine["idx"])], mine["idx"])
        att = view.unit(b, h, given_idx=mine["idx"])
        assert_attention_close(step.out[b, h * G:(h + 1) * G], att["out"], torch.bfloat16)


# the sweep's largest points (up to 64 requests x 128K tokens: 34 GB of K and V), one smaller
# point per k; each as the sweep bench builds it (its seed), checked on sampled units
SWEEP_FULL = [35, 33, 16, 22, 2]


@pytest.mark.parametrize("point", SWEEP_FULL)
def test_full_size_sweep_points_sampled(skv, point):
    B, L, k = workloads.SWEEP_POINTS[point]
    wl = workloads.make_workload("sweep", device="cuda", gen_device="cuda", seed=workloads.seed_for("sweep", point),
                                 B=B, L=L, k=k)
    step = _gpu_step(skv, wl)
    idx = step.idx.cpu().numpy()
    G = wl.G
    for b, h in ((0, 0), (B - 1, wl.H - 1)):
        view = UnitView(wl, b, h)
        full = view.unit()
        check_band(idx[b, h], full, k)
        mine = view.unit(given_scores=step.scores[b, h].cpu().numpy())
        np.testing.assert_array_equal(idx[b, h][: len(mine["idx"])], mine["idx"])
        att = view.unit(given_idx=mine["idx"])
        assert_attention_close(step.out[b, h * G:(h + 1) * G], att["out"], torch.bfloat16)
        np.testing.assert_allclose(step.lse[b, h * G:(h + 1) * G].cpu().numpy(), att["lse"], rtol=1e-5, atol=1e-5)
    del step, wl
    torch.cuda.empty_cache()


def test_full_size_host1m_sampled(skv):
    # 1M-token history: GPU index keys, K/V rows of the selection read from the pinned host pool
    wl = workloads.make_workload("host1m", device="cuda", gen_device="cuda")
    _sampled_check(skv, wl, [(0, 0), (0, 5)])


def test_full_size_mla_sampled(skv):
    # 16 requests x 128K tokens of 576-wide latent rows, 25% in the GPU slot cache, the rest on the host
    wl = workloads.make_workload("mla", device="cuda", gen_device="cuda")
    assert (wl.table < 0).float().mean().item() > 0.7
    _sampled_check(skv, wl, [(0, 0), (9, 0), (15, 0)])
