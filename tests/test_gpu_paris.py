"""ParisKV retrieval (ParisKV notes, §2.2-§2.5) on the GPU against the fp64 oracle.

Encode: centroid ids and codes equal the oracle's except where an fp64 coordinate lies
within 1e-5 of zero or of a quantiser cut (a decision fp32 may take the other way);
weights within 1e-4 relative.  Step: the rotated query within fp32 rounding; the GPU's
centroid similarities within an fp32 bound of the fp64 similarities of its rotated
query; the tier weights, collision scores and candidates bit-exact on the GPU's own
metadata and similarities (the oracle ranks the given values with its plain lexsort);
against the fp64 similarities the ranking may differ only between centroids whose fp64
similarities lie within that bound of each other; rerank scores within an fp32 bound;
the final selection bit-exact on the GPU's rerank scores;
attention on the GPU's selection within the bf16 tolerance; and the whole fp64 chain
selects nearly the same positions."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import paris_oracle as po
from skv_test_utils import OracleView, assert_attention_close, nv

pytestmark = pytest.mark.gpu

LV, TH = po.lloyd_max(8)


@pytest.fixture(scope="module")
def skv():
    import __graft_entry__

    __graft_entry__.build()
    import top_sparse_kv_gb300 as m

    return m


def _keys(view, wl, b, h, positions):
    """fp64 retrieval keys of row (b, h) at `positions` (contiguous index keys, else the K pool)."""
    if view.prob.index_layout == "contig":
        return oracle.as_f64(view.index_keys[b, h][positions])
    return oracle.as_f64(view.kpool.rows(b, h, positions))[:, :128]


def _score_query(view, wl, b, h):
    if view.prob.index_layout == "contig":
        gi = view.q_idx.shape[1] // wl.H
        return view.q_idx[b, h * gi:(h + 1) * gi]
    return view.q[b, h * wl.G:(h + 1) * wl.G]


def _near_boundary(ref):
    """[n, 16]: a coordinate of the subspace within 1e-5 of zero or of a cut (fp64)."""
    au = np.abs(ref["u"])
    close = (au < 1e-5) | (np.min(np.abs(au[..., None] - TH[None, None, None, :]), axis=-1) < 1e-5)
    return close.any(axis=-1)


def _gpu_meta(step, row):
    return dict(cent=step.paris.cent[row].cpu().numpy().astype(np.int64),
                code=step.paris.code[row].cpu().numpy().view(np.uint32).astype(np.int64),
                w=step.paris.w[row].cpu().numpy().astype(np.float64))


def check_encode(step, view, wl, b, h, positions):
    row = b * wl.H + h
    ref = po.encode(_keys(view, wl, b, h, positions), view.sig, 8, LV, TH)
    g = _gpu_meta(step, row)
    near = _near_boundary(ref)
    ok_c = g["cent"][positions] == ref["cent"]
    ok_code = g["code"][positions] == ref["code"]
    assert np.all(ok_c | near) and np.all(ok_code | near), (np.sum(~ok_c & ~near), np.sum(~ok_code & ~near))
    same = ok_code & (ref["w"] > 0)
    np.testing.assert_allclose(g["w"][positions][same], ref["w"][same], rtol=1e-4, atol=1e-6)
    return ref


def check_step(step, view, wl, b, h, params, e2e=True):
    row = b * wl.H + h
    L = int(wl.seq_lens[b])
    s_end, l_start = oracle.regions(L, wl.ns, wl.nl)
    pos = np.arange(s_end, l_start)
    g = _gpu_meta(step, row)
    qt_ref, nq_ref = po.retrieval_query(_score_query(view, wl, b, h), view.sig)
    qt = step.view("qt")[row].cpu().numpy().astype(np.float64)
    nq = float(step.view("nq")[row])
    np.testing.assert_allclose(qt, qt_ref, atol=2e-6)
    assert nq == pytest.approx(nq_ref, rel=1e-5)
    # centroid similarities: fp32 sums of 8 signed coordinates, then a scale, against the
    # fp64 similarities of the same rotated query (ParisKV notes §2.3, Eq. (15))
    sim_gpu = step.view("sim")[row].cpu().numpy().astype(np.float64)
    sim64 = po.centroid_similarity(qt, 8)
    tol = 1.2e-6 * np.abs(qt.reshape(16, 8)).sum(axis=1) / np.sqrt(8) + 1e-30
    assert np.all(np.abs(sim_gpu - sim64) <= tol[:, None]), np.max(np.abs(sim_gpu - sim64) / tol[:, None])
    # the fp32 ranking differs from the fp64 one only between near-ties
    for sub in range(16):
        o32 = np.lexsort((np.arange(256), -sim_gpu[sub]))
        rank64 = np.empty(256, dtype=np.int64)
        rank64[np.lexsort((np.arange(256), -sim64[sub]))] = np.arange(256)
        r = rank64[o32]  # fp64 ranks in fp32 order: an inversion is a pair ranked the other way
        for i in range(255):
            later = o32[i + 1:][r[i + 1:] < r[i]]
            assert np.all(np.abs(sim64[sub, later] - sim64[sub, o32[i]]) <= 2 * tol[sub]), (sub, i)
    # every integer stage on the GPU's own metadata, rotated query and similarities
    cs_gpu = step.view("cand_score")[row].cpu().numpy().astype(np.float64)
    cand_gpu = step.view("cand")[row].cpu().numpy()
    n_c = int(step.view("cand_len")[b])
    given = np.zeros(L)
    given[cand_gpu[:n_c]] = cs_gpu[:n_c]
    sel = po.paris_select(g, pos, qt, nq, wl.k, params, LV, given_rerank=given, given_sim=sim_gpu)
    np.testing.assert_array_equal(step.view("W")[row].cpu().numpy(), sel["W"])
    np.testing.assert_array_equal(step.view("S")[row].cpu().numpy()[pos], sel["S"])
    assert n_c == len(sel["cand"])
    np.testing.assert_array_equal(cand_gpu[:n_c], sel["cand"])
    # rerank within fp32 rounding: |q| sum_s |w_s| |v_s| |qt_s|, a few ulps of it
    v = po.decode_code(g["code"][sel["cand"]], 8, LV)
    bound = nq * np.sum(np.abs(g["w"][sel["cand"]]) * np.linalg.norm(v, axis=-1)
                        * np.linalg.norm(qt.reshape(16, 8), axis=-1)[None, :], axis=1)
    assert np.all(np.abs(cs_gpu[:n_c] - sel["rerank"]) <= 4e-6 * bound + 1e-30)
    idx = step.idx[b, h].cpu().numpy()
    ksel = min(wl.k, n_c)
    np.testing.assert_array_equal(idx[:ksel], sel["idx"])
    assert np.all(idx[ksel:] == -1)
    # attention over sink U selection U local
    res = view.unit(b, h, given_idx=sel["idx"])
    assert_attention_close(step.out[b, h * wl.G:(h + 1) * wl.G], res["out"], wl.dtype)
    np.testing.assert_allclose(step.lse[b, h * wl.G:(h + 1) * wl.G].cpu().numpy(), res["lse"], rtol=1e-5, atol=1e-5)
    if e2e:  # the fp64 chain from the keys selects nearly the same positions
        meta = po.encode(_keys(view, wl, b, h, np.arange(L)), view.sig, 8, LV, TH)
        ref = po.paris_select(meta, pos, qt_ref, nq_ref, wl.k, params, LV)
        both = len(set(ref["idx"].tolist()) & set(sel["idx"].tolist()))
        assert both >= 0.9 * len(ref["idx"]), (both, len(ref["idx"]))
    return sel


def _run(skv, wl, beta_pm=50, rho_pm=100):
    signs = workloads.srht_signs(128, device="cuda")
    step = skv.ParisStep.from_workload(wl, signs, beta_pm, rho_pm)
    step.encode()
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    view = OracleView(wl)
    view.sig = signs.cpu().numpy().astype(np.float64)
    return step, view, po.ParisParams(8, beta_pm, rho_pm)


CASES = [
    ("gqa32b", dict(B=2, H=2, Hq=16, L=3000, k=64), [3000, 1999], 0.0, 50, 100),
    ("gqa32b", dict(B=2, H=2, Hq=8, L=2500, k=40), [2500, 1300], 0.5, 80, 200),   # host tier
    ("host1m", dict(H=2, Hq=8, L=20000, k=100), None, 0.0, 50, 100),              # contiguous index keys
    ("mla", dict(B=2, L=3000, k=256), [3000, 2500], 0.0, 100, 100),                # latent rows, rho = beta
    ("tiny", dict(L=1000), None, 0.0, 1000, 1000),                                 # every key a candidate
]


@pytest.mark.parametrize("name,over,lens,host_frac,beta,rho", CASES)
def test_paris_matches_oracle(skv, name, over, lens, host_frac, beta, rho):
    wl = workloads.make_workload(name, device="cuda", gen_device="cpu", seq_lens=lens, host_frac=host_frac, **over)
    step, view, params = _run(skv, wl, beta, rho)
    hist = step.paris.hist.cpu().numpy()
    for b in range(wl.B):
        L = int(wl.seq_lens[b])
        for h in range(wl.H):
            row = b * wl.H + h
            check_encode(step, view, wl, b, h, np.arange(L))
            cent = step.paris.cent[row, :L].cpu().numpy().astype(np.int64)
            for s in range(16):
                np.testing.assert_array_equal(hist[row, s], np.bincount(cent[:, s], minlength=256))
            check_step(step, view, wl, b, h, params)


def test_paris_short_rows_and_large_k(skv):
    # request 1 has no candidates (L <= sink + local); k above the candidate count on request 0
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=2, H=2, Hq=8, L=1500, k=120,
                                 seq_lens=[1500, 100])
    step, view, params = _run(skv, wl, 50, 100)
    assert int(step.view("cand_len")[1]) == 0
    assert torch.all(step.idx[1] == -1)
    for b in range(2):
        for h in range(2):
            check_step(step, view, wl, b, h, params, e2e=False)


def test_paris_empty_and_one_token_histories(skv):
    # request 0 has no tokens, request 1 one token inside the sink
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=3, H=2, Hq=8, L=1200, k=40,
                                 seq_lens=[0, 1, 1200])
    step, view, params = _run(skv, wl, 50, 100)
    assert int(step.status.item()) == 0
    for b in (0, 1):
        assert int(step.view("cand_len")[b]) == 0 and torch.all(step.idx[b] == -1)
    assert torch.count_nonzero(step.out[0]).item() == 0 and torch.all(torch.isneginf(step.lse[0]))
    for b in range(3):
        for h in range(2):
            check_step(step, view, wl, b, h, params, e2e=(b == 2))


def test_zero_key_encodes_to_zero_weight(skv):
    wl = workloads.make_workload("host1m", device="cuda", gen_device="cpu", H=2, Hq=8, L=3000, k=50)
    wl.index_keys[0, 1, 777].zero_()
    signs = workloads.srht_signs(128, device="cuda")
    step = skv.ParisStep.from_workload(wl, signs)
    step.encode()
    torch.cuda.synchronize()
    assert int(step.paris.cent[1, 777].sum()) == 0 and int(step.paris.code[1, 777].abs().sum()) == 0
    assert float(step.paris.w[1, 777].abs().sum()) == 0.0


def test_encode_flags_bad_slots(skv):
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=1, H=2, Hq=8, L=800, k=10)
    wl.table[0, 5] = 10 ** 6
    signs = workloads.srht_signs(128, device="cuda")
    step = skv.ParisStep.from_workload(wl, signs)
    step.encode()
    torch.cuda.synchronize()
    assert int(step.status.item()) & skv.SKV_DEV_BAD_SLOT


def test_paris_full_size_host1m_sampled(skv):
    wl = workloads.make_workload("host1m", device="cuda", gen_device="cuda")
    step, view, params = _run(skv, wl, 50, 100)
    rng = np.random.default_rng(0)
    for h in (0, 5):
        row = h
        L = int(wl.seq_lens[0])
        check_encode(step, view, wl, 0, h, np.sort(rng.choice(L, 4000, replace=False)))
        cent = step.paris.cent[row, :L].cpu().numpy().astype(np.int64)
        hist = step.paris.hist[row].cpu().numpy()
        for s in (0, 7, 15):
            np.testing.assert_array_equal(hist[s], np.bincount(cent[:, s], minlength=256))
        check_step(step, view, wl, 0, h, params, e2e=(h == 0))


def test_select_then_attend_equals_the_step(skv):
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=2, H=2, Hq=8, L=2000, k=32,
                                 seq_lens=[2000, 1500])
    signs = workloads.srht_signs(128, device="cuda")
    one = skv.ParisStep.from_workload(wl, signs)
    one.encode()
    one.run()
    two = skv.ParisStep.from_workload(wl, signs)
    two.encode()
    two.select()
    two.attend()
    torch.cuda.synchronize()
    assert int(one.status.item()) == 0 and int(two.status.item()) == 0
    assert torch.equal(one.idx, two.idx) and torch.equal(one.out, two.out) and torch.equal(one.lse, two.lse)


def test_paris_step_replays_in_a_cuda_graph(skv):
    wl = workloads.make_workload("host1m", device="cuda", gen_device="cpu", H=2, Hq=8, L=20000, k=100)
    signs = workloads.srht_signs(128, device="cuda")
    eager = skv.ParisStep.from_workload(wl, signs)
    eager.encode()
    eager.run()
    graphed = skv.ParisStep.from_workload(wl, signs)
    graphed.encode()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        graphed.run()
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert int(graphed.status.item()) == 0
        assert torch.equal(eager.idx, graphed.idx) and torch.equal(eager.out, graphed.out)


def test_paris_large_k_takes_the_cluster_path_and_maps_positions(skv):
    # 40,000 candidate slots with k = 6,000: beyond the one-CTA and two-stage selections,
    # so the candidate slots go through the separate position map
    wl = workloads.make_workload("host1m", device="cuda", gen_device="cpu", H=1, Hq=4, L=200000, k=6000)
    step, view, params = _run(skv, wl, 200, 300)
    assert step.offsets[7] >= 40000
    check_step(step, view, wl, 0, 0, params, e2e=False)
