"""Block selection from per-block key summaries (OasisKV notes §3.2) on the GPU against the fp64 oracle."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from skv_test_utils import BAND_REL, OracleView, assert_attention_close, nv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def skv():
    import __graft_entry__

    __graft_entry__.build()
    import top_sparse_kv_gb300 as m

    return m


def _block_rows(view, b, h, blk, L, d):
    toks = np.arange(blk * 16, min(blk * 16 + 16, L))
    return view.kpool.rows(b, h, toks)[:, :d]


def _gpu_block_scores(step):
    """The block scores sit at the start of the workspace: fp32 [rows, ceil(max_len / 16)]."""
    p = step.p
    nb = (p.max_len + 15) // 16
    rows = p.batch * p.n_kv_heads
    return step.ws[: rows * nb * 4].view(torch.float32).view(p.batch, p.n_kv_heads, nb).cpu().numpy()


def _run(skv, wl, K, agg=0):
    step = skv.BlockStep.from_workload(wl, K, group_agg=agg)
    step.summarize()
    step.run()
    torch.cuda.synchronize()
    return step


BLOCK_CASES = [
    ("gqa32b", dict(B=2, H=2, Hq=16, L=3000, k=0), [3000, 1999], 0.0, torch.bfloat16, 20, "mean"),
    ("gqa32b", dict(B=2, H=2, Hq=8, L=1500, k=0), [1500, 777], 0.5, torch.bfloat16, 12, "mean"),  # host tier
    ("gqa32b", dict(B=1, H=4, Hq=8, L=2000, k=0), None, 0.0, torch.float32, 30, "mean"),          # fp32, G = 2
    ("gqa32b", dict(B=2, H=2, Hq=16, L=2500, k=0), [2500, 1000], 0.0, torch.bfloat16, 25, "max"),
    ("tiny", dict(L=1000), [1000], 0.0, torch.bfloat16, 8, "mean"),
    ("gqa32b", dict(B=3, H=2, Hq=8, L=1200, k=0), [0, 1, 1200], 0.0, torch.bfloat16, 10, "mean"),  # no blocks
]


@pytest.mark.parametrize("name,over,lens,host_frac,dtype,K,agg", BLOCK_CASES)
def test_block_decode_matches_oracle(skv, name, over, lens, host_frac, dtype, K, agg):
    wl = workloads.make_workload(name, device="cuda", gen_device="cpu", seq_lens=lens, host_frac=host_frac,
                                 dtype=dtype, **over)
    step = _run(skv, wl, K, skv.SKV_AGG_MAX if agg == "max" else skv.SKV_AGG_MEAN)
    assert int(step.status.item()) == 0
    view = OracleView(wl, group_agg=agg)
    summ = nv(step.summaries)
    bscore = _gpu_block_scores(step)
    bidx = step.block_idx.cpu().numpy()
    att = step.att_idx.cpu().numpy()
    G, d = wl.G, wl.d_qk
    for b in range(wl.B):
        L = int(wl.seq_lens[b])
        for h in range(wl.H):
            # summaries: exact min / max of the block's rows (bf16 in, bf16 out)
            nb, s_blk, l_blk = oracle.block_regions(L, wl.ns, wl.nl, 16)
            for blk in sorted({0, nb // 2, nb - 1}) if nb > 0 else []:
                lo, hi = oracle.block_summary(_block_rows(view, b, h, blk, L, d))
                np.testing.assert_array_equal(oracle.as_f64(summ[b, h, blk, 0]), lo)
                np.testing.assert_array_equal(oracle.as_f64(summ[b, h, blk, 1]), hi)
            ref = oracle.decode_unit_blocks(view.prob, b, h, view.q, view.kpool, view.vpool, K)
            cand = ref["block_positions"]
            # block scores within an fp32 bound of the fp64 box bounds
            qg = oracle.as_f64(view.q[b, h * G:(h + 1) * G])
            mag = np.array([np.abs(qg).max(axis=0) @ np.maximum(np.abs(oracle.block_summary(
                _block_rows(view, b, h, blk, L, d))[0]), np.abs(oracle.block_summary(
                    _block_rows(view, b, h, blk, L, d))[1])) for blk in cand])
            tol = 4.0 * (d + G) * 2.0 ** -24 * mag + 1e-30
            assert np.all(np.abs(bscore[b, h, cand] - ref["block_scores"]) <= tol)
            # the chosen blocks: bit-exact on the GPU's own block scores
            mine = oracle.decode_unit_blocks(view.prob, b, h, view.q, view.kpool, view.vpool, K,
                                             given_block_scores=bscore[b, h])
            ksel = min(K, len(cand))
            np.testing.assert_array_equal(bidx[b, h, :ksel], mine["blocks"])
            assert np.all(bidx[b, h, ksel:K] == -1)
            # ... and the fp64 set apart from blocks whose bound lies within the selection band
            # of the K-th bound: BAND_REL relative to max(|tau|, rms of the row's bounds), the
            # floor the token selection uses
            want, got = set(ref["blocks"].tolist()), set(bidx[b, h, :ksel].tolist())
            if want != got:
                tau = np.sort(ref["block_scores"])[::-1][ksel - 1]
                scale = max(abs(tau), float(np.sqrt(np.mean(ref["block_scores"] ** 2))))
                u = dict(zip(cand.tolist(), ref["block_scores"]))
                for blk in want ^ got:
                    assert abs(u[blk] - tau) <= BAND_REL * scale, (blk, u[blk], tau)
            # the attended list and the attention over it
            att_ref = oracle.block_attended_positions(L, 16, s_blk, l_blk, nb, mine["blocks"])
            row = att[b, h]
            np.testing.assert_array_equal(row[row >= 0], att_ref)
            assert np.all(row[len(att_ref):] == -1)
            res = oracle.decode_unit_blocks(view.prob, b, h, view.q, view.kpool, view.vpool, K,
                                            given_blocks=mine["blocks"])
            assert_attention_close(step.out[b, h * G:(h + 1) * G], res["out"], dtype)
            np.testing.assert_allclose(step.lse[b, h * G:(h + 1) * G].cpu().numpy(), res["lse"], rtol=1e-5,
                                       atol=1e-5)


@pytest.mark.parametrize("K,lens", [(20, [3000, 1999, 0, 1]), (0, [3000, 700, 17, 40]), (500, None)])
def test_decode_step_list_equals_standalone_select(skv, K, lens):
    """The bf16 decode step lists the chosen blocks' tokens inside the attention; the
    standalone selection runs its expansion kernel.  Same chosen blocks, same list, bit
    for bit: ragged and empty rows, K = 0, and K past the candidates (every block; its
    8,160-slot lists take more than 8 splits, so the attention merges through the
    workspace).  The step's output and lse match the oracle on the chosen blocks."""
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=4, H=2, Hq=16, L=3000, k=0,
                                 seq_lens=lens)
    step = skv.BlockStep.from_workload(wl, K)
    step.summarize()
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    fused_blocks, fused_list = step.block_idx.clone(), step.att_idx.clone()
    step.att_idx.fill_(-7)
    step.select()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    assert torch.equal(step.block_idx, fused_blocks)
    assert torch.equal(step.att_idx, fused_list)
    view = OracleView(wl)
    G = wl.G
    step.run()  # the fused step again: its attention output against the oracle on its blocks
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    for b in range(wl.B):
        L = int(wl.seq_lens[b])
        nb, s_blk, l_blk = oracle.block_regions(L, wl.ns, wl.nl, 16)
        for h in range(wl.H):
            ksel = min(K, l_blk - s_blk)
            want = oracle.block_attended_positions(L, 16, s_blk, l_blk, nb, fused_blocks[b, h, :ksel].cpu().numpy())
            row = fused_list[b, h].cpu().numpy()
            np.testing.assert_array_equal(row[row >= 0], want)
            assert np.all(row[len(want):] == -1)
            if L == 0:
                assert torch.count_nonzero(step.out[b, h * G:(h + 1) * G]).item() == 0
                continue
            res = oracle.decode_unit_blocks(view.prob, b, h, view.q, view.kpool, view.vpool, K,
                                            given_blocks=fused_blocks[b, h, :ksel].cpu().numpy())
            assert_attention_close(step.out[b, h * G:(h + 1) * G], res["out"], torch.bfloat16)
            np.testing.assert_allclose(step.lse[b, h * G:(h + 1) * G].cpu().numpy(), res["lse"], rtol=1e-5,
                                       atol=1e-5)


def test_every_block_chosen_is_dense_attention(skv):
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=1, H=2, Hq=16, L=700, k=0,
                                 dtype=torch.float32, keep_logical=True)
    step = _run(skv, wl, K=100)
    assert int(step.status.item()) == 0
    lk, lv = wl.meta["logical_k"].double(), wl.meta["logical_v"].double()
    for h in range(2):
        ref = torch.nn.functional.scaled_dot_product_attention(
            wl.q[0, 8 * h:8 * h + 8].double().cpu()[None], lk[0, h].cpu()[None], lv[0, h].cpu()[None],
            scale=wl.sm_scale)[0]
        assert (step.out[0, 8 * h:8 * h + 8].double().cpu() - ref).abs().max().item() <= 1e-4


def test_block_mode_full_size_gqa32b_sampled(skv):
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cuda")
    K = 205  # 3,280 tokens: the token path's k
    step = _run(skv, wl, K)
    assert int(step.status.item()) == 0
    view = OracleView(wl)
    bscore = _gpu_block_scores(step)
    bidx = step.block_idx.cpu().numpy()
    for b, h in ((0, 0), (4, 6), (7, 7)):
        mine = oracle.decode_unit_blocks(view.prob, b, h, view.q, view.kpool, view.vpool, K,
                                         given_block_scores=bscore[b, h])
        np.testing.assert_array_equal(bidx[b, h], mine["blocks"])
        res = oracle.decode_unit_blocks(view.prob, b, h, view.q, view.kpool, view.vpool, K,
                                        given_blocks=mine["blocks"])
        assert_attention_close(step.out[b, h * 8:(h + 1) * 8], res["out"], torch.bfloat16)


def test_block_summaries_flag_bad_slots(skv):
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=1, H=2, Hq=8, L=800, k=0)
    wl.table[0, 7] = 10 ** 6
    step = skv.BlockStep.from_workload(wl, 10)
    step.summarize()
    torch.cuda.synchronize()
    assert int(step.status.item()) & skv.SKV_DEV_BAD_SLOT
    assert torch.isnan(step.summaries[0, :, 7].float()).all()
    step.status.zero_()
    step.run()
    torch.cuda.synchronize()
    assert not (step.block_idx.cpu().numpy() == 7).any()  # a NaN-bounded block ranks last
    assert torch.isfinite(step.out.float()).all()
