"""skv_topk_static: the top-k entry point that takes no workspace.

Some callers cannot allocate device memory when they select -- a plugin inside
a runtime that owns the memory pool and gives it no allocator, or a serving
loop that must not call cudaMalloc.  This test calls that entry point through
the C ABI several times in a row, each call on a selection path that keeps
state in the library's fixed scratch array (multi-CTA passes, two stages,
8-CTA clusters), and compares every call's selection element by element with
the fp64 oracle's exact top-k and with skv_topk given a caller workspace.  Each
call follows one that left different contents in the shared array, so stale
scratch cannot leak from one call into the next unnoticed.  It is collected
last and is self-contained: it passes alone in a fresh process and after the
rest.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def skv():
    import __graft_entry__

    __graft_entry__.build()
    import top_sparse_kv_gb300 as m

    return m


def _static_fn(skv):
    from top_sparse_kv_gb300 import binding

    fn = skv.lib().skv_topk_static
    fn.argtypes = [ctypes.POINTER(binding.CProblem), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_void_p]
    fn.restype = ctypes.c_int32
    return fn


def _problem(skv, B, H, L, k, lens, ns=4, nl=128):
    return skv.Problem(batch=B, n_kv_heads=H, n_q_heads=H, d_qk=128, d_v=128, max_len=L, topk=k, n_sink=ns,
                       n_local=nl, block_size=16,
                       seq_lens=torch.tensor(lens, dtype=torch.int32, device="cuda"))


def _expect(row, L, k, ns, nl):
    s_end, l_start = oracle.regions(L, ns, nl)
    pos = np.arange(s_end, l_start)
    sel = oracle.exact_topk(row[pos].astype(np.float64), pos, k)
    out = np.full(k, -1, dtype=np.int64)
    out[: len(sel)] = sel
    return out


# (B, H, L, k, lens, seed): every call uses the scratch array; the path it takes is named
CALLS = [
    (1, 2, 300000, 3000, [300000], 11),          # multi-CTA passes (tickets, row state, counts)
    (2, 2, 100000, 2048, [100000, 77777], 12),   # two stages (segment winners)
    (1, 1, 100000, 6000, [100000], 13),          # 8-CTA clusters (row histograms)
    (1, 2, 300000, 3000, [300000], 14),          # multi-CTA again, other scores
    (3, 1, 40960, 4096, [40960, 40000, 5], 15),  # two stages after a multi-CTA call, ragged rows
]


def test_static_scratch_topk_matches_oracle_on_calls_in_a_row(skv):
    fn = _static_fn(skv)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, (B, H, L, k, lens, seed) in enumerate(CALLS):
        rng = np.random.default_rng(seed)
        s = (np.round(rng.standard_normal((B, H, L)) * 3) / 3).astype(np.float32)  # many ties
        scores = torch.from_numpy(s).cuda()
        p = _problem(skv, B, H, L, k, lens)
        cp = p.c()
        got = torch.full((B, H, k), -9, dtype=torch.int32, device="cuda")
        st = torch.zeros((1,), dtype=torch.int32, device="cuda")
        rc = fn(ctypes.byref(cp), scores.data_ptr(), got.data_ptr(), st.data_ptr(), stream)
        assert rc == 0, skv.skv_status_string(rc)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        got_np = got.cpu().numpy()
        for b in range(B):
            for h in range(H):
                want = _expect(s[b, h], lens[b], k, 4, 128)
                np.testing.assert_array_equal(got_np[b, h], want, err_msg=f"call {call}, unit ({b}, {h})")
        # and the same selection as the workspace entry point
        ws = torch.empty((skv.skv_workspace_size(p),), dtype=torch.uint8, device="cuda")
        ref = torch.full((B, H, k), -9, dtype=torch.int32, device="cuda")
        st_ref = torch.zeros((1,), dtype=torch.int32, device="cuda")
        skv.skv_topk(p, scores, ref, ws, st_ref)
        torch.cuda.synchronize()
        assert int(st_ref.item()) == 0
        assert torch.equal(got, ref), f"call {call}: static-scratch selection differs from skv_topk"


def test_static_scratch_rejects_problems_beyond_its_size(skv):
    fn = _static_fn(skv)
    # 1024 rows of 300K keys with k = 3000 (multi-CTA state, ~24 KB a row): more than 16 MiB of scratch
    p = _problem(skv, 128, 8, 300000, 3000, [300000] * 128)
    scores = torch.zeros((1,), dtype=torch.float32, device="cuda")
    idx = torch.zeros((1,), dtype=torch.int32, device="cuda")
    cp = p.c()
    n0 = skv.skv_launch_count()
    rc = fn(ctypes.byref(cp), scores.data_ptr(), idx.data_ptr(), None, None)
    assert rc == 4  # SKV_ERR_WORKSPACE_TOO_SMALL: nothing enqueued
    assert skv.skv_launch_count() == n0
