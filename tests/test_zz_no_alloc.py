"""skv_topk_static: the top-k entry point that takes no workspace.

Some callers cannot allocate device memory when they select -- a plugin inside
a runtime that owns the memory pool and gives it no allocator, or a serving
loop that must not call cudaMalloc.  This test calls that entry point through
the C ABI and checks that it selects exactly what skv_topk (with a caller
workspace) selects, on two calls in a row with different problems, so stale
scratch from the first call cannot leak into the second.  It is collected last
and is self-contained: it passes alone in a fresh process and after the rest.
"""

import ctypes

import numpy as np
import pytest
import torch

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


def _problem(skv, B, H, L, k, lens):
    return skv.Problem(batch=B, n_kv_heads=H, n_q_heads=H, d_qk=128, d_v=128, max_len=L, topk=k, n_sink=4,
                       n_local=128, block_size=16,
                       seq_lens=torch.tensor(lens, dtype=torch.int32, device="cuda"))


def test_static_scratch_topk_matches_workspace_topk(skv):
    fn = _static_fn(skv)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cases = [(2, 4, 6000, 500, [6000, 4100]), (1, 2, 300000, 3000, [300000])]
    for call, (B, H, L, k, lens) in enumerate(cases):
        rng = np.random.default_rng(100 + call)
        s = (np.round(rng.standard_normal((B, H, L)) * 3) / 3).astype(np.float32)  # many ties
        scores = torch.from_numpy(s).cuda()
        p = _problem(skv, B, H, L, k, lens)
        ws = torch.empty((skv.skv_workspace_size(p),), dtype=torch.uint8, device="cuda")
        ref = torch.full((B, H, k), -9, dtype=torch.int32, device="cuda")
        st_ref = torch.zeros((1,), dtype=torch.int32, device="cuda")
        skv.skv_topk(p, scores, ref, ws, st_ref)
        got = torch.full((B, H, k), -9, dtype=torch.int32, device="cuda")
        st = torch.zeros((1,), dtype=torch.int32, device="cuda")
        cp = p.c()
        rc = fn(ctypes.byref(cp), scores.data_ptr(), got.data_ptr(), st.data_ptr(), stream)
        assert rc == 0, skv.skv_status_string(rc)
        torch.cuda.synchronize()
        assert int(st.item()) == 0 and int(st_ref.item()) == 0
        assert torch.equal(got, ref), f"call {call}: static-scratch selection differs"


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
