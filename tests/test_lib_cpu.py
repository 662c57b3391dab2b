"""The C ABI library without a GPU: it builds, loads, exports every declared
symbol, and rejects bad arguments on the host before touching CUDA."""

import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import __graft_entry__

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def skv():
    __graft_entry__.build()
    import top_sparse_kv_gb300 as m

    return m


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "skv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(skv_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("skv_score", "skv_topk", "skv_gather", "skv_sparse_attn", "skv_decode_step", "skv_workspace_size",
              "skv_status_string", "skv_launch_count"):
        assert n in names


def test_library_exports_every_declared_symbol(skv):
    from top_sparse_kv_gb300 import binding

    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (skv_[a-z_]+)\b", out))
    missing = [n for n in declared_symbols() if n not in exported]
    assert not missing, missing
    for n in declared_symbols():
        assert hasattr(skv.lib(), n)


def test_status_strings(skv):
    assert skv.skv_status_string(0) == "ok"
    assert skv.skv_status_string(1) == "invalid argument"
    assert skv.skv_status_string(4) == "workspace too small"
    assert skv.skv_status_string(99) == "unknown status"


FAKE = 1 << 20  # an aligned, never-dereferenced address: validation must reject before use


def _cproblem(skv, **over):
    from top_sparse_kv_gb300 import binding

    d = dict(batch=2, n_kv_heads=2, n_q_heads=8, d_qk=128, d_v=128, d_idx=128, n_idx_q_heads=8, max_len=1000,
             topk=10, n_sink=4, n_local=16, block_size=16, dtype=0, group_agg=0, sm_scale=0.0, n_splits=0,
             seq_lens=FAKE)
    d.update(over)
    return binding.CProblem(**d)


def _call(skv, name, *args):
    return getattr(skv.lib(), name)(*args)


@pytest.mark.parametrize("over", [
    dict(group_agg=1, dtype=1),                              # max: bf16 only (tensor-core scoring)
    dict(group_agg=1, n_q_heads=68, n_idx_q_heads=68),       # max: at most 16 scoring heads per KV head
])
def test_max_aggregation_limits_are_unsupported(skv, over):
    p = _cproblem(skv, **over)
    n = ctypes.c_size_t(0)
    assert _call(skv, "skv_workspace_size", ctypes.byref(p), ctypes.byref(n)) == 2


def test_max_aggregation_accepted_for_bf16(skv):
    p = _cproblem(skv, group_agg=1)
    n = ctypes.c_size_t(0)
    assert _call(skv, "skv_workspace_size", ctypes.byref(p), ctypes.byref(n)) == 0


@pytest.mark.parametrize("over", [
    dict(group_agg=2, dtype=1),                              # per head: bf16 only (tensor-core scoring)
    dict(group_agg=2, n_idx_q_heads=2),                      # per head: the attention heads score
    dict(group_agg=2, n_q_heads=68, n_idx_q_heads=68),       # per head: at most 16 query heads per KV head
])
def test_head_reading_limits_are_unsupported(skv, over):
    p = _cproblem(skv, **over)
    n = ctypes.c_size_t(0)
    assert _call(skv, "skv_workspace_size", ctypes.byref(p), ctypes.byref(n)) == 2


def test_head_reading_sizes_one_row_per_query_head(skv):
    # per query head the selection and attention rows are those of a problem with one
    # query head per KV head, n_q_heads KV heads (the state per row is the same)
    for over in (dict(), dict(max_len=300000, topk=3000), dict(batch=7, n_kv_heads=1, n_q_heads=16,
                                                                n_idx_q_heads=16)):
        head, rows = ctypes.c_size_t(0), ctypes.c_size_t(0)
        p = _cproblem(skv, group_agg=2, **over)
        assert _call(skv, "skv_workspace_size", ctypes.byref(p), ctypes.byref(head)) == 0
        r = _cproblem(skv, **dict(over, n_kv_heads=p.n_q_heads))
        assert _call(skv, "skv_workspace_size", ctypes.byref(r), ctypes.byref(rows)) == 0
        assert head.value == rows.value > 0


def test_head_reading_refused_by_the_other_entry_points(skv):
    from top_sparse_kv_gb300 import binding

    p = _cproblem(skv, group_agg=2)
    n, ln = ctypes.c_size_t(0), ctypes.c_int32(0)
    n0 = skv.skv_launch_count()
    assert _call(skv, "skv_block_workspace_size", ctypes.byref(p), 10, ctypes.byref(n), ctypes.byref(ln)) == 2
    contig = binding.CIndex(1, FAKE)
    pf = binding.CPrefetch(FAKE, FAKE, FAKE, FAKE, FAKE, None, 16, 0.5)
    assert skv.lib().skv_decode_step_prefetch(ctypes.byref(p), FAKE, FAKE, ctypes.byref(contig),
                                              ctypes.byref(_cpool(skv)), FAKE, FAKE, FAKE, None, FAKE, 1 << 30,
                                              ctypes.byref(pf), None, None) == 2
    pool = _cpool(skv, gpu_v=None, n_gpu_blocks=500, host_k=FAKE, n_host_blocks=2000, table_stride=1000)
    assert _call(skv, "skv_cache_workspace_size", ctypes.byref(_cproblem(skv, group_agg=2, block_size=1)),
                 ctypes.byref(pool), 64, ctypes.byref(n)) == 2
    assert skv.lib().skv_paris_workspace_size(ctypes.byref(p), ctypes.byref(binding.CParis(8, 50, 100, FAKE)),
                                              ctypes.byref(n)) == 2
    # the latent layout has one KV head whose rows are shared: no per-head rows
    f = skv.lib().skv_sparse_attn
    lat = _cproblem(skv, group_agg=2, n_kv_heads=1, n_q_heads=16, n_idx_q_heads=16)
    assert f(ctypes.byref(lat), FAKE, ctypes.byref(_cpool(skv, gpu_v=None)), FAKE, FAKE, None, FAKE,
             ctypes.c_size_t(1 << 40), None, None) == 2
    assert skv.skv_launch_count() == n0


@pytest.mark.parametrize("over", [
    dict(batch=0), dict(n_kv_heads=0), dict(n_q_heads=7), dict(topk=-1), dict(n_sink=-2), dict(max_len=-1),
    dict(block_size=0), dict(dtype=5), dict(group_agg=3), dict(seq_lens=0), dict(n_idx_q_heads=3),
    dict(sm_scale=float("nan")), dict(n_splits=-1),
])
def test_workspace_size_rejects_bad_problems(skv, over):
    p = _cproblem(skv, **over)
    n = ctypes.c_size_t(0)
    assert _call(skv, "skv_workspace_size", ctypes.byref(p), ctypes.byref(n)) == 1


def test_workspace_size_grows_with_problem(skv):
    small, big = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert _call(skv, "skv_workspace_size", ctypes.byref(_cproblem(skv)), ctypes.byref(small)) == 0
    assert _call(skv, "skv_workspace_size", ctypes.byref(_cproblem(skv, batch=16, max_len=100000)),
                 ctypes.byref(big)) == 0
    assert 0 < small.value < big.value
    assert _call(skv, "skv_workspace_size", None, ctypes.byref(small)) == 1


def test_topk_rejects_small_workspace_and_nulls(skv):
    p = _cproblem(skv, max_len=300000, topk=3000)  # long rows, large k: multi-CTA state in the workspace
    n = ctypes.c_size_t(0)
    _call(skv, "skv_workspace_size", ctypes.byref(p), ctypes.byref(n))
    f = skv.lib().skv_topk
    assert f(ctypes.byref(p), FAKE, FAKE, FAKE, 16, None, None) == 4  # far below the multi-CTA path's state
    assert f(ctypes.byref(p), None, FAKE, FAKE, n.value, None, None) == 1
    assert f(ctypes.byref(p), FAKE, FAKE, FAKE + 4, n.value, None, None) == 1  # misaligned workspace


def _cpool(skv, **over):
    from top_sparse_kv_gb300 import binding

    d = dict(gpu_k=FAKE, gpu_v=FAKE, n_gpu_blocks=128, host_k=None, host_v=None, n_host_blocks=0,
             slot_table=FAKE, table_stride=63)
    d.update(over)
    return binding.CPool(**d)


def test_score_rejects_unsupported_and_invalid(skv):
    from top_sparse_kv_gb300 import binding

    f = skv.lib().skv_score
    idx = binding.CIndex(0, None)
    ok_pool = _cpool(skv)
    assert f(ctypes.byref(_cproblem(skv, d_idx=64, d_qk=64)), FAKE, ctypes.byref(idx), ctypes.byref(ok_pool),
             FAKE, None, None) == 2
    assert f(ctypes.byref(_cproblem(skv, block_size=8)), FAKE, ctypes.byref(idx),
             ctypes.byref(_cpool(skv, table_stride=125)), FAKE, None, None) == 2
    assert f(ctypes.byref(_cproblem(skv)), FAKE, ctypes.byref(idx), ctypes.byref(_cpool(skv, table_stride=62)),
             FAKE, None, None) == 1  # table too narrow for max_len
    assert f(ctypes.byref(_cproblem(skv)), FAKE + 8, ctypes.byref(idx), ctypes.byref(ok_pool), FAKE, None,
             None) == 1  # misaligned query
    contig = binding.CIndex(1, None)
    assert f(ctypes.byref(_cproblem(skv)), FAKE, ctypes.byref(contig), None, FAKE, None, None) == 1
    assert f(ctypes.byref(_cproblem(skv)), FAKE, ctypes.byref(binding.CIndex(7, FAKE)), ctypes.byref(ok_pool),
             FAKE, None, None) == 1


def test_attention_rejects_unsupported_shapes(skv):
    f = skv.lib().skv_sparse_attn
    big = ctypes.c_size_t(1 << 40)
    assert f(ctypes.byref(_cproblem(skv, n_q_heads=64, n_idx_q_heads=64, n_kv_heads=2)), FAKE,
             ctypes.byref(_cpool(skv)), FAKE, FAKE, None, FAKE, big, None, None) == 2  # G = 32
    assert f(ctypes.byref(_cproblem(skv, d_qk=64, d_v=64)), FAKE, ctypes.byref(_cpool(skv)), FAKE, FAKE, None,
             FAKE, big, None, None) == 2
    assert f(ctypes.byref(_cproblem(skv, n_kv_heads=2)), FAKE, ctypes.byref(_cpool(skv, gpu_v=None)), FAKE, FAKE,
             None, FAKE, big, None, None) == 1  # latent layout needs one KV head
    assert f(ctypes.byref(_cproblem(skv)), FAKE, ctypes.byref(_cpool(skv)), FAKE, FAKE, None, FAKE, 16, None,
             None) == 4


def test_head_table_validation(skv):
    # one slot-table row per (request, KV head): K and V pools only, and only the entry
    # points that resolve rows per head
    from top_sparse_kv_gb300 import binding

    p = _cproblem(skv)
    big = ctypes.c_size_t(1 << 40)
    n0 = skv.skv_launch_count()
    attn = skv.lib().skv_sparse_attn
    assert attn(ctypes.byref(p), FAKE, ctypes.byref(_cpool(skv, table_heads=2)), FAKE, FAKE, None, FAKE, big,
                None, None) == 1
    lat = _cproblem(skv, n_kv_heads=1, n_q_heads=8, d_qk=576, d_v=512, n_idx_q_heads=1, block_size=1,
                    max_len=1000)
    assert attn(ctypes.byref(lat), FAKE, ctypes.byref(_cpool(skv, gpu_v=None, table_heads=1, table_stride=1000)),
                FAKE, FAKE, None, FAKE, big, None, None) == 2
    per_head = _cpool(skv, table_heads=1)
    assert skv.lib().skv_block_summaries(ctypes.byref(p), ctypes.byref(per_head), FAKE, None, None) == 2
    contig = binding.CIndex(1, FAKE)
    pf = binding.CPrefetch(FAKE, FAKE, FAKE, FAKE, FAKE, None, 16, 0.5)
    assert skv.lib().skv_decode_step_prefetch(ctypes.byref(p), FAKE, FAKE, ctypes.byref(contig),
                                              ctypes.byref(per_head), FAKE, FAKE, FAKE, None, FAKE, 1 << 30,
                                              ctypes.byref(pf), None, None) == 2
    # the slot cache takes per-head tables when the host pool backs every block
    n = ctypes.c_size_t(0)
    assert skv.lib().skv_cache_workspace_size(ctypes.byref(p), ctypes.byref(per_head), 64, ctypes.byref(n)) == 2
    backed = _cpool(skv, table_heads=1, host_k=FAKE, host_v=FAKE, n_host_blocks=2 * 63)
    assert skv.lib().skv_cache_workspace_size(ctypes.byref(p), ctypes.byref(backed), 64, ctypes.byref(n)) == 0
    assert n.value > 0
    wide = _cproblem(skv, batch=130, n_kv_heads=8, n_q_heads=64, n_idx_q_heads=64)  # 1,040 units
    assert skv.lib().skv_cache_workspace_size(ctypes.byref(wide), ctypes.byref(
        _cpool(skv, table_heads=1, host_k=FAKE, host_v=FAKE, n_host_blocks=130 * 63)), 64, ctypes.byref(n)) == 2
    ix = binding.CParisIndex(FAKE, FAKE, FAKE)
    assert skv.lib().skv_paris_encode(ctypes.byref(p), ctypes.byref(binding.CParis(8, 50, 100, FAKE)),
                                      ctypes.byref(binding.CIndex(0, None)), ctypes.byref(per_head),
                                      ctypes.byref(ix), None, None) == 2
    assert skv.skv_launch_count() == n0


def test_no_kernel_launched_by_rejected_calls(skv):
    n0 = skv.skv_launch_count()
    test_attention_rejects_unsupported_shapes(skv)
    test_score_rejects_unsupported_and_invalid(skv)
    assert skv.skv_launch_count() == n0


@pytest.mark.parametrize("over,want", [
    (dict(block_size=1), 2), (dict(d_qk=64, d_v=64), 2), (dict(n_idx_q_heads=2), 2), (dict(batch=0), 1),
])
def test_block_workspace_size_validation(skv, over, want):
    p = _cproblem(skv, **over)
    n, ln = ctypes.c_size_t(0), ctypes.c_int32(0)
    assert _call(skv, "skv_block_workspace_size", ctypes.byref(p), 10, ctypes.byref(n), ctypes.byref(ln)) == want


def test_block_workspace_size_and_list_length(skv):
    p = _cproblem(skv)
    n, ln = ctypes.c_size_t(0), ctypes.c_int32(0)
    assert _call(skv, "skv_block_workspace_size", ctypes.byref(p), 10, ctypes.byref(n), ctypes.byref(ln)) == 0
    assert ln.value == 16 * (1 + 10 + 1 + 1)  # sink 4 -> 1 block, k 10, local 16 -> 1 block, + 1 partial
    assert n.value > 0
    assert _call(skv, "skv_block_workspace_size", ctypes.byref(p), -1, ctypes.byref(n), ctypes.byref(ln)) == 1


def test_block_calls_reject_before_enqueuing(skv):
    p = _cproblem(skv)
    n, ln = ctypes.c_size_t(0), ctypes.c_int32(0)
    _call(skv, "skv_block_workspace_size", ctypes.byref(p), 10, ctypes.byref(n), ctypes.byref(ln))
    n0 = skv.skv_launch_count()
    sel = skv.lib().skv_block_select
    assert sel(ctypes.byref(p), 10, FAKE, FAKE, FAKE, FAKE, FAKE, n.value - 1, None, None) == 4
    assert sel(ctypes.byref(p), 10, FAKE, FAKE, None, FAKE, FAKE, n.value, None, None) == 1  # no block_idx
    assert sel(ctypes.byref(p), 10, FAKE + 8, FAKE, FAKE, FAKE, FAKE, n.value, None, None) == 1  # misaligned q
    pool = _cpool(skv)
    assert skv.lib().skv_block_summaries(ctypes.byref(p), ctypes.byref(pool), None, None, None) == 1
    assert skv.skv_launch_count() == n0


def test_prefetch_refuses_unsupported_layouts_before_enqueuing(skv):
    from top_sparse_kv_gb300 import binding

    p = _cproblem(skv)
    pool = _cpool(skv)
    paged_index = binding.CIndex(0, None)
    contig = binding.CIndex(1, FAKE)
    pf = binding.CPrefetch(FAKE, FAKE, FAKE, FAKE, FAKE, None, 16, 0.5)
    n0 = skv.skv_launch_count()
    f = skv.lib().skv_decode_step_prefetch

    def call(prob, index, pool_, pf_):
        return f(ctypes.byref(prob), FAKE, FAKE, ctypes.byref(index), ctypes.byref(pool_), FAKE, FAKE, FAKE, None,
                 FAKE, 1 << 30, pf_, None, None)

    # scoring through the pool itself: the prefetch needs the GPU-resident index keys
    assert call(p, paged_index, pool, ctypes.byref(pf)) == 2
    # paged pools: 16-token blocks of 128-wide K and V rows, bf16, the mean reading
    assert call(_cproblem(skv, block_size=8), contig, _cpool(skv, table_stride=125), ctypes.byref(pf)) == 2
    assert call(_cproblem(skv, dtype=1), contig, pool, ctypes.byref(pf)) == 2
    assert call(_cproblem(skv, group_agg=1), contig, pool, ctypes.byref(pf)) == 2
    assert call(p, contig, pool, None) == 1  # no prefetch state
    bad_alpha = binding.CPrefetch(FAKE, FAKE, FAKE, FAKE, FAKE, None, 16, 0.0)
    assert call(p, contig, pool, ctypes.byref(bad_alpha)) == 1
    assert skv.skv_launch_count() == n0


def _latent(skv, **over):
    d = dict(batch=2, n_kv_heads=1, n_q_heads=128, d_qk=576, d_v=512, d_idx=128, n_idx_q_heads=1, max_len=1000,
             topk=64, n_sink=0, n_local=0, block_size=1)
    d.update(over)
    return _cproblem(skv, **d)


def test_slot_cache_validation_before_enqueuing(skv):
    from top_sparse_kv_gb300 import binding

    pool = _cpool(skv, gpu_v=None, n_gpu_blocks=500, host_k=FAKE, n_host_blocks=2000, table_stride=1000)
    n = ctypes.c_size_t(0)
    f = skv.lib().skv_cache_workspace_size
    assert f(ctypes.byref(_latent(skv)), ctypes.byref(pool), 64, ctypes.byref(n)) == 0 and n.value > 0
    small = n.value
    assert f(ctypes.byref(_latent(skv)), ctypes.byref(pool), 4096, ctypes.byref(n)) == 0 and n.value > small
    assert f(ctypes.byref(_latent(skv)), ctypes.byref(pool), -1, ctypes.byref(n)) == 1
    assert f(ctypes.byref(_latent(skv)), ctypes.byref(_cpool(skv, host_k=FAKE, host_v=FAKE, n_host_blocks=2000,
                                                            table_stride=1000)), 64, ctypes.byref(n)) == 2  # K and V
    short = _cpool(skv, gpu_v=None, n_gpu_blocks=500, host_k=FAKE, n_host_blocks=1999, table_stride=1000)
    assert f(ctypes.byref(_latent(skv)), ctypes.byref(short), 64, ctypes.byref(n)) == 2  # host pool misses rows
    wide = _cpool(skv, gpu_v=None, n_gpu_blocks=500, host_k=FAKE, n_host_blocks=65000, table_stride=1000)
    assert f(ctypes.byref(_latent(skv, batch=65)), ctypes.byref(wide), 64, ctypes.byref(n)) == 2

    g = skv.lib().skv_decode_step_cached
    idx = binding.CIndex(binding.SKV_INDEX_CONTIG, FAKE)
    cache = binding.CSlotCache(FAKE, FAKE, FAKE, 64)
    p = _latent(skv)
    f(ctypes.byref(p), ctypes.byref(pool), 64, ctypes.byref(n))
    n0 = skv.skv_launch_count()
    args = (ctypes.byref(p), FAKE, FAKE, ctypes.byref(idx), ctypes.byref(pool), FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30)
    assert g(*args, None, FAKE, n.value, None, None) == 1                                         # no cache state
    assert g(*args, ctypes.byref(cache), FAKE, n.value - 1, None, None) == 4                      # workspace short
    assert g(*args, ctypes.byref(binding.CSlotCache(FAKE, None, FAKE, 64)), FAKE, n.value, None, None) == 1
    assert g(*args, ctypes.byref(binding.CSlotCache(FAKE, FAKE, FAKE, -3)), FAKE, n.value, None, None) == 1
    u = skv.lib().skv_cache_update
    ws = ctypes.c_size_t(0)
    assert skv.lib().skv_workspace_size(ctypes.byref(p), ctypes.byref(ws)) == 0
    assert u(ctypes.byref(p), ctypes.byref(pool), FAKE, FAKE, ws.value - 1, ctypes.byref(cache), FAKE, n.value,
             None, None) == 4                                                                     # step ws short
    assert u(ctypes.byref(p), ctypes.byref(pool), None, FAKE, ws.value, ctypes.byref(cache), FAKE, n.value,
             None, None) == 1                                                                     # no selection
    assert skv.skv_launch_count() == n0


def test_paris_quantizer_matches_the_oracle(skv):
    from oracle import paris_oracle as po

    for m in (3, 8, 16):
        lv, th = skv.skv_paris_quantizer(m)
        want_lv, want_th = po.lloyd_max(m)
        np.testing.assert_allclose(lv, want_lv, rtol=0, atol=1e-7)
        np.testing.assert_allclose(th, want_th, rtol=0, atol=1e-7)
    from top_sparse_kv_gb300 import binding

    lv, th = (ctypes.c_float * 8)(), (ctypes.c_float * 7)()
    f = skv.lib().skv_paris_quantizer
    assert f(2, ctypes.cast(lv, ctypes.c_void_p), ctypes.cast(th, ctypes.c_void_p)) == 1
    assert f(8, None, ctypes.cast(th, ctypes.c_void_p)) == 1
    del binding


def test_paris_validation_before_enqueuing(skv):
    from top_sparse_kv_gb300 import binding

    p = _cproblem(skv, n_sink=4, n_local=16)
    pool = _cpool(skv)
    ix = binding.CParisIndex(FAKE, FAKE, FAKE)
    paged = binding.CIndex(0, None)
    n0 = skv.skv_launch_count()
    enc = skv.lib().skv_paris_encode

    def call(pr, prob=p, index=paged):
        return enc(ctypes.byref(prob), ctypes.byref(pr), ctypes.byref(index), ctypes.byref(pool), ctypes.byref(ix),
                   None, None)

    assert call(binding.CParis(8, 0, 100, FAKE)) == 1       # beta 0
    assert call(binding.CParis(8, 200, 100, FAKE)) == 1     # rho < beta
    assert call(binding.CParis(8, 50, 1001, FAKE)) == 1     # rho > 1000
    assert call(binding.CParis(8, 50, 100, None)) == 1      # no signs
    assert call(binding.CParis(4, 50, 100, FAKE)) == 2      # m = 4 not built
    assert call(binding.CParis(8, 50, 100, FAKE), prob=_cproblem(skv, dtype=1)) == 2  # fp32 keys not built
    assert call(binding.CParis(8, 50, 100, FAKE), prob=_cproblem(skv, d_qk=64, d_v=64)) == 2
    assert call(binding.CParis(8, 50, 100, FAKE), index=binding.CIndex(1, None)) == 1  # contiguous without keys
    assert call(binding.CParis(8, 50, 100, FAKE), prob=_cproblem(skv, batch=40000, n_kv_heads=2, n_q_heads=8,
                                                                 n_idx_q_heads=8)) == 2  # rows beyond grid.y
    n = ctypes.c_size_t(0)
    assert skv.lib().skv_workspace_size(ctypes.byref(_cproblem(skv, batch=70000)), ctypes.byref(n)) == 2
    n = ctypes.c_size_t(0)
    assert skv.lib().skv_paris_workspace_size(ctypes.byref(p), ctypes.byref(binding.CParis(8, 50, 100, FAKE)),
                                              ctypes.byref(n)) == 0
    wide = ctypes.c_size_t(0)
    assert skv.lib().skv_paris_workspace_size(ctypes.byref(p), ctypes.byref(binding.CParis(8, 500, 500, FAKE)),
                                              ctypes.byref(wide)) == 0 and wide.value > n.value
    step = skv.lib().skv_paris_decode_step
    assert step(ctypes.byref(p), ctypes.byref(binding.CParis(8, 50, 100, FAKE)), FAKE, FAKE, ctypes.byref(paged),
                ctypes.byref(ix), ctypes.byref(pool), FAKE, FAKE, FAKE, FAKE, n.value - 1, None, None) == 4
    assert skv.skv_launch_count() == n0


@pytest.mark.parametrize("limit,arrive,with_status", [
    (0, 0, True), (4_000_000_001, 0, True), (-5, 1, True), (1000, 2, True), (1000, -1, True), (1000, 0, False),
])
def test_wait_check_validates_before_enqueuing(skv, limit, arrive, with_status):
    status = ctypes.c_int32(0)  # never written: every case here is rejected on the host
    ptr = ctypes.cast(ctypes.pointer(status), ctypes.c_void_p) if with_status else None
    n0 = skv.skv_launch_count()
    assert _call(skv, "skv_check_wait_timeout", ctypes.c_int64(limit), ctypes.c_int32(arrive), ptr, None) == 1
    assert skv.skv_launch_count() == n0
