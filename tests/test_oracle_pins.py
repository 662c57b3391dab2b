"""Pins of the fp64 oracle against things other than itself.

Each test ties one oracle function to a fact fixed by the pages or by
mathematics: IEEE bit layouts, brute-force enumeration, closed forms, a library
routine (torch's stable sort, torch's attention), the pages' worked byte counts
and the placement invariances the pages state.  A plausible slip in the oracle
(a dropped term, a wrong sign or index, a transposed operand, a wrong tie rule)
fails at least one of them.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- bf16 decoding


def test_bf16_decode_known_patterns():
    # IEEE binary32 upper halves: sign | 8-bit exponent (bias 127) | 7 mantissa bits
    cases = {
        0x3F80: 1.0, 0xC000: -2.0, 0x3F00: 0.5, 0x4049: 3.140625, 0x0000: 0.0,
        0x7F80: math.inf, 0xFF80: -math.inf, 0x0001: 2.0 ** -133, 0x7F7F: (2 - 2 ** -7) * 2.0 ** 127,
    }
    bits = np.array(list(cases), dtype=np.uint16)
    got = oracle.bf16_bits_to_f64(bits)
    for b, v, g in zip(cases, cases.values(), got):
        assert g == v, hex(b)
    neg_zero = oracle.bf16_bits_to_f64(np.array([0x8000], dtype=np.uint16))[0]
    assert neg_zero == 0.0 and math.copysign(1.0, neg_zero) == -1.0


def test_bf16_decode_matches_torch_on_all_finite_patterns():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    exp = (bits >> 7) & 0xFF
    finite = bits[exp != 0xFF]
    ours = oracle.bf16_bits_to_f64(finite)
    ref = torch.from_numpy(finite.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(ours, ref)


# ---------------------------------------------------------------- regions


@pytest.mark.parametrize("L,ns,nl,want", [
    (100, 4, 10, (4, 90)), (3, 4, 10, (3, 3)), (10, 4, 10, (4, 4)), (0, 4, 64, (0, 0)),
    (14, 4, 10, (4, 4)), (15, 4, 10, (4, 5)), (4096, 0, 0, (0, 4096)),
])
def test_regions_cases(L, ns, nl, want):
    assert oracle.regions(L, ns, nl) == want


def test_regions_partition_invariants():
    for L, ns, nl in itertools.product(range(0, 40), (0, 1, 4, 16), (0, 1, 5, 33)):
        s_end, l_start = oracle.regions(L, ns, nl)
        sink = set(range(0, s_end))
        cand = set(range(s_end, l_start))
        local = set(range(l_start, L))
        assert sink | cand | local == set(range(L))
        assert not (sink & cand or sink & local or cand & local)
        assert len(sink) == min(ns, L)
        assert len(local) == min(nl, L - len(sink))


# ---------------------------------------------------------------- S0 group query


def test_group_query_single_head_is_identity():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((1, 16))
    np.testing.assert_array_equal(oracle.group_query(q), q[0])


def test_group_query_score_is_mean_of_per_head_scores():
    # <mean_g q_g, k> = (1/G) sum_g <q_g, k>: computed head by head with G = 1
    rng = np.random.default_rng(1)
    q = rng.standard_normal((8, 32))
    K = rng.standard_normal((50, 32))
    via_mean = oracle.scores(oracle.group_query(q), K)
    per_head = np.mean([oracle.scores(oracle.group_query(q[g:g + 1]), K) for g in range(8)], axis=0)
    np.testing.assert_allclose(via_mean, per_head, rtol=1e-13, atol=1e-13)


def test_group_to_kv_head_mapping():
    # query head j belongs to KV head j // G: zero every query head except one
    wl = workloads.make_workload("tiny", B=1, H=2, Hq=8, L=64, k=4, ns=0, nl=0, keep_logical=True)
    q = workloads.numpy_view(wl.q).copy()
    q[:] = 0
    q[0, 5] = workloads.numpy_view(wl.q)[0, 5]  # head 5 -> KV head 1 (G = 4)
    prob = _prob(wl)
    pools = _pools(wl)
    r0 = oracle.decode_unit(prob, 0, 0, q, *pools)
    r1 = oracle.decode_unit(prob, 0, 1, q, *pools)
    assert np.all(r0["scores"] == 0.0)
    keys = oracle.as_f64(workloads.numpy_view(wl.meta["logical_k"]))[0, 1]
    want = keys @ oracle.as_f64(q[0, 5]) / 4.0
    np.testing.assert_allclose(r1["scores"], want, rtol=1e-13, atol=1e-12)


# ---------------------------------------------------------------- S2 exact top-k


def _brute_topk(s, k):
    """Enumerate every k-subset; keep those whose every member scores at least as
    high as every non-member (the threshold property); return the lexicographically
    smallest sorted tuple among them (ties to lower positions).  NaN ranks lowest."""
    n = len(s)
    k = min(k, n)

    def key(x):
        return (0, 0.0) if math.isnan(x) else (1, x)

    best = None
    for sub in itertools.combinations(range(n), k):
        inside = set(sub)
        lo = min((key(s[i]) for i in inside), default=None)
        hi = max((key(s[j]) for j in range(n) if j not in inside), default=None)
        if lo is not None and hi is not None and lo < hi:
            continue
        if best is None or sub < best:
            best = sub
    return list(best)


def test_topk_against_brute_force_with_ties():
    rng = np.random.default_rng(2)
    for trial in range(300):
        n = int(rng.integers(0, 10))
        s = rng.integers(-2, 3, size=n).astype(np.float64)  # many ties
        if trial % 5 == 0 and n:
            s[rng.integers(0, n)] = -0.0
        if trial % 7 == 0 and n:
            s[rng.integers(0, n)] = np.nan
        for k in range(0, n + 2):
            got = oracle.exact_topk(s, np.arange(n), k)
            assert list(got) == _brute_topk(list(s), k), (s, k)


def test_topk_maximises_selected_sum():
    rng = np.random.default_rng(3)
    for _ in range(50):
        n = int(rng.integers(1, 11))
        s = rng.standard_normal(n)
        k = int(rng.integers(1, n + 1))
        got = oracle.exact_topk(s, np.arange(n), k)
        best = max(sum(s[list(c)]) for c in itertools.combinations(range(n), k))
        assert abs(s[got].sum() - best) < 1e-12


def test_topk_matches_torch_stable_sort():
    rng = np.random.default_rng(4)
    for n, k in ((1000, 37), (5000, 500), (3000, 3000), (3000, 4000)):
        s = np.round(rng.standard_normal(n) * 4) / 4  # ties
        pos = np.arange(100, 100 + n)
        got = oracle.exact_topk(s, pos, k)
        order = torch.sort(torch.from_numpy(s), descending=True, stable=True).indices.numpy()
        want = np.sort(pos[order[:k]])
        np.testing.assert_array_equal(got, want)


def test_topk_threshold_property_and_order():
    rng = np.random.default_rng(5)
    s = rng.standard_normal(4000)
    pos = np.arange(4000)
    sel = oracle.exact_topk(s, pos, 300)
    assert np.all(np.diff(sel) > 0)
    mask = np.zeros(4000, bool)
    mask[sel] = True
    assert s[mask].min() >= s[~mask].max()


def test_planted_key_is_unique_argmax():
    # closed form: q_bar = e_0, one key = c * e_0, every other key orthogonal to e_0
    d, n = 16, 200
    rng = np.random.default_rng(6)
    K = rng.standard_normal((n, d))
    K[:, 0] = 0.0
    K[123] = 0.0
    K[123, 0] = 2.5
    q = np.zeros((4, d))
    q[:, 0] = 1.0
    s = oracle.scores(oracle.group_query(q), K)
    assert s[123] == 2.5 and np.all(np.delete(s, 123) == 0.0)
    assert list(oracle.exact_topk(s, np.arange(n), 1)) == [123]
    # with k = 2 the tie among the zero scores goes to position 0
    assert list(oracle.exact_topk(s, np.arange(n), 2)) == [0, 123]


# ---------------------------------------------------------------- S4 attention, S5 merge


def test_attention_matches_torch_sdpa_fp64():
    rng = np.random.default_rng(7)
    for G, n, d, dv in ((8, 37, 64, 64), (1, 1, 8, 3), (4, 300, 128, 128), (16, 5, 576, 512)):
        q = rng.standard_normal((G, d))
        K = rng.standard_normal((n, d))
        V = rng.standard_normal((n, dv))
        scale = 1.0 / math.sqrt(d)
        o, lse = oracle.attention(q, K, V, scale)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q)[None], torch.from_numpy(K)[None], torch.from_numpy(V)[None], scale=scale)
        np.testing.assert_allclose(o, ref[0].numpy(), rtol=1e-12, atol=1e-12)
        z = scale * torch.from_numpy(q) @ torch.from_numpy(K).T
        np.testing.assert_allclose(lse, torch.logsumexp(z, dim=1).numpy(), rtol=1e-12, atol=1e-12)


def test_attention_closed_forms():
    # two keys, q = e_0, scale 1: weights e/(1+e) and 1/(1+e)
    q = np.array([[1.0, 0.0]])
    K = np.array([[1.0, 0.0], [0.0, 1.0]])
    V = np.array([[1.0, 2.0], [3.0, 4.0]])
    o, lse = oracle.attention(q, K, V, 1.0)
    e = math.e
    np.testing.assert_allclose(o[0], [(e + 3) / (1 + e), (2 * e + 4) / (1 + e)], rtol=1e-15)
    np.testing.assert_allclose(lse[0], math.log(e + 1.0), rtol=1e-15)
    # equal logits: uniform weights, lse = z + log n
    rng = np.random.default_rng(8)
    Vr = rng.standard_normal((10, 4))
    o, lse = oracle.attention(np.zeros((3, 6)), rng.standard_normal((10, 6)), Vr, 0.3)
    np.testing.assert_allclose(o, np.tile(Vr.mean(0), (3, 1)), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, math.log(10.0), rtol=1e-15)
    # constant V rows -> the constant
    c = rng.standard_normal(5)
    o, _ = oracle.attention(rng.standard_normal((2, 7)), rng.standard_normal((9, 7)), np.tile(c, (9, 1)), 1.0)
    np.testing.assert_allclose(o, np.tile(c, (2, 1)), rtol=1e-13)
    # one dominant logit -> that V row
    K = rng.standard_normal((20, 4)) * 0.01
    K[11] = [50.0, 0, 0, 0]
    o, _ = oracle.attention(np.array([[1.0, 0, 0, 0]]), K, Vr.repeat(2, 0), 1.0)
    np.testing.assert_allclose(o[0], Vr.repeat(2, 0)[11], rtol=1e-15, atol=1e-18)
    # empty attended set
    o, lse = oracle.attention(np.ones((2, 3)), np.zeros((0, 3)), np.zeros((0, 5)), 1.0)
    assert np.all(o == 0) and np.all(lse == -np.inf)


def test_lse_merge_equals_one_softmax():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((8, 32))
    K = rng.standard_normal((103, 32)) * 2
    V = rng.standard_normal((103, 24))
    o_ref, lse_ref = oracle.attention(q, K, V, 0.2)
    for n_split in (1, 2, 7, 103, 150):
        bounds = np.linspace(0, 103, n_split + 1).astype(int)
        parts = [oracle.attention_partial(q, K[a:b], V[a:b], 0.2) for a, b in zip(bounds[:-1], bounds[1:])]
        o, lse = oracle.lse_merge(parts)
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, lse_ref, rtol=1e-13)


# ---------------------------------------------------------------- S3 resolution and whole steps


def _prob(wl, **over):
    d = dict(batch=wl.B, n_kv_heads=wl.H, n_q_heads=wl.Hq, d_qk=wl.d_qk, d_v=wl.d_v, topk=wl.k,
             n_sink=wl.ns, n_local=wl.nl, block_size=wl.bs, seq_lens=[int(x) for x in wl.seq_lens],
             sm_scale=wl.sm_scale, index_layout=wl.index_layout)
    d.update(over)
    return oracle.Problem(**d)


def _pools(wl):
    nv = workloads.numpy_view
    table = nv(wl.table)
    kp = oracle.PagedPool(nv(wl.gpu_k), nv(wl.host_k), table, wl.bs)
    vp = None if wl.gpu_v is None else oracle.PagedPool(nv(wl.gpu_v), nv(wl.host_v), table, wl.bs)
    return kp, vp


def test_resolve_hand_example():
    # vToken Eq. (2): slot = block_id * S + offset; negative entries name host blocks
    gpu = np.arange(3 * 1 * 4 * 2, dtype=np.float64).reshape(3, 1, 4, 2)
    host = -np.arange(1 * 1 * 4 * 2, dtype=np.float64).reshape(1, 1, 4, 2) - 100
    pool = oracle.PagedPool(gpu, host, np.array([[2, -1]]), 4)
    assert pool.resolve(0, 2) == ("gpu", 2, 2)
    assert pool.resolve(0, 5) == ("host", 0, 1)
    np.testing.assert_array_equal(pool.row(0, 0, 2), gpu.reshape(-1, 2)[2 * 4 + 2])
    np.testing.assert_array_equal(pool.row(0, 0, 5), host.reshape(-1, 2)[0 * 4 + 1])
    np.testing.assert_array_equal(pool.rows(0, 0, [5, 2]), np.stack([pool.row(0, 0, 5), pool.row(0, 0, 2)]))
    with pytest.raises(IndexError):
        oracle.PagedPool(gpu, host, np.array([[3, -1]]), 4).row(0, 0, 0)
    with pytest.raises(IndexError):
        oracle.PagedPool(gpu, host, np.array([[0, -2]]), 4).row(0, 0, 4)


@pytest.mark.parametrize("name,over", [
    ("tiny", dict(L=200)),
    ("gqa32b", dict(B=2, H=2, Hq=8, L=300)),
])
def test_resolve_recovers_logical_rows(name, over):
    wl = workloads.make_workload(name, keep_logical=True, host_frac=0.3, **over)
    kp, vp = _pools(wl)
    lk = oracle.as_f64(workloads.numpy_view(wl.meta["logical_k"]))
    lv = oracle.as_f64(workloads.numpy_view(wl.meta["logical_v"]))
    for b in range(wl.B):
        for h in range(wl.H):
            pos = np.arange(wl.L)
            np.testing.assert_array_equal(kp.rows(b, h, pos), lk[b, h])
            np.testing.assert_array_equal(vp.rows(b, h, pos), lv[b, h])


def test_head_table_hand_example():
    # one request, two KV heads, 2-token blocks: head 0 keeps block 0 on GPU block 1 and
    # block 1 on the host; head 1 the other way round, on GPU block 0
    gpu = np.arange(2 * 2 * 3, dtype=np.float64).reshape(2, 2, 3)  # [blocks, bs, d]: one head each
    host = 100 + np.arange(2 * 2 * 2 * 3, dtype=np.float64).reshape(2, 2, 2, 3)  # [blocks, H, bs, d]
    table = np.array([[[1, -2], [-1, 0]]])
    pool = oracle.HeadTablePool(gpu, host, table, 2)
    assert pool.resolve(0, 0, 1) == ("gpu", 1, 1)
    assert pool.resolve(0, 0, 2) == ("host", 1, 0)
    assert pool.resolve(0, 1, 0) == ("host", 0, 0)
    assert pool.resolve(0, 1, 3) == ("gpu", 0, 1)
    np.testing.assert_array_equal(pool.row(0, 0, 1), gpu[1, 1])
    np.testing.assert_array_equal(pool.row(0, 0, 3), host[1, 0, 1])  # the host block keeps head 0's rows
    np.testing.assert_array_equal(pool.row(0, 1, 1), host[0, 1, 1])  # ... and head 1's
    np.testing.assert_array_equal(pool.rows(0, 1, [3, 0]), np.stack([gpu[0, 1], host[0, 1, 0]]))
    with pytest.raises(IndexError):
        oracle.HeadTablePool(gpu, host, np.array([[[2, 0], [0, 0]]]), 2).row(0, 0, 0)
    with pytest.raises(IndexError):
        oracle.HeadTablePool(gpu, host, np.array([[[0, 0], [-3, 0]]]), 2).row(0, 1, 0)


@pytest.mark.parametrize("gpu_frac,host_frac", [(1.0, 0.0), (0.5, 0.3), (0.0, 0.0)])
def test_head_table_layout_recovers_logical_rows(gpu_frac, host_frac):
    wl = workloads.make_workload("gqa32b", B=2, H=3, Hq=6, L=70, k=8, keep_logical=True, host_frac=host_frac)
    lay = workloads.head_table_layout(wl, gpu_frac=gpu_frac, seed=3)
    nv = workloads.numpy_view
    tbl = nv(lay["table"])
    assert tbl.shape == (2, 3, 5)
    if gpu_frac == 1.0:
        assert (tbl >= 0).all() and sorted(tbl.reshape(-1).tolist()) == list(range(30))
    if gpu_frac == 0.0:
        assert (tbl < 0).all()
    kp = oracle.HeadTablePool(nv(lay["gpu_k"]), nv(lay["host_k"]), tbl, wl.bs)
    vp = oracle.HeadTablePool(nv(lay["gpu_v"]), nv(lay["host_v"]), tbl, wl.bs)
    lk = oracle.as_f64(nv(wl.meta["logical_k"]))
    lv = oracle.as_f64(nv(wl.meta["logical_v"]))
    for b in range(2):
        for h in range(3):
            np.testing.assert_array_equal(kp.rows(b, h, np.arange(70)), lk[b, h])
            np.testing.assert_array_equal(vp.rows(b, h, np.arange(70)), lv[b, h])


def test_head_table_step_equals_the_shared_table_step():
    # placement does not change results (vToken notes §3.4): the same logical rows
    # through per-head tables give the same step, bit for bit
    wl = workloads.make_workload("gqa32b", B=2, H=2, Hq=8, L=300, k=20, seq_lens=[300, 211], host_frac=0.2)
    lay = workloads.head_table_layout(wl, gpu_frac=0.6, seed=5)
    nv = workloads.numpy_view
    shared = _pools(wl)
    per_head = (oracle.HeadTablePool(nv(lay["gpu_k"]), nv(lay["host_k"]), nv(lay["table"]), wl.bs),
                oracle.HeadTablePool(nv(lay["gpu_v"]), nv(lay["host_v"]), nv(lay["table"]), wl.bs))
    prob = _prob(wl, seq_lens=[300, 211])
    q = workloads.numpy_view(wl.q)
    for b in range(2):
        for h in range(2):
            r0 = oracle.decode_unit(prob, b, h, q, *shared)
            r1 = oracle.decode_unit(prob, b, h, q, *per_head)
            for key in ("scores", "idx", "out", "lse"):
                np.testing.assert_array_equal(r0[key], r1[key])


def test_latent_token_map_recovers_rows():
    wl = workloads.make_workload("mla", B=2, L=96, k=8, keep_logical=True)
    kp, _ = _pools(wl)
    lat = oracle.as_f64(workloads.numpy_view(wl.meta["logical_latent"]))
    tbl = workloads.numpy_view(wl.table)
    assert (tbl >= 0).sum() == 2 * 24  # 25% of each request's tokens are cached on the GPU
    for b in range(2):
        np.testing.assert_array_equal(kp.rows(b, 0, np.arange(96)), lat[b])


def test_dense_reduction_when_k_covers_candidates():
    # k >= |C| with no sink/local: the step is dense attention over all L positions
    wl = workloads.make_workload("gqa32b", B=1, H=2, Hq=8, L=77, k=1000, ns=0, nl=0, keep_logical=True)
    prob = _prob(wl)
    kp, vp = _pools(wl)
    q = workloads.numpy_view(wl.q)
    lk = oracle.as_f64(workloads.numpy_view(wl.meta["logical_k"]))
    lv = oracle.as_f64(workloads.numpy_view(wl.meta["logical_v"]))
    for h in range(2):
        r = oracle.decode_unit(prob, 0, h, q, kp, vp)
        assert list(r["idx"]) == list(range(77))
        qh = torch.from_numpy(oracle.as_f64(q[0, 4 * h:4 * h + 4]))[None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qh, torch.from_numpy(lk[0, h])[None], torch.from_numpy(lv[0, h])[None], scale=wl.sm_scale)
        np.testing.assert_allclose(r["out"], ref[0].numpy(), rtol=1e-12, atol=1e-12)


def test_sink_and_local_always_attended():
    wl = workloads.make_workload("tiny", L=500, k=10, ns=4, nl=64, seq_lens=[333])
    prob = _prob(wl)
    r = oracle.decode_unit(prob, 0, 0, workloads.numpy_view(wl.q), *_pools(wl))
    att = r["attended"]
    assert set(range(4)) <= set(att) and set(range(333 - 64, 333)) <= set(att)
    assert len(att) == 4 + 10 + 64 and np.all(np.diff(att) > 0)
    assert set(r["idx"]) <= set(range(4, 333 - 64))


def test_placement_invariance():
    # Moving blocks between physical slots or tiers changes no result (vToken notes
    # §3.5 I1/I2; ECHO-OSDI26 wiki: placement never changes the exact top-k).
    base = workloads.make_workload("gqa32b", B=2, H=2, Hq=8, L=400, k=40, ns=4, nl=16)
    moved = workloads.permute_blocks(base, seed=77)
    tiered = workloads.make_workload("gqa32b", B=2, H=2, Hq=8, L=400, k=40, ns=4, nl=16, host_frac=0.5)
    assert not np.array_equal(workloads.numpy_view(base.table), workloads.numpy_view(moved.table))
    assert (workloads.numpy_view(tiered.table) < 0).any()
    q = workloads.numpy_view(base.q)
    np.testing.assert_array_equal(q, workloads.numpy_view(tiered.q))
    for b in range(2):
        for h in range(2):
            r0 = oracle.decode_unit(_prob(base), b, h, q, *_pools(base))
            for other in (moved, tiered):
                r1 = oracle.decode_unit(_prob(other), b, h, q, *_pools(other))
                np.testing.assert_array_equal(r0["idx"], r1["idx"])
                np.testing.assert_array_equal(r0["scores"], r1["scores"])
                np.testing.assert_array_equal(r0["out"], r1["out"])
                np.testing.assert_array_equal(r0["lse"], r1["lse"])


def test_contig_index_and_latent_values():
    # indexer scores come from separate index keys; V is the first d_v latent dims
    wl = workloads.make_workload("mla", B=2, L=128, k=16, keep_logical=True)
    prob = _prob(wl)
    kp, _ = _pools(wl)
    q = workloads.numpy_view(wl.q)
    qi = oracle.as_f64(workloads.numpy_view(wl.q_idx))
    ik = oracle.as_f64(workloads.numpy_view(wl.index_keys))
    lat = oracle.as_f64(workloads.numpy_view(wl.meta["logical_latent"]))
    for b in range(2):
        r = oracle.decode_unit(prob, b, 0, q, kp, None, q_index=workloads.numpy_view(wl.q_idx),
                               index_keys=workloads.numpy_view(wl.index_keys))
        np.testing.assert_allclose(r["scores"], ik[b, 0] @ qi[b, 0], rtol=1e-13, atol=1e-12)
        sel = r["idx"]
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(oracle.as_f64(q[b]))[None], torch.from_numpy(lat[b, sel])[None],
            torch.from_numpy(lat[b, sel, :512])[None], scale=1 / math.sqrt(576))
        np.testing.assert_allclose(r["out"], ref[0].numpy(), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- byte models (worked examples)


def test_ulacache_transfer_example():
    g = json.load(open(os.path.join(GOLDEN, "ulacache_transfer_example.json")))
    for case in g["cases"]:
        v = oracle.step_read_bytes(g["k"], g["s_kv_bytes"], case["hit_rate"])
        assert abs(v - case["bytes"]) < 1e-6 * case["bytes"]
        t_ms = 1e3 * oracle.fetch_time_s(v, g["link_bytes_per_s"])
        assert round(t_ms, 2) == case["time_ms_printed"]


def test_echo_metadata_example():
    g = json.load(open(os.path.join(GOLDEN, "echo_metadata_example.json")))
    per_layer = oracle.echo_metadata_bytes(g["n_host_tokens"], g["n_gpu_tokens"])
    assert per_layer == 10_600_000
    assert round(per_layer / 1e6) == 11 and abs(per_layer / 1e6 - g["per_layer_printed_MB"]) < 1.0
    assert abs(g["layers"] * g["per_layer_printed_MB"] - g["all_layers_printed_MB"]) == 0


def test_step_bytes_model_counts_each_stream_once():
    # hand count for a tiny shape: B1 H1 Hq2 d4 L10 k3 ns1 nl2 bs4 (bf16, fp32 scores)
    # candidates 7 -> keys 7*8 B + scores 7*8 B; attended 1+3+2 = 6 rows of K and V (6*16 B);
    # table 3 entries * 4 B; q and out 2*4*2 B each
    got = oracle.decode_step_hbm_bytes(1, 1, 2, 4, 10, 3, 1, 2, block_size=4)
    assert got == 7 * 8 + 7 * 8 + 6 * 16 + 3 * 4 + 16 + 16
    # per query head: keys once, the scores, attended rows and table row for each of the 2 heads
    got = oracle.decode_step_hbm_bytes(1, 1, 2, 4, 10, 3, 1, 2, block_size=4, per_query_head=True)
    assert got == 7 * 8 + 2 * (7 * 8 + 6 * 16 + 3 * 4) + 16 + 16


# ------------------------------------------------------------------ group aggregation (S0 + S1)


def test_group_scores_unit_vector_closed_form():
    # heads along the first G axes: a head's logit is one coordinate of the key, so the
    # max reading is the largest of those coordinates and the mean their average
    rng = np.random.default_rng(5)
    G, d = 5, 16
    q_group = np.eye(d)[:G]
    keys = rng.standard_normal((40, d))
    np.testing.assert_allclose(oracle.group_scores(q_group, keys, "max"), keys[:, :G].max(axis=1), rtol=0, atol=1e-15)
    np.testing.assert_allclose(oracle.group_scores(q_group, keys, "mean"), keys[:, :G].sum(axis=1) / G,
                               rtol=0, atol=1e-15)


def test_group_scores_brute_force_loops():
    rng = np.random.default_rng(6)
    G, d, n = 3, 4, 5
    q_group = rng.standard_normal((G, d))
    keys = rng.standard_normal((n, d))
    want_max, want_mean = [], []
    for t in range(n):
        logits = []
        for g in range(G):
            acc = 0.0
            for j in range(d):
                acc += float(q_group[g, j]) * float(keys[t, j])
            logits.append(acc)
        best = logits[0]
        for x in logits[1:]:
            best = x if x > best else best
        want_max.append(best)
        want_mean.append(sum(logits) / G)
    np.testing.assert_allclose(oracle.group_scores(q_group, keys, "max"), want_max, rtol=1e-13)
    np.testing.assert_allclose(oracle.group_scores(q_group, keys, "mean"), want_mean, rtol=1e-13)


def test_group_scores_one_head_and_head_order():
    rng = np.random.default_rng(7)
    keys = rng.standard_normal((30, 8))
    q1 = rng.standard_normal((1, 8))
    np.testing.assert_array_equal(oracle.group_scores(q1, keys, "max"), oracle.group_scores(q1, keys, "mean"))
    qg = rng.standard_normal((6, 8))
    np.testing.assert_array_equal(oracle.group_scores(qg, keys, "max"), oracle.group_scores(qg[::-1], keys, "max"))
    assert np.all(oracle.group_scores(qg, keys, "max") >= oracle.group_scores(qg, keys, "mean") - 1e-12)
    with pytest.raises(ValueError):
        oracle.group_scores(qg, keys, "median")


def test_max_and_mean_rank_differently():
    # two heads on two axes; key a = (2, -2): mean 0, max 2; key b = (1, 1): mean 1, max 1
    q = np.zeros((1, 2, 2))
    q[0, 0, 0] = 1.0
    q[0, 1, 1] = 1.0
    rows = np.zeros((1, 1, 4, 2))  # one block of 4 tokens: sink, a, b, local
    rows[0, 0, 1] = [2.0, -2.0]
    rows[0, 0, 2] = [1.0, 1.0]
    pool = oracle.PagedPool(rows, None, np.zeros((1, 1), dtype=np.int64), 4)
    picks = {}
    for agg in ("mean", "max"):
        prob = oracle.Problem(batch=1, n_kv_heads=1, n_q_heads=2, d_qk=2, d_v=2, topk=1, n_sink=1, n_local=1,
                              block_size=4, seq_lens=[4], group_agg=agg)
        picks[agg] = oracle.decode_unit(prob, 0, 0, q, pool, pool)["idx"].tolist()
    assert picks == {"mean": [2], "max": [1]}


# ------------------------------------------------------------------ per-query-head selection


def _head_prob(**over):
    d = dict(batch=1, n_kv_heads=1, n_q_heads=2, d_qk=2, d_v=2, topk=1, n_sink=1, n_local=1, block_size=4,
             seq_lens=[4], group_agg="mean")
    d.update(over)
    return oracle.Problem(**d)


def test_head_reading_hand_example():
    # the two-axis example above: head 0 (axis 0) keeps key a = (2, -2), head 1 (axis 1)
    # keeps key b = (1, 1); sink and local rows are zero, so each head attends {0, its key,
    # 3} with logits s * (0, <q_j, key>, 0) and V = K:
    #   o_j = e^{s x} / (2 + e^{s x}) * key,   lse_j = log(2 + e^{s x}),  s = 1 / sqrt(2)
    q = np.zeros((1, 2, 2))
    q[0, 0, 0] = 1.0
    q[0, 1, 1] = 1.0
    rows = np.zeros((1, 1, 4, 2))
    rows[0, 0, 1] = [2.0, -2.0]
    rows[0, 0, 2] = [1.0, 1.0]
    pool = oracle.PagedPool(rows, None, np.zeros((1, 1), dtype=np.int64), 4)
    prob = _head_prob()
    s = 1.0 / math.sqrt(2.0)
    for j, pos, key, x in ((0, 1, np.array([2.0, -2.0]), 2.0), (1, 2, np.array([1.0, 1.0]), 1.0)):
        r = oracle.decode_head(prob, 0, j, q, pool, pool)
        assert r["idx"].tolist() == [pos]
        assert r["attended"].tolist() == [0, pos, 3]
        e = math.exp(s * x)
        np.testing.assert_allclose(r["out"][0], e / (2.0 + e) * key, rtol=1e-15, atol=1e-15)
        np.testing.assert_allclose(r["lse"][0], math.log(2.0 + e), rtol=1e-15)
    # the group's mean reading keeps b for both heads: the readings differ
    assert oracle.decode_unit(prob, 0, 0, q, pool, pool)["idx"].tolist() == [2]


def test_head_reading_planted_keys_follow_the_kv_head():
    # query head j (G = 4) points along axis j; only KV head j // 4 holds a key along axis
    # j, at position 5 + 7 j.  With k = 1 every head must pick its own planted key: a
    # head mapped to the wrong KV head (j % H) or scored with another head's query misses it.
    rng = np.random.default_rng(11)
    H, G, L, d = 2, 4, 64, 16
    rows = rng.standard_normal((L // 16, H, 16, d))
    q = np.zeros((1, H * G, d))
    for j in range(H * G):
        q[0, j, j] = 10.0
        t = 5 + 7 * j
        rows[t // 16, j // G, t % 16] = 0.0
        rows[t // 16, j // G, t % 16, j] = 10.0
    pool = oracle.PagedPool(rows, None, np.arange(L // 16)[None], 16)
    prob = _head_prob(n_kv_heads=H, n_q_heads=H * G, d_qk=d, d_v=d, n_sink=0, n_local=0, block_size=16,
                      seq_lens=[L])
    for j in range(H * G):
        assert oracle.decode_head(prob, 0, j, q, pool, pool)["idx"].tolist() == [5 + 7 * j]


def test_head_reading_with_one_head_per_group_is_the_kv_head_step():
    # G = 1: the mean and the max of one head are the head, so both readings of the
    # KV-head step give the per-head step, idx bit for bit
    wl = workloads.make_workload("gqa32b", B=2, H=4, Hq=4, L=300, k=20, ns=4, nl=16, host_frac=0.3)
    kp, vp = _pools(wl)
    q = workloads.numpy_view(wl.q)
    for agg in ("mean", "max"):
        prob = _prob(wl, group_agg=agg)
        for b in range(2):
            for j in range(4):
                r_head = oracle.decode_head(prob, b, j, q, kp, vp)
                r_unit = oracle.decode_unit(prob, b, j, q, kp, vp)
                np.testing.assert_array_equal(r_head["idx"], r_unit["idx"])
                np.testing.assert_allclose(r_head["scores"], r_unit["scores"], rtol=1e-14, atol=1e-13)
                np.testing.assert_allclose(r_head["out"], r_unit["out"], rtol=1e-14, atol=1e-14)
                np.testing.assert_allclose(r_head["lse"], r_unit["lse"], rtol=1e-14)


def test_head_reading_dense_when_k_covers_candidates():
    # k >= |C|: every head attends all L rows of its KV head j // G -- torch's attention
    wl = workloads.make_workload("gqa32b", B=1, H=2, Hq=8, L=77, k=1000, ns=0, nl=0, keep_logical=True)
    prob = _prob(wl)
    kp, vp = _pools(wl)
    q = workloads.numpy_view(wl.q)
    lk = oracle.as_f64(workloads.numpy_view(wl.meta["logical_k"]))
    lv = oracle.as_f64(workloads.numpy_view(wl.meta["logical_v"]))
    for j in range(8):
        r = oracle.decode_head(prob, 0, j, q, kp, vp)
        assert list(r["idx"]) == list(range(77))
        qh = torch.from_numpy(oracle.as_f64(q[0, j:j + 1]))[None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qh, torch.from_numpy(lk[0, j // 4])[None], torch.from_numpy(lv[0, j // 4])[None], scale=wl.sm_scale)
        np.testing.assert_allclose(r["out"], ref[0].numpy(), rtol=1e-12, atol=1e-12)


def test_head_reading_with_contiguous_index_keys_equal_to_the_pool():
    # index keys that are the K rows themselves and index queries that are the attention
    # queries: the contiguous-index step is the paged one
    wl = workloads.make_workload("gqa32b", B=2, H=2, Hq=8, L=200, k=15, ns=4, nl=16, keep_logical=True,
                                 host_frac=0.3)
    kp, vp = _pools(wl)
    q = workloads.numpy_view(wl.q)
    keys = workloads.numpy_view(wl.meta["logical_k"])  # [B, H, L, d]
    paged = _prob(wl)
    contig = _prob(wl, index_layout="contig")
    for b in range(2):
        for j in range(8):
            r0 = oracle.decode_head(paged, b, j, q, kp, vp)
            r1 = oracle.decode_head(contig, b, j, q, kp, vp, q_index=q, index_keys=keys)
            for key in ("scores", "idx", "out", "lse"):
                np.testing.assert_array_equal(r0[key], r1[key])


def test_head_reading_ignores_the_other_heads_and_matches_a_uniform_group():
    # a head's step depends on its own query only; a group whose G heads all equal q_j
    # has mean q_j, so the group step selects what head j selects
    wl = workloads.make_workload("gqa32b", B=1, H=2, Hq=8, L=400, k=30, ns=4, nl=32, keep_logical=True)
    prob = _prob(wl)
    kp, vp = _pools(wl)
    q = oracle.as_f64(workloads.numpy_view(wl.q))
    rng = np.random.default_rng(5)
    for j in (1, 6):
        base = oracle.decode_head(prob, 0, j, q, kp, vp)
        other = q.copy()
        mask = np.arange(8) != j
        other[0, mask] = rng.standard_normal((7, q.shape[2]))
        moved = oracle.decode_head(prob, 0, j, other, kp, vp)
        np.testing.assert_array_equal(base["idx"], moved["idx"])
        np.testing.assert_array_equal(base["out"], moved["out"])
        uniform = q.copy()
        h = j // 4
        uniform[0, 4 * h:4 * h + 4] = q[0, j]
        grp = oracle.decode_unit(prob, 0, h, uniform, kp, vp)
        np.testing.assert_allclose(grp["scores"], base["scores"], rtol=1e-13, atol=1e-12)
        np.testing.assert_array_equal(grp["idx"], base["idx"])
        np.testing.assert_allclose(grp["out"][j - 4 * h], base["out"][0], rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------ block selection from key summaries


def test_box_bound_equals_best_corner():
    # the max of a linear function over a box is reached at a corner: enumerate all 2^d corners
    rng = np.random.default_rng(21)
    d = 4
    for _ in range(20):
        q = rng.standard_normal(d)
        a, b = rng.standard_normal(d), rng.standard_normal(d)
        lo, hi = np.minimum(a, b), np.maximum(a, b)
        best = -np.inf
        for bits in itertools.product((0, 1), repeat=d):
            corner = [hi[j] if bits[j] else lo[j] for j in range(d)]
            best = max(best, sum(q[j] * corner[j] for j in range(d)))
        assert abs(oracle.box_bound(q, lo, hi) - best) < 1e-12


def test_block_bound_covers_its_keys_and_is_tight_for_one_key():
    rng = np.random.default_rng(22)
    q_group = rng.standard_normal((4, 32))
    for n in (1, 5, 16):
        rows = rng.standard_normal((n, 32))
        lo, hi = oracle.block_summary(rows)
        for agg in ("mean", "max"):
            u = oracle.block_scores(q_group, lo[None], hi[None], agg)[0]
            assert u >= oracle.group_scores(q_group, rows, agg).max() - 1e-12
            if n == 1:
                assert abs(u - oracle.group_scores(q_group, rows, agg)[0]) < 1e-12
        # the bound is convex in q: the mean's bound never exceeds the largest head's
        assert oracle.block_scores(q_group, lo[None], hi[None], "mean")[0] <= \
            oracle.block_scores(q_group, lo[None], hi[None], "max")[0] + 1e-12


def test_block_regions_hand_examples():
    assert oracle.block_regions(32768, 4, 128, 16) == (2048, 1, 2040)
    assert oracle.block_regions(100, 4, 64, 16) == (7, 1, 2)      # local blocks 2..6 hold tokens 36..99
    assert oracle.block_regions(40, 0, 0, 16) == (3, 0, 3)        # no windows: every block a candidate
    assert oracle.block_regions(10, 40, 5, 16) == (1, 1, 1)       # a sink longer than the history
    att = oracle.block_attended_positions(40, 16, 1, 2, 3, [])
    assert att.tolist() == list(range(0, 16)) + list(range(32, 40))


def test_block_mode_with_every_block_is_dense_attention():
    rng = np.random.default_rng(23)
    L, d, G, bs = 77, 16, 3, 16
    nbk = -(-L // bs)
    perm = rng.permutation(nbk)
    kk = np.zeros((nbk, 1, bs, d))
    vv = np.zeros((nbk, 1, bs, d))
    logical_k = rng.standard_normal((L, d))
    logical_v = rng.standard_normal((L, d))
    for t in range(L):
        kk[perm[t // bs], 0, t % bs] = logical_k[t]
        vv[perm[t // bs], 0, t % bs] = logical_v[t]
    table = perm[None, :].astype(np.int64)
    q = rng.standard_normal((1, G, d))
    prob = oracle.Problem(batch=1, n_kv_heads=1, n_q_heads=G, d_qk=d, d_v=d, topk=0, n_sink=4, n_local=8,
                          block_size=bs, seq_lens=[L])
    r = oracle.decode_unit_blocks(prob, 0, 0, q, oracle.PagedPool(kk, None, table, bs),
                                  oracle.PagedPool(vv, None, table, bs), topk_blocks=100)
    assert r["attended"].tolist() == list(range(L))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q[0])[None], torch.from_numpy(logical_k)[None], torch.from_numpy(logical_v)[None],
        scale=1.0 / math.sqrt(d))[0].numpy()
    np.testing.assert_allclose(r["out"], ref, rtol=1e-12, atol=1e-12)


def test_block_selection_takes_the_highest_bounds():
    # four candidate blocks whose bounds are set by one planted key each
    d, bs = 8, 4
    q = np.zeros((1, 1, d))
    q[0, 0, 0] = 1.0
    L = 6 * bs
    rows = np.zeros((6, 1, bs, d))
    for blk, v in zip(range(1, 5), (0.5, 3.0, -1.0, 2.0)):
        rows[blk, 0, 1, 0] = v
    table = np.arange(6)[None, :]
    prob = oracle.Problem(batch=1, n_kv_heads=1, n_q_heads=1, d_qk=d, d_v=d, topk=0, n_sink=bs, n_local=bs,
                          block_size=bs, seq_lens=[L])
    pool = oracle.PagedPool(rows, None, table, bs)
    r = oracle.decode_unit_blocks(prob, 0, 0, q, pool, pool, topk_blocks=2)
    assert r["blocks"].tolist() == [2, 4]
    np.testing.assert_allclose(r["block_scores"], [0.5, 3.0, 0.0, 2.0])  # block 3: its zero keys bound it


# ------------------------------------------------------------------ GPU slot cache (ECHO wiki, core method 2)


def test_cache_update_hand_example():
    # 3 slots; token 0 in slot 2, token 1 in slot 0, slot 1 free; step 5 attends tokens 0, 4, 5, 6
    L = 8
    table = np.array([[2, 0] + [-(t + 1) for t in range(2, 8)]])
    owner = oracle.cache_owner_from_table(table, 3, L)
    assert owner.tolist() == [1, -1, 0]
    prio = np.array([3, -1, 1])
    t2, o2, p2, promo = oracle.cache_update(table, owner, prio, 5, [[0, 4, 5, 6]], L, budget=3)
    # slot 2 is protected (token 0 used it); the free slot and slot 0 (age 2) take tokens 4 and 5
    assert promo == [(0, 0, 4, 1), (1, 0, 5, 2)]
    assert t2[0].tolist() == [2, -2, -3, -4, 0, 1, -7, -8]  # token 1 back on the host; token 6 still there
    assert o2.tolist() == [4, 5, 0] and p2.tolist() == [5, 5, 5]


def _cache_consistent(table, owner, L):
    b, t = np.nonzero(table[:, :L] >= 0)
    assert sorted(table[b, t].tolist()) == sorted(np.nonzero(owner >= 0)[0].tolist())  # one token per slot
    for bb, tt in zip(b, t):
        assert owner[table[bb, tt]] == bb * L + tt
    hb, ht = np.nonzero(table[:, :L] < 0)
    assert np.all(table[hb, ht] == -(hb * L + ht) - 1)  # host entries name the token's own host row


def test_cache_update_invariants_and_lru():
    rng = np.random.default_rng(31)
    B, L, n = 3, 200, 90
    table = np.array([[-(b * L + t) - 1 for t in range(L)] for b in range(B)])
    cached = rng.choice(B * L, 70, replace=False)
    for sl, tok in enumerate(cached):
        table[tok // L, tok % L] = sl
    owner = oracle.cache_owner_from_table(table, n, L)
    prio = np.where(owner >= 0, rng.integers(0, 10, n), -1)
    for step in range(10, 16):
        attended = [np.sort(rng.choice(L, 25, replace=False)) for _ in range(B)]
        before_prio = prio.copy()
        t2, o2, p2, promo = oracle.cache_update(table, owner, prio, step, attended, L, budget=40)
        _cache_consistent(t2, o2, L)
        used = {int(table[b, t]) for b in range(B) for t in attended[b] if table[b, t] >= 0}
        for sl in used:
            assert o2[sl] == owner[sl] and p2[sl] == step  # protected: kept, marked
        taken = {sl for sl, _, _, _ in promo}
        age = {sl: (np.inf if owner[sl] < 0 else step - before_prio[sl]) for sl in range(n)}
        for sl in range(n):  # LRU: no untaken, unprotected slot is older than a taken one
            if sl not in taken and sl not in used and taken:
                assert age[sl] <= min(age[x] for x in taken)
        n_miss = sum(int((table[b, attended[b]] < 0).sum()) for b in range(B))
        assert len(promo) == min(n_miss, 40, n - len(used))
        table, owner, prio = t2, o2, p2


def test_cache_update_heads_hand_example():
    # one request, two KV heads, 4 blocks of 2 tokens, 3 slots: head 0's block 0 in slot 2,
    # head 1's block 1 in slot 0 (age 2 at step 5), slot 1 free
    table = np.array([[[2, -2, -3, -4], [-1, 0, -3, -4]]])
    owner = np.array([(0 * 2 + 1) * 4 + 1, -1, 0])
    prio = np.array([3, -1, 1])
    attended = [[[0, 1, 5], [6, 7]]]  # head 0: blocks 0 (a hit) and 2; head 1: block 3
    t2, o2, p2, promo = oracle.cache_update_heads(table, owner, prio, 5, attended, 2, budget=3)
    # slot 2 is protected; the free slot and slot 0 take (head 0, block 2) and (head 1, block 3)
    # in slot order, and slot 0's old owner (head 1, block 1) returns to host block 1
    assert promo == [(0, 0, 0, 2), (1, 0, 1, 3)]
    assert t2[0, 0].tolist() == [2, -2, 0, -4] and t2[0, 1].tolist() == [-1, -2, -3, 1]
    assert o2.tolist() == [2, 7, 0] and p2.tolist() == [5, 5, 5]


def test_cache_update_heads_with_one_head_and_one_token_blocks_is_the_token_cache():
    rng = np.random.default_rng(41)
    B, L, n = 3, 120, 50
    table = np.array([[-(b * L + t) - 1 for t in range(L)] for b in range(B)])
    cached = rng.choice(B * L, 40, replace=False)
    for sl, tok in enumerate(cached):
        table[tok // L, tok % L] = sl
    owner = oracle.cache_owner_from_table(table, n, L)
    prio = np.where(owner >= 0, rng.integers(0, 10, n), -1)
    th, oh, ph = table[:, None, :], owner.copy(), prio.copy()
    for step in range(10, 16):
        attended = [np.sort(rng.choice(L, 20, replace=False)) for _ in range(B)]
        t2, o2, p2, promo = oracle.cache_update(table, owner, prio, step, attended, L, budget=15)
        th, oh, ph, promo_h = oracle.cache_update_heads(th, oh, ph, step, [[a] for a in attended], 1, budget=15)
        np.testing.assert_array_equal(th[:, 0, :], t2)
        np.testing.assert_array_equal(oh, o2)
        np.testing.assert_array_equal(ph, p2)
        assert [(sl, b, t) for sl, b, _, t in promo_h] == [(sl, b, t) for sl, b, t, _ in promo]
        table, owner, prio = t2, o2, p2


def test_cache_update_heads_invariants():
    rng = np.random.default_rng(43)
    B, H, S, bs, n = 2, 3, 20, 4, 70
    table = np.array([[[-(b * S + j) - 1 for j in range(S)] for _ in range(H)] for b in range(B)])
    owner = np.full(n, -1)
    cached = rng.choice(B * H * S, 45, replace=False)
    for sl, u in enumerate(cached):
        table.reshape(-1)[u] = sl
        owner[sl] = u
    prio = np.where(owner >= 0, rng.integers(0, 10, n), -1)
    for step in range(10, 18):
        attended = [[np.sort(rng.choice(S * bs, 12, replace=False)) for _ in range(H)] for _ in range(B)]
        t2, o2, p2, promo = oracle.cache_update_heads(table, owner, prio, step, attended, bs, budget=25)
        # one (request, head, block) per slot, and every resident entry names its owner's slot
        flat = t2.reshape(-1)
        res = np.nonzero(flat >= 0)[0]
        assert sorted(flat[res].tolist()) == sorted(np.nonzero(o2 >= 0)[0].tolist())
        assert all(o2[flat[u]] == u for u in res)
        host = np.nonzero(flat < 0)[0]  # entries on the host name their own host block
        assert all(-flat[u] - 1 == (u // (H * S)) * S + u % S for u in host)
        used = {int(table[b, h, t // bs]) for b in range(B) for h in range(H) for t in attended[b][h]
                if table[b, h, t // bs] >= 0}
        for sl in used:
            assert o2[sl] == owner[sl] and p2[sl] == step
        misses = {(b, h, t // bs) for b in range(B) for h in range(H) for t in attended[b][h]
                  if table[b, h, t // bs] < 0}
        assert len(promo) == min(len(misses), 25, n - len(used))
        assert {(b, h, j) for _, b, h, j in promo} <= misses
        table, owner, prio = t2, o2, p2


def test_cache_update_reaches_a_fixed_point():
    L, n = 50, 30
    table = np.array([[-(t + 1) for t in range(L)]])
    owner = np.full(n, -1)
    prio = np.full(n, -1)
    attended = [np.arange(5, 25)]
    for step in range(4):
        table, owner, prio, promo = oracle.cache_update(table, owner, prio, step, attended, L, budget=8)
    assert promo == [] and np.all(table[0, 5:25] >= 0)


# --------------------------------------------------------------------------------------
# threshold prediction (ECHO-OSDI26 wiki, core method 3: an EMA, alpha = 0.5, of the
# k-th score predicts the next step's threshold; keys above it are fetched early)
# --------------------------------------------------------------------------------------


def test_prefetch_prediction_hand_worked_three_steps():
    # six candidates, k = 2, alpha = 0.5; rows 1 and 4 live in HBM, the others on the host
    pos = np.arange(6)
    host = np.array([True, False, True, True, False, True])
    # step 0: no prediction yet, nothing qualifies; top-2 = {5: 5.0, 1: 4.0}, so tau = 4.0
    r0 = oracle.prefetch_step(float("nan"), np.array([1.0, 4.0, 3.0, 0.5, 2.0, 5.0]), pos, host, 2)
    assert r0["eligible"].tolist() == [] and r0["kth"] == 4.0 and r0["tau"] == 4.0
    # step 1: above 4.0 on the host only position 0 (4.5); 2 equals it, 1 and 4 are in HBM;
    # top-2 = {4: 7.0, 1: 6.0}: tau = (6 + 4) / 2 = 5.0
    r1 = oracle.prefetch_step(r0["tau"], np.array([4.5, 6.0, 4.0, 1.0, 7.0, 3.0]), pos, host, 2)
    assert r1["eligible"].tolist() == [0] and r1["kth"] == 6.0 and r1["tau"] == 5.0
    # step 2: above 5.0 on the host: 2 (5.5), 3 (6.5), 5 (9.0); 0 equals it; a cap of 2
    # stages two of them; top-2 = {5: 9.0, 3: 6.5}: tau = (6.5 + 5) / 2 = 5.75
    r2 = oracle.prefetch_step(r1["tau"], np.array([5.0, 1.0, 5.5, 6.5, 0.0, 9.0]), pos, host, 2, cap=2)
    assert r2["eligible"].tolist() == [2, 3, 5] and r2["n_staged"] == 2
    assert r2["kth"] == 6.5 and r2["tau"] == 5.75


def test_prefetch_prediction_limits():
    rng = np.random.default_rng(41)
    pos = np.arange(10, 60)
    host = rng.random(50) < 0.5
    s = rng.standard_normal(50)
    kth = np.sort(s)[::-1][6]
    # alpha = 1: the prediction is the last step's k-th score, whatever came before
    assert oracle.prefetch_step(123.0, s, pos, host, 7, alpha=1.0)["tau"] == kth
    # nothing selected (k = 0, or no candidates): the prediction stays
    assert oracle.prefetch_step(0.25, s, pos, host, 0)["tau"] == 0.25
    assert oracle.prefetch_step(0.25, s[:0], pos[:0], host[:0], 5)["tau"] == 0.25
    assert math.isnan(oracle.prefetch_step(float("nan"), s[:0], pos[:0], host[:0], 5)["tau"])
    # k >= |C|: the k-th score is the smallest candidate score
    assert oracle.prefetch_step(float("nan"), s, pos, host, 500)["kth"] == s.min()
    # -0 and +0 compare equal; the threshold reads +0
    z = oracle.prefetch_step(float("nan"), np.array([-0.0, -0.0, -1.0]), np.arange(3), np.ones(3, bool), 2)
    assert z["kth"] == 0.0 and math.copysign(1.0, z["kth"]) == 1.0
    # a prediction below every score: every host row qualifies; HBM rows never do
    r = oracle.prefetch_step(-np.inf, s, pos, host, 7, cap=5)
    assert r["eligible"].tolist() == pos[host].tolist() and r["n_staged"] == min(5, int(host.sum()))
