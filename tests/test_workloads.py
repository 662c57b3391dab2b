"""The seeded generator: determinism, shapes and the recipe's structure."""

import numpy as np
import pytest
import torch

import workloads


def test_deterministic_per_seed():
    a = workloads.make_workload("gqa32b", B=2, H=2, Hq=8, L=256, k=20)
    b = workloads.make_workload("gqa32b", B=2, H=2, Hq=8, L=256, k=20)
    c = workloads.make_workload("gqa32b", B=2, H=2, Hq=8, L=256, k=20, seed=5)
    for name in ("q", "table", "gpu_k", "gpu_v"):
        assert torch.equal(getattr(a, name), getattr(b, name))
    assert not torch.equal(a.gpu_k, c.gpu_k)


def test_shapes_and_permutation():
    wl = workloads.make_workload("gqa32b", B=3, H=2, Hq=16, L=100, k=10)
    nblk = 7
    assert wl.table.shape == (3, nblk) and wl.table.dtype == torch.int32
    assert wl.gpu_k.shape == (3 * nblk, 2, 16, 128) and wl.gpu_k.dtype == torch.bfloat16
    assert sorted(wl.table.view(-1).tolist()) == list(range(3 * nblk))
    assert wl.table.view(-1).tolist() != list(range(3 * nblk))  # permuted


def test_heavy_keys_align_with_group_query():
    wl = workloads.make_workload("tiny", L=4096, keep_logical=True)
    keys = wl.meta["logical_k"].float()[0, 0]
    qbar = wl.q.float()[0].mean(0)
    s = keys @ (qbar / qbar.norm())
    top = s.topk(41).values
    assert top.min() > 2.0 and s.median().abs() < 0.2  # 41 planted keys stand out by ~3


def test_host_paged_layout():
    wl = workloads.make_workload("host1m", L=4096, k=10, ns=16, nl=64)
    t = wl.table[0]
    assert (t[:1] >= 0).all() and (t[-4:] >= 0).all() and (t[1:-4] < 0).all()
    assert wl.host_k.shape[0] == 256 and wl.gpu_k.shape[0] == 5
    assert wl.index_keys.shape == (1, 8, 4096, 128)


def test_latent_layout():
    wl = workloads.make_workload("mla", B=2, L=64, k=8)
    assert wl.gpu_v is None and wl.host_k.shape == (128, 1, 1, 576)
    assert wl.gpu_k.shape == (32, 1, 1, 576) and wl.q.shape == (2, 128, 576)
    assert wl.q_idx.shape == (2, 1, 128) and wl.index_keys.shape == (2, 1, 64, 128)
    slots = wl.table[wl.table >= 0]
    assert sorted(slots.tolist()) == list(range(32))


def test_sweep_points():
    assert len(workloads.SWEEP_POINTS) == 36
    assert workloads.seed_for("sweep", 3) == 2003 and workloads.seed_for("gqa32b") == 1001


@pytest.mark.parametrize("host_frac", [0.0, 0.4])
def test_unit_view_equals_the_whole_workload_view(host_frac):
    """The one-unit oracle view used for full-size workloads gives the whole view's results."""
    from skv_test_utils import OracleView, UnitView

    wl = workloads.make_workload("sweep", device="cpu", gen_device="cpu", B=3, L=3000, k=200,
                                 seq_lens=[3000, 2017, 140], host_frac=host_frac)
    whole = OracleView(wl)
    for b, h in ((0, 0), (1, 5), (2, 7)):
        a, u = whole.unit(b, h), UnitView(wl, b, h).unit()
        for key in ("idx", "out", "lse"):
            np.testing.assert_array_equal(a[key], u[key])


def test_head_table_layout_is_seeded_and_backs_every_block():
    wl = workloads.make_workload("gqa32b", B=2, H=2, Hq=4, L=100, k=8, host_frac=0.25)
    a = workloads.head_table_layout(wl, gpu_frac=0.5, seed=9)
    b = workloads.head_table_layout(wl, gpu_frac=0.5, seed=9)
    c = workloads.head_table_layout(wl, gpu_frac=0.5, seed=10)
    for key in ("gpu_k", "gpu_v", "host_k", "host_v", "table"):
        assert torch.equal(a[key], b[key])
    assert not torch.equal(a["table"], c["table"])
    stride = wl.table.shape[1]
    assert tuple(a["table"].shape) == (2, 2, stride)
    assert tuple(a["host_k"].shape) == (2 * stride, 2, wl.bs, wl.d_qk)  # every block backed, every head
    t = a["table"].reshape(-1).long()
    res = t[t >= 0]
    assert sorted(res.tolist()) == list(range(a["gpu_k"].shape[0]))  # one block a slot, all slots used
    bj = torch.arange(2).view(2, 1, 1) * stride + torch.arange(stride).view(1, 1, stride)
    host_entry = (-bj - 1).expand(2, 2, stride).reshape(-1)
    assert torch.equal(t[t < 0], host_entry[t < 0])  # a host entry names its own block
    with pytest.raises(ValueError):
        workloads.head_table_layout(workloads.make_workload("mla", B=1, L=64, k=4))
