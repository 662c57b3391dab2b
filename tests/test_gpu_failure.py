"""The bounded waits of the pipelined kernels: a wait that nothing completes gives up,
reports SKV_DEV_TIMEOUT in the status word and leaves the context usable -- no trap and
no hang (the failure is made by withholding an arrival, not by a fault)."""

import time

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def skv():
    import __graft_entry__

    __graft_entry__.build()
    import top_sparse_kv_gb300 as m

    return m


LIMIT = 2_000_000  # SM clocks: about a millisecond


def test_a_wait_that_nothing_completes_reports_a_timeout(skv):
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    skv.skv_check_wait_timeout(LIMIT, 0, status)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 5.0
    assert int(status.item()) == skv.SKV_DEV_TIMEOUT


def test_a_completed_wait_reports_nothing(skv):
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    skv.skv_check_wait_timeout(LIMIT, 1, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_the_context_stays_usable_after_a_timeout(skv):
    wl = workloads.make_workload("tiny", device="cuda", gen_device="cpu")
    step = skv.DecodeStep.from_workload(wl)
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    before = (step.idx.clone(), step.out.clone(), step.lse.clone())
    skv.skv_check_wait_timeout(LIMIT, 0, step.status)
    torch.cuda.synchronize()
    assert int(step.status.item()) == skv.SKV_DEV_TIMEOUT
    step.status.zero_()
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    assert torch.equal(step.idx, before[0]) and torch.equal(step.out, before[1]) and torch.equal(step.lse, before[2])
