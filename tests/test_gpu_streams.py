"""The library keeps no per-call state on the device: steps enqueued on two streams at
once, and steps replayed from a CUDA graph, give the results of eager steps run one at a
time, bit for bit."""

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


def _outputs(step):
    return step.idx.clone(), step.out.clone(), step.lse.clone()


def _steps(skv):
    a = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=3, H=2, Hq=16, L=5000, k=300,
                                seq_lens=[5000, 4100, 777])
    b = workloads.make_workload("mla", device="cuda", gen_device="cpu", B=2, L=6000, k=512, seq_lens=[6000, 3500])
    c = workloads.make_workload("host1m", device="cuda", gen_device="cpu", H=2, Hq=8, L=70000, k=100)
    return [skv.DecodeStep.from_workload(w) for w in (a, b, c)]


def test_concurrent_streams_match_one_at_a_time(skv):
    steps = _steps(skv)
    want = []
    for s in steps:
        s.run()
        torch.cuda.synchronize()
        assert int(s.status.item()) == 0
        want.append(_outputs(s))
        s.idx.fill_(-7)
        s.out.zero_()
        s.lse.zero_()
    streams = [torch.cuda.Stream() for _ in steps]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    for _ in range(4):  # interleaved enqueues: the three steps' kernels overlap on the GPU
        for s, st in zip(steps, streams):
            s.run(stream=st)
    torch.cuda.synchronize()
    for s, w in zip(steps, want):
        assert int(s.status.item()) == 0
        for got, ref in zip(_outputs(s), w):
            assert torch.equal(got, ref)


def test_graph_replay_matches_eager_steps(skv):
    for s in _steps(skv):
        s.run()
        torch.cuda.synchronize()
        want = _outputs(s)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            s.run()
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            s.run()
        s.idx.fill_(-7)
        s.out.zero_()
        s.lse.zero_()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        assert int(s.status.item()) == 0
        for got, ref in zip(_outputs(s), want):
            assert torch.equal(got, ref)
