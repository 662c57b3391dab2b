"""Child process of test_gpu_capture.py: the library's very first calls in this process
are made inside a CUDA graph capture (so the per-context kernel preparation, including the
attention's cluster-occupancy query, happens while a stream is capturing); the replayed
graph must give the eager call's results.  Prints OK."""

import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import top_sparse_kv_gb300 as skv  # noqa: E402
import workloads  # noqa: E402


def capture_first(run, outputs, status):
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        run()
    g.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, int(status.item())
    got = [t.clone() for t in outputs()]
    run()  # the same call, eager
    torch.cuda.synchronize()
    assert int(status.item()) == 0, int(status.item())
    for a, b in zip(got, outputs()):
        assert torch.equal(a, b)


def main():
    # a decode step whose attention merges its splits in a cluster, then a block step
    wl = workloads.make_workload("gqa32b", device="cuda", gen_device="cpu", B=2, H=2, Hq=16, L=3000, k=300,
                                 seq_lens=[3000, 2100])
    step = skv.DecodeStep.from_workload(wl)
    capture_first(step.run, lambda: (step.idx, step.out, step.lse), step.status)
    blk = skv.BlockStep.from_workload(wl, 20)
    blk.summarize()
    torch.cuda.synchronize()
    capture_first(blk.run, lambda: (blk.block_idx, blk.att_idx, blk.out, blk.lse), blk.status)
    print("OK")


if __name__ == "__main__":
    main()
