"""Benchmark of one sparse-decode step (score -> exact top-k -> slot-table gather ->
split-K attention) on the 32B-class GQA workload, printed as one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload (seeded, synthetic): batch 8, 8 KV heads x 64 query heads, head dim 128,
history 32768, top-k 3277 + 4 sink + 128 local, bf16 K/V in a paged GPU pool of
16-token blocks with a random physical block permutation, 1% planted heavy keys.

One step = one skv_decode_step over all (request, KV head) units, replayed from a
CUDA graph.  The K/V pool (1.07 GB) is larger than L2, so every step streams its
keys and rows from HBM.  With N GPUs (torchrun) every rank runs its own copy of
the workload (weak scaling, no collective on the data path); the time is the
max over ranks.

--impl reference times the fp64 CPU oracle on the host cores: each step is a
bounded sample of the same workload's (request, KV head) units, processed by a
pool of worker processes, scaled to whole steps.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse decode steps/s (all heads, 1 GB300) and achieved % of HBM/PCIe roofline"
UNIT = "steps/s"
WORKLOAD = "gqa32b"
WORKLOAD_DESC = ("32B-class GQA decode: batch 8, 8 KV x 64 q heads, d128, L32768, top-k 3277 + 4 sink + 128 local, "
                 "bf16 paged GPU pool (16-token blocks, random permutation), 1% heavy keys")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle subprocess (profiling runs)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads' entries on the headline line (profiling runs)")
    ap.add_argument("--sample-units", type=int, default=0, help="reference arm: units per step (0 = one per core)")
    ap.add_argument("--json-only", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="extra line for another workload (tiny, host1m, mla); the default is the headline")
    ap.add_argument("--hostlink", action="store_true", help="host-link ceiling through skv_gather")
    ap.add_argument("--sweep", action="store_true", help="one line per sweep point (batch x history x k)")
    ap.add_argument("--blocks", type=int, default=0,
                    help="block-selection line: choose this many 16-token blocks from per-block key summaries")
    ap.add_argument("--prefetch", type=int, default=0,
                    help="host1m or mla workload: threshold prefetch of host rows with this many staging rows per unit")
    ap.add_argument("--paris", action="store_true",
                    help="ParisKV retrieval in place of exact scoring and top-k (host1m unless --workload)")
    ap.add_argument("--paris-beta", type=int, default=50, help="ParisKV candidates, per mille")
    ap.add_argument("--paris-rho", type=int, default=100, help="ParisKV collision fraction, per mille")
    ap.add_argument("--cache", type=int, default=0,
                    help="manage the GPU slot pool as a cache, promoting up to this many entries a step: the latent "
                         "workload's rows, or with --workload host1m one-head blocks of a per-head table layout")
    ap.add_argument("--agg", choices=("mean", "max", "head"), default="mean",
                    help="how a group's scoring heads combine: mean (the headline), max over the heads, or "
                         "head (every query head selects its own top-k)")
    return ap.parse_args()


# ------------------------------------------------------------------------------------ distributed


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


def rank_seed(rank: int) -> int:
    """Each rank draws its own copy of the workload (weak scaling)."""
    import workloads

    return workloads.seed_for(WORKLOAD) + 100 * rank


def reduce_max(value: float, world: int) -> float:
    """Max of a float over all ranks (the slowest rank sets the time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def job_rate(steps_per_rank: int, seconds: float, world: int):
    """Whole-job rate: every rank runs `steps_per_rank` steps on its own replica; the
    job takes as long as its slowest rank.  Returns (slowest seconds, steps/s over all ranks)."""
    slowest = reduce_max(seconds, world)
    return slowest, world * steps_per_rank / slowest


def sum_over_ranks(count: int, world: int) -> int:
    """Sum of an integer over all ranks."""
    if world <= 1:
        return count
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([count], dtype=torch.int64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return int(t.item())


# ------------------------------------------------------------------------------------ byte counts
# The benchmark's own bookkeeping for the roofline: region sizes and algorithmic bytes,
# written out here so that the timed arm uses nothing from the oracle.


def regions(L: int, n_sink: int, n_local: int) -> tuple[int, int]:
    """(s_end, l_start): sink [0, s_end), candidates [s_end, l_start), local [l_start, L)."""
    s_end = min(n_sink, L)
    return s_end, max(s_end, L - n_local)


def block_regions(L: int, n_sink: int, n_local: int, bs: int) -> tuple[int, int, int]:
    """(nb, s_blk, l_blk): blocks [s_blk, l_blk) of the nb blocks over [0, L) are candidates."""
    nb = -(-L // bs)
    s_blk = min(-(-n_sink // bs), nb)
    l_blk = nb if n_local <= 0 else max(s_blk, max(L - n_local, 0) // bs)
    return nb, s_blk, l_blk


def decode_step_hbm_bytes(B, H, Hq, d, L, k, ns, nl, elem=2, score_bytes=4, table_entry=4, block_size=16,
                          per_query_head=False):
    """Algorithmic HBM bytes of one paged decode step: candidate keys read once (per KV
    head), scores written and read once, the attended K and V rows read once, the
    slot-table row once per selection row, queries read and outputs written.  The
    selection rows are the KV heads, or every query head when each selects its own."""
    s_end, l_start = regions(L, ns, nl)
    n_c = l_start - s_end
    n_att = s_end + min(k, n_c) + (L - l_start)
    rows = Hq if per_query_head else H
    per_row = n_c * 2 * score_bytes + n_att * 2 * d * elem + (-(-L // block_size)) * table_entry
    return B * H * n_c * d * elem + B * rows * per_row + 2 * B * Hq * d * elem


# ------------------------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons around a region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # the raw samples (the JSON line carries their summary); SKV_CLOCKS_DIR keeps them elsewhere
        out_dir = os.environ.get("SKV_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"skv_clocks_rank{index}.csv")
        self.t0 = self.t1 = None

    def start(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
            self.started = time.time()
        except (OSError, FileNotFoundError):
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), active=parts[4], hw=parts[5],
                                 hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return None
        # samples are 200 ms apart; keep those inside the timed region (by count from the start)
        n_before = int(max(0.0, (self.t0 - self.started)) / 0.2)
        n_in = max(1, int(round((self.t1 - self.t0) / 0.2)) + 1)
        inside = rows[n_before:n_before + n_in] or rows[-1:]
        reasons = set()
        for r in inside:
            if r["hw"] == "Active":
                reasons.add("hw_slowdown")
            if r["hwt"] == "Active":
                reasons.add("hw_thermal_slowdown")
            if r["swt"] == "Active":
                reasons.add("sw_thermal_slowdown")
            if r["pcap"] == "Active":
                reasons.add("sw_power_cap")
        return {"sm_mhz": statistics.median(r["sm"] for r in inside), "sm_max_mhz": max(r["smax"] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside)}


# ------------------------------------------------------------------------------------ our arm


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except OSError:
        return None


def stored_traffic(kernel: str):
    """dram bytes per launch from the committed ncu summary, if taken on the current source."""
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))[kernel]
    except (OSError, KeyError, ValueError):
        return None
    src = os.path.join(ROOT, "top_sparse_kv_gb300", "csrc", rec["source"])
    try:
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    return rec["dram_bytes_per_launch"] if h == rec["source_sha256"] else None


def agg_code(skv, name):
    """The library's SKV_AGG_* code of a --agg name."""
    return {"mean": skv.SKV_AGG_MEAN, "max": skv.SKV_AGG_MAX, "head": skv.SKV_AGG_HEAD}[name]


def headline_config(wl, agg, world):
    """The headline workload's config, the same dict in both arms."""
    return {"workload": WORKLOAD_DESC, "batch": wl.B, "kv_heads": wl.H, "q_heads": wl.Hq, "head_dim": 128,
            "history": wl.L, "topk": wl.k, "sink": wl.ns, "local": wl.nl, "block_size": wl.bs, "group_agg": agg,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    import __graft_entry__

    __graft_entry__.build()
    import top_sparse_kv_gb300 as skv
    import workloads

    wl = workloads.make_workload(WORKLOAD, device="cuda", gen_device="cuda", seed=rank_seed(rank))
    step = skv.DecodeStep.from_workload(wl, group_agg=agg_code(skv, args.agg))
    stream = torch.cuda.current_stream()

    # one direct call: counts the kernels of a step and checks the device status
    n0 = skv.skv_launch_count()
    step.run()
    torch.cuda.synchronize()
    kernels_per_step = skv.skv_launch_count() - n0
    if int(step.status.item()) != 0:
        raise RuntimeError(f"device status {int(step.status.item())}")

    # capture the step as a graph (one replay = one whole decode step)
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for _ in range(2):
            step.run()
    stream.wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step.run()
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.5)
    clocks.mark("t0")
    # K replays per repeat; repeats until the region lasts >= 0.5 s; the median repeat counts
    reps = timed_repeats(graph.replay, args.steps, stream, world)
    clocks.mark("t1")
    clock_rec = clocks.stop()
    ms = statistics.median(reps) * args.steps
    s_max, value = job_rate(args.steps, ms / 1e3, world)
    ms_max = s_max * 1e3

    dist_stats = step_distribution(graph.replay, min(args.steps, 500), stream)
    read_gbs, read_detail = read_stream_gbs(stream)

    # dominant kernel (scoring) timed alone, and the other phases for the breakdown:
    # each from a CUDA graph of 20 calls, CUDA events on the launch stream
    score_ms = graph_call_ms(step.score, stream)
    phase = {"topk": graph_call_ms(step.topk, stream),
             "attention": graph_call_ms(step.attend, stream, cold_l2=True)}

    lens = [int(x) for x in wl.seq_lens.cpu()]
    s_end, l_start = regions(lens[0], wl.ns, wl.nl)
    n_c = l_start - s_end
    units = wl.B * wl.H
    sel_rows = wl.B * (wl.Hq if args.agg == "head" else wl.H)  # score rows written
    score_bytes = units * n_c * wl.d_qk * 2 + sel_rows * n_c * 4  # keys read once + fp32 scores written
    step_bytes = decode_step_hbm_bytes(wl.B, wl.H, wl.Hq, wl.d_qk, lens[0], wl.k, wl.ns, wl.nl,
                                       per_query_head=args.agg == "head")
    pk = peaks()
    hbm_peak = pk["hbm_gbs"] if pk else 6800.0
    achieved = score_bytes / (score_ms * 1e-3) / 1e9
    sga_bytes = step_bytes - sel_rows * n_c * 4  # everything but the top-k's read of the scores
    traffic = stored_traffic("score_kernel")

    # end to end through the public call with host buffers
    # the serving loop runs long enough that filling and draining its two-deep pipeline is noise
    e2e = run_e2e(step, wl, max(args.steps, 1000), world)
    # every repeat of the timed region replays K steps: all of them count
    launches = sum_over_ranks(kernels_per_step * args.steps * len(reps), world)

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": headline_config(wl, args.agg, world),
        "l2": "inputs larger than L2 (1.07 GB K/V pool streamed per step)",
        "timing": {"how": "CUDA graph replay of skv_decode_step, CUDA events on the launch stream; K replays "
                          "per repeat, repeated until the repeats last >= 0.5 s; the median repeat is reported",
                   "repeats": len(reps), "timed_steps_total": args.steps * len(reps),
                   "repeat_ms_per_step": {"min": round(min(reps), 6),
                                                                 "median": round(statistics.median(reps), 6),
                                                                 "max": round(max(reps), 6)}},
        "roofline": {"bound": "hbm", "kernel": "score_kernel (S0+S1)", "achieved": round(achieved, 1),
                     "peak": hbm_peak, "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                     "traffic": traffic, "bytes_per_launch": score_bytes, "ms_per_launch": round(score_ms, 5),
                     "peak_source": "measured" if pk else "fallback",
                     "read_stream_gbs": read_gbs, "read_stream_detail": read_detail,
                     "frac_of_read_stream": round(achieved / read_gbs, 4)},
        "step_times": dist_stats,
        "score_gather_attention": {
            "bytes_per_step": sga_bytes, "ms": round(score_ms + phase["attention"], 5),
            "achieved_gbs": round(sga_bytes / ((score_ms + phase["attention"]) * 1e-3) / 1e9, 1),
            "frac": round(sga_bytes / ((score_ms + phase["attention"]) * 1e-3) / 1e9 / hbm_peak, 4),
            "what": "the step's bytes without the top-k's read of the scores, over the scoring and the "
                    "gather + attention kernel times (attention timed after an L2-evicting write, as in a step)"},
        "step_roofline": {"bytes_per_step": step_bytes,
                          "achieved_gbs": round(step_bytes / (ms_max / args.steps * 1e-3) / 1e9, 1),
                          "frac": round(step_bytes / (ms_max / args.steps * 1e-3) / 1e9 / hbm_peak, 4),
                          "phase_ms": {"score": round(score_ms, 5), **{k: round(v, 5) for k, v in phase.items()}}},
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clock_rec,
    }
    if world == 1 and not args.no_configs and args.agg == "mean":
        del step, graph, wl
        torch.cuda.empty_cache()
        line["configs"] = run_configs(args, stream, hbm_peak)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_subprocess(args.agg)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(step, wl, n, world=1):
    """Steps/s through skv_decode_step with the step's inputs in pinned host memory:
    every step copies q, the slot table and seq_lens host->device, runs the step and
    reads the attention output back device->host.  Two steps are in flight, as in a
    serving loop: the host enqueues step i+1 before it waits for step i's output (two
    pinned output buffers; the device orders every copy after the previous step's
    kernels on the one stream).  With several ranks the region is bracketed by barriers
    and the rate is over all ranks, timed by the slowest.  Also reported: the same loop
    waiting for every step's output before enqueueing the next."""
    import torch

    h_q = wl.q.cpu().pin_memory()
    h_table = wl.table.cpu().pin_memory()
    h_lens = wl.seq_lens.cpu().pin_memory()
    h_out = [torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory() for _ in range(2)]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    stream = torch.cuda.current_stream()

    def enqueue(i):
        step.q.copy_(h_q, non_blocking=True)
        step.pool.slot_table.copy_(h_table, non_blocking=True)
        step.p.seq_lens.copy_(h_lens, non_blocking=True)
        step.run()
        h_out[i % 2].copy_(step.out, non_blocking=True)
        done[i % 2].record(stream)

    checksum = 0.0

    def loop(in_flight, enq):
        nonlocal checksum
        barrier(world)
        t0 = time.perf_counter()
        for i in range(n):
            enq(i)
            j = i - (in_flight - 1)
            if j >= 0:
                done[j % 2].synchronize()
                checksum += float(h_out[j % 2].view(-1)[0])  # the host reads the step's output
        for j in range(max(0, n - (in_flight - 1)), n):
            done[j % 2].synchronize()
            checksum += float(h_out[j % 2].view(-1)[0])
        dt = time.perf_counter() - t0
        barrier(world)
        return dt

    for i in range(3):
        enqueue(i)
    stream.synchronize()
    dt_eager = loop(2, enqueue)
    dt_sync = loop(1, enqueue)
    # the same step captured once per output buffer: (H2D copies, skv_decode_step, D2H copy)
    graphs = []
    for i in range(2):
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            enqueue(i)
        stream.wait_stream(side)
        with torch.cuda.graph(g):
            step.q.copy_(h_q, non_blocking=True)
            step.pool.slot_table.copy_(h_table, non_blocking=True)
            step.p.seq_lens.copy_(h_lens, non_blocking=True)
            step.run()
            h_out[i].copy_(step.out, non_blocking=True)
        graphs.append(g)
    torch.cuda.synchronize()

    def enqueue_graph(i):
        graphs[i % 2].replay()
        done[i % 2].record(stream)

    dt_graph = loop(2, enqueue_graph)
    del graphs
    dt = run_e2e_overlapped(wl, n, world, h_q, h_table, h_lens, step.p.group_agg)
    _, rate = job_rate(n, dt, world)
    _, rate_graph = job_rate(n, dt_graph, world)
    _, rate_eager = job_rate(n, dt_eager, world)
    _, rate_sync = job_rate(n, dt_sync, world)
    h2d = h_q.numel() * h_q.element_size() + h_table.numel() * 4 + h_lens.numel() * 4
    d2h = h_out[0].numel() * h_out[0].element_size()
    return {"value": round(rate, 3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": n, "timing": "wall clock; every step copies its inputs from pinned memory and reads its "
                                  "output back, on a copy stream that overlaps the previous step's kernels "
                                  "(two device buffer sets, each set's step replayed from a CUDA graph); the "
                                  "host reads every step's output",
            "one_stream_graph_two_in_flight": round(rate_graph, 3),
            "one_stream_eager_two_in_flight": round(rate_eager, 3), "one_stream_eager_one_in_flight": round(rate_sync, 3)}


def run_e2e_overlapped(wl, n, world, h_q, h_table, h_lens, group_agg=0):
    """Wall-clock seconds for n steps of a serving loop whose copies overlap compute:
    two device buffer sets (query, slot table, lengths, outputs, workspace) over the
    one K/V pool, each set's skv_decode_step captured in a CUDA graph; a copy stream
    brings step i's inputs in while step i-1 computes and takes step i-1's output out
    while step i computes; events keep a buffer set from being refilled before the step
    that used it is done."""
    import copy

    import torch

    import top_sparse_kv_gb300 as skv

    steps = []
    for _ in range(2):
        w = copy.copy(wl)
        w.q, w.table, w.seq_lens = wl.q.clone(), wl.table.clone(), wl.seq_lens.clone()
        steps.append(skv.DecodeStep.from_workload(w, group_agg=group_agg))
    h_out = [torch.empty(steps[0].out.shape, dtype=steps[0].out.dtype).pin_memory() for _ in range(2)]
    comp, cs = torch.cuda.current_stream(), torch.cuda.Stream()
    # each buffer set's skv_decode_step captured once: a replay is one call's kernels
    graphs = []
    for st in steps:
        side = torch.cuda.Stream()
        side.wait_stream(comp)
        with torch.cuda.stream(side):
            st.run()
        comp.wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            st.run()
        graphs.append(g)
    torch.cuda.synchronize()
    in_ready = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_ready = [torch.cuda.Event() for _ in range(2)]
    sink = 0.0

    def step_in(i):
        x, st = i % 2, steps[i % 2]
        with torch.cuda.stream(cs):
            cs.wait_event(comp_done[x])  # the step that last used this buffer set is done
            st.q.copy_(h_q, non_blocking=True)
            st.pool.slot_table.copy_(h_table, non_blocking=True)
            st.p.seq_lens.copy_(h_lens, non_blocking=True)
            in_ready[x].record(cs)
        comp.wait_event(in_ready[x])
        with torch.cuda.stream(comp):
            graphs[x].replay()
        comp_done[x].record(comp)

    def step_out(i):
        x = i % 2
        with torch.cuda.stream(cs):
            cs.wait_event(comp_done[x])
            h_out[x].copy_(steps[x].out, non_blocking=True)
            out_ready[x].record(cs)

    def read(i):
        nonlocal sink
        out_ready[i % 2].synchronize()
        sink += float(h_out[i % 2].view(-1)[0])  # the host reads the step's output

    for i in range(4):  # warm-up
        step_in(i)
        step_out(i)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for i in range(n):
        step_in(i)           # step i's inputs (overlapping step i-1's kernels), then its kernels
        if i >= 1:
            step_out(i - 1)  # step i-1's output (overlapping step i's kernels)
        if i >= 2:
            read(i - 2)
    step_out(n - 1)
    for j in range(max(0, n - 2), n):
        read(j)
    dt = time.perf_counter() - t0
    barrier(world)
    for st in steps:
        assert int(st.status.item()) == 0
    return dt


def cpu_baseline_subprocess(agg="mean"):
    cmd = [sys.executable, os.path.abspath(__file__), "--impl", "reference", "--steps", "3", "--warmup", "1",
           "--json-only", "--agg", agg]
    env = dict(os.environ)
    env["CUDA_VISIBLE_DEVICES"] = ""
    try:
        r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env)
        line = json.loads(r.stdout.strip().splitlines()[-1])
        return line["cpu_baseline"]
    except Exception as e:  # noqa: BLE001  (reported, never fatal)
        return {"value": None, "unit": UNIT, "error": str(e)[:200]}


# ------------------------------------------------------------------------------------ reference arm

_REF = {}


def _ref_unit(bh):
    import oracle

    v = _REF["view"]
    b, h = bh
    if v["per_head"]:  # h is a query head
        return float(oracle.decode_head(v["prob"], b, h, v["q"], v["kpool"], v["vpool"])["out"][0, 0])
    r = oracle.decode_unit(v["prob"], b, h, v["q"], v["kpool"], v["vpool"])
    return float(r["out"][0, 0])


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return  # the reference arm runs on rank 0 only
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"  # one thread per worker process
    import multiprocessing as mp

    import numpy as np  # noqa: F401
    import oracle
    import workloads

    t_gen = time.perf_counter()
    wl = workloads.make_workload(WORKLOAD, device="cpu", gen_device="cpu", seed=rank_seed(0))
    nv = workloads.numpy_view
    table = nv(wl.table)
    _REF["view"] = dict(
        prob=oracle.Problem(batch=wl.B, n_kv_heads=wl.H, n_q_heads=wl.Hq, d_qk=wl.d_qk, d_v=wl.d_v, topk=wl.k,
                            n_sink=wl.ns, n_local=wl.nl, block_size=wl.bs, seq_lens=[wl.L] * wl.B,
                            sm_scale=wl.sm_scale, group_agg="mean" if args.agg == "head" else args.agg),
        per_head=args.agg == "head",
        q=nv(wl.q), kpool=oracle.PagedPool(nv(wl.gpu_k), None, table, wl.bs),
        vpool=oracle.PagedPool(nv(wl.gpu_v), None, table, wl.bs))
    t_gen = time.perf_counter() - t_gen
    cores = os.cpu_count() or 1
    units = [(b, h) for b in range(wl.B) for h in range(wl.Hq if args.agg == "head" else wl.H)]
    unit_name = "(request, query head)" if args.agg == "head" else "(request, KV head)"
    per_step = args.sample_units or cores
    per_step = max(1, min(per_step, len(units)))
    ctx = mp.get_context("fork")  # this process never touches CUDA
    times = []
    budget_s = 120.0  # the timed steps stop once they have taken this long (at least 3 run)
    t_start = None
    with ctx.Pool(cores) as pool:
        for i in range(args.warmup + args.steps):
            sample = [units[(i * per_step + j) % len(units)] for j in range(per_step)]
            t0 = time.perf_counter()
            pool.map(_ref_unit, sample, chunksize=1)
            dt = time.perf_counter() - t0
            if i >= args.warmup:
                t_start = t_start if t_start is not None else t0
                times.append(dt * len(units) / per_step)  # scaled to a whole step
                if len(times) >= 3 and time.perf_counter() - t_start > budget_s:
                    break
    ms = sum(times) / len(times) * 1e3
    value = 1e3 / ms
    # one core: a few units in this process (one BLAS thread), scaled to a whole step
    n1 = min(4, len(units))
    t0 = time.perf_counter()
    for bh in units[:n1]:
        _ref_unit(bh)
    single = 1.0 / ((time.perf_counter() - t0) * len(units) / n1)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": len(times), "steps_requested": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": headline_config(wl, args.agg, world),
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": min(cores, per_step), "kind": "oracle",
                         "sample": f"{per_step} of {len(units)} {unit_name} units per step, one per worker "
                                   f"process, each the full oracle path (fp64 scores, full sort, slot-table gather, "
                                   f"softmax attention); step time scaled by {len(units)}/{per_step}; "
                                   f"{len(times)} timed steps (stopped after {budget_s:.0f} s); input "
                                   f"generation {t_gen:.1f} s not timed",
                         "single_thread_value": round(single, 6),
                         "single_thread_sample": f"{n1} units in one process, one BLAS thread, scaled by "
                                                 f"{len(units)}/{n1}"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def time_calls(fn, n, stream):
    import torch

    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def timed_repeats(fn, steps, stream, world=1, min_s=0.5, max_repeats=5000):
    """Device time of `steps` back-to-back calls of fn, between CUDA events on the launch
    stream with a barrier and a synchronize on both sides, repeated until the repeats
    together last at least min_s (so the clock sampler sees the region).  Returns the
    per-repeat milliseconds per call."""
    import torch

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    out, total = [], 0.0
    while (total < min_s * 1e3 or not out) and len(out) < max_repeats:
        barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        ms = e0.elapsed_time(e1)
        out.append(ms / steps)
        total += ms
    return out


def step_distribution(fn, n, stream):
    """Per-call device times (ms) of n back-to-back calls, one event between calls:
    median, p10 and p90."""
    import torch

    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    evs[0].record(stream)
    for i in range(n):
        fn()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    t = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(n))
    pick = lambda f: t[min(n - 1, int(f * n))]  # noqa: E731
    return {"median_ms": round(pick(0.5), 5), "p10_ms": round(pick(0.1), 5), "p90_ms": round(pick(0.9), 5),
            "n": n}


def graph_call_ms(fn, stream, calls=20, reps=10, cold_l2=False):
    """Device time of one call of fn: `calls` calls captured in one CUDA graph,
    replayed `reps` times between CUDA events on the launch stream (no host
    launch cost inside the timed region).  cold_l2: every call is preceded by a
    256 MiB read that evicts L2 (129 MB) with clean lines, as the key stream of a
    step does, and a graph of the reads alone is timed the same way and
    subtracted -- the call as it runs inside a step."""
    import torch

    flush = torch.ones((64 << 20,), dtype=torch.float32, device=stream.device) if cold_l2 else None
    sink = torch.empty((), dtype=torch.float32, device=stream.device) if cold_l2 else None

    def timed(body):
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for _ in range(3):
                body()
        stream.wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(calls):
                body()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        del g
        return e0.elapsed_time(e1) / (calls * reps)

    if not cold_l2:
        return timed(fn)

    def sweep():
        torch.sum(flush, dim=0, out=sink)

    def both():
        sweep()
        fn()

    t = timed(both) - timed(sweep)
    del flush, sink
    torch.cuda.empty_cache()
    return t


def read_stream_gbs(stream):
    """Read-mostly HBM bandwidth of library kernels, best of two: a torch sum over
    2 GiB of bf16, and a cuBLAS bf16 matrix-vector product over a [8M, 128] matrix
    (the library form of scoring every key against one query: 2 GiB read, 32 MiB
    written).  Best of 5 each.  The copy peak counts read + write bytes."""
    import torch

    x = torch.ones((1 << 30,), dtype=torch.bfloat16, device="cuda")
    sum_ms = min(time_calls(lambda: x.sum(dtype=torch.float32), 1, stream) for _ in range(5))
    a = x.view(1 << 23, 128)
    v = torch.ones((128,), dtype=torch.bfloat16, device="cuda")
    mv_ms = min(time_calls(lambda: torch.mv(a, v), 1, stream) for _ in range(5))
    del x, a, v
    torch.cuda.empty_cache()
    sum_gbs = (1 << 31) / (sum_ms * 1e-3) / 1e9
    mv_gbs = ((1 << 31) + (1 << 24)) / (mv_ms * 1e-3) / 1e9
    return round(max(sum_gbs, mv_gbs), 1), {"sum_gbs": round(sum_gbs, 1), "mv_gbs": round(mv_gbs, 1)}


def step_bytes(wl, idx):
    """Algorithmic bytes of one step split by where they live: (HBM bytes, host bytes).

    HBM: the scored keys of every candidate (read once per KV head), the fp32 scores
    (written and read once per selection row), queries and outputs, and the attended
    K/V rows that sit in the GPU pool (for latent rows also the gathered copy, written
    and read once).  Host: the attended rows read from the pinned host pool over the
    host link.  The selection rows are idx's second dimension: the KV heads, or the
    query heads when each selects its own."""
    import torch

    d_row = wl.d_qk * 2 + (0 if wl.gpu_v is None else wl.d_v * 2)
    lens = [int(x) for x in wl.seq_lens.cpu()]
    rows = idx.shape[1]
    hbm = wl.B * wl.Hq * (wl.d_qk + wl.d_v) * 2
    host = 0
    for b in range(wl.B):
        s_end, l_start = regions(lens[b], wl.ns, wl.nl)
        n_c = l_start - s_end
        hbm += wl.H * n_c * wl.d_idx * 2 + rows * n_c * 8
        for h in range(rows):
            sel = idx[b, h]
            sel = sel[sel >= 0].long()
            pos = torch.cat([torch.arange(0, s_end, device=sel.device), sel,
                             torch.arange(l_start, lens[b], device=sel.device)])
            ent = wl.table[b].long()[pos // wl.bs]
            n_host = int((ent < 0).sum())
            n_gpu = pos.numel() - n_host
            hbm += n_gpu * d_row
            host += n_host * d_row
            if wl.gpu_v is None:
                hbm += 2 * pos.numel() * d_row
    return hbm, host


CONFIG_DESC = {
    "tiny": "tiny: batch 1, 1 KV x 8 q heads, d128, L4096, top-k 256 + 4 sink + 64 local, bf16, identity "
            "16-token blocks, 1% heavy keys",
    "host1m": "8B-class long context host pool: batch 1, 8 KV x 32 q heads, d128, L1048576, top-k 100 + 16 sink "
              "+ 512 local; K/V in pinned host memory read over UVA (sink/local blocks in HBM); GPU-resident index "
              "keys from a drifting 64-component mixture",
    "mla": "MLA-style latent: batch 16, L131072, 576-wide latent rows (512 + 64 rope), 128 q heads, single-head "
           "d128 indexer, top-k 2048; latent pool in pinned host memory, GPU slot cache of 25% of tokens",
    "sweep": "sweep point: 8 KV x 64 q heads, d128, 4 sink + 128 local, bf16 paged GPU pool, random block "
             "permutation, 1% heavy keys",
}

# the sweep's four corners measured on the headline line
SWEEP_CORNERS = ((1, 8192, 256), (64, 131072, 4096), (64, 8192, 4096), (16, 32768, 1024))
L2_BYTES = 129 * 10 ** 6


def measure_config(name, stream, steps, hbm_peak, link=None, prefetch=0, seed=None, phases=True, group_agg="mean",
                   **over):
    """One workload's decode step, measured like the headline: a CUDA graph of the step,
    K replays per repeat until the repeats last >= 0.5 s (median repeat), the clock
    sampler around them.  Working sets under 4x L2 run after an L2-evicting 256 MiB read
    inside the graph, whose own time is measured the same way and subtracted.  Returns
    the entry: steps/s, HBM and host-link bytes and fractions, phase times, clocks."""
    import torch

    import top_sparse_kv_gb300 as skv
    import workloads

    wl = workloads.make_workload(name, device="cuda", gen_device="cuda", seed=seed, **over)
    step = skv.DecodeStep.from_workload(wl, group_agg=agg_code(skv, group_agg))
    run = step.run
    if prefetch > 0:  # threshold prefetch: its state persists across the replays
        step.enable_prefetch(prefetch)
        run = lambda: step.run_prefetch(stats=False)  # noqa: E731
    run()
    torch.cuda.synchronize()
    if int(step.status.item()) != 0:
        raise RuntimeError(f"{name}: device status {int(step.status.item())}")
    hbm, host = step_bytes(wl, step.idx)
    cold = hbm < 4 * L2_BYTES
    flush = torch.ones((64 << 20,), dtype=torch.float32, device="cuda") if cold else None
    sink = torch.empty((), dtype=torch.float32, device="cuda") if cold else None

    def graph_of(body, calls):
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for _ in range(2):
                body()
        stream.wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(calls):
                body()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        return g

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    if cold:
        def both():
            torch.sum(flush, dim=0, out=sink)
            run()

        g_both = graph_of(both, steps)
        g_flush = graph_of(lambda: torch.sum(flush, dim=0, out=sink), steps)
        clocks.mark("t0")
        reps_both = timed_repeats(g_both.replay, 1, stream, min_s=0.5)
        reps_flush = timed_repeats(g_flush.replay, 1, stream, min_s=0.2)
        clocks.mark("t1")
        reps = [(x - statistics.median(reps_flush)) / steps for x in reps_both]
        del g_both, g_flush
    else:
        g = graph_of(run, 1)
        clocks.mark("t0")
        reps = timed_repeats(g.replay, steps, stream, min_s=0.5)
        clocks.mark("t1")
        del g
    clock_rec = clocks.stop()
    ms = statistics.median(reps)
    entry = {"workload": CONFIG_DESC.get(name, name), "value": round(1e3 / ms, 3), "unit": UNIT,
             "ms_per_step": round(ms, 6), "repeats": len(reps),
             "l2": "an L2-evicting 256 MiB read before every step (subtracted)" if cold else
                   "inputs larger than 4x L2",
             "hbm": {"bytes_per_step": hbm, "achieved_gbs": round(hbm / ms / 1e6, 1),
                     "frac": round(hbm / ms / 1e6 / hbm_peak, 4)},
             "clocks": clock_rec}
    if host > 0:
        entry["host_link"] = {"bytes_per_step": host, "achieved_gbs_over_step": round(host / ms / 1e6, 1)}
    if phases and prefetch == 0:
        entry["phase_ms"] = {"score": round(graph_call_ms(step.score, stream), 5),
                             "topk": round(graph_call_ms(step.topk, stream), 5),
                             "attention": round(graph_call_ms(step.attend, stream, cold_l2=True), 5)}
    if host > 0 and link is not None:
        # the step's own attended rows through skv_gather: host bytes over its time
        n_att = wl.ns + wl.k + wl.nl
        k_out = torch.empty((wl.B, wl.H, n_att, wl.d_qk), dtype=wl.dtype, device="cuda")
        v_out = None if wl.gpu_v is None else torch.empty((wl.B, wl.H, n_att, wl.d_v), dtype=wl.dtype,
                                                          device="cuda")
        # a graph of 20 calls: a small gather's time is the kernel's, not the host's launch rate
        g_ms = graph_call_ms(lambda: skv.skv_gather(step.p, step.pool, step.idx, k_out, v_out, step.status), stream)
        gbs = host / g_ms / 1e6
        entry["host_gather"] = {"host_bytes": host, "ms": round(g_ms, 5), "gbs": round(gbs, 1),
                                "frac_of_copy_engine": round(gbs / link["copy_engine_h2d_1GiB"]["gbs"], 4),
                                "frac_of_sm_sequential_read": round(gbs / link["seq_rows_256B"]["gbs"], 4),
                                "how": "skv_gather of the step's attended rows (its own selection), host-resident "
                                       "bytes over the kernel time (a CUDA graph of 20 calls)"}
        del k_out, v_out
    if prefetch > 0:
        step.pf.stats.zero_()
        step.run_prefetch(stats=True)
        torch.cuda.synchronize()
        hits, misses = (int(x) for x in step.pf.stats.cpu())
        entry["prefetch"] = {"staging_rows": prefetch, "host_rows_staged": hits, "host_rows_read_after": misses,
                             "staged_frac": round(hits / max(1, hits + misses), 4),
                             "note": "the same query every replay: the threshold EMA settles on the step's own "
                                     "k-th score"}
    del step, wl, flush, sink
    torch.cuda.empty_cache()
    return entry


def link_ceilings(stream):
    """Host-link ceilings: one 1 GiB pinned host -> device copy on the copy engine, and
    the path's own gather (skv_gather, SM loads over UVA) from fully host-resident pinned
    pools: 16-token blocks read in order, random 256-byte rows, random 1152-byte rows."""
    import torch

    import top_sparse_kv_gb300 as skv
    import workloads

    out = {}
    h = torch.empty((1 << 30,), dtype=torch.uint8).pin_memory()
    d = torch.empty((1 << 30,), dtype=torch.uint8, device="cuda")
    ms_ce = min(time_calls(lambda: d.copy_(h, non_blocking=True), 2, stream) for _ in range(3))
    ce_gbs = (1 << 30) / ms_ce / 1e6
    out["copy_engine_h2d_1GiB"] = {"gbs": round(ce_gbs, 1), "ms": round(ms_ce, 4), "bytes": 1 << 30}
    del h, d
    torch.cuda.empty_cache()
    cases = [("seq_rows_256B", dict(name="gqa32b", B=1, H=1, Hq=8, L=1 << 20, k=(1 << 20), ns=0, nl=0), "all"),
             ("random_rows_256B", dict(name="gqa32b", B=1, H=1, Hq=8, L=1 << 20, k=65536, ns=0, nl=0), "random"),
             ("random_rows_1152B", dict(name="mla", B=4, L=131072, k=16384, gpu_cache_frac=0.0), "random")]
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    for label, cfg, kind in cases:
        cfg = dict(cfg)
        name = cfg.pop("name")
        wl = workloads.make_workload(name, device="cuda", gen_device="cuda",
                                     host_frac=0.9999 if name != "mla" else 0.0, **cfg)
        step = skv.DecodeStep.from_workload(wl)
        n_c = wl.L - wl.ns - wl.nl
        if kind == "all":
            idx = torch.arange(wl.ns, wl.ns + wl.k, device="cuda", dtype=torch.int32).repeat(wl.B, wl.H, 1)
        else:
            r = torch.rand((wl.B * wl.H, n_c), generator=g, device="cuda")
            idx = (r.argsort(dim=1)[:, :wl.k].sort(dim=1).values + wl.ns).to(torch.int32).view(wl.B, wl.H, wl.k)
        idx = idx.contiguous()
        n_att = wl.ns + wl.k + wl.nl
        k_out = torch.empty((wl.B, wl.H, n_att, wl.d_qk), dtype=wl.dtype, device="cuda")
        v_out = None if wl.gpu_v is None else torch.empty((wl.B, wl.H, n_att, wl.d_v), dtype=wl.dtype, device="cuda")
        fn = lambda: skv.skv_gather(step.p, step.pool, idx, k_out, v_out, step.status)  # noqa: E731
        ms = time_calls(fn, 20, stream)
        host_rows = wl.B * wl.H * wl.k
        row_bytes = wl.d_qk * 2 + (0 if v_out is None else wl.d_v * 2)
        gbs = host_rows * row_bytes / ms / 1e6
        out[label] = {"gbs": round(gbs, 1), "ms": round(ms, 4), "bytes": host_rows * row_bytes,
                      "frac_of_copy_engine": round(gbs / ce_gbs, 4)}
        del wl, step, k_out, v_out, idx
        torch.cuda.empty_cache()
    return out


def run_configs(args, stream, hbm_peak):
    """Every other workload, measured in the same run as the headline (each entry with its
    own clock record): tiny, host1m (with the host gather against the link ceilings
    measured here) plain and with threshold prefetch, mla plain and with threshold
    prefetch, and the sweep's four corners."""
    steps = max(3, args.steps)
    out = {"host_link_ceilings": link_ceilings(stream)}
    link = out["host_link_ceilings"]
    out["tiny"] = measure_config("tiny", stream, steps, hbm_peak)
    out["host1m"] = measure_config("host1m", stream, steps, hbm_peak, link=link)
    out["host1m_prefetch"] = measure_config("host1m", stream, steps, hbm_peak, prefetch=4096)
    out["mla"] = measure_config("mla", stream, steps, hbm_peak, link=link)
    out["mla_prefetch"] = measure_config("mla", stream, steps, hbm_peak, prefetch=4096)
    import workloads

    for B, L, k in SWEEP_CORNERS:
        i = workloads.SWEEP_POINTS.index((B, L, k))
        e = measure_config("sweep", stream, steps, hbm_peak, seed=workloads.seed_for("sweep", i), B=B, L=L, k=k)
        e["point"] = {"batch": B, "history": L, "topk": k}
        out[f"sweep_B{B}_L{L // 1024}K_k{k}"] = e
    return out


def run_workload(args):
    """One line for a named workload (tiny, host1m, mla; --prefetch for the latent one), measured
    as the headline line's configs entries are."""
    import torch

    import __graft_entry__

    __graft_entry__.build()
    pk = peaks()
    hbm_peak = pk["hbm_gbs"] if pk else 6800.0
    stream = torch.cuda.current_stream()
    entry = measure_config(args.workload, stream, max(3, args.steps), hbm_peak, prefetch=args.prefetch,
                           group_agg=args.agg)
    print(json.dumps({"metric": METRIC, "workload": args.workload, "group_agg": args.agg, "dtype": "bf16",
                      "data": "synthetic", **entry}), flush=True)


def run_cache(args):
    """Latent workload with the GPU slot pool managed as a cache over the host pool
    (skv_decode_step_cached), on a drifting query trajectory: the cached step
    against the uncached one on the same queries.

    Trajectory: every query tensor follows q_{s+1} = r q_s + sqrt(1 - r^2) n_s with
    fresh standard normal n_s and r = cos(2 pi / 64), so each step's query keeps the
    workload's distribution while consecutive queries stay correlated (the step-to-step
    reuse that a cache over decode steps relies on).  The first 64 steps warm the cache
    untimed; the next `timed` steps are captured in one CUDA graph, replayed four times
    from the same cache state (the first replay uncounted, the median of the others)."""
    import copy
    import math

    import torch

    import __graft_entry__

    __graft_entry__.build()
    import top_sparse_kv_gb300 as skv
    from top_sparse_kv_gb300 import binding as B
    import workloads

    wl = workloads.make_workload("mla", device="cuda", gen_device="cuda")
    twin = copy.copy(wl)
    twin.table, twin.gpu_k = wl.table.clone(), wl.gpu_k.clone()
    n_warm, timed = 64, 256
    r = math.cos(2 * math.pi / 64)
    g = torch.Generator(device="cuda").manual_seed(4242)

    def walk(x0, n):
        out = torch.empty((n,) + tuple(x0.shape), dtype=x0.dtype, device="cuda")
        x = x0.float()
        for i in range(n):
            out[i] = x.to(x0.dtype)
            x = r * x + math.sqrt(1.0 - r * r) * torch.randn(x0.shape, generator=g, device="cuda")
        return out

    qs, qis = walk(wl.q, n_warm + timed), walk(wl.q_idx, n_warm + timed)
    step = skv.DecodeStep.from_workload(wl)
    plain = skv.DecodeStep.from_workload(twin)
    cache = step.enable_cache(args.cache)
    stream = torch.cuda.current_stream()

    def cached(i):
        B.skv_decode_step_cached(step.p, qs[i], qis[i], step.index, step.pool, step.scores, step.idx, step.out,
                                 step.lse, step.ws, cache, step.status)  # the current stream (capture too)

    def uncached(i):
        B.skv_decode_step(plain.p, qs[i], qis[i], plain.index, plain.pool, plain.scores, plain.idx, plain.out,
                          plain.lse, plain.ws, plain.status)

    for i in range(n_warm):
        cached(i)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    span = range(n_warm, n_warm + timed)
    gc, gp = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(gc):
        for i in span:
            cached(i)
    with torch.cuda.graph(gp):
        for i in span:
            uncached(i)
    # the trajectory moves the cache state: every timed replay starts from the same
    # snapshot (restored outside the timed region); the first replay is not counted
    snap = [t.clone() for t in (wl.table, wl.gpu_k, cache.owner, cache.prio, cache.step)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    trials = []
    for trial in range(4):
        for dst, src in zip((wl.table, wl.gpu_k, cache.owner, cache.prio, cache.step), snap):
            dst.copy_(src)
        cache.stats.zero_()
        torch.cuda.synchronize()
        e0.record(stream)
        gc.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        if trial > 0:
            trials.append(e0.elapsed_time(e1) / timed)
    ms_c = sorted(trials)[len(trials) // 2]
    hits, misses, promos = (int(x) for x in cache.stats.cpu())
    assert int(step.status.item()) == 0
    gp.replay()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(3):
        gp.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms_p = e0.elapsed_time(e1) / (3 * timed)
    # the uncached step's host rows on the same trajectory (its table never changes)
    p_host = p_all = 0
    for i in span:
        uncached(i)
        idx = plain.idx[:, 0].long()
        ok = idx >= 0
        ent = twin.table.long().gather(1, idx.clamp(min=0))
        p_host += int(((ent < 0) & ok).sum())
        p_all += int(ok.sum())
    assert int(plain.status.item()) == 0
    cache.count = False
    upd = graph_call_ms(step.cache_update, stream)
    row = wl.d_qk * 2
    line = {"metric": METRIC, "workload": "mla", "value": round(1e3 / ms_c, 3), "unit": UNIT,
            "ms_per_step": round(ms_c, 6), "dtype": "bf16", "data": "synthetic",
            "cache": {"budget_per_step": args.cache, "gpu_slots": int(wl.gpu_k.shape[0]),
                      "timed_steps": timed, "warm_steps": n_warm, "query_step_correlation": round(r, 6),
                      "hit_frac": round(hits / max(1, hits + misses), 4),
                      "promotions_per_step": round(promos / timed, 1),
                      "host_bytes_per_step": misses * row // timed,
                      "update_ms": round(upd, 5),
                      "replays_ms_per_step": [round(x, 5) for x in trials],
                      "timing": "median of 3 replays of the trajectory graph, each from the same cache state"},
            "uncached": {"value": round(1e3 / ms_p, 3), "ms_per_step": round(ms_p, 6),
                         "hit_frac": round(1 - p_host / max(1, p_all), 4),
                         "host_bytes_per_step": p_host * row // timed}}
    print(json.dumps(line), flush=True)


def run_cache_heads(args):
    """host1m with one slot-table row per (request, KV head) and the GPU slots managed as a
    per-head block cache (skv_decode_step_cached) over the host pool that backs every
    block, on the drifting query trajectory of run_cache; against the uncached step on
    host1m's own layout (sink and local blocks in HBM, the rest read from the host) on the
    same queries.  Slots: 16,384 one-head blocks (2,048 a head), empty at the start."""
    import math

    import torch

    import __graft_entry__

    __graft_entry__.build()
    import top_sparse_kv_gb300 as skv
    from top_sparse_kv_gb300 import binding as B
    import workloads

    wl = workloads.make_workload("host1m", device="cuda", gen_device="cuda")
    lay = workloads.head_table_layout(wl, gpu_frac=0.0, seed=4243)
    n_slots = 16384
    shape_k, shape_v = tuple(lay["gpu_k"].shape[1:]), tuple(lay["gpu_v"].shape[1:])
    gpu_k = torch.zeros((n_slots,) + shape_k, dtype=wl.dtype, device="cuda")
    gpu_v = torch.zeros((n_slots,) + shape_v, dtype=wl.dtype, device="cuda")
    n_warm, timed = 64, 256
    r = math.cos(2 * math.pi / 64)
    g = torch.Generator(device="cuda").manual_seed(4242)
    qs = torch.empty((n_warm + timed,) + tuple(wl.q.shape), dtype=wl.q.dtype, device="cuda")
    x = wl.q.float()
    for i in range(n_warm + timed):
        qs[i] = x.to(wl.q.dtype)
        x = r * x + math.sqrt(1.0 - r * r) * torch.randn(wl.q.shape, generator=g, device="cuda")
    plain = skv.DecodeStep.from_workload(wl)
    pool = skv.Pool(gpu_k, gpu_v, lay["table"], lay["host_k"], lay["host_v"], table_heads=1)
    step = skv.DecodeStep(plain.p, pool, plain.q, plain.index, q_score=plain.q_score)
    cache = step.enable_cache(args.cache)
    stream = torch.cuda.current_stream()

    def cached(i):  # host1m scores with the attention query itself (contiguous index keys)
        B.skv_decode_step_cached(step.p, qs[i], qs[i], step.index, step.pool, step.scores, step.idx, step.out,
                                 step.lse, step.ws, cache, step.status)

    def uncached(i):
        B.skv_decode_step(plain.p, qs[i], qs[i], plain.index, plain.pool, plain.scores, plain.idx, plain.out,
                          plain.lse, plain.ws, plain.status)

    for i in range(n_warm):
        cached(i)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    span = range(n_warm, n_warm + timed)
    gc, gp = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(gc):
        for i in span:
            cached(i)
    with torch.cuda.graph(gp):
        for i in span:
            uncached(i)
    state = (lay["table"], gpu_k, gpu_v, cache.owner, cache.prio, cache.step)
    snap = [t.clone() for t in state]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    trials = []
    for trial in range(4):
        for dst, src in zip(state, snap):
            dst.copy_(src)
        cache.stats.zero_()
        torch.cuda.synchronize()
        e0.record(stream)
        gc.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        if trial > 0:
            trials.append(e0.elapsed_time(e1) / timed)
    ms_c = sorted(trials)[len(trials) // 2]
    hits, misses, promos = (int(x) for x in cache.stats.cpu())
    assert int(step.status.item()) == 0
    gp.replay()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(3):
        gp.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms_p = e0.elapsed_time(e1) / (3 * timed)
    assert int(plain.status.item()) == 0
    block_bytes = wl.bs * (wl.d_qk + wl.d_v) * 2
    line = {"metric": METRIC, "workload": "host1m, one slot-table row per (request, KV head)",
            "value": round(1e3 / ms_c, 3), "unit": UNIT, "ms_per_step": round(ms_c, 6), "dtype": "bf16",
            "data": "synthetic",
            "cache": {"budget_per_step": args.cache, "gpu_slots": n_slots, "slot": "one KV head's 16-token block",
                      "timed_steps": timed, "warm_steps": n_warm, "query_step_correlation": round(r, 6),
                      "block_hit_frac": round(hits / max(1, hits + misses), 4),
                      "blocks_used_per_step": round((hits + misses) / timed, 1),
                      "promotions_per_step": round(promos / timed, 1),
                      "promotion_bytes_per_step": promos * block_bytes // timed,
                      "replays_ms_per_step": [round(x, 5) for x in trials],
                      "timing": "median of 3 replays of the trajectory graph, each from the same cache state"},
            "uncached": {"value": round(1e3 / ms_p, 3), "ms_per_step": round(ms_p, 6),
                         "layout": "host1m's own: sink and local blocks in HBM, the rest read from the host"}}
    print(json.dumps(line), flush=True)


def run_paris(args):
    """ParisKV retrieval (skv_paris_decode_step) in place of exact scoring and top-k, on a
    named workload (host1m unless --workload names another), against the exact step on
    the same inputs: steps/s, phase times, the selection phase's HBM fraction, and the
    recall of the exact top-k."""
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import top_sparse_kv_gb300 as skv
    import workloads

    name = args.workload if args.workload != WORKLOAD else "host1m"
    wl = workloads.make_workload(name, device="cuda", gen_device="cuda")
    stream = torch.cuda.current_stream()
    signs = workloads.srht_signs(128, device="cuda")
    ps = skv.ParisStep.from_workload(wl, signs, args.paris_beta, args.paris_rho)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    ps.encode()
    e1.record(stream)
    torch.cuda.synchronize()
    enc_ms = e0.elapsed_time(e1)
    assert int(ps.status.item()) == 0

    def graph_ms(fn):
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return time_calls(g.replay, max(20, min(args.steps, 2000)), stream)

    ms = graph_ms(ps.run)
    assert int(ps.status.item()) == 0
    exact = skv.DecodeStep.from_workload(wl)
    ms_exact = graph_ms(exact.run)
    rows = wl.B * wl.H
    got, want = ps.idx.view(rows, -1).cpu().numpy(), exact.idx.view(rows, -1).cpu().numpy()
    recall = sum(len(set(got[r][got[r] >= 0].tolist()) & set(want[r][want[r] >= 0].tolist()))
                 for r in range(rows)) / max(1, int((want >= 0).sum()))
    sel_ms = graph_call_ms(ps.select, stream, cold_l2=True)
    att_ms = graph_call_ms(ps.attend, stream, cold_l2=True)
    # algorithmic bytes of the selection: 16 centroid bytes read and one score byte written
    # per candidate-region key, 64 + 64 bytes of codes and weights per candidate, its
    # position and score written and read once, the rows' small tables
    n_keys = 0
    for b in range(wl.B):
        s_end, l_start = regions(int(wl.seq_lens[b]), wl.ns, wl.nl)
        n_keys += wl.H * (l_start - s_end)
    n_cand = int(ps.view("cand_len").sum().item()) * wl.H
    sel_bytes = n_keys * 17 + n_cand * (128 + 16) + rows * (16 * 256 * 5 + 1024)
    pk = peaks()
    hbm_peak = pk["hbm_gbs"] if pk else 6800.0
    line = {"metric": METRIC, "workload": name, "retrieval": "paris", "value": round(1e3 / ms, 3), "unit": UNIT,
            "ms_per_step": round(ms, 6), "dtype": "bf16", "data": "synthetic",
            "paris": {"beta_permille": args.paris_beta, "rho_permille": args.paris_rho,
                      "candidates_per_row": n_cand // rows, "recall_of_exact_topk": round(recall, 4),
                      "encode_ms": round(enc_ms, 3),
                      "index_bytes_per_key": 16 + 64 + 64},
            "phase_ms": {"select": round(sel_ms, 5), "attention": round(att_ms, 5)},
            "select_hbm": {"bytes": sel_bytes, "achieved_gbs": round(sel_bytes / sel_ms / 1e6, 1),
                           "frac": round(sel_bytes / sel_ms / 1e6 / hbm_peak, 4)},
            "exact": {"value": round(1e3 / ms_exact, 3), "ms_per_step": round(ms_exact, 6)}}
    print(json.dumps(line), flush=True)


def run_blocks(args):
    """One line for block selection from per-block min/max key summaries on the gqa32b workload:
    steps/s of skv_block_decode_step (CUDA graph), its HBM bytes and roofline fraction."""
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import top_sparse_kv_gb300 as skv
    import workloads

    if args.agg == "head":
        raise SystemExit("block selection ranks blocks per KV head: --agg mean or max")
    wl = workloads.make_workload(WORKLOAD, device="cuda", gen_device="cuda")
    agg = skv.SKV_AGG_MAX if args.agg == "max" else skv.SKV_AGG_MEAN
    step = skv.BlockStep.from_workload(wl, args.blocks, group_agg=agg)
    stream = torch.cuda.current_stream()
    step.summarize()
    step.run()
    torch.cuda.synchronize()
    if int(step.status.item()) != 0:
        raise RuntimeError(f"device status {int(step.status.item())}")
    # a step's inputs (summaries and attended rows, ~180 MB) are close to L2's 129 MB: every timed
    # step runs after an L2-evicting read, as it would after the rest of a model's layer
    ms = graph_call_ms(step.run, stream, calls=20, reps=max(5, min(args.steps, 200) // 20), cold_l2=True)
    t_sel = graph_call_ms(step.select, stream, cold_l2=True)
    t_sum = graph_call_ms(step.summarize, stream)
    nb, s_blk, l_blk = block_regions(wl.L, wl.ns, wl.nl, 16)
    n_cand = l_blk - s_blk
    n_tok = int((step.att_idx[0, 0] >= 0).sum())
    units = wl.B * wl.H
    hbm = units * (n_cand * (2 * wl.d_qk * 2 + 8) + n_tok * 2 * wl.d_qk * 2) + 2 * wl.B * wl.Hq * wl.d_qk * 2
    pk = peaks()
    hbm_peak = pk["hbm_gbs"] if pk else 6800.0
    line = {"metric": "block-selection decode steps/s (all heads, 1 GB300)", "workload": WORKLOAD, "value":
            round(1e3 / ms, 3), "unit": UNIT, "ms_per_step": round(ms, 6), "dtype": "bf16", "data": "synthetic",
            "group_agg": args.agg, "blocks": args.blocks, "attended_tokens": n_tok,
            "hbm": {"bytes_per_step": hbm, "achieved_gbs": round(hbm / ms / 1e6, 1),
                    "frac": round(hbm / ms / 1e6 / hbm_peak, 4)},
            "phase_ms": {"select": round(t_sel, 5), "attention": round(ms - t_sel, 5)},
            "summaries_ms": round(t_sum, 5),
            "timing": "CUDA graph of 20 steps, each after a 256 MiB L2-evicting read (subtracted)",
            "note": "summaries are maintenance (run when blocks fill), not part of a step"}
    print(json.dumps(line), flush=True)


def run_hostlink(args):
    """Host-link ceilings through the path's own gather (skv_gather) and the copy engine."""
    import torch

    import __graft_entry__

    __graft_entry__.build()
    print(json.dumps({"hostlink": link_ceilings(torch.cuda.current_stream()),
                      "how": "skv_gather from a fully host-resident pinned pool, CUDA events; one 1 GiB "
                             "pinned host -> device copy on the copy engine"}), flush=True)


def run_sweep(args):
    """One line per sweep point: batch x history x k on the paged GPU pool."""
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import workloads

    stream = torch.cuda.current_stream()
    pk = peaks()
    hbm_peak = pk["hbm_gbs"] if pk else 6800.0
    for i, (B, L, k) in enumerate(workloads.SWEEP_POINTS):
        e = measure_config("sweep", stream, max(3, args.steps), hbm_peak, seed=workloads.seed_for("sweep", i),
                           phases=False, B=B, L=L, k=k)
        print(json.dumps({"sweep_point": i, "batch": B, "history": L, "topk": k, **e}), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.blocks > 0:
        run_blocks(args)
    elif args.cache > 0 and args.workload == "host1m":
        run_cache_heads(args)
    elif args.cache > 0:
        run_cache(args)
    elif args.paris:
        run_paris(args)
    elif args.hostlink:
        run_hostlink(args)
    elif args.sweep:
        run_sweep(args)
    elif args.workload != WORKLOAD:
        run_workload(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
