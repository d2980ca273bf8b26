"""Benchmark of one paged-KV decode step on GB300: slot write + decode attention.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload 3]

A step is one pass of the whole hot path over one batch of synthetic input, through
paged_decode_step: the slot-mapping KV write of the step's new tokens, then decode
attention (launched as a programmatic dependent of the write) as the
launcher plans it (one kernel: one CTA per partition; split sequences are merged by
their last partition).

Default workload: the largest single-GPU step, a decode batch of 64 sequences with
ragged contexts uniform in [128, 4096], 24 query / 8 kv heads, head_dim 128, bf16,
block_size 16, block tables drawn from a shuffled pool of 1.25x the blocks in use,
64 new tokens written per step (about 554 MB of K/V read per step).  The other
workloads (--workload 1..5) are the batch-1 / batch-16 / continuous-batching /
long-context shapes of the same path.

Timing (ours): inputs are resident in HBM; the pool is replicated R times so that
the copies together exceed 3x the L2 size, and step i uses copy i mod R (so every
step reads its K/V from DRAM, not L2).  The K timed steps are replayed from CUDA
graphs (one graph of R steps, one of the remainder), bracketed by a barrier and
torch.cuda.synchronize() and timed with CUDA events on the launching stream; the
max over ranks is reported.  `value` is algorithmic HBM bytes per step / time,
in GB/s (whole job: all ranks' bytes / the slowest rank's time).

`roofline` covers the dominant kernel (the decode kernel), timed alone by
the same method; `e2e` runs the same step through the public API with the step's
inputs in pinned host memory and the output read back into pinned host memory each
step; `cpu_baseline` is the CPU oracle (fp64, all host cores) on the same workload.
`e2e` hands paged_decode_step the pinned host buffers themselves (zero-copy: the
kernels read the inputs and write the output over the host link), one CUDA graph
replayed and synchronised per step (the eager time is reported beside it); the
breakdown also gives the same step with an explicit copy in and copy out as graph
nodes.

`--impl reference` times that oracle as the reference arm (rank 0 only).

Other modes, each printing one JSON line of its own: `--kernel prefill | rope_write |
rope_step` time those entry points on the workload's shapes; `--kernel split
--partition P` times paged_decode_split + paged_decode_combine at a fixed partition
size; `--consumer fma` switches the partition decode kernel's consumer warps to their
CUDA-core form (pkv_set_decode_consumer) for comparison with the default tensor form.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_decode_mapping_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode attention µs/step and achieved HBM GB/s (% of GB300 peak)"


# ----------------------------------------------------------------------------- bytes
def algorithmic_bytes(inp: dict) -> dict:
    """Bytes the operations must move, per step (no re-reads, no workspace)."""
    w = inp["workload"]
    lens = inp["context_lens"].long()
    nblk = (lens + w.BS - 1) // w.BS
    kv = int(lens.sum()) * w.Hkv * w.D * 2 * 2             # K and V rows read once
    qo = w.B * w.Hq * w.D * 2                                # q read, out written (each)
    tables = 4 * int(nblk.sum()) + 4 * w.B                   # table entries + context_lens
    T = int(inp["slot_mapping"].numel())
    write = 2 * (2 * T * w.Hkv * w.D * 2) + 8 * T            # k/v read + cache rows written + slots
    decode = kv + qo + tables                                # what the decode kernel reads
    return {"kv": kv, "decode_kernel": decode, "step": decode + qo + write, "write": write}


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- setup
def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


DECODE_SOURCES = ("pkv_decode.cu", "attn_device.cuh", "pkv_internal.h")


def decode_source_sha() -> str:
    """sha256 over the decode kernel's device source files, in a fixed order."""
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        h.update(open(os.path.join(ROOT, "paged_kv_decode_mapping_gb300", "csrc", name), "rb").read())
    return h.hexdigest()


def recorded_traffic(workload: int) -> float | None:
    """Per-launch DRAM bytes of the decode kernel on this workload from the committed ncu
    summary, if it was taken on the current kernel source (same sha256 over
    DECODE_SOURCES); else None."""
    path = os.path.join(ROOT, "profiles", f"ncu_decode_kernel_workload{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_tr or m_sha.group(1) != decode_source_sha():
        return None
    return float(m_tr.group(1))


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ----------------------------------------------------------------------------- CPU oracle
def time_oracle(inp: dict, budget_s: float, max_reps: int = 1000) -> dict:
    """Oracle write+decode on the host cores for up to ~budget_s: GB/s of algorithmic bytes."""
    import oracle

    orc = oracle.get()
    nbytes = algorithmic_bytes(inp)["step"]
    t0 = time.perf_counter()
    reps = 0
    while True:
        orc.step(inp)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= max_reps:
            break
    per = el / reps
    # the same step on one thread (a fifth of the budget, at least one step)
    t1, reps1 = time.perf_counter(), 0
    while True:
        orc.step(inp, num_threads=1)
        reps1 += 1
        el1 = time.perf_counter() - t1
        if el1 >= budget_s / 5 or reps1 >= max_reps:
            break
    per1 = el1 / reps1
    return {"value": nbytes / per / 1e9, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
            "value_1_thread": nbytes / per1 / 1e9,
            "sample": f"{reps} full write+decode steps of the workload, fp64, OpenMP over "
                      f"(sequence, head) rows on {os.cpu_count()} threads; {per * 1e3:.1f} ms/step "
                      f"({per1 * 1e3:.1f} ms/step on one thread, {reps1} steps)"}


def run_reference(args, w) -> None:
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle

    inp = W.make_inputs(w)
    orc = oracle.get()
    B, Hq = w.B, w.Hq
    rows_all = torch.tensor([[b, h] for b in range(B) for h in range(Hq)], dtype=torch.int32)
    # calibrate one full step, then size each step's sample so the run stays within ~2 minutes
    t0 = time.perf_counter()
    orc.step(inp)
    t_full = time.perf_counter() - t0
    budget = 120.0
    frac = min(1.0, budget / max(1e-9, t_full * (args.steps + args.warmup)))
    n_rows = max(1, int(round(frac * len(rows_all))))
    step_bytes = algorithmic_bytes(inp)["step"]
    kv_cache, v_cache = orc.kv_write(inp["k_new"], inp["v_new"], inp["slot_mapping"],
                                     inp["k_cache"], inp["v_cache"])

    def one(i):
        sel = rows_all[(torch.arange(n_rows) + i * n_rows) % len(rows_all)]
        if n_rows == len(rows_all):
            orc.step(inp)
            return step_bytes
        orc.decode(inp["q"], kv_cache, v_cache, inp["block_tables"], inp["context_lens"],
                   inp["scale"], rows=sel)
        return step_bytes * n_rows / len(rows_all)  # the sampled share of the step

    for i in range(args.warmup):
        one(i)
    t0 = time.perf_counter()
    nbytes = 0
    for i in range(args.steps):
        nbytes += one(i)
    el = time.perf_counter() - t0
    value = nbytes / el / 1e9
    sample = (f"each step: the full write+decode step" if n_rows == len(rows_all) else
              f"each step: {n_rows} of {len(rows_all)} (sequence, query head) rows of the decode, "
              f"round robin") + f"; fp64 oracle, {os.cpu_count()} threads"
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "impl": "reference", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(w, inp, args, world=1),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_dict(w, inp, args, world: int) -> dict:
    return {"workload": w.name, "batch": w.B, "q_heads": w.Hq, "kv_heads": w.Hkv,
            "head_dim": w.D, "block_size": w.BS, "context": f"{w.lens}:{int(inp['context_lens'].min())}"
            f"..{int(inp['context_lens'].max())}", "pool_blocks": inp["num_blocks"],
            "new_tokens_per_step": int(inp["slot_mapping"].numel()), "seed": w.seed,
            "l2": "rotating pool copies > 3x L2 between steps", "parallelism": f"replicas x{world}",
            "consumer": args.consumer}


# ----------------------------------------------------------------------------- ours
def run_ours(args, w) -> None:
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=device)
    from paged_kv_decode_mapping_gb300 import binding as B

    inp = W.make_inputs(w, seed=w.seed + 7919 * rank)
    nb = algorithmic_bytes(inp)
    Bn, Hq, D = inp["q"].shape
    NB, Hkv, BS, _ = inp["k_cache"].shape
    max_len = inp["max_context_len"]
    scale = inp["scale"]
    P = B.paged_decode_plan(Bn, Hq, Hkv, D, max_len)
    path = B.paged_decode_path(Bn, Hq, Hkv, D, max_len)

    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    pool_bytes = 2 * inp["k_cache"].numel() * 2
    R = max(2, math.ceil(3 * l2 / pool_bytes))
    kcs = [inp["k_cache"].to(device) for _ in range(R)]
    vcs = [inp["v_cache"].to(device) for _ in range(R)]
    q = inp["q"].to(device)
    bt = inp["block_tables"].to(device)
    cl = inp["context_lens"].to(device)
    kn, vn, sm = inp["k_new"].to(device), inp["v_new"].to(device), inp["slot_mapping"].to(device)
    out = torch.empty_like(q)
    ws_bytes = B.paged_decode_workspace_size(Bn, Hq, Hkv, D, max_len)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=device)  # counters start at 0

    def step(r):
        B.paged_decode_step(out, q, kn, vn, sm, kcs[r], vcs[r], bt, cl, max_len, scale, workspace=ws)

    def decode_only(r):
        B.paged_decode_attention(out, q, kcs[r], vcs[r], bt, cl, max_len, scale, workspace=ws)

    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i % R)
            decode_only(i % R)
    torch.cuda.synchronize()
    assert B.pkv_device_errors() == 0

    def graphs_for(fn):
        full = torch.cuda.CUDAGraph()
        with torch.cuda.graph(full, stream=stream):
            for r in range(R):
                fn(r)
        rem = args.steps % R
        part = None
        if rem:
            part = torch.cuda.CUDAGraph()
            with torch.cuda.graph(part, stream=stream):
                for r in range(rem):
                    fn(r)
        return full, part

    def timed(full, part) -> float:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(args.steps // R):
                full.replay()
            if part is not None:
                part.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return e0.elapsed_time(e1) / 1e3  # seconds

    g_step = graphs_for(step)
    g_dec = graphs_for(decode_only)
    for g in (g_step, g_dec):  # warm replays of the graphs themselves
        with torch.cuda.stream(stream):
            g[0].replay()
        torch.cuda.synchronize()

    clocks = ClockSampler(local)
    t_step = timed(*g_step)
    clk_timed = clocks.stop()
    t_dec = timed(*g_dec)

    # Clock record: the timed region above can be far shorter than nvidia-smi's 100 ms
    # sampling period, so the same step graph is also replayed back to back for a window
    # of about 1.5 s (outside the timed region) while the clocks are sampled; its own
    # step time is reported beside the clocks as a cross-check of the timed number.
    def clock_window(full, seconds=1.5):
        sampler = ClockSampler(local)
        time.sleep(0.25)  # let nvidia-smi start before the load
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 0
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            e0.record(stream)
            while time.perf_counter() - t0 < seconds:
                for _ in range(20):
                    full.replay()
                reps += 20
                stream.synchronize()
            e1.record(stream)
        torch.cuda.synchronize()
        c = sampler.stop()
        c["window_s"] = round(time.perf_counter() - t0, 3)
        c["window_us_per_step"] = e0.elapsed_time(e1) * 1e3 / (reps * R)
        c["timed_region_samples"] = clk_timed.get("samples", 0)
        c["timed_region_reasons"] = clk_timed.get("reasons", [])
        return c

    clk = clock_window(g_step[0])

    # spread of the step time: 200 replays of the R-step graph, each timed by its own
    # events on the stream (outside the timed region above)
    def spread(full, n=200):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        with torch.cuda.stream(stream):
            evs[0].record(stream)
            for i in range(n):
                full.replay()
                evs[i + 1].record(stream)
        torch.cuda.synchronize()
        per = sorted(evs[i].elapsed_time(evs[i + 1]) * 1e3 / R for i in range(n))
        pick = lambda f: per[min(n - 1, int(f * n))]
        return {"p10_us": pick(0.1), "p50_us": pick(0.5), "p90_us": pick(0.9), "samples": n,
                "steps_per_sample": R}

    step_spread = spread(g_step[0])
    t_step_max = reduce_max(t_step, world, device)
    bytes_all = reduce_sum(nb["step"] * args.steps, world, device)
    value = bytes_all / t_step_max / 1e9
    us_step = t_step_max / args.steps * 1e6
    dec_s = t_dec / args.steps
    achieved = nb["decode_kernel"] / dec_s / 1e9

    # end to end through the public API: pinned host inputs in, output back, every step.
    # The step's inputs sit in one pinned host buffer and its output in another;
    # paged_decode_step takes them as they are (zero-copy: the kernels read the inputs and
    # write the output over the host link), captured once as a CUDA graph and replayed,
    # then synchronised, each step; the same step run eagerly is reported beside it.  The
    # same step with a host-to-device copy of the inputs before it and a device-to-host
    # copy of out after it (three graph nodes) is measured too, for the breakdown.
    # (256-byte aligned pieces of one buffer: one copy in the copy-node form)
    names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")
    offs, total = [], 0
    for k in names:
        offs.append(total)
        total += -(-inp[k].numel() * inp[k].element_size() // 256) * 256
    stage_h = torch.empty(total, dtype=torch.uint8).pin_memory()
    stage_d = torch.empty(total, dtype=torch.uint8, device=device)

    def view(buf, k, o):
        t = inp[k]
        n = t.numel() * t.element_size()
        return buf[o:o + n].view(t.dtype).view(t.shape)

    for k, o in zip(names, offs):
        view(stage_h, k, o).copy_(inp[k])
    dq, dkn, dvn, dsm, dbt, dcl = (view(stage_d, k, o) for k, o in zip(names, offs))
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(inp[k].numel() * inp[k].element_size() for k in names)
    d2h = out_h.numel() * out_h.element_size()
    e2e_steps = max(20, min(args.steps, 2000))

    hq, hkn, hvn, hsm, hbt, hcl = (view(stage_h, k, o) for k, o in zip(names, offs))

    def e2e_body(r):  # zero-copy
        B.paged_decode_step(out_h, hq, hkn, hvn, hsm, kcs[r], vcs[r], hbt, hcl, max_len, scale,
                            workspace=ws)

    def copy_body(r):  # copy nodes
        stage_d.copy_(stage_h, non_blocking=True)
        B.paged_decode_step(out, dq, dkn, dvn, dsm, kcs[r], vcs[r], dbt, dcl, max_len, scale,
                            workspace=ws)
        out_h.copy_(out, non_blocking=True)

    def time_e2e(run) -> float:
        with torch.cuda.stream(stream):
            for i in range(3):
                run(i % R)
                stream.synchronize()
            barrier(world)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(e2e_steps):
                run(i % R)
                stream.synchronize()  # the host reads the step's output
            e1.record(stream)
        torch.cuda.synchronize()
        return reduce_max(e0.elapsed_time(e1) / 1e3 / e2e_steps, world, device)

    def graphs_of(body):
        gs = []
        for r in range(R):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                body(r)
            gs.append(gr)
        return gs

    e2e_graphs = graphs_of(e2e_body)
    t_e2e = time_e2e(lambda r: e2e_graphs[r].replay())
    t_e2e_eager = time_e2e(e2e_body)
    e2e_value = reduce_sum(nb["step"], world, device) / t_e2e / 1e9
    copy_graphs = graphs_of(copy_body)
    t_copy_e2e = time_e2e(lambda r: copy_graphs[r].replay())

    def replays_us(gs, n=200) -> float:  # device time per step, replays back to back
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for i in range(R):
                gs[i].replay()
            e0.record(stream)
            for i in range(n):
                gs[i % R].replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / n

    zc_step_us = replays_us(e2e_graphs)

    # Where the end-to-end time goes: the device time of the two copies (each measured
    # as 20 copies in one graph, back to back), the device time of the step (the timed
    # region above), the step alone replayed and synchronised per step (no copies), and
    # the rest -- graph launch, host synchronise and the gaps between -- as the remainder.
    def copies_us(fn, n=20) -> float:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for _ in range(n):
                fn()
        with torch.cuda.stream(stream):
            gr.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(10):
                gr.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (10 * n)

    h2d_us = copies_us(lambda: stage_d.copy_(stage_h, non_blocking=True))
    d2h_us = copies_us(lambda: out_h.copy_(out, non_blocking=True))
    step_graphs = []
    for r in range(R):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            step(r)
        step_graphs.append(gr)
    t_step_sync = time_e2e(lambda r: step_graphs[r].replay())
    breakdown = {"zero_copy_step_us": zc_step_us,
                 "launch_sync_us": t_e2e * 1e6 - zc_step_us,
                 "step_us": us_step,
                 "step_alone_replayed_and_synchronised_us": t_step_sync * 1e6,
                 "copy_nodes_e2e_us": t_copy_e2e * 1e6,
                 "copy_nodes_h2d_us": h2d_us, "copy_nodes_d2h_us": d2h_us,
                 "copy_nodes_launch_sync_us": t_copy_e2e * 1e6 - (h2d_us + us_step + d2h_us)}

    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or 6800.0
    traffic = recorded_traffic(args.workload)
    launches_per_step = 2  # kv_write_kernel + the fused decode (one launch, merge included)
    decode_name = {B.PATH_PARTITIONS: "decode_kernel (one CTA per partition, merge by the last)",
                   B.PATH_CLUSTER: "decode_kernel (partitions of a unit in one cluster, DSMEM merge)",
                   B.PATH_PERSISTENT: "decode_persistent_kernel (work items, longest first)"}[path]

    if rank != 0:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
        return
    cpu = time_oracle(inp, budget_s=args.cpu_budget) if (world == 1 and args.cpu_budget > 0) else None
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": us_step / 1e3, "us_per_step": us_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_dict(w, inp, args, world),
        "hbm_frac_of_peak": value / peak,
        "spread": step_spread,
        "plan": {"partition_tokens": P, "n_parts": math.ceil(max_len / P), "path": path,
                 "pool_copies": R},
        "roofline": {"bound": "hbm", "kernel": decode_name,
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_src} hbm_gbs (copy, burst)",
                     "bytes_per_launch": nb["decode_kernel"], "us_per_launch": dec_s * 1e6,
                     "traffic": traffic},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "us_per_step": t_e2e * 1e6,
                "how": "paged_decode_step on pinned host inputs and a pinned host output "
                       "(zero-copy: the kernels read and write them over the host link), one CUDA "
                       "graph replayed and synchronised per step; breakdown copy_nodes_*: the same "
                       "step with one H2D copy of the inputs and one D2H copy of out as graph nodes",
                "eager_us_per_step": t_e2e_eager * 1e6, "breakdown": breakdown},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


# ----------------------------------------------------------------------------- other kernels
def run_kernel(args, w) -> None:
    """Times one of the other kernels on the workload's shapes (graph replays, rotating
    pool copies, CUDA events) and prints one JSON line for it."""
    import itertools

    from paged_kv_decode_mapping_gb300 import binding as B

    device = torch.device("cuda", 0)
    inp = W.make_inputs(w)
    Bn, Hq, D = inp["q"].shape
    NB, Hkv, BS, _ = inp["k_cache"].shape
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    R = max(2, math.ceil(3 * l2 / (2 * inp["k_cache"].numel() * 2)))
    kcs = [inp["k_cache"].to(device) for _ in range(R)]
    vcs = [inp["v_cache"].to(device) for _ in range(R)]
    bt, cl = inp["block_tables"].to(device), inp["context_lens"].to(device)
    gen = torch.Generator().manual_seed(w.seed + 1)
    peaks = measured_peaks()
    line = {"n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "data": "synthetic",
            "dtype": "bf16", "vs_baseline": None, "scaling": "weak",
            "config": config_dict(w, inp, args, 1)}
    if args.kernel == "prefill":
        lens = inp["context_lens"].long()
        chunks = torch.clamp(lens, max=args.chunk)
        qs = torch.tensor([0] + list(itertools.accumulate(chunks.tolist())), dtype=torch.int32)
        nq = int(qs[-1])
        q = torch.randn(nq, Hq, D, generator=gen).to(torch.bfloat16).to(device)
        out = torch.empty_like(q)
        qsd = qs.to(device)
        # useful flops: each query at position p does (p+1) keys x (QK + PV) x 2 flops x D
        keys = sum(int(L * n - n * (n - 1) // 2) for L, n in zip(lens.tolist(), chunks.tolist()))
        flops = keys * Hq * D * 4

        def fn(r):
            B.paged_prefill_attention(out, q, kcs[r], vcs[r], bt, cl, inp["max_context_len"], qsd,
                                      int(chunks.max()), inp["scale"])
        unit, per = "TFLOP/s", flops / 1e12
        bound, peak = "tensor", peaks.get("bf16_tflops") or 1900.0
        metric = f"paged prefill attention (last min(L, {args.chunk}) tokens of each sequence) TFLOP/s"
    elif args.kernel == "rope_step":
        nb = algorithmic_bytes(inp)
        kn, vn = inp["k_new"].to(device), inp["v_new"].to(device)
        sm = inp["slot_mapping"].to(device)
        qd = inp["q"].to(device)  # rotated in place by every call
        out = torch.empty_like(qd)
        pos = (inp["context_lens"].long() - 1).clamp(min=0).to(device)
        maxpos = int(inp["max_context_len"]) + 1
        half = D // 2
        inv = 10000.0 ** (-torch.arange(half, dtype=torch.float64) * 2.0 / D)
        ang = torch.arange(maxpos, dtype=torch.float64)[:, None] * inv[None, :]
        cs = torch.cat([ang.cos(), ang.sin()], 1).float().to(device)
        ws = torch.zeros(max(B.paged_decode_workspace_size(Bn, Hq, Hkv, D, inp["max_context_len"]), 16),
                         dtype=torch.uint8, device=device)
        # the step's bytes plus the in-place q rotation (read + write) and two table rows a token
        nbytes = nb["step"] + Bn * Hq * D * 2 * 2 + Bn * D * 4 * 2

        def fn(r):
            B.paged_decode_step_rope(out, qd, kn, vn, sm, pos, cs, kcs[r], vcs[r], bt, cl,
                                     inp["max_context_len"], inp["scale"], workspace=ws)
        unit, per = "GB/s", nbytes / 1e9
        bound, peak = "hbm", peaks.get("hbm_gbs") or 6800.0
        metric = "decode step with RoPE (rotary write + fused decode) GB/s"
    elif args.kernel == "split":
        nb = algorithmic_bytes(inp)
        P = args.partition
        n = math.ceil(inp["max_context_len"] / P)
        qd = inp["q"].to(device)
        o_part = torch.empty(Bn, Hq, n, D, device=device)
        lse = torch.empty(Bn, Hq, n, device=device)
        out = torch.empty_like(qd)

        def fn(r):
            B.paged_decode_split(o_part, lse, qd, kcs[r], vcs[r], bt, cl, inp["max_context_len"],
                                 inp["scale"], P)
            B.paged_decode_combine(out, o_part, lse, cl, inp["max_context_len"], P)
        unit, per = "GB/s", nb["decode_kernel"] / 1e9
        bound, peak = "hbm", peaks.get("hbm_gbs") or 6800.0
        metric = f"decode attention as paged_decode_split (P={P}) + paged_decode_combine GB/s"
    else:  # rope_write
        T = Bn
        kn = torch.randn(T, Hkv, D, generator=gen).to(torch.bfloat16).to(device)
        vn = torch.randn(T, Hkv, D, generator=gen).to(torch.bfloat16).to(device)
        q = inp["q"].to(device)
        sm = inp["slot_mapping"][:T].to(device) if inp["slot_mapping"].numel() >= T else \
            torch.arange(T, dtype=torch.int64, device=device)
        pos = (inp["context_lens"].long() - 1).clamp(min=0).to(device)
        maxpos = int(inp["max_context_len"]) + 1
        half = D // 2
        inv = 10000.0 ** (-torch.arange(half, dtype=torch.float64) * 2.0 / D)
        ang = torch.arange(maxpos, dtype=torch.float64)[:, None] * inv[None, :]
        cs = torch.cat([ang.cos(), ang.sin()], 1).float().to(device)
        nbytes = T * (Hkv * D * 2 * 4 + Hq * D * 2 * 2 + 16 + D * 4 * 2)

        def fn(r):
            B.paged_kv_write_rope(kn, vn, sm, pos, cs, kcs[r], vcs[r], q=q)
        unit, per = "GB/s", nbytes / 1e9
        bound, peak = "hbm", peaks.get("hbm_gbs") or 6800.0
        metric = "fused RoPE + slot write GB/s"
    stream = torch.cuda.Stream(device)
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            fn(i % R)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for r in range(R):
            fn(r)
    reps = max(1, args.steps // R)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(0)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    clk_timed = clocks.stop()
    t = e0.elapsed_time(e1) / 1e3 / (reps * R)
    value = per / t
    # Clock record: the timed region can be shorter than nvidia-smi's sampling period, so
    # the same graph is replayed back to back for about 1.5 s more (outside the timed
    # region) while the clocks are sampled; that window's own time per call is reported
    # beside them as a cross-check.
    sampler = ClockSampler(0)
    time.sleep(0.25)  # let nvidia-smi start before the load
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wreps, t0 = 0, time.perf_counter()
    with torch.cuda.stream(stream):
        w0.record(stream)
        while time.perf_counter() - t0 < 1.5:
            for _ in range(20):
                g.replay()
            wreps += 20
            stream.synchronize()
        w1.record(stream)
    torch.cuda.synchronize()
    clk = sampler.stop()
    clk["window_s"] = round(time.perf_counter() - t0, 3)
    clk["window_ms_per_call"] = w0.elapsed_time(w1) / (wreps * R)
    clk["timed_region_samples"] = clk_timed.get("samples", 0)
    clk["timed_region_reasons"] = clk_timed.get("reasons", [])
    assert B.pkv_device_errors() == 0
    line.update({"metric": metric, "value": value, "unit": unit, "ms_per_step": t * 1e3,
                 "steps": reps * R, "higher_is_better": True,
                 "roofline": {"bound": bound, "achieved": value, "peak": peak, "unit": unit,
                              "frac": value / peak, "traffic": None},
                 "gpu_launches": (2 if args.kernel in ("rope_step", "split") else 1) * reps * R,
                 "clocks": clk})
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=3, choices=sorted(W.WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle time for the cpu_baseline object (0: skip)")
    ap.add_argument("--kernel", choices=["step", "prefill", "rope_write", "rope_step", "split"],
                    default="step",
                    help="step: the decode step (the benchmark line); others time one kernel; "
                         "split: paged_decode_split + paged_decode_combine at --partition")
    ap.add_argument("--chunk", type=int, default=512, help="prefill: query tokens per sequence")
    ap.add_argument("--consumer", choices=["tensor", "fma"], default="tensor",
                    help="arithmetic of the partition decode kernel's consumer warps")
    ap.add_argument("--partition", type=int, default=1024,
                    help="split: partition size in tokens (a multiple of 64)")
    args = ap.parse_args()
    w = W.WORKLOADS[args.workload]
    if args.consumer != "tensor":
        from paged_kv_decode_mapping_gb300 import binding as B

        B.pkv_set_decode_consumer(B.CONSUMER_FMA)
    if args.kernel != "step":
        run_kernel(args, w)
    elif args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
