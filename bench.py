"""Benchmark of the MLA tree-verify path on GB300.

One step = one pass of the whole verify path on one batch of seeded
synthetic input, through one C-ABI call (mla_verify_attention_paged): the
split-KV partial kernel, which reads each key's pool slot from the page
table and builds the tree masks as it stages rows (the index build fused
in), and the log-sum-exp combine, on one stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C]
                    [--impl ours|reference] [--no-extras] [--next-rows ...]

The headline workload is the batched mixed verify (batch 8, 64 heads,
prefix lengths uniform in [1024, 131072], 16-node random trees, nsplit 64,
a 1.2M-slot pool): the largest of the five workloads on one GPU. The line
also carries, for every other workload, the same timings, and for the mid
and long workloads the roofline block, the end-to-end time and a CPU-oracle
sample. Inputs are resident in HBM when the timed region starts; each timed
step is preceded (outside its events) by a write of a buffer larger than
L2, so every step reads the KV rows from HBM.

--impl reference times the CPU fp64 oracle (the only reference that exists
for this method) on the machine's host cores, on a bounded sample of the same
workload.
"""

from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import CONFIGS, make_config  # noqa: E402

METRIC = "MLA tree-verify attention µs/call and KV GB/s vs HBM/tensor roofline (1×GB300)"
UNIT = "us/call"
ROW_BYTES = 576 * 2          # one latent row, bf16
FLOPS_PER_PAIR = 2 * 576 + 2 * 512   # QK^T over 576 dims + PV over 512 dims
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------- workload arithmetic
def workload_name(idx):
    """What a verify workload is, with its sizes (e.g. "long verify: 1 x
    prefix 184728, T=64, H=8, nsplit 64")."""
    c = CONFIGS[idx]
    kind, _, rest = c["prefix"].partition(":")
    prefix = rest if kind == "fixed" else "U[" + rest.replace(":", ", ") + "]"
    return (f"{c['name']} verify: {c['batch']} x prefix {prefix}, T={c['T']}, "
            f"H={c['num_heads']}, nsplit {c['nsplit']}")


def workload_figures(inp):
    """Algorithmic bytes and flops of one verify call (each KV row read once;
    flops count only visible (row, key) pairs)."""
    L = inp.prefix_lens.astype(np.int64)
    T, H, B = inp.T, inp.num_heads, inp.batch
    keys = int(L.sum() + B * T)
    kv_bytes = keys * ROW_BYTES
    q_bytes = B * T * H * ROW_BYTES
    out_bytes = B * T * H * (512 * 2 + 4)
    idx_bytes = keys * 4
    depth = np.zeros((B, T), dtype=np.int64)
    for b in range(B):
        for t in range(T):
            p = int(inp.tree_parent[b, t])
            depth[b, t] = depth[b, p] + 1 if p >= 0 else 0
    vis = (L[:, None] + depth + 1).sum() * H  # visible keys summed over rows
    flops = int(vis) * FLOPS_PER_PAIR
    return dict(keys=keys, kv_bytes=kv_bytes, bytes=kv_bytes + q_bytes + out_bytes + idx_bytes,
                flops=flops, visible_pairs=int(vis), rows=B * T * H)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def roofline_us(fig, peaks):
    t_mem = fig["bytes"] / (peaks["hbm_gbs"] * 1e9) * 1e6
    t_flop = fig["flops"] / (peaks["bf16_tflops"] * 1e12) * 1e6
    return max(t_mem, t_flop), ("tensor" if t_flop > t_mem else "hbm"), t_mem, t_flop


# The partial kernel each committed ncu record was taken on, by its source file.
KERNEL_SOURCES = {"partial_quad_kernel": "partial_quad.cu", "partial_pair_kernel": "partial_pair.cu"}


def _code_only(text):
    """Source text without comments and trailing blanks (a comment edit does
    not change the kernel the counters were taken on)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(kernel="partial_quad_kernel"):
    """Hash of the code of the kernel's source file and the headers it shares."""
    files = (KERNEL_SOURCES[kernel], "partial_kernels.cuh", "tc_ptx.cuh", "common.cuh", "partition.h")
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_speculative_decoding_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name in files:
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(config_idx, kernel):
    """DRAM bytes per launch of the workload's partial kernel from a committed
    ncu summary, if it was taken on that kernel's current source; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    e = t.get(str(config_idx))
    if not e or e.get("kernel") != kernel or kernel not in KERNEL_SOURCES:
        return None
    if e.get("kernel_hash") != kernel_source_hash(e["kernel"]):
        return None
    return e.get("dram_bytes_per_launch")


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id=None):
        self.samples = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in self.samples:
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
            except ValueError:
                continue
            for name, v in zip(names, p[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- distributed helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value, world, backend_device=None):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=backend_device if backend_device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- CPU oracle timing
def time_oracle(inp, target_s=10.0, max_rows=None):
    """Oracle (as it stands) on a bounded row sample; returns (us per full call,
    sample description, threads)."""
    import oracle
    ip, ix, _ = oracle.build_meta(inp)
    threads = oracle.max_threads()
    H, T = inp.num_heads, inp.T
    L = inp.prefix_lens.astype(np.int64)
    depth = np.zeros((inp.batch, T), dtype=np.int64)
    for b in range(inp.batch):
        for t in range(T):
            p = int(inp.tree_parent[b, t])
            depth[b, t] = depth[b, p] + 1 if p >= 0 else 0
    vis_row = np.repeat((L[:, None] + depth + 1).reshape(-1), H)  # visible keys per row
    total_vis = float(vis_row.sum())
    rng = np.random.default_rng(1234)
    order = rng.permutation(inp.num_rows)
    # Calibrate on a few rows, then size the sample to ~target_s.
    n0 = min(len(order), max(threads, 4))
    t0 = time.perf_counter()
    oracle.verify_attention(inp, ip, ix, rows=order[:n0])
    dt0 = time.perf_counter() - t0
    per_vis = dt0 / float(vis_row[order[:n0]].sum())
    want = int(target_s / max(per_vis * float(vis_row.mean()), 1e-9))
    n = max(n0, min(len(order), want if max_rows is None else min(want, max_rows)))
    rows = order[:n]
    t0 = time.perf_counter()
    oracle.verify_attention(inp, ip, ix, rows=rows)
    dt = time.perf_counter() - t0
    us = dt * 1e6 * total_vis / float(vis_row[rows].sum())
    return us, f"{n} of {inp.num_rows} query rows (random), scaled by visible keys", threads, dt


# ----------------------------------------------------------------- GPU arm
class L2Flush:
    """Evicts the inputs from L2 between timed steps: writes a buffer of 4x L2,
    then reads its first 2x L2, so that L2 ends up holding clean lines of
    that buffer only (a write-only flush would leave L2 full of dirty lines,
    whose write-back the next timed kernel would pay for)."""

    DESCRIPTION = ("flushed before every timed step: a 4x L2 buffer written, then 2x L2 of "
                   "it read back, so no input line and no dirty line stays in L2")

    def __init__(self, l2_bytes, dev):
        import torch
        self.l2 = int(l2_bytes)
        self.buf = torch.empty(max(4 * self.l2, 512 << 20), dtype=torch.uint8, device=dev)

    def __call__(self):
        self.buf.zero_()
        self.buf[:2 * self.l2].sum()


def time_steps(fn, flush, steps, warmup, stream):
    """Device time (µs) of each of `steps` calls of fn, L2 flushed before
    every call (outside the events); `warmup` untimed calls first."""
    import torch
    for _ in range(warmup):
        flush()
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        flush()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) * 1e3 for a, b in ev]


def split_times(d, flush, steps, stream):
    """The paged call's two launches timed apart (events between them keep
    the second from starting early, so this is kept out of the timed step)."""
    import torch
    for _ in range(2):
        flush()
        d.partial_paged()
        d.combine()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for e in ev:
        flush()
        e[0].record(stream)
        d.partial_paged()
        e[1].record(stream)
        d.combine()
        e[2].record(stream)
    torch.cuda.synchronize()
    part = statistics.mean(e[0].elapsed_time(e[1]) * 1e3 for e in ev)
    comb = statistics.mean(e[1].elapsed_time(e[2]) * 1e3 for e in ev)
    return part, comb


def graph_time(fn, flush, steps, dev, stream):
    """Median device time of a CUDA-graph replay of fn (the pages' deployment
    mode); fn must launch on the current stream (it is captured on a side
    stream)."""
    import torch
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    # the mean: CUDA events tick in ~2 us steps, which a median of a few replays keeps
    return statistics.mean(time_steps(g.replay, flush, steps, 3, stream))


def e2e_time(d, flush, steps, warmup, stream):
    """End to end through the public API with host buffers: per step the H2D
    copy of that step's inputs from pinned memory (queries, tree, prefix
    lengths, table rows, draft slots; the KV pool and req_to_token are
    resident device state), the verify call, the D2H copy of out and lse,
    and a synchronize, timed on the host clock. A second pass with events
    between the pieces splits the time."""
    import torch
    call = d.bound_step_paged()
    h_in = d.step_in.cpu().pin_memory()
    h_out = d.step_out.cpu().pin_memory()

    def one():
        d.step_in.copy_(h_in, non_blocking=True)
        call()
        h_out.copy_(d.step_out, non_blocking=True)

    walls = []
    for k in range(warmup + steps):
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        one()
        torch.cuda.synchronize()
        if k >= warmup:
            walls.append((time.perf_counter() - t0) * 1e6)
    # breakdown pass (events between the pieces)
    parts = {"h2d": [], "verify": [], "d2h": [], "issue": []}
    for _ in range(steps):
        flush()
        torch.cuda.synchronize()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        t0 = time.perf_counter()
        e[0].record(stream)
        d.step_in.copy_(h_in, non_blocking=True)
        e[1].record(stream)
        call()
        e[2].record(stream)
        h_out.copy_(d.step_out, non_blocking=True)
        e[3].record(stream)
        parts["issue"].append((time.perf_counter() - t0) * 1e6)
        torch.cuda.synchronize()
        parts["h2d"].append(e[0].elapsed_time(e[1]) * 1e3)
        parts["verify"].append(e[1].elapsed_time(e[2]) * 1e3)
        parts["d2h"].append(e[2].elapsed_time(e[3]) * 1e3)
    wall = statistics.mean(walls)
    br = {k: round(statistics.mean(v), 2) for k, v in parts.items()}
    br["host_and_sync"] = round(wall - br["h2d"] - br["verify"] - br["d2h"], 2)
    br["note"] = ("h2d / verify / d2h: device time between events (each after a flush); "
                  "issue: host time to enqueue the three calls; host_and_sync: the rest of "
                  "the wall time (launch latency before the first copy, gaps, synchronize)")
    return wall, int(h_in.numel()), int(h_out.numel()), br


def roofline_block(fig, peaks, peak_src, part_us, traffic, kernel):
    """Roofline of the dominant (partial) kernel: algorithmic flops or bytes
    of one launch over its measured device time."""
    roof_us, bound, _, _ = roofline_us(fig, peaks)
    if bound == "tensor":
        achieved, peak, unit = fig["flops"] / (part_us * 1e-6) / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    else:
        achieved, peak, unit = fig["bytes"] / (part_us * 1e-6) / 1e9, peaks["hbm_gbs"], "GB/s"
    return {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic, "kernel": kernel,
            "peak_source": f"{peak_src} (burst)",
            "frac_of_sustained": (round(achieved / peaks["bf16_tflops_sustained"], 4)
                                  if bound == "tensor" and "bf16_tflops_sustained" in peaks
                                  else None),
            "algorithmic": {"bytes": fig["bytes"], "flops": fig["flops"]}}


def default_kernel(inp):
    return "partial_pair_kernel" if inp.T * inp.num_heads <= 128 else "partial_quad_kernel"


def measure_workload(idx, inp, mv, dev, flush, peaks, peak_src, steps, warmup, full):
    """One workload: the paged verify call (the benchmark's step) timed with
    events after an L2 flush, its graph replay, the list-form call (builder +
    mla_verify_attention, the boundary's own signature), the per-kernel
    split; with `full`, also the roofline block, the end-to-end time and a
    CPU-oracle sample."""
    import torch
    stream = torch.cuda.current_stream()
    fig = workload_figures(inp)
    d = mv.to_device(inp, device=dev)
    call = d.bound_step_paged()
    us = statistics.mean(time_steps(call, flush, steps, warmup, stream))
    part, comb = split_times(d, flush, min(steps, 10), stream)
    gus = graph_time(d.step_paged, flush, min(steps, 10), dev, stream)
    lus = statistics.mean(time_steps(lambda: (d.build(), d.attention(use_anc=False)), flush,
                                     min(steps, 10), 3, stream))
    roof, bound, _, _ = roofline_us(fig, peaks)
    res = {"us": round(us, 3), "graph_us": round(gus, 3), "list_form_us": round(lus, 3),
           "breakdown_us": {"build": "fused into the partial kernel", "partial": round(part, 3),
                            "combine": round(comb, 3)},
           "roofline_us": round(roof, 3), "frac": round(roof / us, 4), "bound": bound,
           "kv_gbps": round(fig["kv_bytes"] / (us * 1e-6) / 1e9, 1)}
    if full:
        kernel = default_kernel(inp)
        res["roofline"] = roofline_block(fig, peaks, peak_src, part, ncu_traffic(idx, kernel), kernel)
        wall, bi, bo, br = e2e_time(d, flush, steps, 3, stream)
        res["e2e"] = {"value": round(wall, 3), "unit": UNIT, "h2d_bytes_per_step": bi,
                      "d2h_bytes_per_step": bo, "breakdown_us": br}
    res["status_ok"] = int(d.status.item()) == 0
    del d, call
    torch.cuda.empty_cache()
    return res


def run_ours(args):
    import torch

    import mla_speculative_decoding_gb300 as mv

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    mv.mla_verify_init(local)
    peaks, peak_src = load_peaks()

    idx = args.config
    t0 = time.time()
    inp = make_config(idx)
    log(f"[bench] config {idx} generated in {time.time() - t0:.1f}s")
    fig = workload_figures(inp)
    d = mv.to_device(inp, device=dev)
    stream = torch.cuda.current_stream()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    flush = L2Flush(l2, dev)

    # One step = the whole verify path through one C-ABI call: the paged
    # entry point, whose partial kernels fetch each key's pool slot from the
    # page table as they stage rows (the index build fused in) and build the
    # tree masks in-kernel, then the combine: two launches.
    step_call = d.bound_step_paged()

    for _ in range(args.warmup):
        flush()
        step_call()
    torch.cuda.synchronize()
    assert int(d.status.item()) == 0, "device status word set during warm-up"

    gpu_id = None
    try:
        gpu_id = str(props.uuid)
        if not gpu_id.startswith("GPU-"):
            gpu_id = "GPU-" + gpu_id
    except Exception:
        gpu_id = None
    clocks = ClockSampler(gpu_id)
    time.sleep(0.3)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for k in range(args.steps):
        flush()
        evs[k][0].record(stream)
        step_call()
        evs[k][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    step_us = [evs[k][0].elapsed_time(evs[k][1]) * 1e3 for k in range(args.steps)]
    mean_step = statistics.mean(step_us)
    mean_step_max = max_over_ranks(mean_step, world, dev if world > 1 else None)
    value = mean_step_max / world  # whole-job: calls of all ranks over the slowest rank's time
    assert int(d.status.item()) == 0

    part_us, comb_us = split_times(d, flush, args.steps, stream)
    graph_us = None
    try:
        graph_us = graph_time(d.step_paged, flush, args.steps, dev, stream)
    except Exception as e:  # reported, not hidden
        log(f"[bench] graph replay failed: {e!r}")
    list_us = statistics.mean(time_steps(lambda: (d.build(), d.attention(use_anc=False)), flush,
                                         args.steps, 3, stream))
    e2e_wall, h2d, d2h, e2e_br = e2e_time(d, flush, args.steps, args.warmup, stream)
    e2e = max_over_ranks(e2e_wall, world, dev if world > 1 else None) / world
    assert int(d.status.item()) == 0
    del step_call, d
    torch.cuda.empty_cache()

    roof_us, bound, t_mem, t_flop = roofline_us(fig, peaks)
    kernel = default_kernel(inp)
    result = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(mean_step_max / 1e3, 6),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 q and latent KV; random trees; scattered slots)",
        "config": {"workload": workload_name(idx), "batch": inp.batch,
                   "heads": inp.num_heads, "prefix_lens": [int(x) for x in inp.prefix_lens][:8],
                   "T": inp.T, "nsplit": inp.nsplit, "pool_slots": inp.pool_slots,
                   "call": "mla_verify_attention_paged (partial + combine, two launches)",
                   "l2": L2Flush.DESCRIPTION,
                   "parallelism": "replicas" if world > 1 else "single-gpu"},
        "kv_gbps": round(fig["kv_bytes"] / (value * 1e-6) / 1e9, 1),
        "roofline_frac": round(roof_us / value, 4),
        "roofline_us": round(roof_us, 3),
        "breakdown_us": {"build": "fused into the partial kernel", "partial": round(part_us, 3),
                         "combine": round(comb_us, 3)},
        "graph_us": None if graph_us is None else round(graph_us, 3),
        "list_form_us": round(list_us, 3),
        "roofline": roofline_block(fig, peaks, peak_src, part_us, ncu_traffic(idx, kernel), kernel),
        "e2e": {"value": round(e2e, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "breakdown_us": e2e_br},
        "gpu_launches": 2 * args.steps,  # partial + combine per step
        "clocks": clk,
        "wall_s_timed_region": round(wall, 4),
    }

    if args.extras and rank == 0:
        per = {}
        for j in sorted(CONFIGS):
            if j == idx:
                continue
            try:
                per[str(j)] = measure_workload(j, make_config(j), mv, dev, flush, peaks, peak_src,
                                               10, 3, full=j >= 3)
            except Exception as e:
                per[str(j)] = {"error": repr(e)}
        per[str(idx)] = {"us": result["value"], "graph_us": result["graph_us"],
                         "list_form_us": result["list_form_us"], "roofline_us": round(roof_us, 3),
                         "frac": result["roofline_frac"], "bound": bound,
                         "kv_gbps": result["kv_gbps"], "headline": True}
        # the mid workload once more with its keys in contiguous slots (the
        # defragmented placement), to compare gather cost
        try:
            per["3c"] = measure_workload(3, make_config(3, placement="contiguous"), mv, dev, flush,
                                         peaks, peak_src, 10, 3, full=False)
        except Exception as e:
            per["3c"] = {"error": repr(e)}
        result["per_config"] = {k: per[k] for k in sorted(per)}
        try:
            result["next_rows"] = measure_next_rows(mv, dev, flush, peaks)
        except Exception as e:
            result["next_rows"] = {"error": repr(e)}

    if rank == 0 and world == 1 and args.cpu_baseline:
        us, sample, threads, dt = time_oracle(inp, target_s=args.cpu_seconds)
        result["cpu_baseline"] = {"value": round(us, 1), "unit": UNIT, "cores": threads,
                                  "kind": "oracle", "sample": sample,
                                  "sample_seconds": round(dt, 2)}
        if args.extras:
            for j in (3, 4):
                if j == idx or str(j) not in result.get("per_config", {}):
                    continue
                us, sample, threads, dt = time_oracle(make_config(j), target_s=3.0)
                result["per_config"][str(j)]["cpu_baseline"] = {
                    "value": round(us, 1), "unit": UNIT, "cores": threads, "kind": "oracle",
                    "sample": sample, "sample_seconds": round(dt, 2)}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def _time_us(fn, flush, steps=10, warm=3):
    """Mean device time of fn() over `steps` runs, L2 flushed before each
    (outside the events)."""
    import torch
    stream = torch.cuda.current_stream()
    for _ in range(warm):
        flush()
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for k in range(steps):
        flush()
        ev[k][0].record(stream)
        fn()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) * 1e3 for a, b in ev)


NEXT_ROWS = ("sparse_decode", "kv_relocate", "tree_accept", "fp8_indexer")


def measure_next_rows(mv, dev, flush, peaks, which=NEXT_ROWS):
    """The steps beside the verify attention, each on a workload of the pages'
    shape: µs per call and the fraction of its roofline (algorithmic bytes at
    the measured HBM bandwidth, flops at the measured bf16 peak)."""
    import torch
    from workloads import (make_accept_inputs, make_indexer_inputs, make_relocate_inputs,
                           make_sparse_decode)
    hbm = peaks["hbm_gbs"] * 1e9
    res = {}
    st = torch.zeros(1, dtype=torch.int32, device=dev)

    if "sparse_decode" in which:
        # f1: sparse-MLA decode (16 requests x 64 heads over 512 top-k slots + self)
        inp = make_sparse_decode()
        fig = workload_figures(inp)
        d = mv.to_device(inp, device=dev)
        us = _time_us(d.step_paged, flush)
        roof, bound, _, _ = roofline_us(fig, peaks)
        res["sparse_decode"] = {"workload": "batch 16, H=64, top-k 512 + self, nsplit 8",
                                "us": round(us, 2), "roofline_us": round(roof, 3),
                                "frac": round(roof / us, 4), "bound": bound,
                                "status_ok": int(d.status.item()) == 0}
        del d

    if "kv_relocate" in which:
        # f2: KV relocation, 8 requests x 16384 scattered rows into contiguous ranges, one call
        x = make_relocate_inputs(batch=8, prefix="fixed:16384", pool_slots=600_000, seed=11,
                                 poison=False)
        pool = torch.from_numpy(x.kv_pool.view(np.int16)).to(dev).view(torch.bfloat16)
        r2t0 = torch.from_numpy(x.req_to_token).to(dev)
        r2t = r2t0.clone()
        rpi = torch.from_numpy(x.req_pool_indices).to(dev)
        lens = torch.from_numpy(x.prefix_lens).to(dev)
        dst = torch.from_numpy(x.dst_start).to(dev)
        prog = torch.zeros(8, dtype=torch.int32, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)

        def reloc():
            r2t.copy_(r2t0)
            prog.zero_()
            mv.mla_kv_relocate(pool, r2t, rpi, lens, dst, prog, 16384, st)
        t_copy = _time_us(lambda: (r2t.copy_(r2t0), prog.zero_()), flush)
        us = _time_us(reloc, flush) - t_copy
        rows = 8 * 16384
        nbytes = rows * (2 * 1152 + 8)
        res["kv_relocate"] = {"workload": "8 x 16384 scattered rows, one call", "us": round(us, 2),
                              "gbps": round(nbytes / (us * 1e-6) / 1e9, 1),
                              "roofline_us": round(nbytes / hbm * 1e6, 2),
                              "frac": round(nbytes / hbm * 1e6 / us, 4), "bound": "hbm",
                              "status_ok": int(st.item()) == 0}
        del pool

    if "tree_accept" in which:
        # f3: greedy acceptance, 64 requests x 64-node trees
        a = make_accept_inputs(batch=64, T=64, seed=12)
        tens = [torch.from_numpy(v).to(dev) for v in (a.tree_parent, a.draft_tokens, a.target_argmax,
                                                      a.out_cache_loc)]
        outs = [torch.zeros(64, dtype=torch.int32, device=dev)] + \
            [torch.zeros(64, 64, dtype=torch.int32, device=dev) for _ in range(3)]
        us = _time_us(lambda: mv.mla_tree_accept(*tens, *outs, st), flush)
        res["tree_accept"] = {"workload": "64 requests x 64-node trees", "us": round(us, 2),
                              "bound": "latency"}

    if "fp8_indexer" in which:
        # f4: fp8 indexer, 16 requests x 32768 positions (512 pages) over a 4097-entry table
        ix = make_indexer_inputs(batch=16, num_heads=64, seq_lens="fixed:32768", max_pages=4097,
                                 seed=13)
        q = torch.from_numpy(ix.q).to(dev)
        w = torch.from_numpy(ix.weights).to(dev)
        kv = torch.from_numpy(ix.kv_blocks).to(dev)
        bt = torch.from_numpy(ix.block_table).to(dev)
        sl = torch.from_numpy(ix.seq_lens).to(dev)
        out = torch.empty(16, 4097 * 64, dtype=torch.float32, device=dev)
        us = _time_us(lambda: mv.mla_fp8_indexer_logits(q, w, kv, bt, sl, out, st), flush)
        pages = int(((ix.seq_lens + 63) // 64).sum())
        nbytes = pages * 8448 + q.numel() + w.numel() * 4 + out.numel() * 4 + bt.numel() * 4
        flops = 2 * int(ix.seq_lens.sum()) * 64 * 128
        t_mem = nbytes / hbm * 1e6
        t_flop = flops / (peaks["bf16_tflops"] * 2 * 1e12) * 1e6   # fp8 tensor rate = 2 x bf16
        roof = max(t_mem, t_flop)
        res["fp8_indexer"] = {"workload": "16 x 32768 positions, H=64, 4097-page table",
                              "us": round(us, 2), "roofline_us": round(roof, 2),
                              "frac": round(roof / us, 4), "bound": "hbm" if t_mem >= t_flop else "tensor",
                              "gflops": round(flops / (us * 1e-6) / 1e9, 1),
                              "status_ok": int(st.item()) == 0}
        del kv, out
    torch.cuda.empty_cache()
    return res


def run_next_rows(which):
    import torch

    import mla_speculative_decoding_gb300 as mv
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    mv.mla_verify_init(0)
    peaks, _ = load_peaks()
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20))
    flush = L2Flush(l2, dev)
    print(json.dumps(measure_next_rows(mv, dev, flush, peaks, which)), flush=True)


# ----------------------------------------------------------------- reference arm
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return  # the CPU oracle runs once, on rank 0
    idx = args.config
    inp = make_config(idx)
    per_step = []
    sample = threads = None
    # Each step: the oracle on a bounded random row sample (~cpu_step_s of CPU
    # work), scaled to the whole call by visible keys.
    for k in range(args.warmup + args.steps):
        us, sample, threads, _ = time_oracle(inp, target_s=args.cpu_step_s)
        if k >= args.warmup:
            per_step.append(us)
    value = statistics.mean(per_step)
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(value / 1e3, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(idx), "batch": inp.batch,
                   "heads": inp.num_heads, "T": inp.T, "nsplit": inp.nsplit},
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=5, choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extras", dest="extras", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-step-s", type=float, default=4.0)
    ap.add_argument("--next-rows", nargs="*", choices=NEXT_ROWS, default=None,
                    help="time only these steps beside the verify attention (all if none named) "
                         "and print their JSON instead of the bench line")
    args = ap.parse_args()
    if args.next_rows is not None:
        run_next_rows(args.next_rows or NEXT_ROWS)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
