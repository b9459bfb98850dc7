"""Benchmark of the MLA tree-verify path on GB300.

One step = one pass of the whole verify path on one batch of seeded
synthetic input: the index/tree-mask builder, the split-KV partial kernel
and the log-sum-exp combine, launched through the C ABI on one stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C]
                    [--impl ours|reference] [--no-extras]

The headline workload is the long-context verify (batch 1, 8 heads,
prefix 184,728 keys, 64-node random tree, nsplit 64): the pages' longest
measured context. Inputs are resident in HBM when the timed region starts;
each timed step is preceded (outside its events) by a write of a buffer
larger than L2, so every step reads the KV rows from HBM.

--impl reference times the CPU fp64 oracle (the only reference that exists
for this method) on the machine's host cores, on a bounded sample of the same
workload.
"""

from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
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
    files = (KERNEL_SOURCES[kernel], "partial_tc.cuh", "tc_ptx.cuh", "common.cuh", "partition.h")
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_speculative_decoding_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name in files:
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(config_idx):
    """DRAM bytes per launch of the partial kernel from a committed ncu summary,
    if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    e = t.get(str(config_idx))
    if not e or e.get("kernel") not in KERNEL_SOURCES:
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
    # tree masks in-kernel, then the combine. (With --simt: the builder and
    # the CUDA-core partial kernel, through the combined key list.)
    def step_call():
        if args.flags:
            d.build()
            d.partial(flags=args.flags)
            d.combine()
        else:
            d.step_paged()

    def one_step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        step_call()
        if ev is not None:
            ev[1].record(stream)

    # The same path with events between its launches, for the per-kernel
    # breakdown (kept out of the timed step: an event between two kernels
    # keeps the second from starting early).
    def split_step(ev):
        ev[0].record(stream)
        if args.flags:
            d.build()
            ev[1].record(stream)
            d.partial(flags=args.flags)
        else:
            ev[1].record(stream)
            d.partial_paged()
        ev[2].record(stream)
        d.combine()
        ev[3].record(stream)

    for _ in range(args.warmup):
        flush()
        one_step()
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
        one_step(evs[k])
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    step_us = [evs[k][0].elapsed_time(evs[k][1]) * 1e3 for k in range(args.steps)]
    sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush()
        split_step(sevs[k])
    torch.cuda.synchronize()
    part_us = [sevs[k][1].elapsed_time(sevs[k][2]) * 1e3 for k in range(args.steps)]
    build_us = [sevs[k][0].elapsed_time(sevs[k][1]) * 1e3 for k in range(args.steps)]
    comb_us = [sevs[k][2].elapsed_time(sevs[k][3]) * 1e3 for k in range(args.steps)]
    mean_step = statistics.mean(step_us)
    mean_step_max = max_over_ranks(mean_step, world, dev if world > 1 else None)
    value = mean_step_max / world  # whole-job: calls of all ranks over the slowest rank's time

    # CUDA-graph replay of the same step (deployment mode on the pages).
    graph_us = None
    try:
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            step_call()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            step_call()
        ge = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for _ in range(3):
            flush()
            g.replay()
        for k in range(args.steps):
            flush()
            ge[k][0].record(stream)
            g.replay()
            ge[k][1].record(stream)
        torch.cuda.synchronize()
        graph_us = statistics.median(a.elapsed_time(b) * 1e3 for a, b in ge)
    except Exception as e:  # reported, not hidden
        log(f"[bench] graph replay failed: {e!r}")

    # End to end through the public API with host buffers: per step, H2D of the
    # step's inputs (queries, tree, prefix lengths, table rows, draft slots) from
    # pinned memory, the verify path, D2H of out and lse. The KV pool and the
    # req_to_token table are resident device state.
    # The step's inputs live in one device buffer (d.step_in) and its outputs
    # in another (d.step_out), so each direction is one copy.
    h_in = d.step_in.cpu().pin_memory()
    h_out = d.step_out.cpu().pin_memory()
    h2d = h_in.numel()
    d2h = h_out.numel()
    e2e_us = []
    for k in range(args.warmup + args.steps):
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        d.step_in.copy_(h_in, non_blocking=True)
        step_call()
        h_out.copy_(d.step_out, non_blocking=True)
        torch.cuda.synchronize()
        if k >= args.warmup:
            e2e_us.append((time.perf_counter() - t0) * 1e6)
    e2e = max_over_ranks(statistics.mean(e2e_us), world, dev if world > 1 else None) / world
    assert int(d.status.item()) == 0

    roof_us, bound, t_mem, t_flop = roofline_us(fig, peaks)
    part_mean = statistics.mean(part_us)
    if bound == "tensor":
        achieved = fig["flops"] / (part_mean * 1e-6) / 1e12
        peak = peaks["bf16_tflops"]
        runit = "TFLOP/s"
    else:
        achieved = fig["bytes"] / (part_mean * 1e-6) / 1e9
        peak = peaks["hbm_gbs"]
        runit = "GB/s"

    result = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(mean_step_max / 1e3, 6),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 q and latent KV; random trees; scattered slots)",
        "config": {"workload": workload_name(idx), "batch": inp.batch,
                   "heads": inp.num_heads, "prefix_lens": [int(x) for x in inp.prefix_lens][:8],
                   "T": inp.T, "nsplit": inp.nsplit, "pool_slots": inp.pool_slots,
                   "l2": L2Flush.DESCRIPTION,
                   "parallelism": "replicas" if world > 1 else "single-gpu",
                   "kernel": "simt" if args.flags else "default"},
        "kv_gbps": round(fig["kv_bytes"] / (value * 1e-6) / 1e9, 1),
        "roofline_frac": round(roof_us / value, 4),
        "roofline_us": round(roof_us, 3),
        "breakdown_us": ({"build": round(statistics.mean(build_us), 3)} if args.flags else
                         {"build": "fused into the partial kernel"}) |
                        {"partial": round(part_mean, 3), "combine": round(statistics.mean(comb_us), 3)},
        "graph_us": None if graph_us is None else round(graph_us, 3),
        "roofline": {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": runit,
                     "frac": round(achieved / peak, 4), "traffic": ncu_traffic(idx),
                     "kernel": "partial", "peak_source": f"{peak_src} (burst)",
                     "algorithmic": {"bytes": fig["bytes"], "flops": fig["flops"]}},
        "e2e": {"value": round(e2e, 3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": (3 if args.flags else 2) * args.steps,  # partial + combine (+ build)
        "clocks": clk,
        "wall_s_timed_region": round(wall, 4),
    }

    if args.extras and rank == 0:
        per = {}
        for j in sorted(CONFIGS):
            if j == idx:
                continue
            try:
                per[j] = measure_config(j, mv, dev, flush, peaks, args)
            except Exception as e:
                per[j] = {"error": repr(e)}
        per[idx] = {"us": round(value, 3), "roofline_us": round(roof_us, 3),
                    "frac": round(roof_us / value, 4), "bound": bound}
        result["per_config"] = {str(k): per[k] for k in sorted(per)}
        # the mid workload once more with its keys in contiguous slots (the
        # defragmented placement), to compare gather cost
        try:
            result["per_config"]["3c"] = measure_config(3, mv, dev, flush, peaks, args,
                                                        placement="contiguous")
        except Exception as e:
            result["per_config"]["3c"] = {"error": repr(e)}
        try:
            result["next_rows"] = measure_next_rows(mv, dev, flush, peaks)
        except Exception as e:
            result["next_rows"] = {"error": repr(e)}

    if rank == 0 and world == 1 and args.cpu_baseline:
        us, sample, threads, dt = time_oracle(inp, target_s=args.cpu_seconds)
        result["cpu_baseline"] = {"value": round(us, 1), "unit": UNIT, "cores": threads,
                                  "kind": "oracle", "sample": sample,
                                  "sample_seconds": round(dt, 2)}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def measure_config(j, mv, dev, flush, peaks, args, steps=10, placement="scattered"):
    import torch
    inp = make_config(j, placement=placement)
    fig = workload_figures(inp)
    d = mv.to_device(inp, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        flush()
        d.step_paged()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for k in range(steps):
        flush()
        ev[k][0].record(stream)
        d.step_paged()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    us = statistics.mean(a.elapsed_time(b) * 1e3 for a, b in ev)
    roof, bound, _, _ = roofline_us(fig, peaks)
    ok = int(d.status.item()) == 0
    del d
    torch.cuda.empty_cache()
    return {"us": round(us, 3), "roofline_us": round(roof, 3), "frac": round(roof / us, 4),
            "bound": bound, "kv_gbps": round(fig["kv_bytes"] / (us * 1e-6) / 1e9, 1),
            "status_ok": ok}


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


# ----------------------------------------------------------------- building-block probes
PROBES = ("mma", "gather", "blocks", "dsmem", "mbar")


def run_probes(which=PROBES):
    """Microbenchmarks of the building blocks the kernels rely on (test-only
    library libmlaselftest.so): 2-SM MMA issue rate, scattered-row gather
    throughput, contiguous 8 KB block streams by copy method, mbarrier
    operation costs and producer/consumer hand-over. Prints one table; not
    part of the bench contract."""
    import ctypes
    import torch
    from mla_speculative_decoding_gb300 import build as mbuild

    lib = ctypes.CDLL(mbuild.build_selftest())
    torch.cuda.set_device(0)
    cyc = torch.zeros(1, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    if "mma" in which:
        _probe_mma(lib, cyc, err)
    if "gather" in which:
        _probe_gather(lib, err)
    if "blocks" in which:
        _probe_blocks(lib, err)
    if "dsmem" in which:
        _probe_dsmem(lib, err)
    if "mbar" in which:
        _probe_mbar(lib, cyc, err)


def _probe_mma(lib, cyc, err):
    import ctypes
    import torch
    # 2-SM MMA (M = 256, K = 16), single accumulator chain, tight issue loop.
    f = lib.mlav_pair_probe
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 + [ctypes.c_void_p] * 3
    g = torch.Generator().manual_seed(1)
    A = torch.randn(256, 64, generator=g).to(torch.bfloat16).cuda()
    addr = torch.zeros(2, dtype=torch.int32, device="cuda")
    print("pair MMA (cta_group::2, M=256, K=16), cycles per MMA; peak = 128 (N=256) / 64 (N=128)")
    for mode, N, label in ((1, 256, "A TMEM, B K-major"), (0, 256, "A smem, B K-major"),
                           (2, 256, "A smem, B MN-major"), (1, 128, "A TMEM, B K-major")):
        Bm = (torch.randn(N, 64, generator=g) if mode in (0, 1) else torch.randn(64, N, generator=g))
        Bm = Bm.to(torch.bfloat16).cuda()
        D = torch.zeros(256, N, dtype=torch.float32, device="cuda")
        row = []
        for var in (0, 2):
            rc = f(A.data_ptr(), Bm.data_ptr(), D.data_ptr(), N, mode, 256, var, addr.data_ptr(),
                   cyc.data_ptr(), err.data_ptr())
            assert rc == 0 and int(err.item()) == 0
            row.append(int(cyc.item()) / (4 * 256))
        print(f"  N={N:3d} {label:20s}: plain {row[0]:6.1f}   with per-4-MMA barrier test, fences, commit {row[1]:6.1f}")



def _probe_gather(lib, err):
    import ctypes
    import torch
    # Scattered 128-byte row segments into shared memory, all SMs.
    f = lib.mlav_gather_rate
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_void_p] + [ctypes.c_int] * 5 + \
        [ctypes.c_void_p] * 2
    pool = 1_200_000
    kv = torch.randn(pool, 576, device="cuda", dtype=torch.bfloat16)
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    cyc_sm = torch.zeros(nsm, dtype=torch.int64, device="cuda")
    print("gather: bytes per clock per SM, 256 keys x 9 segments per tile, all SMs")
    for label, hi in (("rows in HBM (1.2M-slot pool)", pool), ("rows L2-resident (20k slots)", 20000)):
        rng = np.random.default_rng(0)
        slots = torch.from_numpy(rng.integers(0, hi, size=nsm * 8 * 256).astype(np.int32)).cuda()
        parts = []
        for method, nw, tr in ((0, 2, 0), (0, 4, 0), (0, 8, 0), (0, 12, 0), (2, 1, 0), (4, 4, 32)):
            for _ in range(2):
                rc = f(kv.data_ptr(), pool, slots.data_ptr(), nsm, 8, method, nw, tr, cyc_sm.data_ptr(),
                       err.data_ptr())
            assert rc == 0 and int(err.item()) == 0
            c = cyc_sm.float().mean().item()
            name = {0: f"cp.async x{nw} warps", 2: "TMA gather4", 4: "cp.async x4 + gather4 1/8"}[method]
            parts.append(f"{name} {8 * 9 * 256 * 128 / c:5.1f}")
        print(f"  {label}: " + "; ".join(parts))

    del kv
    torch.cuda.empty_cache()


def _probe_blocks(lib, err):
    import ctypes
    import torch
    # Contiguous 8 KB blocks (the fp8 indexer cache) into a swizzled ring, all SMs.
    f = lib.mlav_block_rate
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_void_p] + [ctypes.c_int] * 4 + \
        [ctypes.c_longlong] + [ctypes.c_void_p] * 2
    nblk = 120_000                      # ~1 GB pool
    rows = nblk * 8448 // 1152          # the same bytes as latent-cache rows
    kv = torch.zeros(nblk * 8448, dtype=torch.uint8, device="cuda")
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    cyc_sm = torch.zeros(nsm, dtype=torch.int64, device="cuda")
    ntile = 512
    rng = np.random.default_rng(1)
    blocks = torch.from_numpy(rng.integers(0, nblk, size=nsm * ntile * 2).astype(np.int32)).cuda()
    row_slots = torch.from_numpy(rng.integers(0, rows, size=nsm * 128 * 126).astype(np.int32)).cuda()
    print("8 KB blocks: bytes per clock per SM (and GB/s over all SMs), 2 blocks per 16 KB stage, "
          "8-stage ring, all SMs")
    for method, nw, label in ((0, 1, "TMA 3-D boxes"), (2, 1, "1-D bulk copies"),
                              (1, 4, "cp.async x4 warps"), (1, 8, "cp.async x8 warps"),
                              (3, 4, "TMA + cp.async x4 (half each)"),
                              (3, 8, "TMA + cp.async x8 (half each)"),
                              (4, 4, "ld.global x4 warps"), (4, 8, "ld.global x8 warps"),
                              (5, 1, "TMA boxes + 256 B bulk scales"),
                              (6, 1, "TMA boxes + 256 B TMA scale boxes"),
                              (7, 8, "whole 1152 B rows, cp.async x8"),
                              (7, 12, "whole 1152 B rows, cp.async x12"),
                              (8, 8, "128 B of each row, cp.async x8"),
                              (8, 12, "128 B of each row, cp.async x12"),
                              (9, 1, "whole 1152 B rows, 1-D bulk copies")):
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        nt = ntile if method < 7 else 128
        idx = blocks if method < 7 else row_slots
        for rep in range(2):
            ev[0].record()
            rc = f(kv.data_ptr(), nblk, idx.data_ptr(), nsm, nt, method, nw, rows,
                   cyc_sm.data_ptr(), err.data_ptr())
            ev[1].record()
        assert rc == 0 and int(err.item()) == 0
        torch.cuda.synchronize()
        c = cyc_sm.float().mean().item()
        stage = 16128 if method >= 7 else 16384
        gbs = nsm * nt * stage / (ev[0].elapsed_time(ev[1]) * 1e-3) / 1e9
        print(f"  {label:34s} {nt * stage / c:6.1f} B/clk   {gbs:7.0f} GB/s")
    del kv
    torch.cuda.empty_cache()


def _probe_dsmem(lib, err):
    import ctypes
    import torch
    # Bulk copies from one CTA's shared memory into its cluster peer's, through
    # a 4-slot ring released by remote arrives (2-CTA clusters).
    f = lib.mlav_bulk_rate
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int] * 3 + [ctypes.c_void_p] * 2
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    cyc = torch.zeros(nsm, dtype=torch.int64, device="cuda")
    print("DSMEM bulk copy CTA -> peer: bytes per clock per sending SM")
    for ncl in (1, nsm // 2):
        parts = []
        for chunk in (4096, 16384, 32768):
            n = (64 << 20) // chunk // max(1, ncl) + 64
            rc = f(ncl, chunk, n, cyc.data_ptr(), err.data_ptr())
            assert rc == 0 and int(err.item()) == 0
            c = cyc[:ncl].float().mean().item()
            parts.append(f"{chunk // 1024} KB chunks {n * chunk / c:5.1f}")
        print(f"  {ncl:3d} cluster(s): " + "; ".join(parts))


def _probe_mbar(lib, cyc, err):
    import ctypes
    import torch
    # mbarrier operations (one thread) and a producer/consumer ring.
    f = lib.mlav_mbar_cost
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    names = ["try_wait, phase complete", "test_wait, phase complete", "arrive",
             "try_wait.acquire.cluster, complete", "arrive + try_wait"]
    print("mbarrier, cycles per operation (one thread)")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    for op in range(5):
        rc = f(op, 4096, cyc.data_ptr(), sink.data_ptr())
        assert rc == 0
        print(f"  {names[op]:36s} {int(cyc.item()) / 4096:6.1f}")
    f = lib.mlav_ring_probe
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int] * 4 + [ctypes.c_void_p] * 2
    print("empty ring (producer warp -> consumer thread, parking try_wait), cycles per stage")
    for depth in (1, 8):
        for pm in (0, 1):
            for cm in (0, 1):
                rc = f(depth, 4096, pm, cm, cyc.data_ptr(), err.data_ptr())
                assert rc == 0 and int(err.item()) == 0
                print(f"  depth {depth} producer {'cp.async arrive' if pm else 'arrive':15s} "
                      f"consumer {'tcgen05.commit' if cm else 'arrive':14s} {int(cyc.item()) / 4096:6.1f}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=4, choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--simt", action="store_true", help="force the CUDA-core partial kernel")
    ap.add_argument("--no-extras", dest="extras", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-step-s", type=float, default=4.0)
    ap.add_argument("--probes", nargs="*", choices=PROBES, default=None,
                    help="run these building-block microbenchmarks (all if none named) "
                         "instead of the bench")
    ap.add_argument("--next-rows", nargs="*", choices=NEXT_ROWS, default=None,
                    help="time only these steps beside the verify attention (all if none named) "
                         "and print their JSON instead of the bench line")
    args = ap.parse_args()
    if args.probes is not None:
        run_probes(args.probes or PROBES)
        return
    if args.next_rows is not None:
        run_next_rows(args.next_rows or NEXT_ROWS)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    args.flags = 1 if args.simt else 0
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
