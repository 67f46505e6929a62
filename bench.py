#!/usr/bin/env python
"""Benchmark of selected-token log-probabilities on one GB300 (or N replicas).

A step is one pass of the hot path over one batch of synthetic input: the
forward (online log-sum-exp + target gather) and the backward ((onehot -
softmax) * g / T) of the logits-input path on the c151k workload
(N=4096 tokens, V=151936, bf16 logits), through the C ABI of libslp.so.
Prints ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl slp|reference]

Under torchrun (N > 1) every rank runs an independent replica of the same
workload on its own GPU (rows are independent: no data-path collective); the
timed region is bracketed by barriers and the max time over ranks is used.
``--impl reference`` times the CPU oracle on a bounded sample of the same
workload instead (rank 0 only).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "selected-logprob fwd+bwd tokens/s and HBM GB/s (% of roofline) at V=151936, 1 GB300"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["slp", "reference"], default="slp")
    p.add_argument("--config", default="c151k", choices=["c151k", "packed", "stability", "tiny"])
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--no-extra", action="store_true", help="skip the other workloads' lines")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--lmhead-only", action="store_true",
                   help="time only the fused LM-head path and print its numbers")
    p.add_argument("--lmhead-rows", type=int, default=None)
    p.add_argument("--fused-only", action="store_true",
                   help="time only the fused forward+backward on --config (and --rows)")
    p.add_argument("--vocab", type=int, default=None,
                   help="override V (same recipe), with --fused-only, e.g. for long-row profiling")
    p.add_argument("--rows", type=int, default=None,
                   help="override N (same recipe), e.g. for a small profiling case")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def traffic_table():
    """Per-launch DRAM bytes from the committed ncu summary (kernel, workload,
    bytes, source hash of the kernel file when captured)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    out = {}
    if os.path.exists(path):
        for line in open(path):
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, w, b, h = line.split()[:4]
            out[(k, w)] = (float(b), h)
    return out


def code_text(src):
    """C++/CUDA source with its comments, trailing blanks and empty lines
    removed: what a change to the compiled kernels must touch."""
    out, i, n = [], 0, len(src)
    quote = None
    while i < n:
        ch = src[i]
        if quote:
            out.append(ch)
            if ch == "\\" and i + 1 < n:
                out.append(src[i + 1])
                i += 2
                continue
            if ch == quote:
                quote = None
            i += 1
        elif ch in "\"'":
            quote = ch
            out.append(ch)
            i += 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(ch)
            i += 1
    lines = [ln.rstrip() for ln in "".join(out).split("\n")]
    return "\n".join(ln for ln in lines if ln.strip())


def source_hash(fname):
    """sha1 (12 hex digits) of a csrc file's code, comments excluded, so the
    DRAM-traffic record stays tied to the kernels rather than their prose."""
    import hashlib
    p = os.path.join(ROOT, "vocab_selected_token_gb300", "csrc", fname)
    return hashlib.sha1(code_text(open(p).read()).encode()).hexdigest()[:12]


# ---------------------------------------------------------------- distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "slp" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif args.impl == "slp":
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world, device):
    """The slowest rank's time (measurement only: no data-path collective)."""
    if world == 1:
        return v
    import torch.distributed as dist
    on = device if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([v], dtype=torch.float64, device=on)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(tokens_per_rank, world, ms_per_step_max):
    """Weak scaling: every rank processes its own replica of the workload, so
    the job's throughput is all ranks' tokens over the slowest rank's time."""
    return world * tokens_per_rank * 1000.0 / ms_per_step_max


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device, interval_ms=200):
        self.proc = None
        self.interval_ms = int(interval_ms)
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            ident = os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0]
        self.ident = ident

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.ident, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
                power.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- workloads
def logits_bytes(x, mask):
    N, V = x.shape
    es = x.element_size()
    na = N if mask is None else int(mask.sum().item())
    fwd = na * V * es + N * (4 + 4 + 4 + (0 if mask is None else 1))
    bwd = na * V * es + N * V * es + N * (4 * 3 + (0 if mask is None else 1))
    return fwd, bwd, na


def time_logits(inp, steps, warmup, world, device, clocks=None):
    """Device-timed forward+backward steps through the C ABI.  Returns a dict
    with ms/step and the average duration of each kernel (CUDA events on the
    launching stream)."""
    from vocab_selected_token_gb300 import _lib
    lib = _lib.load()
    x, t, mask, T, g = inp.x, inp.t, inp.mask, inp.T, inp.g
    N, V = x.shape
    dt = _lib.SLP_BF16 if x.dtype == torch.bfloat16 else _lib.SLP_F32
    lp = torch.empty(N, dtype=torch.float32, device=device)
    lse = torch.empty_like(lp)
    gx = torch.empty_like(x)
    stream = torch.cuda.current_stream(device)
    sh = stream.cuda_stream
    mp = None if mask is None else mask.data_ptr()
    fargs = (x.data_ptr(), dt, N, V, x.stride(0), t.data_ptr(), mp, float(T), lp.data_ptr(),
             lse.data_ptr(), None, sh)
    bargs = (x.data_ptr(), dt, N, V, x.stride(0), t.data_ptr(), mp, float(T), lse.data_ptr(),
             g.data_ptr(), gx.data_ptr(), gx.stride(0), None, sh)

    def step():
        assert lib.slp_forward(*fargs) == 0
        assert lib.slp_backward(*bargs) == 0

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(device)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize(device)
    if clocks:
        clocks.start()
    for i in range(steps):
        ev[i][0].record(stream)
        assert lib.slp_forward(*fargs) == 0
        ev[i][1].record(stream)
        assert lib.slp_backward(*bargs) == 0
        ev[i][2].record(stream)
    torch.cuda.synchronize(device)
    barrier(world)
    clk = clocks.stop() if clocks else None
    total_ms = ev[0][0].elapsed_time(ev[-1][2])
    fwd = [e[0].elapsed_time(e[1]) for e in ev]
    bwd = [e[1].elapsed_time(e[2]) for e in ev]
    total_ms = max_over_ranks(total_ms, world, device)
    return {"ms_per_step": total_ms / steps, "fwd_ms": sum(fwd) / steps,
            "bwd_ms": sum(bwd) / steps, "clocks": clk, "launches": 2 * steps,
            "outputs": (lp, lse, gx)}


def host_topology(device):
    """Where the host buffers live relative to the GPU: the CPUs this process
    may run on, the host's NUMA nodes with their CPUs, and the GPU's PCI
    NUMA node and local CPUs (from sysfs; None where not exposed)."""
    def read(path):
        try:
            with open(path) as f:
                return f.read().strip()
        except OSError:
            return None
    info = {"process_cpus": len(os.sched_getaffinity(0))}
    root = "/sys/devices/system/node"
    nodes = {}
    try:
        for n in sorted(os.listdir(root)):
            if n.startswith("node") and n[4:].isdigit():
                nodes[n] = read(os.path.join(root, n, "cpulist"))
    except OSError:
        pass
    info["numa_nodes"] = nodes
    try:
        pr = torch.cuda.get_device_properties(device)
        bus = "%04x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
        dev = os.path.join("/sys/bus/pci/devices", bus)
        info["gpu_pci"] = bus
        info["gpu_numa_node"] = read(os.path.join(dev, "numa_node"))
        info["gpu_local_cpus"] = read(os.path.join(dev, "local_cpulist"))
    except Exception:
        info["gpu_pci"] = None
    return info


def host_link_rates(device, nbytes=1 << 29, reps=4):
    """This machine's host link from page-locked memory: GB/s host->device,
    device->host, and both directions at once (two streams), best of two
    rounds of `reps` copies of `nbytes`."""
    hs = [torch.empty(nbytes, dtype=torch.uint8).pin_memory() for _ in range(2)]
    ds = [torch.empty(nbytes, dtype=torch.uint8, device=device) for _ in range(2)]
    st = [torch.cuda.Stream(device=device) for _ in range(2)]

    def timed(jobs):
        best = None
        for _ in range(2):
            torch.cuda.synchronize(device)
            t0 = time.perf_counter()
            for j, (dst, src) in enumerate(jobs):
                with torch.cuda.stream(st[j]):
                    for _ in range(reps):
                        dst.copy_(src, non_blocking=True)
            torch.cuda.synchronize(device)
            dt = time.perf_counter() - t0
            best = dt if best is None else min(best, dt)
        return len(jobs) * reps * nbytes / best / 1e9

    out = {"h2d_gbs": timed([(ds[0], hs[0])]), "d2h_gbs": timed([(hs[0], ds[0])]),
           "both_gbs": timed([(ds[0], hs[0]), (hs[1], ds[1])])}
    del hs, ds
    return out


def e2e_logits(inp, steps, device):
    """Same metric through the public API for host-resident data:
    vocab_selected_token_gb300.streaming.forward_backward_from_host streams the
    step's logits, targets and upstream gradient from pinned host memory and
    returns logprob, lse and grad_x in pinned host memory (copies in both
    directions overlap the kernels).  Wall time around the whole call, which
    returns only when the results are on the host."""
    from vocab_selected_token_gb300.streaming import forward_backward_from_host
    xh = inp.x.cpu().pin_memory()
    th = inp.t.cpu().pin_memory()
    gh = inp.g.cpu().pin_memory()
    mh = None if inp.mask is None else inp.mask.cpu().pin_memory()
    N, V = xh.shape
    lp_h = torch.empty(N, dtype=torch.float32).pin_memory()
    lse_h = torch.empty(N, dtype=torch.float32).pin_memory()
    gx_h = torch.empty((N, V), dtype=xh.dtype).pin_memory()
    h2d = xh.numel() * xh.element_size() + th.numel() * 4 + gh.numel() * 4 + (0 if mh is None else N)
    d2h = 2 * N * 4 + gx_h.numel() * gx_h.element_size()

    def step():
        forward_backward_from_host(xh, th, gh, mh, inp.T, logprob=lp_h, lse=lse_h, grad_x=gx_h,
                                   device=device)

    for _ in range(3):
        step()
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    ms = (time.perf_counter() - t0) * 1000.0 / steps
    link = host_link_rates(device)
    link["e2e_frac_of_both"] = (h2d + d2h) / (ms * 1e-3) / 1e9 / link["both_gbs"]
    return {"value": N * 1000.0 / ms, "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "api": "streaming.forward_backward_from_host -> slp_forward_backward_host "
                   "(native 3-stream pipeline, ~64 MB chunks, fused forward+backward)",
            "host": host_topology(device), "host_link": link}


# ---------------------------------------------------------------- oracle arm
def oracle_rows_per_second(inp, seconds, max_rows=4096):
    """The CPU oracle as it stands (fp64 numpy, one core), forward+backward on
    consecutive rows of the workload until `seconds` of CPU work are done."""
    from oracle import slp_oracle as O
    N = inp.x.shape[0]
    rows_done, t_total, r = 0, 0.0, 0
    while (t_total < seconds and rows_done < max_rows) or rows_done == 0:
        blk = slice(r, min(r + 4, N))
        x64 = inp.x[blk].double().cpu().numpy()
        tt = inp.t[blk].cpu().numpy()
        mm = None if inp.mask is None else inp.mask[blk].cpu().numpy()
        gg = inp.g[blk].double().cpu().numpy()
        t0 = time.perf_counter()
        lp, lse = O.selected_logprob_forward(x64, tt, mm, inp.T)
        O.selected_logprob_backward(x64, tt, mm, inp.T, lse, gg)
        t_total += time.perf_counter() - t0
        rows_done += x64.shape[0]
        r = (r + 4) % N
    return rows_done / t_total, rows_done, t_total


def oracle_rows_per_second_all_cores(inp, seconds, rows_per_thread=32):
    """The CPU oracle as it stands on every host core this process may use:
    one thread per core, each running forward+backward on its own block of
    consecutive rows of the workload for about `seconds`.  numpy releases the
    GIL inside its array loops, so the threads compute in parallel; they are
    released together by a barrier."""
    import threading
    from oracle import slp_oracle as O
    n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    N = inp.x.shape[0]
    blocks = []
    for i in range(n):
        r0 = (i * rows_per_thread) % N
        blk = slice(r0, min(r0 + rows_per_thread, N))
        blocks.append((inp.x[blk].double().cpu().numpy(), inp.t[blk].cpu().numpy(),
                       None if inp.mask is None else inp.mask[blk].cpu().numpy(),
                       inp.g[blk].double().cpu().numpy()))
    done = [0] * n
    gate = threading.Barrier(n + 1)
    stop_at = [0.0]

    def work(i):
        x64, tt, mm, gg = blocks[i]
        gate.wait()
        while time.perf_counter() < stop_at[0]:
            lp, lse = O.selected_logprob_forward(x64, tt, mm, inp.T)
            O.selected_logprob_backward(x64, tt, mm, inp.T, lse, gg)
            done[i] += x64.shape[0]

    threads = [threading.Thread(target=work, args=(i,)) for i in range(n)]
    for th in threads:
        th.start()
    t0 = time.perf_counter()
    stop_at[0] = t0 + seconds
    gate.wait()
    for th in threads:
        th.join()
    el = time.perf_counter() - t0
    return sum(done) / el, sum(done), el, n


def workload_desc(name, inp, na):
    N, V = inp.x.shape
    from vocab_selected_token_gb300.workloads import WORKLOADS
    dt = "bf16" if inp.x.dtype == torch.bfloat16 else "f32"
    return {"workload": f"{name}: N={N} tokens, V={V}, {dt} logits, T={inp.T}; "
                        + WORKLOADS[name]["recipe"],
            "N": N, "V": V, "active_rows": na, "temperature": inp.T,
            "l2": f"inputs exceed L2 (logits {N * V * inp.x.element_size() / 1e9:.3f} GB > 129 MB); no flush"}


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle as it stands on every host core this
    process may use.  Each step is a bounded sample of the workload: `rows`
    consecutive rows per core, one thread per core (numpy releases the GIL
    inside its array loops)."""
    import threading
    from vocab_selected_token_gb300 import workloads as W
    if rank != 0:
        return
    inp = W.make_logits_inputs(args.config, device="cpu", N=args.rows)
    n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    # size one step so the whole run stays within about two minutes
    r1, _, t1 = oracle_rows_per_second(inp, 0.0, max_rows=4)
    per_row = 1.0 / r1
    rows = max(1, min(32, int(120.0 / max(1, args.steps + args.warmup) / per_row)))
    from oracle import slp_oracle as O
    N = inp.x.shape[0]

    def block(i, j):
        r0 = ((i * n + j) * rows) % N
        blk = slice(r0, min(r0 + rows, N))
        x64 = inp.x[blk].double().numpy()
        tt = inp.t[blk].numpy()
        mm = None if inp.mask is None else inp.mask[blk].numpy()
        lp, lse = O.selected_logprob_forward(x64, tt, mm, inp.T)
        O.selected_logprob_backward(x64, tt, mm, inp.T, lse, inp.g[blk].double().numpy())
        return x64.shape[0]

    def step(i):
        counts = [0] * n

        def run(j):
            counts[j] = block(i, j)

        threads = [threading.Thread(target=run, args=(j,)) for j in range(n)]
        for th in threads:
            th.start()
        for th in threads:
            th.join()
        return sum(counts)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    done = sum(step(i) for i in range(args.steps))
    el = time.perf_counter() - t0
    v = done / el
    _, _, na = logits_bytes(inp.x, inp.mask)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1000 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded generators, CPU)",
            "config": {**workload_desc(args.config, inp, na),
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": n, "kind": "oracle",
                             "sample": f"{rows} consecutive rows per core per step ({n} threads), "
                                       "fp64 numpy forward+backward including each row's "
                                       "conversion to fp64; value = rows done / wall time "
                                       "(a per-core row sample scaled to tokens/s, not the "
                                       "whole workload)"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- main
def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    import __graft_entry__
    __graft_entry__.build()
    from vocab_selected_token_gb300 import workloads as W
    device = torch.device("cuda", torch.cuda.current_device())
    hbm, bf16_burst, bf16_sus, peak_src = peaks()
    if args.lmhead_only:
        r = time_lmhead(device, steps=args.steps, warmup=args.warmup, N=args.lmhead_rows)
        if rank == 0:
            print(json.dumps({"lmhead": r}), flush=True)
        return
    if args.fused_only:
        r = time_fused(device, hbm, steps=args.steps, warmup=args.warmup, names=(args.config,),
                       rows=args.rows, vocab=args.vocab)
        if rank == 0:
            print(json.dumps({"fused_fwd_bwd": r}), flush=True)
        return

    inp = W.make_logits_inputs(args.config, device=device, N=args.rows)
    fwd_b, bwd_b, na = logits_bytes(inp.x, inp.mask)
    N, V = inp.x.shape
    torch.cuda.reset_peak_memory_stats(device)
    base_mem = torch.cuda.memory_allocated(device)
    res = time_logits(inp, args.steps, args.warmup, world, device, ClockSampler(device))
    extra_mem = torch.cuda.max_memory_allocated(device) - base_mem
    value = whole_job_tokens_per_s(N, world, res["ms_per_step"])

    kern = "slp_bwd_kernel" if res["bwd_ms"] >= res["fwd_ms"] else "slp_fwd_kernel"
    k_bytes, k_ms = (bwd_b, res["bwd_ms"]) if kern == "slp_bwd_kernel" else (fwd_b, res["fwd_ms"])
    achieved = k_bytes / (k_ms * 1e-3) / 1e9
    tt = traffic_table().get((kern, args.config))
    traffic = None
    if tt is not None and tt[1] == source_hash("slp_logits.cu"):
        traffic = tt[0]
    step_gbs = (fwd_b + bwd_b) / (res["ms_per_step"] * 1e-3) / 1e9

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if inp.x.dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded generators on the device)",
        "config": {**workload_desc(args.config, inp, na),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "hbm": {"step_gbs": step_gbs, "step_frac_of_measured": step_gbs / hbm,
                "step_frac_of_8tbs": step_gbs / 8000.0,
                "fwd_ms": res["fwd_ms"], "bwd_ms": res["bwd_ms"],
                "fwd_gbs": fwd_b / (res["fwd_ms"] * 1e-3) / 1e9,
                "bwd_gbs": bwd_b / (res["bwd_ms"] * 1e-3) / 1e9,
                "bytes_per_step": fwd_b + bwd_b},
        "roofline": {"kernel": kern, "bound": "hbm", "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic,
                     "algorithmic_bytes_per_launch": k_bytes, "peak_source": peak_src},
        "clocks": res["clocks"],
        "gpu_launches": res["launches"],
        "peak_extra_device_bytes": int(extra_mem),  # beyond the inputs, outputs included
        "peak_workspace_bytes": int(extra_mem - (2 * N * 4 + N * V * inp.x.element_size())),
    }
    if rank == 0:
        line["e2e"] = e2e_logits(inp, args.e2e_steps, device)
        if world == 1:
            v1, rows1, secs1 = oracle_rows_per_second(inp, args.cpu_seconds)
            va, rowsa, secsa, cores = oracle_rows_per_second_all_cores(
                inp, max(1.0, args.cpu_seconds / 2))
            line["cpu_baseline"] = {
                "value": va, "unit": UNIT, "cores": cores, "kind": "oracle",
                "sample": f"{rowsa} rows of {args.config} (forward+backward, fp64 numpy, one "
                          f"thread per core on its own 32-row block, {secsa:.1f} s)",
                "single_core": {"value": v1, "unit": UNIT, "cores": 1,
                                "sample": f"{rows1} consecutive rows, {secs1:.1f} s"}}
        if not args.no_extra:
            del inp
            torch.cuda.empty_cache()
            line["other_workloads"] = other_workloads(device, hbm)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def other_workloads(device, hbm):
    """Shorter timings of the other logits-input workloads (and the fused LM
    head once present), for the record."""
    from vocab_selected_token_gb300 import workloads as W
    out = {}
    for name in ("packed", "stability"):
        inp = W.make_logits_inputs(name, device=device)
        fwd_b, bwd_b, na = logits_bytes(inp.x, inp.mask)
        r = time_logits(inp, 30, 3, 1, device)
        out[name] = {"N": inp.x.shape[0], "V": inp.x.shape[1], "active_rows": na,
                     "ms_per_step": r["ms_per_step"], "fwd_ms": r["fwd_ms"], "bwd_ms": r["bwd_ms"],
                     "tokens_per_s": inp.x.shape[0] * 1000.0 / r["ms_per_step"],
                     "step_gbs": (fwd_b + bwd_b) / (r["ms_per_step"] * 1e-3) / 1e9,
                     "fwd_gbs": fwd_b / (r["fwd_ms"] * 1e-3) / 1e9,
                     "bwd_gbs": bwd_b / (r["bwd_ms"] * 1e-3) / 1e9}
        out[name]["step_frac_of_measured"] = out[name]["step_gbs"] / hbm
        del inp, r
        torch.cuda.empty_cache()
    out["fused_fwd_bwd"] = time_fused(device, hbm)
    out["short_rows"] = time_short_rows(device, hbm)
    out["small_n"] = time_small_n(device, hbm)
    out["entropy"] = time_entropy(device, hbm)
    out["topk_kl"] = time_topk(device, hbm)
    out["lmhead"] = time_lmhead(device)
    return out


def time_small_n(device, hbm, steps=30, warmup=3):
    """Few rows (c151k recipe, N = 256 and 1024 at V = 32768 and 151936): the
    separate forward + backward step and the fused call.  Most of these inputs
    fit in L2, so L2 is flushed (a 256 MB write) before every timed step, and
    each step is timed on its own with CUDA events (the flush outside them)."""
    import vocab_selected_token_gb300 as slp
    from vocab_selected_token_gb300 import workloads as W
    out = {}
    s = torch.cuda.current_stream(device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    for N, V in ((256, 32768), (256, 151936), (1024, 32768), (1024, 151936)):
        inp = W.make_logits_inputs("c151k", device=device, N=N, V=V)
        nb = N * V * inp.x.element_size()
        lp = torch.empty(N, device=device)
        lse = torch.empty(N, device=device)
        gx = torch.empty_like(inp.x)

        def sep():
            slp.slp_forward(inp.x, inp.t, None, inp.T, logprob=lp, lse=lse)
            slp.slp_backward(inp.x, inp.t, None, inp.T, lse, inp.g, grad_x=gx)

        def fused():
            slp.slp_forward_backward(inp.x, inp.t, None, inp.T, inp.g, logprob=lp, lse=lse,
                                     grad_x=gx)

        res = {"N": N, "V": V, "l2": "flushed before every timed step"}
        for key, fn, passes in (("step", sep, 3), ("fused", fused, 2)):
            for _ in range(warmup):
                fn()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(steps)]
            for e0, e1 in ev:
                flush.fill_(1)
                e0.record(s)
                fn()
                e1.record(s)
            torch.cuda.synchronize(device)
            ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / steps
            gbs = passes * nb / (ms * 1e-3) / 1e9
            res[key] = {"ms": ms, "tokens_per_s": N * 1000.0 / ms, "gbs": gbs,
                        "frac_of_measured": gbs / hbm}
        out[f"N{N}_V{V}"] = res
        del inp, gx
        torch.cuda.empty_cache()
    del flush
    torch.cuda.empty_cache()
    return out


def time_short_rows(device, hbm, steps=30, warmup=3):
    """Small vocabularies (c151k recipe at V = 4096 and 32768, 1 GB of bf16
    logits each): the separate forward + backward step and the fused call.
    Rows of a few KB run on the warp-per-row kernels."""
    import vocab_selected_token_gb300 as slp
    from vocab_selected_token_gb300 import workloads as W
    out = {}
    s = torch.cuda.current_stream(device)
    for V, N in ((4096, 131072), (32768, 16384)):
        inp = W.make_logits_inputs("c151k", device=device, N=N, V=V)
        nb = N * V * inp.x.element_size()
        lp = torch.empty(N, device=device)
        lse = torch.empty(N, device=device)
        gx = torch.empty_like(inp.x)

        def sep():
            slp.slp_forward(inp.x, inp.t, None, inp.T, logprob=lp, lse=lse)
            slp.slp_backward(inp.x, inp.t, None, inp.T, lse, inp.g, grad_x=gx)

        def fused():
            slp.slp_forward_backward(inp.x, inp.t, None, inp.T, inp.g, logprob=lp, lse=lse,
                                     grad_x=gx)

        res = {"N": N, "V": V}
        for key, fn, passes in (("step", sep, 3), ("fused", fused, 2)):
            for _ in range(warmup):
                fn()
            torch.cuda.synchronize(device)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(steps):
                fn()
            e1.record(s)
            torch.cuda.synchronize(device)
            ms = e0.elapsed_time(e1) / steps
            gbs = passes * nb / (ms * 1e-3) / 1e9
            res[key] = {"ms": ms, "tokens_per_s": N * 1000.0 / ms, "gbs": gbs,
                        "frac_of_measured": gbs / hbm}
        out[f"V{V}"] = res
        del inp, gx
        torch.cuda.empty_cache()
    return out


def time_entropy(device, hbm, steps=30, warmup=3):
    """slp_forward_entropy + slp_backward_entropy on c151k (same bytes as the
    plain step: the entropy is one more accumulator in the same pass)."""
    import vocab_selected_token_gb300 as slp
    from vocab_selected_token_gb300 import workloads as W
    inp = W.make_logits_inputs("c151k", device=device)
    N, V = inp.x.shape
    fwd_b, bwd_b, _ = logits_bytes(inp.x, inp.mask)
    gH = torch.rand(N, device=device)
    lp = torch.empty(N, device=device)
    lse = torch.empty(N, device=device)
    H = torch.empty(N, device=device)
    gx = torch.empty_like(inp.x)
    s = torch.cuda.current_stream(device)

    def step():
        slp.slp_forward_entropy(inp.x, inp.t, None, inp.T, logprob=lp, lse=lse, entropy=H)
        slp.slp_backward_entropy(inp.x, inp.t, None, inp.T, lse, H, inp.g, gH, grad_x=gx)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        step()
    e1.record(s)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / steps

    def fused():
        slp.slp_forward_backward_entropy(inp.x, inp.t, None, inp.T, inp.g, gH, logprob=lp,
                                         lse=lse, entropy=H, grad_x=gx)

    for _ in range(warmup):
        fused()
    torch.cuda.synchronize(device)
    e0.record(s)
    for _ in range(steps):
        fused()
    e1.record(s)
    torch.cuda.synchronize(device)
    ms_f = e0.elapsed_time(e1) / steps
    fb = 2 * N * V * inp.x.element_size()  # one read of the logits, one write of the gradient
    del inp, gx
    torch.cuda.empty_cache()
    return {"workload": "c151k", "ms_per_step": ms, "tokens_per_s": N * 1000.0 / ms,
            "gbs": (fwd_b + bwd_b) / (ms * 1e-3) / 1e9,
            "frac_of_measured": (fwd_b + bwd_b) / (ms * 1e-3) / 1e9 / hbm,
            "fused": {"ms_per_step": ms_f, "tokens_per_s": N * 1000.0 / ms_f,
                      "algorithmic_bytes": fb, "gbs": fb / (ms_f * 1e-3) / 1e9,
                      "frac_of_measured": fb / (ms_f * 1e-3) / 1e9 / hbm}}


def time_topk(device, hbm, steps=20, warmup=3):
    """Top-k forward KL on the distillation workload (N=4096, V=248320, K=128,
    clamp -10): the forward reads the logits once (+ K gathers per row), the
    backward reads them once and writes the gradient."""
    import vocab_selected_token_gb300 as slp
    from vocab_selected_token_gb300 import workloads as W
    a = W.make_topk_inputs(device=device)
    N, V = a.x.shape
    K = a.ids.shape[1]
    s = torch.cuda.current_stream(device)
    gx = torch.empty_like(a.x)
    res = {}
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for i in range(warmup + steps):
        if i == warmup:
            ev[0].record(s)
        kl, sm, tm, lse = slp.slp_topk_kl_forward(a.x, a.ids, a.lt, None, a.T, a.clamp)
        if i == warmup + steps - 1:
            ev[1].record(s)
        slp.slp_topk_kl_backward(a.x, a.ids, a.lt, None, a.T, a.clamp, lse, a.g, grad_x=gx)
    ev[2].record(s)
    torch.cuda.synchronize(device)
    # forward-only timing: a second loop
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        slp.slp_topk_kl_forward(a.x, a.ids, a.lt, None, a.T, a.clamp)
    e1.record(s)
    torch.cuda.synchronize(device)
    step_ms = ev[0].elapsed_time(ev[2]) / steps
    fwd_ms = e0.elapsed_time(e1) / steps
    nb = N * V * a.x.element_size()
    res = {"N": N, "V": V, "K": K, "ms_per_step": step_ms, "fwd_ms": fwd_ms,
           "bwd_ms": step_ms - fwd_ms, "tokens_per_s": N * 1000.0 / step_ms,
           "step_gbs": 3 * nb / (step_ms * 1e-3) / 1e9,
           "frac_of_measured": 3 * nb / (step_ms * 1e-3) / 1e9 / hbm}
    del a, gx
    torch.cuda.empty_cache()
    return res


def time_fused(device, hbm, steps=30, warmup=3, names=("c151k", "packed", "stability"),
               rows=None, vocab=None):
    """slp_forward_backward (upstream gradient known at forward time): one
    read of the active rows and one write of the gradient per step."""
    from vocab_selected_token_gb300 import _lib
    from vocab_selected_token_gb300 import workloads as W
    lib = _lib.load()
    out = {}
    for name in names:
        inp = W.make_logits_inputs(name, device=device, N=rows, V=vocab)
        x = inp.x
        N, V = x.shape
        es = x.element_size()
        na = N if inp.mask is None else int(inp.mask.sum().item())
        nbytes = na * V * es + N * V * es
        lp = torch.empty(N, device=device)
        lse = torch.empty(N, device=device)
        gx = torch.empty_like(x)
        s = torch.cuda.current_stream(device)
        args = (x.data_ptr(), _lib.SLP_BF16 if x.dtype == torch.bfloat16 else _lib.SLP_F32, N, V,
                x.stride(0), inp.t.data_ptr(), None if inp.mask is None else inp.mask.data_ptr(),
                float(inp.T), inp.g.data_ptr(), lp.data_ptr(), lse.data_ptr(), gx.data_ptr(),
                gx.stride(0), None, s.cuda_stream)
        for _ in range(warmup):
            assert lib.slp_forward_backward(*args) == 0
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            assert lib.slp_forward_backward(*args) == 0
        e1.record(s)
        torch.cuda.synchronize(device)
        ms = e0.elapsed_time(e1) / steps
        out[name] = {"ms_per_step": ms, "tokens_per_s": N * 1000.0 / ms,
                     "algorithmic_bytes": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9,
                     "frac_of_measured": nbytes / (ms * 1e-3) / 1e9 / hbm}
        del inp, x, gx
        torch.cuda.empty_cache()
    return out


def time_lmhead(device, steps=40, warmup=3, N=None):
    """Fused LM-head forward and backward on the lmhead workload (N=8192,
    d=2560, V=151936, Bernoulli(0.5) mask), each call timed whole with CUDA
    events; TFLOP/s counts 2*Na*V*d for the forward and 6*Na*V*d for the
    backward (logits recompute, dh and dW GEMMs).  SM clocks are sampled
    every 50 ms during the timed steps (about 0.3 s of back-to-back GEMMs)."""
    from vocab_selected_token_gb300 import _lib
    from vocab_selected_token_gb300 import workloads as W
    lib = _lib.load()
    a = W.make_lmhead_inputs(device=device, N=N)
    Nn, d = a.h.shape
    V = a.W.shape[0]
    na = int(a.mask.sum().item())
    ws_b = lib.slp_lmhead_workspace_size(Nn, V, d)
    ws = torch.empty(ws_b, dtype=torch.uint8, device=device)
    lp = torch.empty(Nn, device=device)
    lse = torch.empty(Nn, device=device)
    dh = torch.empty((Nn, d), dtype=torch.bfloat16, device=device)
    dW = torch.empty((V, d), dtype=torch.bfloat16, device=device)
    sh = torch.cuda.current_stream(device).cuda_stream
    s = torch.cuda.current_stream(device)
    fa = (a.h.data_ptr(), a.W.data_ptr(), Nn, V, d, a.t.data_ptr(), a.mask.data_ptr(), float(a.T),
          lp.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws_b, None, sh)
    ba = (a.h.data_ptr(), a.W.data_ptr(), Nn, V, d, a.t.data_ptr(), a.mask.data_ptr(), float(a.T),
          lse.data_ptr(), a.g.data_ptr(), dh.data_ptr(), dW.data_ptr(), ws.data_ptr(), ws_b, None, sh)
    for _ in range(warmup):
        assert lib.slp_lmhead_forward(*fa) == 0
        assert lib.slp_lmhead_backward(*ba) == 0
    torch.cuda.synchronize(device)
    clocks = ClockSampler(device, interval_ms=50)
    clocks.start()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(s)
        assert lib.slp_lmhead_forward(*fa) == 0
        ev[i][1].record(s)
        assert lib.slp_lmhead_backward(*ba) == 0
        ev[i][2].record(s)
    torch.cuda.synchronize(device)
    clk = clocks.stop()
    f_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
    b_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / steps
    flop_f = 2.0 * na * V * d
    _, peak, peak_sus, src = peaks()
    res = {"N": Nn, "V": V, "d": d, "active_rows": na, "fwd_ms": f_ms, "bwd_ms": b_ms,
           "fwd_tflops": flop_f / (f_ms * 1e-3) / 1e12,
           "bwd_tflops": 3 * flop_f / (b_ms * 1e-3) / 1e12,
           "step_tflops": 4 * flop_f / ((f_ms + b_ms) * 1e-3) / 1e12,
           # the same step counted without the backward's logits recompute
           # (6 Na V d: the forward, dh and dW GEMMs)
           "step_tflops_useful": 3 * flop_f / ((f_ms + b_ms) * 1e-3) / 1e12,
           "peak_bf16_tflops": peak, "peak_bf16_tflops_sustained": peak_sus, "peak_source": src,
           "workspace_bytes": int(ws_b), "clocks": clk}
    # the forward (~2 ms) is a burst against the burst peak; the backward and
    # the whole step (6-8 ms of back-to-back GEMMs under the power cap) are
    # also given against the sustained peak
    res["fwd_frac"] = res["fwd_tflops"] / peak
    res["bwd_frac"] = res["bwd_tflops"] / peak
    res["step_frac"] = res["step_tflops"] / peak
    res["bwd_frac_sustained"] = res["bwd_tflops"] / peak_sus
    res["step_frac_sustained"] = res["step_tflops"] / peak_sus
    # NVIDIA's dense bf16 figure for one GB300 (half its 2:4-sparse figure)
    res["peak_bf16_tflops_datasheet"] = 2250.0
    res["step_frac_datasheet"] = res["step_tflops"] / 2250.0
    # The same calls with 50 ms of idle GPU before each step, so the clock
    # recovers from the power cap between steps: the kernels' rate at the
    # clock they start at, beside the back-to-back rate above.
    fs = bs = 0.0
    for _ in range(10):
        torch.cuda.synchronize(device)
        time.sleep(0.05)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(s)
        assert lib.slp_lmhead_forward(*fa) == 0
        e[1].record(s)
        assert lib.slp_lmhead_backward(*ba) == 0
        e[2].record(s)
        torch.cuda.synchronize(device)
        fs += e[0].elapsed_time(e[1])
        bs += e[1].elapsed_time(e[2])
    fs /= 10
    bs /= 10
    res["spaced"] = {"how": "10 steps, 50 ms idle before each", "fwd_ms": fs, "bwd_ms": bs,
                     "fwd_tflops": flop_f / (fs * 1e-3) / 1e12,
                     "bwd_tflops": 3 * flop_f / (bs * 1e-3) / 1e12}
    res["spaced"]["fwd_frac"] = res["spaced"]["fwd_tflops"] / peak
    res["spaced"]["bwd_frac"] = res["spaced"]["bwd_tflops"] / peak
    # the backward against its workspace: the chunk width follows the bytes
    # given (16384 columns at the minimum, 65536 by default, the whole
    # vocabulary at the maximum)
    del ws
    torch.cuda.empty_cache()
    curve = []
    for name, fn in (("min", lib.slp_lmhead_workspace_size_min),
                     ("default", lib.slp_lmhead_workspace_size),
                     ("max", lib.slp_lmhead_workspace_size_max)):
        nb = int(fn(Nn, V, d))
        wsx = torch.empty(nb, dtype=torch.uint8, device=device)
        bx = ba[:12] + (wsx.data_ptr(), nb) + ba[14:]
        for _ in range(2):
            assert lib.slp_lmhead_backward(*bx) == 0
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        e0.record(s)
        for _ in range(10):
            assert lib.slp_lmhead_backward(*bx) == 0
        e1.record(s)
        torch.cuda.synchronize(device)
        ms = e0.elapsed_time(e1) / 10
        curve.append({"workspace": name, "workspace_bytes": nb, "bwd_ms": ms,
                      "bwd_tflops": 3 * flop_f / (ms * 1e-3) / 1e12})
        del wsx
        torch.cuda.empty_cache()
    res["bwd_by_workspace"] = curve
    # for scale: the bf16 logits of every row, which the fused path never stores
    res["bf16_logits_bytes_all_rows"] = 2 * Nn * V
    del a, dh, dW
    torch.cuda.empty_cache()
    return res


if __name__ == "__main__":
    main()
