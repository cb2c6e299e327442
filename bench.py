"""Benchmark: EF Top-k (0.1%) + int8 compression of a Llama-3-8B-shaped fp32
gradient arena (291 tensors, 8,030,261,248 elements) on one GB300.

One step = one gc_ef_topk_compress call over the whole arena: acc = g + e,
per-tensor Top-k by |acc|, int8 stochastic rounding of the kept values,
index/code payload, residual update.  Inputs (g, e: 64.2 GB) are resident in
HBM and larger than L2, so no L2 flush is needed between steps.

The default run prints ONE JSON line (rank 0) with the headline and, under
"rows", every other compression path measured on its own workload (the flat
2^20 tensor, ResNet-50, BERT-large, GPT-2-medium, the Llama arena's
receiver), and under "cpu_baseline" the oracle timed on the host cores over a
full iteration of the Llama arena (checked against the GPU's output) and over
the other workloads.  `--op <row>` measures one row alone; `--impl reference`
times the CPU oracle instead, on a bounded sample of the headline workload.

Multi-GPU: the compression of one worker's gradient does not shard (each
data-parallel worker compresses its own gradient with its own residual), so
N > 1 runs N independent replicas, one per GPU; value = all ranks' elements
over the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import os
import platform
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "EF Top-k compress gradient GB/s (elems/s) at 1 GB300; % of HBM roofline"
UNIT = "GB/s"
# workload name -> (generator config id, density, int8, reference-arm tensors)
WORKLOADS = {
    "llama3_8b": (5, 0.001, True, list(range(1, 17))),
    "bert_large": (3, 0.001, True, list(range(0, 16))),
    "resnet50": (2, 0.01, False, list(range(0, 161))),
    "flat_2p20": (1, 0.001, False, [0]),
}
CFG, RHO, INT8 = 5, 0.001, True
# kernels libgc launches per gc_ef_topk_compress call (Top-k mode): the
# workspace zeroing, plan, the sampled threshold estimate, the streaming
# pass, the level-1 select, three histogram passes (full-pass level 1,
# candidate levels 2 and 3) with their selects, count, scan, write
LAUNCHES_PER_STEP = 14
# bytes the streaming pass must move per element: read g, read e, write e
STREAM_BYTES_PER_ELEM = 12
# integer multiplies of one Philox4x32-10 word (random-k keys, QSGD rounding)
IMAD_PER_ELEMENT = 10
L2_BYTES = 129 * 2 ** 20

GRADIENT = {1: "student_t_nu3_x1e-3", 2: "laplace_loguniform_scale", 3: "student_t_nu2.5_x1e-3",
            4: "gaussian_mixture_0.999N(0,1e-4)_0.001N(0,1e-2)", 5: "student_t_nu3_x1e-3"}


def workload_config(layout, k):
    big = 8 * layout.numel > 129e6
    return {"workload": "%s_arena_ef_topk_%gpct%s" % (layout.name, 100 * RHO, "_int8" if INT8 else ""),
            "tensors": layout.num_tensors, "elements": layout.numel, "kept": int(k.sum()), "density": RHO,
            "ef": True, "int8": INT8, "gradient": GRADIENT[CFG],
            "l2": ("inputs (g + e, %.1f GB) larger than L2; no flush" % (8 * layout.numel / 1e9)) if big
            else "inputs fit in L2 (not flushed): latency-bound case",
            "parallelism": "replicas"}


def max_over_ranks(ms: float, device) -> float:
    """The slowest rank's time (replicas run independently; the job ends with the last)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gradient_gbs(elements_per_rank: int, world_size: int, ms_per_step: float) -> float:
    """Whole-job gradient GB/s: every rank compresses its own arena of fp32 elements."""
    return world_size * 4.0 * elements_per_rank / (ms_per_step * 1e-3) / 1e9


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def code_text(src):
    """C/C++/CUDA source without comments, trailing blanks and empty lines."""
    text = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.split("\n"))
    return "\n".join(ln for ln in lines if ln)


def kernel_source_hash():
    """Hash of the streaming pass's source files as code_text: a change to
    the code voids the recorded traffic, an edit of a comment does not."""
    h = hashlib.sha256()
    for f in ("gc_topk.cu", "gc_common.cuh"):
        with open(os.path.join(ROOT, "gradient_compression_gb300", "csrc", f)) as fh:
            h.update(code_text(fh.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per element of the streaming pass from the committed ncu summary;
    None if missing or taken on different kernel source."""
    p = os.path.join(ROOT, "profiles", "k_stream_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    if d.get("source_hash") != kernel_source_hash():
        return None
    return float(d["bytes_per_element"])


def host_description():
    model = platform.processor() or platform.machine()
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                low = line.lower()
                if low.startswith("model name") or low.startswith("cpu part") or low.startswith("hardware"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    try:
        lscpu = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in lscpu.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return {"nproc": os.cpu_count(), "cpu_model": model, "machine": platform.machine(),
            "mem_available_gb": round(mem_available() / 1e9, 1)}


def mem_available() -> int:
    try:
        with open("/proc/meminfo") as fh:
            for line in fh:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 16 * 2 ** 30


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-i", str(gpu_index), "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 10:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]), "util": float(parts[4]),
                             "hw": parts[6], "hwt": parts[7], "swt": parts[8], "pcap": parts[9]})
            except ValueError:
                continue
        if not rows:
            return None
        load = [r for r in rows if r["util"] >= 50]
        if not load:
            return {"sm_mhz": None, "sm_max_mhz": max(r["max"] for r in rows), "reasons": [], "samples": 0,
                    "note": "no sample under load: the timed region is shorter than the 100 ms sampling period"}
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load), "sm_max_mhz": max(r["max"] for r in load),
                "reasons": sorted(reasons), "samples": len(load)}


# ---------------------------------------------------------------------------- CPU oracle

class ByteBudget:
    """Bounds the host memory held by concurrent oracle tasks."""

    def __init__(self, limit):
        self.limit, self.used = limit, 0
        self.cv = threading.Condition()

    def acquire(self, n):
        n = min(n, self.limit)
        with self.cv:
            while self.used > 0 and self.used + n > self.limit:
                self.cv.wait()
            self.used += n
        return n

    def release(self, n):
        with self.cv:
            self.used -= n
            self.cv.notify_all()


def oracle_threads():
    return max(1, min(os.cpu_count() or 1, 64))


def run_tensor_tasks(tasks, threads):
    """Runs (bytes, fn) tasks on a thread pool, the largest first, within a host
    memory budget; the oracle's C calls release the GIL.  Returns the results
    in task order and the wall time."""
    budget = ByteBudget(int(0.5 * mem_available()))
    order = sorted(range(len(tasks)), key=lambda i: -tasks[i][0])
    results = [None] * len(tasks)

    def run(i):
        held = budget.acquire(tasks[i][0])
        try:
            results[i] = tasks[i][1]()
        finally:
            budget.release(held)

    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        for f in [ex.submit(run, i) for i in order]:
            f.result()
    return results, time.perf_counter() - t0


def oracle_full_iteration(gc, layout, k, g_dev, dev, threads):
    """The oracle over every tensor of one iteration (e = 0, iteration 0) on the
    host cores, against a GPU call on the same gradient: returns the oracle's
    GB/s of gradient, its wall time and whether every tensor's payload, scale
    and residual agree bit for bit."""
    import oracle
    oracle.lib()
    L = gc.Layout(layout.off, k, device=dev)
    N, T = layout.numel, layout.num_tensors
    flags = gc.GC_EF | gc.GC_INT8
    comp = gc.TopkCompressor(L, flags, device=dev)
    e = torch.zeros(N, dtype=torch.float32, device=dev)
    comp(g_dev, e, 1234, 0)
    torch.cuda.synchronize()
    K = L.total_k
    gi, gq, gs = comp.idx[:K].cpu().numpy(), comp.q[:K].cpu().numpy(), comp.scale.cpu().numpy()
    off, koff = layout.off, L.koff
    lock = threading.Lock()
    secs = []

    def task(t):
        a, b = int(off[t]), int(off[t + 1])
        with lock:                      # device -> host copies one at a time
            g_h = g_dev[a:b].cpu().numpy()
            e_gpu = e[a:b].cpu().numpy()
        e_h = np.zeros(b - a, np.float32)
        t0 = time.perf_counter()
        ri, _, rq, rs = oracle.ef_topk_tensor(g_h, e_h, int(k[t]), base=a, int8=True, seed=1234, it=0)
        dt = time.perf_counter() - t0
        with lock:
            secs.append(dt)
        ka, kb = int(koff[t]), int(koff[t + 1])
        return (np.array_equal(ri, gi[ka:kb]) and np.array_equal(rq, gq[ka:kb])
                and np.float32(rs).view(np.uint32) == gs[t:t + 1].view(np.uint32)[0]
                and np.array_equal(e_h.view(np.uint32), e_gpu.view(np.uint32)))

    tasks = [(28 * layout.sizes[t], (lambda t=t: task(t))) for t in range(T)]
    agree, wall = run_tensor_tasks(tasks, threads)
    del e, comp
    torch.cuda.empty_cache()
    return {"gbs": 4.0 * N / wall / 1e9, "wall_s": wall, "cpu_s": sum(secs), "agrees": bool(all(agree)),
            "tensors": T, "elements": N}


def oracle_config_workloads(dev, threads):
    """The oracle over the whole workload of each smaller configuration (every
    iteration, state carried), tensors in parallel on the host cores.  The
    gradients are generated on the GPU with the bench's recipe and copied to
    the host; only the oracle calls are timed."""
    import oracle
    oracle.lib()
    specs = [  # name, cfg, iterations, call
        ("flat_2p20_ef_topk_0.1pct", 1, 10, "topk", 0.001),
        ("resnet50_ef_topk_1pct", 2, 20, "topk", 0.01),
        ("resnet50_randk_1pct", 2, 20, "randk", 0.01),
        ("bert_large_ef_topk_0.1pct_int8", 3, 10, "topk8", 0.001),
        ("gpt2_medium_sign_ef", 4, 10, "sign", None),
        ("gpt2_medium_qsgd16", 4, 10, "qsgd", None),
        ("gpt2_medium_momentum_topk_0.5pct", 4, 10, "momentum", 0.005),
    ]
    out = {}
    lock = threading.Lock()
    for name, cfg, iters, call, rho in specs:
        layout = workloads.LAYOUTS[cfg]()
        k = workloads.k_per_tensor(layout.sizes, rho) if rho else None
        off = layout.off
        secs = []

        def task(t, cfg=cfg, iters=iters, call=call, k=k, layout=layout, off=off, secs=secs):
            n, a = layout.sizes[t], int(off[t])
            s1 = np.zeros(n, np.float32)
            s2 = np.zeros(n, np.float32)
            spent = 0.0
            for it in range(iters):
                with lock:
                    g = workloads.tensor_grad(cfg, layout, it, t, device=dev).cpu().numpy()
                t0 = time.perf_counter()
                if call in ("topk", "topk8"):
                    oracle.ef_topk_tensor(g, s1, int(k[t]), base=a, int8=call == "topk8", seed=5, it=it)
                elif call == "randk":
                    oracle.randk_tensor(g, s1, int(k[t]), base=a, seed=5, it=it)
                elif call == "sign":
                    oracle.sign_tensor(g, s1)
                elif call == "qsgd":
                    oracle.quantize_tensor(g, None, "qsgd", 16, base=a, seed=5, it=it)
                else:
                    oracle.momentum_topk_tensor(g, s1, s2, int(k[t]), 0.9, base=a, seed=5, it=it)
                spent += time.perf_counter() - t0
            with lock:
                secs.append(spent)
            return True

        tasks = [(40 * layout.sizes[t], (lambda t=t: task(t))) for t in range(layout.num_tensors)]
        _, wall = run_tensor_tasks(tasks, threads)
        out[name] = {"iterations": iters, "elements": layout.numel, "wall_s": round(wall, 3),
                     "cpu_s": round(sum(secs), 3), "gbs": 4.0 * layout.numel * iters / wall / 1e9}
    return out


def run_reference(args):
    """The oracle as it stands, on the host cores: each step runs the oracle on
    16 tensors of the headline arena in parallel (one per thread)."""
    ws, rank, _ = dist_info()
    if rank != 0:
        return
    import oracle
    oracle.lib()
    layout = workloads.LAYOUTS[CFG]()
    k = workloads.k_per_tensor(layout.sizes, RHO)
    sample_t = WORKLOADS[args.workload][3]
    threads = min(oracle_threads(), len(sample_t))
    grads = {t: workloads.tensor_grad(CFG, layout, 0, t, device="cpu").numpy() for t in sample_t}
    n = sum(layout.sizes[t] for t in sample_t)
    off = layout.off

    def one(it):
        def task(t):
            e = np.zeros_like(grads[t])
            oracle.ef_topk_tensor(grads[t], e, int(k[t]), base=int(off[t]), int8=INT8, seed=0, it=it)
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(task, sample_t))

    for w in range(args.warmup):
        one(w)
    t0 = time.perf_counter()
    for s in range(args.steps):
        one(args.warmup + s)
    secs = time.perf_counter() - t0
    value = 4.0 * n * args.steps / secs / 1e9
    sample = "tensors %d..%d of the arena (%d elements) per step, one per thread" % (sample_t[0], sample_t[-1], n)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": workload_config(layout, k),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample,
                             "host": host_description()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- headline

def run_ours(args):
    import gradient_compression_gb300 as gc

    ws, rank, local = dist_info()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    layout = workloads.LAYOUTS[CFG]()
    k = workloads.k_per_tensor(layout.sizes, RHO)
    N = layout.numel
    flags = gc.GC_EF | (gc.GC_INT8 if INT8 else 0)
    L = gc.Layout(layout.off, k, device=dev)
    # two resident gradients, alternated step by step (a fresh gradient each
    # step as far as the EF state can tell; 2 x 32 GB + e fits in HBM)
    grads = [workloads.make_grad(CFG, layout, i, device=dev) for i in range(2)]
    e = torch.zeros(N, dtype=torch.float32, device=dev)
    comp = gc.TopkCompressor(L, flags, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(it, e_buf, events=None):
        gi = grads[it % 2]
        if events is None:
            gc.ef_topk_compress(L, gi, e_buf, comp.idx, comp.val, comp.q, comp.scale, 1234, it, flags,
                                comp.workspace)
        else:
            gc.ef_topk_compress_profiled(L, gi, e_buf, comp.idx, comp.val, comp.q, comp.scale, 1234, it, flags,
                                         comp.workspace, events)

    for w in range(args.warmup):
        step(w, e)
    torch.cuda.synchronize()
    e_start = e.clone()            # for the untimed replay of the timed steps below

    ph = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    t_begin, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_begin.record(stream)
    for s in range(args.steps):
        step(args.warmup + s, e, ph[s])
    t_end.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    total_ms = t_begin.elapsed_time(t_end)
    stream_ms = [p[1].elapsed_time(p[2]) for p in ph]
    phase = {"sample_ms": statistics.mean(p[0].elapsed_time(p[1]) for p in ph),
             "stream_ms": statistics.mean(stream_ms),
             "select_ms": statistics.mean(p[2].elapsed_time(p[3]) for p in ph),
             "write_ms": statistics.mean(p[3].elapsed_time(p[4]) for p in ph)}
    total_ms = max_over_ranks(total_ms, dev)
    ms_per_step = total_ms / args.steps
    value = job_gradient_gbs(N, ws, ms_per_step)
    peak, peak_kind = measured_peaks()
    t_stream = statistics.mean(stream_ms) * 1e-3
    achieved = STREAM_BYTES_PER_ELEM * N / t_stream / 1e9
    bpe = profiled_traffic()
    algo_step_bytes = 12 * N + (5 * int(k.sum()) + 4 * layout.num_tensors if INT8 else 8 * int(k.sum()))

    # The timed steps again, untimed, from the same residual: each step's
    # selection diagnostics (the calls are deterministic), and the final
    # residual must be bit-identical to the timed run's.
    exact, overflow = [], []
    for s in range(args.steps):
        step(args.warmup + s, e_start)
        d = gc.get_device_status(comp.workspace)
        exact.append(int(d.exact_tensors))
        overflow.append(int(d.overflow_tensors))
    replay_identical = bool(torch.equal(e_start.view(torch.int32), e.view(torch.int32)))
    del e_start
    torch.cuda.empty_cache()

    lazy = measure_lazy(gc, L, layout, k, grads, comp, flags, dev, args, algo_step_bytes, peak)

    e2e = None
    if not args.no_e2e:
        g_keep = grads[0]
        del grads[1:]
        torch.cuda.empty_cache()
        e2e = measure_e2e(gc, L, layout, k, g_keep, e, comp, flags, dev, args)
    del e, comp
    torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        threads = oracle_threads()
        it0 = oracle_full_iteration(gc, layout, k, grads[0], dev, threads)
        cpu = {"value": it0["gbs"], "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": "the whole arena (%d tensors, %d elements), iteration 0 with e = 0, tensors in "
                         "parallel, one per thread; %.1f s wall, %.1f s of oracle time"
                         % (it0["tensors"], it0["elements"], it0["wall_s"], it0["cpu_s"]),
               "agrees_with_gpu": it0["agrees"], "host": host_description()}
    del grads
    torch.cuda.empty_cache()

    rows = None
    if not args.no_rows and ws == 1:
        rows = measure_rows(gc, dev, args)
        if cpu is not None:
            cpu["config_workloads"] = oracle_config_workloads(dev, oracle_threads())

    if rank != 0:
        return
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": workload_config(layout, k),
            "elems_per_s": ws * N / (ms_per_step * 1e-3),
            "hbm_roofline_frac_step": (algo_step_bytes / (ms_per_step * 1e-3) / 1e9) / peak,
            "roofline": {"bound": "hbm", "kernel": "k_stream (acc = g + e, e write-back, candidate emission)",
                         "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": achieved / peak,
                         "traffic": None if bpe is None else bpe * N,
                         "algorithmic_bytes": STREAM_BYTES_PER_ELEM * N},
            "phases_ms": phase,
            "timed_steps_selection": {"exact_tensors": exact, "overflow_tensors": overflow,
                                      "replay_bit_identical": replay_identical},
            "lazy_residual": lazy,
            "gpu_launches": LAUNCHES_PER_STEP * args.steps, "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu,
            "rows": rows}
    print(json.dumps(line), flush=True)


def measure_lazy(gc, L, layout, k, grads, comp, flags, dev, args, algo_step_bytes, peak):
    """The same steps through gc_ef_topk_compress_lazy (residual update deferred
    into the next call's streaming pass; payloads bit-identical)."""
    N = layout.numel
    e = torch.zeros(N, dtype=torch.float32, device=dev)
    rd = gc.alloc_residual_desc(L, device=dev)

    def one(it):
        gc.ef_topk_compress_lazy(L, grads[it % 2], e, rd, comp.idx, comp.val, comp.q, comp.scale, 1234, it,
                                 flags & ~gc.GC_EF, comp.workspace)

    for w in range(args.warmup):
        one(w)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for s in range(args.steps):
        one(args.warmup + s)
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / args.steps
    del e
    return {"ms_per_step": ms, "value": 4.0 * N / (ms * 1e-3) / 1e9, "unit": UNIT,
            "hbm_roofline_frac_step": (algo_step_bytes / (ms * 1e-3) / 1e9) / peak,
            "entry": "gc_ef_topk_compress_lazy"}


def measure_e2e(gc, L, layout, k, g, e, comp, flags, dev, args):
    """Same metric through the public API with the gradient in pinned host
    memory: each step the library's kernels read g in place from host memory
    (zero-copy over NVLink-C2C, 4N bytes host -> device), compress, and the
    payload (indices, codes, scales) is copied back to pinned host memory.
    Timed over the same number of steps as the device-resident value."""
    N = layout.numel
    K = int(k.sum())
    try:
        g_host = torch.empty(N, dtype=torch.float32, pin_memory=True)
    except RuntimeError as exc:
        return {"value": None, "unit": UNIT, "error": "pinned host buffer: %s" % str(exc)[:120]}
    g_host.copy_(g, non_blocking=False)
    idx_h = torch.empty(K, dtype=torch.int32, pin_memory=True)
    q_h = torch.empty(K, dtype=torch.int8 if INT8 else torch.float32, pin_memory=True)
    sc_h = torch.empty(layout.num_tensors, dtype=torch.float32, pin_memory=True)
    steps = args.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def one(it):
        gc.ef_topk_compress(L, g_host, e, comp.idx, comp.val, comp.q, comp.scale, 99, it, flags, comp.workspace)
        idx_h.copy_(comp.idx[:K], non_blocking=True)
        if INT8:
            q_h.copy_(comp.q[:K], non_blocking=True)
            sc_h.copy_(comp.scale, non_blocking=True)
        else:
            q_h.copy_(comp.val[:K], non_blocking=True)

    one(0)
    torch.cuda.synchronize()
    t0.record()
    for s in range(steps):
        one(1 + s)
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    del g_host
    return {"value": 4.0 * N / (ms * 1e-3) / 1e9, "unit": UNIT, "ms_per_step": ms, "steps": steps,
            "h2d_bytes_per_step": 4 * N,
            "d2h_bytes_per_step": (5 * K + 4 * layout.num_tensors) if INT8 else 8 * K,
            "h2d": "g read in place from pinned host memory by the kernels (NVLink-C2C)"}


# ---------------------------------------------------------------------------- other rows

# layout name -> generator config of workloads.LAYOUTS
LAYOUT_CFG = {"flat": 1, "resnet50": 2, "bert_large": 3, "gpt2_medium": 4, "llama3_8b": 5}

# row -> (layout, op, density, steps (the configuration's iterations), what)
ROWS = {
    "flat_2p20_ef_topk_0.1pct": ("flat", "topk", 0.001, 10, "EF Top-k, k = 1049 of 2^20 (one tensor; L2 flushed "
                                 "between steps; latency-bound)"),
    "resnet50_ef_topk_1pct": ("resnet50", "topk", 0.01, 20, "per-tensor EF Top-k at 1%"),
    "resnet50_randk_1pct": ("resnet50", "randk", 0.01, 20, "random-k (Philox keys) with EF at 1%"),
    "bert_large_ef_topk_0.1pct_int8": ("bert_large", "topk_int8", 0.001, 10,
                                       "EF Top-k 0.1% + int8 stochastic rounding of the kept values"),
    "bert_large_ef_topk_0.1pct_qsgd16": ("bert_large", "topk_qsgd", 0.001, 10,
                                         "EF Top-k 0.1% + QSGD s = 16 of the kept values (norm of the kept set)"),
    "bert_large_ef_topk_0.1pct_sign": ("bert_large", "topk_sign", 0.001, 10,
                                       "EF Top-k 0.1% + sign bits of the kept values (mean |kept| scale)"),
    "gpt2_medium_sign_ef": ("gpt2_medium", "sign", None, 10, "1-bit sign + EF, mean-|acc| scale per tensor"),
    "gpt2_medium_sign_ef_one_pass": ("gpt2_medium", "sign_lazy", None, 10,
                                     "1-bit sign + EF, one pass (residual applied by the next call)"),
    "gpt2_medium_qsgd16": ("gpt2_medium", "qsgd", None, 10, "QSGD s = 16 (Philox stochastic rounding), no EF"),
    "gpt2_medium_int8_sr_ef": ("gpt2_medium", "int8", None, 10, "dense int8 stochastic rounding + EF"),
    "gpt2_medium_momentum_topk_0.5pct": ("gpt2_medium", "momentum", 0.005, 10,
                                         "DGC momentum correction + Top-k 0.5%, beta 0.9, factor masking"),
    "llama3_8b_decompress_w8": ("llama3_8b", "decompress", 0.001, 10,
                                "scatter-add of W = 8 workers' sparse fp32 payloads (0.1% each)"),
    "bert_large_threshold": ("bert_large", "threshold", 0.002, 10,
                             "threshold |acc| >= 1e-2 with EF, capped at 0.2% per tensor"),
    "bert_large_clip_ef_topk_0.1pct": ("bert_large", "clip", 0.001, 10,
                                       "DGC local clipping (max norm = half of ||g_t||) + EF Top-k 0.1%"),
    "bert_large_powersgd_r4": ("bert_large", "powersgd", None, 10, "PowerSGD rank 4 with EF on every weight matrix"),
    "bert_large_powersgd_r4_lazy": ("bert_large", "powersgd_lazy", None, 10,
                                    "PowerSGD rank 4 with EF, residual kept pending (two passes over M per call)"),
}
# --op name -> row (the short names of the single-row mode)
OPS = {"flat": "flat_2p20_ef_topk_0.1pct", "resnet_topk": "resnet50_ef_topk_1pct", "randk": "resnet50_randk_1pct",
       "bert_topk_int8": "bert_large_ef_topk_0.1pct_int8", "topk_qsgd": "bert_large_ef_topk_0.1pct_qsgd16",
       "topk_sign": "bert_large_ef_topk_0.1pct_sign", "sign": "gpt2_medium_sign_ef",
       "sign_lazy": "gpt2_medium_sign_ef_one_pass", "qsgd": "gpt2_medium_qsgd16", "int8": "gpt2_medium_int8_sr_ef",
       "momentum": "gpt2_medium_momentum_topk_0.5pct", "decompress": "llama3_8b_decompress_w8",
       "threshold": "bert_large_threshold", "clip": "bert_large_clip_ef_topk_0.1pct",
       "powersgd": "bert_large_powersgd_r4", "powersgd_lazy": "bert_large_powersgd_r4_lazy"}


def measure_row(gc, dev, name, warmup, steps=None, layout_name=None):
    """One compression path on its own workload: per-call device time (CUDA
    events around each call on its stream), gradient GB/s and the fraction of
    the measured HBM copy peak reached with the row's algorithmic bytes."""
    lname, op, rho, row_steps, what = ROWS[name]
    if layout_name:
        lname = layout_name
    steps = steps or row_steps
    cfg = LAYOUT_CFG[lname]
    layout = workloads.LAYOUTS[cfg]()
    N, T = layout.numel, layout.num_tensors
    k = workloads.k_per_tensor(layout.sizes, rho) if rho else np.zeros(T, np.int64)
    L = gc.Layout(layout.off, k, device=dev)
    K = int(k.sum())
    flush = None
    if 12 * N < 2 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    if op == "decompress":
        grads = []
    elif lname == "flat":
        grads = [workloads.make_grad(cfg, layout, i, device=dev) for i in range(warmup + steps)]
    else:
        grads = [workloads.make_grad(cfg, layout, i, device=dev) for i in range(2)]
    extra = {}
    if op in ("topk", "topk_int8", "randk", "momentum", "clip", "threshold"):
        int8 = op == "topk_int8"
        flags = {"topk": gc.GC_EF, "topk_int8": gc.GC_EF | gc.GC_INT8, "randk": gc.GC_EF | gc.GC_RANDK,
                 "momentum": 0, "clip": gc.GC_EF, "threshold": gc.GC_EF}[op]
        ws = gc.alloc_workspace(L, gc.GC_OP_MOMENTUM if op == "momentum" else gc.GC_OP_TOPK, flags)
        idx = torch.empty(max(K, 1), dtype=torch.int32, device=dev)
        val = None if int8 else torch.empty(max(K, 1), dtype=torch.float32, device=dev)
        q = torch.empty(max(K, 1), dtype=torch.int8, device=dev) if int8 else None
        sc = torch.empty(T, dtype=torch.float32, device=dev) if int8 else None
        a = torch.zeros(N, device=dev)
        b = torch.zeros(N, device=dev) if op == "momentum" else None
        cnt = torch.zeros(T, dtype=torch.int64, device=dev)
        norm = torch.empty(T, device=dev)
        tau = torch.full((T,), 1e-2, device=dev)
        cap = None
        if op == "clip":
            cap = torch.stack([0.5 * torch.linalg.vector_norm(grads[0][int(L.off[t]):int(L.off[t + 1])])
                               for t in range(T)]).float()

        def step(it):
            g = grads[it % len(grads)]
            if op == "momentum":
                gc.ef_topk_compress_momentum(L, g, a, b, 0.9, idx, val, None, None, 5, it, 0, ws)
            elif op == "clip":
                gc.ef_topk_compress_clipped(L, g, a, cap, norm, idx, val, None, None, 5, it, flags, ws)
            elif op == "threshold":
                gc.ef_threshold_compress(L, g, a, tau, cnt, idx, val, None, None, 5, it, flags, ws)
            else:
                gc.ef_topk_compress(L, g, a, idx, val, q, sc, 5, it, flags, ws)
        per_elem = {"momentum": 20, "clip": 16}.get(op, 12)
        if op == "threshold":
            step(0)
            torch.cuda.synchronize()
            K = int(cnt.sum())
            extra["kept_per_step"] = K
        algo = per_elem * N + ((5 * K + 4 * T) if int8 else 8 * K)
    elif op in ("topk_qsgd", "topk_sign"):
        kind = gc.GC_KEPT_QSGD if op == "topk_qsgd" else gc.GC_KEPT_SIGN
        ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, gc.GC_EF)
        idx = torch.empty(max(K, 1), dtype=torch.int32, device=dev)
        q = torch.empty(max(K, 1), dtype=torch.int8, device=dev) if op == "topk_qsgd" else None
        bits = torch.empty(max(L.kept_words, 1), dtype=torch.int32, device=dev) if op == "topk_sign" else None
        sc = torch.empty(T, dtype=torch.float32, device=dev)
        e = torch.zeros(N, device=dev)

        def step(it):
            gc.ef_topk_compress_quantized(L, grads[it % 2], e, idx, None, q, bits, sc, kind, 16, 5, it, gc.GC_EF, ws)
        algo = 12 * N + (5 * K if op == "topk_qsgd" else 4 * K + 4 * L.kept_words) + 4 * T
    elif op in ("powersgd", "powersgd_lazy"):
        mats = workloads.matrices_of(layout)
        ml = gc.MatrixLayout([int(layout.off[t]) for t, _, _ in mats], [m for _, m, _ in mats],
                             [n for _, _, n in mats], device=dev)
        R = 4
        e = torch.zeros(N, device=dev)
        qv = torch.randn(int(ml.qoff[-1]) * R, device=dev)
        pv = torch.empty(int(ml.poff[-1]) * R, device=dev)
        ws = gc.powersgd_workspace(ml, R)
        pvs = [pv, torch.empty_like(pv)]

        def step(it):
            if op == "powersgd":
                gc.powersgd_compress(ml, R, grads[it % 2], e, qv, pv, None, ws)
            else:
                gc.powersgd_compress_lazy(ml, R, grads[it % 2], e, qv, pvs[it % 2], None if it == 0 else pvs[(it - 1) % 2],
                                          None, ws)
        melems = sum(m * n for _, m, n in mats)
        algo = 12 * melems + 4 * R * (int(ml.poff[-1]) + int(ml.qoff[-1]))
        extra = {"matrices": len(mats), "matrix_elements": melems, "rank": R,
                 "passes": ("M = G + E and P = MQ (12 B/elt), Q = M^T P (4), E = M - PQ^T (8)" if op == "powersgd"
                            else "E = M_prev - P_prev Q_prev^T, M = G + E and P = MQ (12 B/elt), Q = M^T P (4)")}
    elif op in ("sign", "sign_lazy", "qsgd", "int8"):
        ws = gc.alloc_workspace(L, gc.GC_OP_QUANTIZE if op in ("qsgd", "int8") else gc.GC_OP_SIGN)
        sc = torch.empty(T, device=dev)
        e = torch.zeros(N, device=dev)
        if op == "sign_lazy":
            bits = torch.empty(L.words, dtype=torch.int32, device=dev)
            mus = [torch.empty(T, device=dev) for _ in range(2)]

            def step(it):
                gc.sign_compress_lazy(L, grads[it % 2], e, None if it == 0 else mus[(it - 1) % 2], bits,
                                      mus[it % 2], ws)
        elif op == "sign":
            bits = torch.empty(L.words, dtype=torch.int32, device=dev)

            def step(it):
                gc.sign_compress(L, grads[it % 2], e, bits, sc, ws)
        else:
            codes = torch.empty(N, dtype=torch.int8, device=dev)
            mode = gc.GC_Q_QSGD if op == "qsgd" else gc.GC_Q_INT8

            def step(it):
                gc.quantize_stochastic(L, grads[it % 2], None if op == "qsgd" else e, codes, sc, mode, 16, 5, it, ws)
        algo = {"sign": 12.125, "sign_lazy": 12.125, "qsgd": 5, "int8": 13}[op] * N + 4 * T
    else:  # decompress
        W = 8
        pays = [workloads.make_sparse_payload(layout, k, w, device=dev, cfg=cfg) for w in range(W)]
        out = torch.zeros(N, device=dev)
        ws = gc.alloc_workspace(L, gc.GC_OP_DECOMPRESS)
        idxs, vals = [p[0] for p in pays], [p[1] for p in pays]
        touched = 0
        for t in range(T):
            a0, b0 = int(L.koff[t]), int(L.koff[t + 1])
            if b0 > a0:
                touched += int(torch.unique(torch.cat([ix[a0:b0] for ix in idxs])).numel())

        def step(it):
            gc.sparse_decompress_accumulate(L, idxs, vals, None, None, out, ws)
        algo = 8 * touched + 8 * K * W
        extra = {"workers": W, "touched_elements": touched, "payload_entries": K * W,
                 "sector_bound_bytes": 64 * K * W + 8 * K * W}
    for w in range(warmup):
        step(w)
    torch.cuda.synchronize()
    if op in ("topk", "randk") and lname in ("flat", "resnet50"):
        extra["graph_replay"] = graph_replay(gc, L, grads, a, idx, val, flags, ws, warmup, steps, flush)
    if op in ("topk", "topk_int8", "randk", "momentum", "clip", "threshold", "topk_qsgd", "topk_sign"):
        d = gc.get_device_status(ws)
        extra["last_warmup_call"] = {"exact_tensors": int(d.exact_tensors), "overflow_tensors": int(d.overflow_tensors)}
    if op == "topk":
        extra["one_launch"] = int(gc.get_device_status(ws).one_launch)
        if extra["one_launch"]:
            extra["multi_kernel"] = multi_kernel_time(gc, L, grads, a, idx, val, flags, ws, warmup, steps, flush)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for s_ in range(steps):
        if flush is not None:
            flush.zero_()
        evs[s_][0].record()
        step(warmup + s_)
        evs[s_][1].record()
    torch.cuda.synchronize()
    times = [a_.elapsed_time(b_) for a_, b_ in evs]
    ms = statistics.mean(times)
    peak, peak_kind = measured_peaks()
    achieved = algo / (ms * 1e-3) / 1e9
    row = {"what": what, "layout": lname, "tensors": T, "elements": N, "kept": K, "density": rho, "steps": steps,
           "ms_per_call": ms, "ms_min": min(times), "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak,
                                                                 "peak_kind": peak_kind, "unit": "GB/s",
                                                                 "frac": achieved / peak, "algorithmic_bytes": algo},
           "l2": "flushed between calls" if flush is not None else "inputs larger than L2"}
    if op == "decompress":
        row.update(value=K * extra["workers"] / (ms * 1e-3) / 1e9, unit="G entries/s")
        row["sector_bound_frac"] = extra["sector_bound_bytes"] / (ms * 1e-3) / 1e9 / peak
        extra["random_access_reference"] = random_access_reference(L, k, idxs, vals, out, ms)
    else:
        row.update(value=4.0 * N / (ms * 1e-3) / 1e9, unit=UNIT, elems_per_s=N / (ms * 1e-3))
    if op in ("qsgd", "randk"):
        # Philox4x32-10 draws one 32-bit word per element: 10 rounds of two
        # 32x32 -> 64-bit products per block of 4 words, each product an
        # integer multiply-high and multiply-low, so 10 integer multiplies
        # per element; the integer multiply-add rate is 64 per SM per clock.
        sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
        imad_peak = sm_count * 64 * 2070.0 * 1e6
        imad_done = IMAD_PER_ELEMENT * N / (ms * 1e-3)
        row["alu"] = {"bound": "alu", "unit": "G int-mul/s", "per_element": IMAD_PER_ELEMENT,
                      "achieved": imad_done / 1e9, "peak": imad_peak / 1e9, "frac": imad_done / imad_peak,
                      "peak_from": "%d SMs x 64 per clock x 2070 MHz" % sm_count}
    row.update(extra)
    return row


def random_access_reference(L, k, idxs, vals, out, ms, reps=5):
    """What the memory system gives for the receiver's access pattern with
    PyTorch's own kernels, on the same arena and the same W payloads'
    positions (arena-global, worker after worker): a plain gather (random
    reads only) and index_add_ (random read-modify-writes).  A yardstick for
    the receiver, not part of any path."""
    dev = out.device
    base = torch.repeat_interleave(torch.as_tensor(np.asarray(L.off[:-1], np.int64), device=dev),
                                   torch.as_tensor(np.asarray(k, np.int64), device=dev))
    gidx = torch.cat([ix.long() + base for ix in idxs])
    v = torch.cat(vals)
    buf = torch.empty_like(v)
    res = {}
    for name, fn in (("gather_ms", lambda: torch.index_select(out, 0, gidx, out=buf)),
                     ("index_add_ms", lambda: out.index_add_(0, gidx, v))):
        fn()
        fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        torch.cuda.synchronize()
        for a_, b_ in evs:
            a_.record()
            fn()
            b_.record()
        torch.cuda.synchronize()
        res[name] = statistics.mean(a_.elapsed_time(b_) for a_, b_ in evs)
    del gidx, v, buf
    torch.cuda.empty_cache()
    res["receiver_ms"] = ms
    res["how"] = ("torch.index_select (random reads) and Tensor.index_add_ (random read-modify-writes) of the "
                  "same payload positions in the same arena, mean of %d calls" % reps)
    return res


def multi_kernel_time(gc, L, grads, e, idx, val, flags, ws, warmup, steps, flush):
    """The same calls through the multi-kernel pipeline (GC_MULTI_KERNEL), for
    comparison with the one-launch path.  Runs on a copy of the state."""
    e = e.clone()
    fl = flags | gc.GC_MULTI_KERNEL
    for w in range(warmup):
        gc.ef_topk_compress(L, grads[w % len(grads)], e, idx, val, None, None, 5, w, fl, ws)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for s_ in range(steps):
        if flush is not None:
            flush.zero_()
        evs[s_][0].record()
        gc.ef_topk_compress(L, grads[(warmup + s_) % len(grads)], e, idx, val, None, None, 5, warmup + s_, fl, ws)
        evs[s_][1].record()
    torch.cuda.synchronize()
    times = [a_.elapsed_time(b_) for a_, b_ in evs]
    return {"ms_per_call": statistics.mean(times), "ms_min": min(times),
            "how": "the same calls with GC_MULTI_KERNEL (14 chained kernels)"}


def graph_replay(gc, L, grads, e, idx, val, flags, ws, warmup, steps, flush):
    """The same call captured once per resident gradient into a CUDA graph
    (gc_ef_topk_compress_dev_iter: the iteration counter lives on the device
    and advances per replay) and replayed alternately: the per-call time
    without the host's per-launch work.  Runs on copies of the state."""
    dev = grads[0].device
    e = e.clone()
    it_dev = torch.zeros(1, dtype=torch.int64, device=dev)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graphs = []
    for g in grads[:2]:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                gc.ef_topk_compress_dev_iter(L, g, e, idx, val, None, None, 5, it_dev, flags, ws)
        graphs.append(graph)
    torch.cuda.synchronize()
    for w in range(warmup):
        graphs[w % 2].replay()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for s_ in range(steps):
        if flush is not None:
            flush.zero_()
        evs[s_][0].record()
        graphs[s_ % 2].replay()
        evs[s_][1].record()
    torch.cuda.synchronize()
    times = [a_.elapsed_time(b_) for a_, b_ in evs]
    del graphs
    return {"ms_per_call": statistics.mean(times), "ms_min": min(times),
            "how": "one CUDA-graph capture of gc_ef_topk_compress_dev_iter per resident gradient, replayed "
                   "alternately (two of the gradients)"}


def measure_rows(gc, dev, args):
    sampler = ClockSampler(0)
    time.sleep(0.2)
    rows = {}
    t0 = time.perf_counter()
    for name in ROWS:
        rows[name] = measure_row(gc, dev, name, max(3, args.warmup))
        torch.cuda.empty_cache()
    rows["clocks"] = sampler.stop()
    rows["wall_s"] = round(time.perf_counter() - t0, 1)
    return rows


def run_op(args):
    """Measures one of the other compression rows on its own workload (one JSON line)."""
    import gradient_compression_gb300 as gc

    dev = torch.device("cuda", 0)
    name = OPS[args.op]
    sampler = ClockSampler(0)
    time.sleep(0.2)
    row = measure_row(gc, dev, name, args.warmup, steps=args.steps, layout_name=args.layout)
    clocks = sampler.stop()
    line = {"metric": "%s (%s)" % (name, row["unit"]), "value": row["value"], "unit": row["unit"], "n_gpus": 1,
            "steps": row["steps"], "warmup": args.warmup, "ms_per_step": row["ms_per_call"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": name, "what": row["what"], "layout": row["layout"], "tensors": row["tensors"],
                       "elements": row["elements"], "kept": row["kept"], "density": row["density"]},
            "roofline": row["roofline"], "clocks": clocks, "row": row}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="llama3_8b",
                    help="the measured workload is llama3_8b; the others are smaller cases for profiling")
    ap.add_argument("--op", choices=("topk",) + tuple(OPS), default="topk",
                    help="topk is the measured headline (with every row); the others measure one row alone")
    ap.add_argument("--layout", choices=sorted(LAYOUT_CFG), default=None,
                    help="with --op: run that row on another layout (smaller cases for profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rows", action="store_true", help="headline only")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    global CFG, RHO, INT8
    CFG, RHO, INT8 = WORKLOADS[args.workload][:3]
    if args.impl == "reference":
        run_reference(args)
    elif args.op != "topk":
        run_op(args)
    else:
        if args.workload != "llama3_8b":
            args.no_rows = True
        run_ours(args)


if __name__ == "__main__":
    main()
