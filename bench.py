"""Benchmark: EF Top-k (0.1%) + int8 compression of a Llama-3-8B-shaped fp32
gradient arena (291 tensors, 8,030,261,248 elements) on one GB300.

One step = one gc_ef_topk_compress call over the whole arena: acc = g + e,
per-tensor Top-k by |acc|, int8 stochastic rounding of the kept values,
index/code payload, residual update.  Inputs (g, e: 64.2 GB) are resident in
HBM and larger than L2, so no L2 flush is needed between steps.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle
instead, on a bounded sample of the same workload.

Multi-GPU: the compression of one worker's gradient does not shard (each
data-parallel worker compresses its own gradient with its own residual), so
N > 1 runs N independent replicas, one per GPU; value = all ranks' elements
over the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "EF Top-k compress gradient GB/s (elems/s) at 1 GB300; % of HBM roofline"
UNIT = "GB/s"
# workload name -> (generator config id, density, int8, oracle-baseline tensors, reference-arm tensor)
WORKLOADS = {
    "llama3_8b": (5, 0.001, True, list(range(1, 10)), 1),
    "bert_large": (3, 0.001, True, list(range(0, 3)), 0),
    "resnet50": (2, 0.01, False, list(range(0, 161)), 160),
    "flat_2p20": (1, 0.001, False, [0], 0),
}
CFG, RHO, INT8 = 5, 0.001, True
# kernels libgc launches per gc_ef_topk_compress call (Top-k mode): plan,
# the sampled threshold estimate, the streaming pass, the level-1 select,
# three histogram passes (full-pass level 1, candidate levels 2 and 3) with
# their selects, count, scan, write
LAUNCHES_PER_STEP = 13
# bytes the streaming pass must move per element: read g, read e, write e
STREAM_BYTES_PER_ELEM = 12
# integer multiplies of one Philox4x32-10 word (random-k keys, QSGD rounding)
IMAD_PER_ELEMENT = 10


GRADIENT = {1: "student_t_nu3_x1e-3", 2: "laplace_loguniform_scale", 3: "student_t_nu2.5_x1e-3",
            5: "student_t_nu3_x1e-3"}


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


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("gc_topk.cu", "gc_common.cuh"):
        with open(os.path.join(ROOT, "gradient_compression_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the streaming pass from the committed ncu summary,
    scaled to this workload; None if missing or taken on different kernel source."""
    p = os.path.join(ROOT, "profiles", "k_stream_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    if d.get("source_hash") != kernel_source_hash():
        return None
    return float(d["bytes_per_element"])


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
        load = [r for r in rows if r["util"] >= 50] or rows
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load), "sm_max_mhz": max(r["max"] for r in load),
                "reasons": sorted(reasons), "samples": len(load)}


def oracle_baseline(layout, k, tensors, it=0, seed=0):
    """Times the oracle (single thread) on the given tensors; returns (GB/s, seconds, elements)."""
    import oracle
    oracle.lib()
    n_tot, secs = 0, 0.0
    off = layout.off
    for t in tensors:
        g = workloads.tensor_grad(CFG, layout, it, t, device="cpu").numpy()
        e = np.zeros_like(g)
        t0 = time.perf_counter()
        oracle.ef_topk_tensor(g, e, int(k[t]), base=int(off[t]), int8=INT8, seed=seed, it=it)
        secs += time.perf_counter() - t0
        n_tot += g.size
    return 4.0 * n_tot / secs / 1e9, secs, n_tot


def run_reference(args):
    ws, rank, _ = dist_info()
    if rank != 0:
        return
    layout = workloads.LAYOUTS[CFG]()
    k = workloads.k_per_tensor(layout.sizes, RHO)
    sample_t = [WORKLOADS[args.workload][4]]
    sample = "tensor %d (%d elements) of the arena per step" % (sample_t[0], layout.sizes[sample_t[0]])
    for w in range(args.warmup):
        oracle_baseline(layout, k, sample_t, it=w)
    vals, secs_all = [], 0.0
    for s in range(args.steps):
        v, secs, n = oracle_baseline(layout, k, sample_t, it=args.warmup + s)
        vals.append(v)
        secs_all += secs
    value = 4.0 * n * args.steps / secs_all / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs_all / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": workload_config(layout, k),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


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
    g = grads[0]
    e = torch.zeros(N, dtype=torch.float32, device=dev)
    comp = gc.TopkCompressor(L, flags, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(it, events=None):
        gi = grads[it % 2]
        if events is None:
            gc.ef_topk_compress(L, gi, e, comp.idx, comp.val, comp.q, comp.scale, 1234, it, flags, comp.workspace)
        else:
            gc.ef_topk_compress_profiled(L, gi, e, comp.idx, comp.val, comp.q, comp.scale, 1234, it, flags,
                                         comp.workspace, events)

    for w in range(args.warmup):
        step(w)
    torch.cuda.synchronize()
    diag = gc.get_device_status(comp.workspace)

    ph = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    t_begin, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_begin.record(stream)
    for s in range(args.steps):
        step(args.warmup + s, ph[s])
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

    lazy = measure_lazy(gc, L, layout, k, grads, comp, flags, dev, args, algo_step_bytes, peak)

    e2e = None
    if not args.no_e2e:
        del grads[1:]
        torch.cuda.empty_cache()
        e2e = measure_e2e(gc, L, layout, k, g, e, comp, flags, dev, args)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        tensors = WORKLOADS[args.workload][3]
        v, secs, n = oracle_baseline(layout, k, tensors)
        cpu = {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": "tensors %d..%d of the arena (%d elements), one iteration, %.1f s"
               % (tensors[0], tensors[-1], n, secs)}

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
            "phases_ms": phase, "exact_tensors_warmup": int(diag.exact_tensors), "lazy_residual": lazy,
            "gpu_launches": LAUNCHES_PER_STEP * args.steps, "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu}
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
    The gradient is regenerated host-side copies of the resident ones."""
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
    steps = max(2, min(args.steps, 5))
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
    return {"value": 4.0 * N / (ms * 1e-3) / 1e9, "unit": UNIT, "ms_per_step": ms, "steps": steps,
            "h2d_bytes_per_step": 4 * N,
            "d2h_bytes_per_step": (5 * K + 4 * layout.num_tensors) if INT8 else 8 * K,
            "h2d": "g read in place from pinned host memory by the kernels (NVLink-C2C)"}


# ---------------------------------------------------------------------------- other rows

# layout name -> generator config of workloads.LAYOUTS
LAYOUT_CFG = {"resnet50": 2, "bert_large": 3, "gpt2_medium": 4, "llama3_8b": 5}

OPS = {
    # op: (generator config, layout, density, what, algorithmic bytes per element, per kept, per tensor)
    "randk": (2, "resnet50", 0.01, "random-k (Philox keys) with EF", 12, 8, 0),
    "momentum": (4, "gpt2_medium", 0.005, "DGC momentum correction + Top-k, beta 0.9, factor masking", 20, 8, 0),
    "sign": (4, "gpt2_medium", None, "1-bit sign + EF, mean-|acc| scale per tensor", 12.125, 0, 4),
    "sign_lazy": (4, "gpt2_medium", None, "1-bit sign + EF, one pass (residual applied by the next call)",
                  12.125, 0, 4),
    "qsgd": (4, "gpt2_medium", None, "QSGD s = 16 (Philox stochastic rounding), no EF", 5, 0, 4),
    "decompress": (5, "llama3_8b", 0.001, "scatter-add of W = 8 workers' sparse fp32 payloads", 0, 0, 0),
    "threshold": (3, "bert_large", 0.002, "threshold |acc| >= 1e-2 with EF, capped at 0.2% per tensor", 12, 8, 0),
    "clip": (3, "bert_large", 0.001, "DGC local clipping (max norm = half of ||g_t||) + EF Top-k 0.1%", 16, 8, 0),
    "powersgd": (3, "bert_large", None, "PowerSGD rank 4 with EF on every weight matrix", 12, 0, 0),
}


def run_op(args):
    """Measures one of the other compression rows on its own workload (one JSON line)."""
    import gradient_compression_gb300 as gc
    import oracle

    dev = torch.device("cuda", 0)
    cfg, lname, rho, what, b_elem, b_kept, b_tensor = OPS[args.op]
    if args.layout:
        cfg, lname = LAYOUT_CFG[args.layout], args.layout
    layout = workloads.LAYOUTS[cfg]()
    N, T = layout.numel, layout.num_tensors
    k = workloads.k_per_tensor(layout.sizes, rho) if rho else np.zeros(T, np.int64)
    L = gc.Layout(layout.off, k, device=dev)
    K = int(k.sum())
    grads = [workloads.make_grad(cfg, layout, i, device=dev) for i in range(2)] if args.op != "decompress" else []
    extra = {}
    if args.op in ("randk", "momentum"):
        flags = (gc.GC_EF | gc.GC_RANDK) if args.op == "randk" else 0
        op = gc.GC_OP_TOPK if args.op == "randk" else gc.GC_OP_MOMENTUM
        ws = gc.alloc_workspace(L, op, flags)
        idx = torch.empty(K, dtype=torch.int32, device=dev)
        val = torch.empty(K, dtype=torch.float32, device=dev)
        a = torch.zeros(N, device=dev)
        b = torch.zeros(N, device=dev) if args.op == "momentum" else None

        def step(it):
            if args.op == "randk":
                gc.ef_topk_compress(L, grads[it % 2], a, idx, val, None, None, 5, it, flags, ws)
            else:
                gc.ef_topk_compress_momentum(L, grads[it % 2], a, b, 0.9, idx, val, None, None, 5, it, 0, ws)
        algo = b_elem * N + b_kept * K
    elif args.op == "powersgd":
        mats = workloads.matrices_of(layout)
        ml = gc.MatrixLayout([int(layout.off[t]) for t, _, _ in mats], [m for _, m, _ in mats],
                             [n for _, _, n in mats], device=dev)
        R = 4
        e = torch.zeros(N, device=dev)
        qv = torch.randn(int(ml.qoff[-1]) * R, device=dev)
        pv = torch.empty(int(ml.poff[-1]) * R, device=dev)
        ws = gc.powersgd_workspace(ml, R)

        def step(it):
            gc.powersgd_compress(ml, R, grads[it % 2], e, qv, pv, None, ws)
        melems = sum(m * n for _, m, n in mats)
        algo = 12 * melems + 4 * R * (int(ml.poff[-1]) + int(ml.qoff[-1]))
        extra = {"matrices": len(mats), "matrix_elements": melems, "rank": R,
                 "passes": "M = G + E and P = MQ (12 B/elt), Q = M^T P (4), E = M - PQ^T (8)"}
    elif args.op in ("threshold", "clip"):
        ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, gc.GC_EF)
        idx = torch.empty(K, dtype=torch.int32, device=dev)
        val = torch.empty(K, dtype=torch.float32, device=dev)
        e = torch.zeros(N, device=dev)
        cnt = torch.zeros(T, dtype=torch.int64, device=dev)
        norm = torch.empty(T, device=dev)
        tau = torch.full((T,), 1e-2, device=dev)
        cap = torch.stack([0.5 * torch.linalg.vector_norm(grads[0][int(L.off[t]):int(L.off[t + 1])])
                           for t in range(T)]).float()

        def step(it):
            if args.op == "threshold":
                gc.ef_threshold_compress(L, grads[it % 2], e, tau, cnt, idx, val, None, None, 5, it, gc.GC_EF, ws)
            else:
                gc.ef_topk_compress_clipped(L, grads[it % 2], e, cap, norm, idx, val, None, None, 5, it, gc.GC_EF, ws)
        step(0)
        torch.cuda.synchronize()
        kept = int(cnt.sum()) if args.op == "threshold" else K
        algo = b_elem * N + b_kept * kept
        extra = {"kept_per_step": kept}
    elif args.op in ("sign", "sign_lazy", "qsgd"):
        ws = gc.alloc_workspace(L, gc.GC_OP_QUANTIZE if args.op == "qsgd" else gc.GC_OP_SIGN)
        sc = torch.empty(T, device=dev)
        if args.op == "sign_lazy":
            e = torch.zeros(N, device=dev)
            bits = torch.empty(L.words, dtype=torch.int32, device=dev)
            mus = [torch.empty(T, device=dev) for _ in range(2)]

            def step(it):
                gc.sign_compress_lazy(L, grads[it % 2], e, None if it == 0 else mus[(it - 1) % 2], bits,
                                      mus[it % 2], ws)
        elif args.op == "sign":
            e = torch.zeros(N, device=dev)
            bits = torch.empty(L.words, dtype=torch.int32, device=dev)

            def step(it):
                gc.sign_compress(L, grads[it % 2], e, bits, sc, ws)
        else:
            codes = torch.empty(N, dtype=torch.int8, device=dev)

            def step(it):
                gc.quantize_stochastic(L, grads[it % 2], None, codes, sc, gc.GC_Q_QSGD, 16, 5, it, ws)
        algo = b_elem * N + b_tensor * T
    else:
        W = 8
        pays = [workloads.make_sparse_payload(layout, k, w, device=dev, cfg=cfg) for w in range(W)]
        out = torch.zeros(N, device=dev)
        ws = gc.alloc_workspace(L, gc.GC_OP_DECOMPRESS)
        idxs, vals = [p[0] for p in pays], [p[1] for p in pays]
        # touched elements: the union of the workers' index sets (counted once)
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
    for w in range(args.warmup):
        step(w)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(0)
    time.sleep(0.3)
    t0.record()
    for s_ in range(args.steps):
        step(args.warmup + s_)
    t1.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = t0.elapsed_time(t1) / args.steps
    if args.op == "randk":
        extra["graph_replay"] = graph_replay_randk(gc, L, grads, a, idx, val, flags, ws, args, N)
    peak, peak_kind = measured_peaks()
    achieved = algo / (ms * 1e-3) / 1e9
    if args.op == "decompress":
        value, unit, metric = K * W / (ms * 1e-3) / 1e9, "G entries/s", "sparse decompress/scatter-add throughput"
    else:
        value, unit, metric = 4.0 * N / (ms * 1e-3) / 1e9, UNIT, "%s compress gradient GB/s" % args.op
    line = {"metric": metric, "value": value, "unit": unit, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "%s_%s" % (lname, args.op), "what": what, "tensors": T, "elements": N,
                       "kept": K, "density": rho},
            "roofline": {"bound": "hbm", "kernel": "whole call", "achieved": achieved, "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                         "algorithmic_bytes": algo}, "clocks": clocks}
    if args.op in ("qsgd", "randk"):
        # Philox4x32-10 draws one 32-bit word per element: 10 rounds of two
        # 32x32 -> 64-bit products per block of 4 words, each product an
        # integer multiply-high and multiply-low, so 10 integer multiplies
        # per element; the integer multiply-add rate is 64 per SM per clock.
        sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
        mhz = (clocks or {}).get("sm_mhz") or 2070.0
        imad_peak = sm_count * 64 * mhz * 1e6
        imad_done = IMAD_PER_ELEMENT * N / (ms * 1e-3)
        line["alu"] = {"bound": "alu", "unit": "G int-mul/s", "per_element": IMAD_PER_ELEMENT,
                       "achieved": imad_done / 1e9, "peak": imad_peak / 1e9, "frac": imad_done / imad_peak,
                       "peak_from": "%d SMs x 64 per clock x %.0f MHz" % (sm_count, mhz)}
    line.update(extra)
    print(json.dumps(line), flush=True)


def graph_replay_randk(gc, L, grads, e, idx, val, flags, ws, args, N):
    """The same random-k call captured once per resident gradient into a CUDA
    graph (device-resident iteration counter) and replayed alternately: the
    per-call time without per-launch host work."""
    dev = grads[0].device
    it_dev = torch.zeros(1, dtype=torch.int64, device=dev)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graphs = []
    for g in grads:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                gc.ef_topk_compress_dev_iter(L, g, e, idx, val, None, None, 5, it_dev, flags, ws)
        graphs.append(graph)
    torch.cuda.synchronize()
    for w in range(args.warmup):
        graphs[w % 2].replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for s_ in range(args.steps):
        graphs[s_ % 2].replay()
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / args.steps
    return {"ms_per_step": ms, "value": 4.0 * N / (ms * 1e-3) / 1e9, "unit": UNIT,
            "how": "one CUDA-graph capture of gc_ef_topk_compress_dev_iter per resident gradient, replayed "
                   "alternately"}


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="llama3_8b",
                    help="the measured workload is llama3_8b; the others are smaller cases for profiling")
    ap.add_argument("--op", choices=("topk",) + tuple(OPS), default="topk",
                    help="topk is the measured headline; the others measure the remaining compression rows")
    ap.add_argument("--layout", choices=sorted(LAYOUT_CFG), default=None,
                    help="with --op: run that row on another layout (smaller cases for profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
        run_ours(args)


if __name__ == "__main__":
    main()
