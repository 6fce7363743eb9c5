"""Benchmark: embedding backward + fused optimizer step through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload dlrm|tiny|mixed|lm|large] [--no-cpu-baseline]

One step = one whole pass of the hot path (linearise, sort, run-length encode,
long-run partition, fused reduce + optimizer) over one synthetic batch. The
default workload is the large skewed one, the largest that fits one GPU (64
tables x 2M rows, D=128 fp16 weights + fp32 row-wise state, B=65536, bag length
power law on [1, 500] with mean 30, Zipf(1.2) ids, ~1.26e8 lookups, drawn on the
device). Its inputs (37 GB) are far larger than L2; a 256 MB buffer is still
written between timed steps, as for the small workloads, whose working sets fit
in L2.

Prints one JSON line (rank 0). Under torchrun each rank runs its own batch on
its own GPU (weak scaling, no collective: tables are independent).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "embedding bwd+update: lookups/sec and achieved HBM GB/s vs GB300 peak"
DESCR = {
    "dlrm": "DLRM-like: T=8 x 100k rows, D=64 fp32, B=2048, L~U{1..20}, Zipf(1.05) ids, sum, "
            "row-wise Adagrad lr=0.01 eps=1e-8",
    "tiny": "tiny pooled: T=2 (1000, 500 rows), D=16 fp32, B=64, L~U{0..4}, uniform ids, sum, SGD",
    "mixed": "mixed tables: T=26, rows log-uniform 1e3..1e6, D in {32,64,128,256}, fp16 weights, "
             "fp32 grad, B=16384, L~Poisson(15), weighted, mean, row-wise Adagrad",
    "lm": "unpooled LM: vocab 128256, D=4096 fp32 weights, bf16 grad, 32768 tokens, Zipf(1.1), SGD",
    "large": "large skewed: T=64 x 2M rows, D=128 fp16 weights, B=65536, L power law mean 30 max 500, "
             "Zipf(1.2) ids, sum, row-wise Adagrad",
}
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the
# dominant kernel, from ncu captures of the current kernels (the large workload at
# full size, in the metric's single pass; the others from full section captures);
# a workload without an entry reports null.
TRAFFIC = {
    ("large", "reduce_update"): 8_431_475_200 + 2_477_187_584,
    ("dlrm", "reduce_update"): 21_103_360 + 1_792,
    ("mixed", "reduce_update"): 686_832_384 + 196_421_632,
    ("lm", "reduce_update"): 399_733_760 + 85_272_576,
    ("lm", "atomic_scatter"): 418_342_144 + 114_398_976,
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="large", choices=list(DESCR))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-pdl", action="store_true", help="plain launches instead of programmatic dependent launches")
    ap.add_argument("--front", default="auto", choices=["auto", "multiblock"],
                    help="multiblock: sort every call with the multi-block front (A/B timing of the small-batch front)")
    ap.add_argument("--path", default="auto", choices=["auto", "sorted", "atomic"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--op", default="bwd", choices=["bwd", "fwd", "shard"],
                    help="bwd: backward + update (the headline); fwd: forward pooled lookup; "
                         "shard: row-sharded step of one rank (W ranks emulated on one GPU)")
    ap.add_argument("--variant", default="update", choices=["update", "dense", "adagrad", "sr"],
                    help="bwd: update = the workload's optimizer; dense = dense-gradient mode; "
                         "adagrad = elementwise Adagrad; sr = the update with stochastic rounding")
    ap.add_argument("--shards", type=int, default=8, help="ranks W of --op shard")
    ap.add_argument("--tables", type=int, default=None,
                    help="large workload only: draw just its first K tables (a cut-down case of the "
                         "same kernels, e.g. for profiler captures)")
    ap.add_argument("--shard-map", default="cyclic", choices=["cyclic", "ranges"],
                    help="row map of --op shard: rows modulo W, or contiguous ranges")
    return ap.parse_args()


def make_workload(name, seed, device, tables=None):
    from sparse_embedding_bag_gb300 import synth
    if name == "large":
        return synth.large_on_device(seed, device=device, tables=tables)
    return synth.BY_NAME[name](seed)


def host_arrays(w):
    """Host copies of a workload's step inputs (device-drawn workloads are copied back)."""
    import torch
    conv = lambda x: None if x is None else (x.cpu().numpy() if isinstance(x, torch.Tensor) else x)
    return conv(w.indices), conv(w.offsets), conv(w.grad_output), conv(w.per_sample_weights)


# Largest batch the library sorts with its one-launch small-batch front (a cluster of
# CTAs per table); above it, or with EMB_FLAG_NO_CLUSTER_FRONT, the multi-block front.
SMALL_FRONT_MAX_N = 1 << 16


def step_stages(atomic, small_front, passes, reduce_launches=1):
    """Kernels of one step by profiled stage (the five stages of emb_plan_stage_ms),
    the stages' names, and the kernels per step. small_front: the call took the
    one-launch small-batch front (its sort and run-length stages are empty)."""
    if atomic:
        return [1, 0, 0, 0, 1], ["index_check", "-", "-", "-", "atomic_scatter"], 2
    if small_front:
        return ([1, 0, 0, 0, reduce_launches], ["cluster_front", "-", "-", "-", "reduce_update"],
                1 + reduce_launches)
    return ([1, passes, 1, 0, reduce_launches], ["linearise_hist", "radix_sort", "run_length", "-", "reduce_update"],
            2 + passes + reduce_launches)


def radix_passes(w):
    """Radix passes of the sort: the row index of the largest table in digits of at most 9 bits."""
    row_bits = max(int(np.ceil(np.log2(max(int(np.max(w.rows)), 2)))), 1)
    return min(-(-row_bits // 9), 4)


def algorithmic_bytes(w, variant="update"):
    """Minimal bytes of one step: int64 indices, the gradient row read per lookup,
    and one read + one write of every unique row (and its fp32 state for Adagrad:
    8 bytes per row row-wise, 8 per element elementwise). The dense-gradient mode
    writes every unique row once and clears the whole weights-sized buffer.
    Counted with torch on the device that holds the workload's arrays (host numpy
    arrays are counted on the CPU). Returns (step bytes, reduce-kernel bytes,
    unique rows)."""
    import torch
    from sparse_embedding_bag_gb300 import synth
    on_dev = isinstance(w.indices, torch.Tensor)
    dev = w.indices.device if on_dev else torch.device("cpu")
    idx = torch.as_tensor(w.indices, device=dev)
    off = torch.as_tensor(w.offsets, device=dev)
    hsc = torch.as_tensor(np.asarray(w.hash_size_cumsum, np.int64), device=dev)
    dims = torch.as_tensor(np.asarray(w.dims, np.int64), device=dev)
    t_of_lookup = torch.repeat_interleave(torch.arange(w.T * w.B, device=dev) // w.B, off[1:] - off[:-1])
    uniq = torch.unique(hsc[t_of_lookup] + idx)
    t_of_row = torch.searchsorted(hsc, uniq, right=True) - 1
    gsize = 4 if w.grad_dtype == synth.F32 else 2
    wsize = 4 if w.weight_dtype == synth.F32 else 2
    grad_bytes = int(dims[t_of_lookup].sum()) * gsize
    row_elems = int(dims[t_of_row].sum())
    n_uniq, N = int(uniq.numel()), int(idx.numel())
    del t_of_lookup, uniq, t_of_row
    row_bytes = row_elems * 2 * wsize
    state = 8 * n_uniq if w.optimizer == synth.ROWWISE_ADAGRAD else 0
    if variant == "adagrad":
        state = 8 * row_elems
    if variant == "dense":
        reduce_bytes = grad_bytes + row_elems * wsize
        return 8 * N + reduce_bytes + int(w.weights.numel() if on_dev else np.asarray(w.weights).size) * wsize, \
            reduce_bytes, n_uniq
    reduce_bytes = grad_bytes + row_bytes + state
    return 8 * N + reduce_bytes, reduce_bytes, n_uniq


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        # raw samples (the summary goes into the JSON line); BENCH_CLOCKS_DIR keeps them
        out_dir = os.environ.get("BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"embbwd_clocks_rank{gpu_index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def host_subset(w, tables=1):
    """A workload drawn on the device, cut to its first `tables` tables on the host
    (tables are independent, so the oracle's rate per lookup carries over)."""
    import dataclasses
    T2 = min(tables, w.T)
    off = w.offsets[:T2 * w.B + 1].cpu().numpy()
    n2 = int(off[-1])
    wend = int(w.weights_offsets[T2 - 1]) + int(w.rows[T2 - 1]) * int(w.dims[T2 - 1])
    conv = lambda x: None if x is None else x.cpu().numpy()
    weights = w.weights[:wend].cpu()
    weights = weights.view(torch_int16()).numpy().view(np.uint16) if str(weights.dtype) == "torch.bfloat16" \
        else weights.numpy()
    return dataclasses.replace(
        w, T=T2, rows=w.rows[:T2], dims=w.dims[:T2], hash_size_cumsum=w.hash_size_cumsum[:T2 + 1],
        D_offsets=w.D_offsets[:T2 + 1], weights_offsets=w.weights_offsets[:T2],
        momentum_offsets=None if w.momentum_offsets is None else w.momentum_offsets[:T2],
        indices=w.indices[:n2].cpu().numpy(), offsets=off,
        grad_output=w.grad_output[:, :int(w.D_offsets[T2])].contiguous().cpu().numpy(),
        weights=weights,
        momentum=None if w.momentum is None else w.momentum[:int(w.hash_size_cumsum[T2])].cpu().numpy(),
        per_sample_weights=None if w.per_sample_weights is None else conv(w.per_sample_weights[:n2]))


def torch_int16():
    import torch
    return torch.int16


def cpu_baseline(w, budget_s, variant="update"):
    """The oracle, as it stands (single thread), on the same workload for ~budget_s seconds
    (for a workload drawn on the device, on its first table)."""
    import oracle
    from sparse_embedding_bag_gb300 import synth
    subset = not isinstance(w.indices, np.ndarray)
    w_full_T = w.T
    if subset:
        w = host_subset(w)
    indices, offsets, grad, psw = host_arrays(w)
    n_done, el, runs = 0, 0.0, 0
    wts = np.asarray(w.weights)
    while el < budget_s:
        weights = np.array(wts, copy=True)
        mom = None if w.momentum is None else np.array(w.momentum, copy=True)
        kw = dict(per_sample_weights=psw, mean=(w.pooling == synth.MEAN), nobag=w.nobag,
                  grad_dtype=w.grad_dtype)
        t1 = time.perf_counter()
        if variant == "dense":
            oracle.dense_grad(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets, wts.size,
                              indices, offsets, grad, out_dtype=w.weight_dtype, **kw)
        elif variant == "adagrad":
            m = np.zeros(wts.size, np.float32)
            oracle.backward(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets, weights,
                            indices, offsets, grad, optimizer=oracle.ADAGRAD, lr=w.lr, eps=w.eps,
                            momentum=m, **kw)
        else:
            oracle.backward(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets, weights,
                            indices, offsets, grad, optimizer=w.optimizer, lr=w.lr, eps=w.eps,
                            momentum=mom, momentum_offsets=w.momentum_offsets,
                            stochastic_rounding=(1, runs) if variant == "sr" else None, **kw)
        el += time.perf_counter() - t1
        n_done += indices.size
        runs += 1
    what = (f"the first {w.T} of the {w_full_T} tables of the same workload" if subset else "the same workload")
    return {"value": n_done / el, "unit": "lookups/s", "cores": 1, "host_cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{runs} full step(s) of {what} ({indices.size} lookups each), "
                      f"{el:.1f} s, single-threaded C++ oracle (double accumulation)"}


def run_reference(args):
    """Reference arm: the CPU oracle timed on the same workload, metric and unit.
    The large workload (32.8 GB of weights) is timed on its first table, drawn on
    the device when there is one, so that it is exactly the first table of the
    workload the GPU arm times (tables are independent: the rate per lookup
    carries over); one step of it is a few seconds of one host core."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from sparse_embedding_bag_gb300 import synth
    oracle.build()
    if args.workload == "large":
        import torch
        gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
        w = host_subset(make_workload("large", 0, gen_dev, tables=1), tables=1)
        sample = (f"table 1 of the 64 tables of the same workload ({w.N} lookups per step)" +
                  ("" if gen_dev == "cuda" else ", drawn with the CPU generator (same recipe, other draws)"))
    else:
        w = make_workload(args.workload, 0, "cpu")
        sample = f"the whole workload ({w.N} lookups per step)"
    indices, offsets, grad, psw = host_arrays(w)

    def one():
        weights = np.array(w.weights, copy=True)
        mom = None if w.momentum is None else np.array(w.momentum, copy=True)
        t = time.perf_counter()
        oracle.backward(w.T, w.B, w.hash_size_cumsum, w.D_offsets, w.weights_offsets, weights,
                        indices, offsets, grad, optimizer=w.optimizer, lr=w.lr, eps=w.eps,
                        momentum=mom, momentum_offsets=w.momentum_offsets, per_sample_weights=psw,
                        mean=(w.pooling == synth.MEAN), nobag=w.nobag, grad_dtype=w.grad_dtype)
        return time.perf_counter() - t

    for _ in range(args.warmup):
        one()
    times = [one() for _ in range(args.steps)]
    ms = 1e3 * sum(times) / len(times)
    value = indices.size / (ms / 1e3)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "lookups/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": DESCR[args.workload], "N": int(indices.size)},
        "cpu_baseline": {"value": value, "unit": "lookups/s", "cores": 1, "host_cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"{args.steps} steps of {sample}, single-threaded C++ oracle "
                                   f"(double accumulation)"},
        "e2e": {"value": value, "unit": "lookups/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def run_forward(args):
    """Forward pooled lookup on one GPU: the same timing rules as the backward."""
    import torch
    from sparse_embedding_bag_gb300 import build as b
    from sparse_embedding_bag_gb300 import device as dev
    from sparse_embedding_bag_gb300 import embbwd as E
    from sparse_embedding_bag_gb300 import synth
    torch.cuda.set_device(0)
    b.build()
    E.load()
    w = make_workload(args.workload, 0, "cuda:0")
    if w.nobag:
        raise SystemExit("the forward pooled lookup needs a pooled workload")
    indices_h, offsets_h, _, psw_h = host_arrays(w)
    dw = dev.to_device(w, "cuda:0")
    plan = dev.make_plan(w, flags=E.EMB_FLAG_NO_PDL if args.no_pdl else 0)
    out = torch.empty((w.B, int(w.D_offsets[-1])), dtype=torch.float32, device="cuda:0")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda:0")

    def call():
        dev.forward(plan, dw, 0, out)

    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize()
    if E.emb_plan_status(plan) != E.EMB_OK:
        raise SystemExit("device status error")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    with ClockSampler(0) as clocks:
        t_soak = time.perf_counter()
        while time.perf_counter() - t_soak < 0.6:
            for _ in range(50):
                flush.zero_()
                graph.replay()
            torch.cuda.synchronize()
        for k in range(K):
            flush.zero_()
            starts[k].record()
            graph.replay()
            ends[k].record()
        torch.cuda.synchronize()
    ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / K
    N = int(indices_h.size)
    lengths = np.diff(offsets_h)
    t_of_lookup = np.repeat(np.arange(w.T * w.B) // w.B, lengths)
    wsize = 4 if w.weight_dtype == synth.F32 else 2
    fbytes = (8 * N + int(np.sum(w.dims[t_of_lookup].astype(np.int64))) * wsize +
              w.B * int(w.D_offsets[-1]) * 4 + (4 * N if psw_h is not None else 0))
    peak, peak_kind = peaks()
    achieved = fbytes / (ms * 1e-3) / 1e9
    # end to end: inputs from pinned host memory, the call, the output back to the host
    pin = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    h_idx, h_off, h_psw = pin(indices_h), pin(offsets_h), pin(psw_h)
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (h_idx, h_off, h_psw) if x is not None)
    e2e = []
    for k in range(min(max(3, K // 2), 200) + 2):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        dw.indices.copy_(h_idx, non_blocking=True)
        dw.offsets.copy_(h_off, non_blocking=True)
        if h_psw is not None:
            dw.per_sample_weights.copy_(h_psw, non_blocking=True)
        call()
        h_out.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
        e2e.append(time.perf_counter() - t0)
    e2e_s = statistics.median(e2e[2:])
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        subset = not isinstance(w.indices, np.ndarray)
        wc = host_subset(w) if subset else w  # drawn on the device: its first table
        ic, oc, _, pc = host_arrays(wc)
        n_done, el, runs = 0, 0.0, 0
        while el < min(args.cpu_seconds, 10.0):
            t1 = time.perf_counter()
            oracle.forward(wc.T, wc.B, wc.hash_size_cumsum, wc.D_offsets, wc.weights_offsets,
                           np.asarray(wc.weights), ic, oc, per_sample_weights=pc,
                           mean=(wc.pooling == synth.MEAN))
            el += time.perf_counter() - t1
            n_done += int(ic.size)
            runs += 1
        what = f"the first {wc.T} tables of the same workload" if subset else "the same workload"
        cpu = {"value": n_done / el, "unit": "lookups/s", "cores": 1, "host_cores": os.cpu_count(),
               "kind": "oracle", "sample": f"{runs} full forward(s) of {what}, {el:.1f} s, single-threaded"}
    print(json.dumps({
        "metric": "embedding bag forward: lookups/sec and achieved HBM GB/s vs GB300 peak",
        "op": "fwd", "value": N / (ms * 1e-3), "unit": "lookups/s", "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": DESCR[args.workload], "N": N, "output": "fp32 [B, sum D]",
                   "l2": "256 MB buffer written between timed steps", "cuda_graph": True},
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "kernel": "k_bag_fwd", "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None},
        "cpu_baseline": cpu,
        "e2e": {"value": N / e2e_s, "unit": "lookups/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(out.numel() * out.element_size())},
        "gpu_launches": K,
        "clocks": clocks.summary(),
    }, default=float))


def timed(fn, K, flush, stream):
    """Mean device ms of fn over K runs (CUDA events on the launching stream, L2
    flushed before each run)."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for k in range(K):
        flush.zero_()
        starts[k].record(stream)
        fn()
        ends[k].record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / K


def run_shard(args):
    """One rank's row-sharded step, W ranks emulated on one GPU: every rank's batch
    is bucketed by row owner, the all-to-all is replaced by device copies (on a
    deployment NCCL moves these bytes), and the most loaded owner merges what it
    receives and runs its backward (B' = W*B). Timed per stage, excluding the
    exchange itself: bucketize (rank 0's batch; it synchronises for the sizes),
    merge and backward (the most loaded owner)."""
    import torch
    from sparse_embedding_bag_gb300 import build as b
    from sparse_embedding_bag_gb300 import embbwd as E
    from sparse_embedding_bag_gb300 import shard as S
    from sparse_embedding_bag_gb300 import synth
    if args.workload not in ("dlrm", "tiny"):
        raise SystemExit("--op shard needs a workload whose tables do not depend on the seed (dlrm, tiny)")
    torch.cuda.set_device(0)
    b.build()
    E.load()
    W, K = args.shards, max(args.steps // 10, 20)
    srcs = [make_workload(args.workload, s, "cpu") for s in range(W)]
    w = srcs[0]
    T, B = w.T, w.B
    rb = S.even_row_bounds(w.rows, W)
    cyclic = args.shard_map == "cyclic"
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda:0")
    dev_in = [(torch.from_numpy(x.indices).cuda(), torch.from_numpy(x.offsets).cuda()) for x in srcs]
    maxN = max(x.N for x in srcs)
    sh = E.emb_shard_create_cyclic(0, T, W, w.rows, B) if cyclic else E.emb_shard_create(0, T, W, rb, B)
    sends = []
    for (idx, off), x in zip(dev_in, srcs):
        so = torch.empty((W, T * B + 1), dtype=torch.int64, device="cuda:0")
        si = torch.empty(maxN, dtype=torch.int64, device="cuda:0")
        cnt = E.emb_shard_bucketize(sh, idx, off, x.N, B, None, E.EMB_POOL_SUM, so, si, None)
        sends.append((so, si, cnt))
    recv_counts = np.sum([c for _, _, c in sends], axis=0)
    r = int(np.argmax(recv_counts))  # the most loaded owner
    ro = torch.stack([so[r] for so, _, _ in sends]).contiguous()
    ri = torch.cat([si[int(c[:r].sum()):int(c[:r].sum()) + int(c[r])] for _, si, c in sends])
    n = int(ri.numel())
    mo = torch.empty(T * W * B + 1, dtype=torch.int64, device="cuda:0")
    mi = torch.empty(max(n, 1), dtype=torch.int64, device="cuda:0")
    local, hsc, Do, wo = S.local_tables(w.rows, w.dims, rb, r, W, cyclic)
    plan = E.emb_bwd_plan(0, T, hsc, Do, wo, None, w.weight_dtype, w.grad_dtype, max(n, 1), W * B, 0, 0)
    own = S.owned_rows(w.rows, rb, r, W, cyclic)
    wl = torch.from_numpy(np.concatenate([w.weights[(w.weights_offsets[t] + own[t][:, None] * w.dims[t] +
                                                     np.arange(w.dims[t])).reshape(-1)]
                                          for t in range(T)])).cuda()
    ml = torch.full((int(hsc[-1]),), 0.0, dtype=torch.float32, device="cuda:0")
    grad = torch.from_numpy(np.concatenate([x.grad_output for x in srcs])).cuda()
    so0, si0 = torch.empty_like(sends[0][0]), torch.empty_like(sends[0][1])

    def bucketize():
        E.emb_shard_bucketize(sh, dev_in[0][0], dev_in[0][1], srcs[0].N, B, None, E.EMB_POOL_SUM,
                              so0, si0, None)

    def merge():
        E.emb_shard_merge(sh, ro, ri, None, n, B, mo, mi, None)

    def backward():
        if w.optimizer == synth.SGD:
            E.emb_bag_bwd_sgd(plan, wl, mi, mo, n, W * B, None, grad, E.EMB_POOL_SUM, w.lr)
        else:
            E.emb_bag_bwd_rowwise_adagrad(plan, wl, ml, mi, mo, n, W * B, None, grad,
                                          E.EMB_POOL_SUM, w.lr, w.eps)

    for _ in range(max(args.warmup, 3)):
        bucketize(); merge(); backward()
    torch.cuda.synchronize()
    if E.emb_shard_status(sh) != E.EMB_OK or E.emb_plan_status(plan) != E.EMB_OK:
        raise SystemExit("device status error")
    with ClockSampler(0) as clocks:
        ms_b = timed(bucketize, K, flush, stream)
        ms_m = timed(merge, K, flush, stream)
        ms_r = timed(backward, K, flush, stream)
    N0, BT = srcs[0].N, T * B
    bytes_b = 16 * N0 + 8 * (BT + 1) + 8 * W * (BT + 1)       # indices in/out, offsets, per-owner offsets
    bytes_m = 8 * W * (BT + 1) + 16 * n + 8 * (T * W * B + 1)  # received offsets, indices in/out, merged offsets
    peak, peak_kind = peaks()
    stages = {"bucketize": (ms_b, bytes_b), "merge": (ms_m, bytes_m)}
    dom = max(stages, key=lambda k: stages[k][0])
    ach = stages[dom][1] / (stages[dom][0] * 1e-3) / 1e9
    ms = ms_b + ms_m + ms_r
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        # the oracle on the same step: rank 0's bucketize, the owner's merge and backward
        parts = [oracle.bucketize(T, B, rb, x.indices, x.offsets, cyclic=cyclic) for x in srcs]
        el, runs = 0.0, 0
        while el < min(args.cpu_seconds, 10.0) or runs == 0:
            t1 = time.perf_counter()
            oracle.bucketize(T, B, rb, srcs[0].indices, srcs[0].offsets, cyclic=cyclic)
            ro_h = np.stack([p[0][r] for p in parts])
            ri_h = np.concatenate([p[1][int(p[3][:r].sum()):int(p[3][:r].sum()) + int(p[3][r])] for p in parts])
            mo_h, mi_h, _ = oracle.merge(T, B, W, ro_h, ri_h, np.ones(ri_h.size, np.float32))
            wl_h = wl.cpu().numpy().copy()
            ml_h = np.zeros(int(hsc[-1]), np.float32)
            oracle.backward(T, W * B, hsc, Do, wo, wl_h, mi_h, mo_h, grad.cpu().numpy(),
                            optimizer=w.optimizer, lr=w.lr, eps=w.eps, momentum=ml_h)
            el += time.perf_counter() - t1
            runs += 1
        cpu = {"value": int(recv_counts.sum()) * runs / el, "unit": "lookups/s", "cores": 1,
               "host_cores": os.cpu_count(), "kind": "oracle", "sample": f"{runs} step(s): rank 0's bucketize, owner {r}'s merge and "
                                           f"backward, {el:.1f} s, single-threaded"}
    print(json.dumps({
        "metric": "row-sharded embedding step, W ranks (exchange kernels + the most loaded owner's "
                  "backward, communication excluded): all ranks' lookups/sec",
        "op": "shard", "value": int(recv_counts.sum()) / (ms * 1e-3), "unit": "lookups/s", "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": DESCR[args.workload] + " per rank", "ranks_emulated": W,
                   "row_split": "rows modulo W" if cyclic else "even contiguous ranges of every table",
                   "owner": r, "lookups_received": n, "lookups_per_owner": recv_counts.tolist(),
                   "excluded": "the all-to-all and all-gather themselves (device copies here)",
                   "l2": "256 MB buffer written before each timed call"},
        "stage_ms": {"bucketize": ms_b, "merge": ms_m, "backward_owner": ms_r},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": ach / peak, "traffic": None},
        "cpu_baseline": cpu,
        # bucketize: count, three scan phases, scatter; merge: bases, copy; backward:
        # histogram, radix passes, run-length, reduce
        "gpu_launches": K * (5 + 2 + 3 + min(-(-max(int(np.max(np.diff(hsc)) - 1).bit_length(), 1) // 9), 4)),
        "clocks": clocks.summary(),
    }, default=float))
    E.emb_plan_destroy(plan)
    E.emb_shard_destroy(sh)


def run_shard_dist(args, device=None, ops_factory=None, workload=None):
    """The row-sharded step over WORLD_SIZE ranks (one per GPU, NCCL): every rank
    has its own batch and owns the rows congruent to its rank modulo W of every
    table; per step the lookups are routed to their owners (bucketize, three
    all-to-alls, merge), the forward runs on the owners and a reduce-scatter
    returns each rank its bags, and the backward all-gathers grad_output and
    updates each owner's rows. Each stage is timed on its own (the max over
    ranks); value = all ranks' lookups / the max step time.

    device / ops_factory / workload let the CPU test drive the same code over gloo
    with other implementations of the library steps (None: the GPU and the library)."""
    import torch
    import torch.distributed as dist
    from sparse_embedding_bag_gb300 import embbwd as E
    from sparse_embedding_bag_gb300 import shard as S
    from sparse_embedding_bag_gb300 import synth
    world = int(os.environ["WORLD_SIZE"])
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    on_gpu = device is None
    if on_gpu:
        torch.cuda.set_device(local)
        device = f"cuda:{local}"
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        from sparse_embedding_bag_gb300 import build as b
        b.build()
        E.load()
    elif not dist.is_initialized():
        dist.init_process_group("gloo")
    name = workload or args.workload
    if name not in ("dlrm", "tiny"):
        raise SystemExit("--op shard needs a workload whose table shapes do not depend on the seed (dlrm, tiny)")
    w = synth.BY_NAME[name](rank)  # this rank's batch; every rank has the same table shapes
    T, B = w.T, w.B
    n_all = torch.tensor([w.N], dtype=torch.int64, device=device)
    dist.all_reduce(n_all)
    max_N = int(n_all.item())  # an owner receives at most every rank's lookups
    sb = S.RowShardedBags(w.rows, w.dims, rank, world, B, max_N, cyclic=True, device=device,
                          weight_dtype=w.weight_dtype, grad_dtype=w.grad_dtype,
                          ops=None if ops_factory is None else ops_factory(w, rank, world))
    own = S.owned_rows(w.rows, None, rank, world, cyclic=True)
    wl = torch.from_numpy(np.concatenate([w.weights[(w.weights_offsets[t] + own[t][:, None] * w.dims[t] +
                                                     np.arange(w.dims[t])).reshape(-1)]
                                          for t in range(T)])).to(device)
    ml = torch.zeros(int(sb.hsc[-1]), dtype=torch.float32, device=device)
    idx = torch.from_numpy(w.indices).to(device)
    off = torch.from_numpy(w.offsets).to(device)
    grad = torch.from_numpy(np.ascontiguousarray(w.grad_output)).to(device)
    sync = torch.cuda.synchronize if on_gpu else (lambda: None)

    def step(times=None):
        t0 = time.perf_counter()
        routed = sb.route(idx, off, w.N, B)
        sync()
        t1 = time.perf_counter()
        sb.forward(wl, routed)
        sync()
        t2 = time.perf_counter()
        if w.optimizer == synth.SGD:
            sb.backward_sgd(wl, routed, grad, w.lr)
        else:
            sb.backward_rowwise_adagrad(wl, ml, routed, grad, w.lr, w.eps)
        sync()
        t3 = time.perf_counter()
        if times is not None:
            times.append((t1 - t0, t2 - t1, t3 - t2))

    for _ in range(max(args.warmup, 3)):
        step()
    dist.barrier()
    sync()
    times = []
    with ClockSampler(local) if on_gpu else _NoClocks() as clocks:
        t_start = time.perf_counter()
        for _ in range(args.steps):
            step(times)
        sync()
        dist.barrier()
        wall = time.perf_counter() - t_start
    mean = np.mean(np.array(times), axis=0) * 1e3  # ms: exchange, forward, backward
    stats = torch.tensor([wall * 1e3 / args.steps, *mean.tolist()], dtype=torch.float64, device=device)
    dist.all_reduce(stats, op=dist.ReduceOp.MAX)
    ms, ex_ms, fw_ms, bw_ms = (float(x) for x in stats.tolist())
    sb.close()
    if rank == 0:
        print(json.dumps({
            "metric": "row-sharded embedding step (route, forward, backward with update): "
                      "all ranks' lookups/sec",
            "op": "shard", "value": int(n_all.item()) / (ms * 1e-3), "unit": "lookups/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": DESCR[name] + " per rank", "parallelism": f"row-sharded, {world} ranks",
                       "row_map": "rows modulo W", "N_all_ranks": int(n_all.item()),
                       "collectives": "all_to_all_single x3, reduce_scatter_tensor, all_gather_into_tensor"},
            "stage_ms": {"exchange": ex_ms, "forward": fw_ms, "backward": bw_ms},
            "e2e": None, "gpu_launches": args.steps * (7 + 1 + 3 + radix_passes(w)) if on_gpu else 0,
            "clocks": clocks.summary(),
        }, default=float))


class _NoClocks:
    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False

    def summary(self):
        return None


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.op == "fwd":
        return run_forward(args)
    if args.op == "shard":
        if int(os.environ.get("WORLD_SIZE", "1")) > 1:
            return run_shard_dist(args)
        return run_shard(args)
    import torch
    import torch.distributed as dist

    from sparse_embedding_bag_gb300 import build as b
    from sparse_embedding_bag_gb300 import device as dev
    from sparse_embedding_bag_gb300 import embbwd as E
    from sparse_embedding_bag_gb300 import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    b.build()
    E.load()

    w = make_workload(args.workload, rank, f"cuda:{local}", tables=args.tables)
    variant = args.variant
    if variant == "sr" and w.weight_dtype == synth.F32:
        raise SystemExit("--variant sr needs a workload with fp16 / bf16 weights (mixed, large)")
    if variant == "adagrad" and w.nobag:
        raise SystemExit("--variant adagrad needs a pooled workload")
    indices_h, offsets_h, grad_h, psw_h = host_arrays(w)
    step_bytes, reduce_bytes, uniq = algorithmic_bytes(w, variant)
    dw = dev.to_device(w, f"cuda:{local}")
    flags = (E.EMB_FLAG_NO_PDL if args.no_pdl else 0) | (E.EMB_FLAG_STOCHASTIC_ROUNDING if variant == "sr" else 0) \
        | (E.EMB_FLAG_NO_CLUSTER_FRONT if args.front == "multiblock" else 0)
    plan = dev.make_plan(w, device_index=local, flags=flags)
    path = {"auto": E.EMB_NOBAG_AUTO, "sorted": E.EMB_NOBAG_SORTED, "atomic": E.EMB_NOBAG_ATOMIC}[args.path]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=f"cuda:{local}")
    dense_buf = torch.empty_like(dw.weights) if variant == "dense" else None
    ew_state = torch.zeros(dw.weights.numel(), dtype=torch.float32, device=f"cuda:{local}") \
        if variant == "adagrad" else None

    def call(d=None, stream=None):  # stream None: torch's current stream
        d = dw if d is None else d
        if variant == "dense":
            if w.nobag:
                E.emb_nobag_bwd_dense_grad(plan, dense_buf, d.indices, d.offsets, w.N, w.B,
                                           d.grad_output, stream)
            else:
                E.emb_bag_bwd_dense_grad(plan, dense_buf, d.indices, d.offsets, w.N, w.B,
                                         d.per_sample_weights, d.grad_output, w.pooling, stream)
        elif variant == "adagrad":
            E.emb_bag_bwd_adagrad(plan, d.weights, ew_state, d.indices, d.offsets, w.N, w.B,
                                  d.per_sample_weights, d.grad_output, w.pooling, w.lr, w.eps, stream)
        else:
            dev.step(plan, d, path=path, stream=stream)

    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize()
    st = E.emb_plan_status(plan)
    if st != E.EMB_OK:
        raise SystemExit(f"device status {E.status_string(st)}")

    use_graph = not args.no_graph
    graph = None
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            call()
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()

    def one_step():
        graph.replay() if use_graph else call()

    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    with ClockSampler(local) as clocks:
        # keep the GPU busy for ~0.6 s before the timed region so that the
        # 200 ms clock samples cover the load (the steps themselves are short)
        t_soak = time.perf_counter()
        while time.perf_counter() - t_soak < 0.6:
            for _ in range(50):
                flush.zero_()
                one_step()
            torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        for k in range(K):
            flush.zero_()
            starts[k].record()
            one_step()
            ends[k].record()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    ms_list = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = sum(ms_list) / K
    st = E.emb_plan_status(plan)
    if st != E.EMB_OK:
        raise SystemExit(f"device status {E.status_string(st)}")
    n_local = int(indices_h.size)
    if world > 1:
        t = torch.tensor([ms, float(n_local)], device=f"cuda:{local}", dtype=torch.float64)
        mx = t.clone()
        dist.all_reduce(mx, op=dist.ReduceOp.MAX)
        sm = t.clone()
        dist.all_reduce(sm, op=dist.ReduceOp.SUM)
        ms_job, n_job = float(mx[0]), float(sm[1])
    else:
        ms_job, n_job = ms, float(n_local)

    # ---- per-stage times (profiled replays, same work) -> dominant kernel roofline
    E.emb_plan_set_profiling(plan, True)
    stage_runs = []
    if use_graph:
        gprof = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gprof):
            call()
        run_prof = gprof.replay
    else:
        run_prof = call
    for k in range(min(K, 200)):
        flush.zero_()
        run_prof()
        torch.cuda.synchronize()
        stage_runs.append(E.emb_plan_stage_ms(plan))
    E.emb_plan_set_profiling(plan, False)
    stage = np.mean(np.array(stage_runs), axis=0)
    atomic = w.nobag and path == E.EMB_NOBAG_ATOMIC
    passes = radix_passes(w)
    # the small-batch front: one launch, so the sort and run-length stages record nothing
    small_front = (not atomic and args.front == "auto" and n_local <= SMALL_FRONT_MAX_N
                   and float(stage[1] + stage[2]) < 0.006)
    # row-wise Adagrad on rows wider than 1024 elements launches the reduce twice
    reduce_launches = 2 if (variant == "update" and not w.nobag and w.optimizer == synth.ROWWISE_ADAGRAD
                            and int(np.max(w.dims)) > 1024) else 1
    # launches per stage: the dominant kernel is the one with the longest launch
    launches, names, kernels_per_step = step_stages(atomic, small_front, passes, reduce_launches)
    per_launch = [t / n if n else 0.0 for t, n in zip(stage, launches)]
    dom = int(np.argmax(per_launch))
    peak, peak_kind = peaks()
    vbytes = 8 if (w.per_sample_weights is not None or w.pooling == synth.MEAN) else 4
    N = n_local
    stage_bytes = {
        "linearise_hist": 8 * N + 8 * (w.T * w.B + 1),
        "radix_sort": N * (8 + 4 + vbytes) + (passes - 1) * N * 2 * (4 + vbytes),
        "run_length": 4 * N + 8 * uniq,
        "reduce_update": reduce_bytes,
        "index_check": 8 * N,
        "atomic_scatter": reduce_bytes,
    }
    stage_bytes["cluster_front"] = stage_bytes["linearise_hist"] + stage_bytes["radix_sort"] + stage_bytes["run_length"]
    dom_name = names[dom]
    achieved = stage_bytes.get(dom_name, 0) / launches[dom] / (per_launch[dom] * 1e-3) / 1e9
    # measured DRAM bytes of one launch of the dominant kernel (null without a capture
    # of the current kernels on this workload); its rate over the event-timed launch
    traffic = TRAFFIC.get((args.workload, dom_name)) if (args.tables is None and variant == "update") else None
    dram_gbs = traffic / (per_launch[dom] * 1e-3) / 1e9 if traffic else None
    red_achieved = reduce_bytes / (stage[4] * 1e-3) / 1e9

    # ---- end to end through the public API with host buffers: every step copies its
    # inputs (indices, offsets, gradient, per-sample weights) from pinned host memory
    # and reads the 4-byte status word back. As a training loop prefetches its next
    # batch, step k+1's inputs are copied on a copy stream into a second set of
    # device buffers while step k computes; a buffer set is refilled only after the
    # step that read it has finished. The time of the whole run (every copy, call and
    # status read) divided by its steps is the step time; nothing is written between
    # steps to evict L2 (each step's inputs are new copies). The library's calls run
    # on torch's default stream (passed explicitly), the copies on a second stream.
    pin = lambda a: None if a is None else torch.from_numpy(
        np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a)).pin_memory()
    h_idx, h_off, h_grad, h_psw = pin(indices_h), pin(offsets_h), pin(grad_h), pin(psw_h)
    h2d = sum(x.numel() * x.element_size() for x in (h_idx, h_off, h_grad, h_psw) if x is not None)
    spare = lambda t: None if t is None else torch.empty_like(t)
    bufs = [dw, dataclasses.replace(dw, indices=spare(dw.indices), offsets=spare(dw.offsets),
                                    grad_output=spare(dw.grad_output),
                                    per_sample_weights=spare(dw.per_sample_weights))]
    copies = [[(b.indices, h_idx), (b.offsets, h_off), (b.grad_output, h_grad)] +
              ([(b.per_sample_weights, h_psw)] if h_psw is not None else []) for b in bufs]
    copy_stream = torch.cuda.Stream(device=f"cuda:{local}")
    compute_stream = torch.cuda.default_stream(torch.device(f"cuda:{local}"))
    copied = [torch.cuda.Event() for _ in bufs]
    used = [torch.cuda.Event() for _ in bufs]

    def issue_copies(k):  # on the copy stream (the current torch stream of e2e_run)
        copy_stream.wait_event(used[k % 2])  # the step that last read this buffer set is done
        for dst, src in copies[k % 2]:
            dst.copy_(src, non_blocking=True)
        copied[k % 2].record(copy_stream)

    def e2e_run(steps):
        with torch.cuda.stream(copy_stream):
            issue_copies(0)
            for k in range(steps):
                if k + 1 < steps:
                    issue_copies(k + 1)
                compute_stream.wait_event(copied[k % 2])
                call(bufs[k % 2], compute_stream)
                used[k % 2].record(compute_stream)
                st = E.emb_plan_status(plan)  # waits for step k and reads the 4-byte status word back
                if st != E.EMB_OK:
                    raise SystemExit(f"device status {E.status_string(st)}")

    e2e_steps = min(max(3, K // 2), 200)
    e2e_run(2)  # warm-up
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e2e_run(e2e_steps)
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    e2e_val = n_local / e2e_s
    if world > 1:
        t = torch.tensor([e2e_s], device=f"cuda:{local}", dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_val = n_job / float(t[0])

    result = {
        "metric": METRIC,
        "value": n_job / (ms_job * 1e-3),
        "unit": "lookups/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms_job,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": DESCR[args.workload] + (f" (first {w.T} tables only)" if args.tables else ""),
                   "N": n_local, "unique_rows": uniq,
                   "variant": {"update": "the workload's optimizer", "dense": "dense-gradient mode",
                               "adagrad": "elementwise Adagrad",
                               "sr": "the workload's optimizer, stochastic rounding"}[variant],
                   "l2": "256 MB buffer written between timed steps", "cuda_graph": use_graph, "pdl": not args.no_pdl,
                   "front": args.front, "parallelism": f"{world} independent shard(s), no collective"},
        "hbm_gbs": step_bytes / (ms_job * 1e-3) / 1e9,
        "step_bytes": step_bytes,
        "roofline": {"bound": "hbm", "kernel": dom_name, "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "dram_gbs": dram_gbs,
                     "dram_frac": None if dram_gbs is None else dram_gbs / peak},
        "reduce_update": {"ms": float(stage[4]), "gbs": red_achieved, "frac": red_achieved / peak,
                          "bytes": reduce_bytes},
        "stage_ms": {n: float(v) for n, v in zip(names, stage) if n != "-"},
        "e2e": {"value": e2e_val, "unit": "lookups/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": 4,
                "overlap": "step k+1's inputs copied on a copy stream into a second buffer set while step k "
                           "computes; status read back every step; no L2 flush between steps"},
        "gpu_launches": kernels_per_step * K,
        "clocks": clocks.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        result["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds, variant)
    E.emb_plan_destroy(plan)
    if rank == 0:
        print(json.dumps(result, default=float))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
