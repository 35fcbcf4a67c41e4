"""Benchmark of the pack -> ragged attention -> unpack path on one or more GPUs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl rra|reference]
                    [--workload serving|tiny|batched|hires] [--sweep]

One step = one pass of the whole path (pack, then attention with the unpack
fused into its epilogue) over one batch of the workload.  Default workload:
the serving case, DeiT-S-shaped B=4, N=197, H=6, d=64, bf16, 80% of patches
pruned (39 +- 4 tokens per image).  Inputs are seeded synthetic data resident
in HBM; R copies of the input set rotate so that their total size exceeds L2
and every step reads cold inputs.

Printed (rank 0, one JSON line): kept tokens/s of the path (value), the
host-timed latency of one rra_attend call at BS=1/2/4, end-to-end tokens/s
from pinned host buffers (through rra_pipeline_mapped, which reads the kept
rows over the CPU-GPU link, and through rra_pipeline_host's copies), the dominant kernel's
roofline fraction, the CPU oracle's throughput on a bounded sample, SM clocks
sampled during the run and the number of kernel launches.

--impl reference times the CPU oracle (the only reference implementation:
the pages ship no code) on the same workload and prints the same line shape.
Under torchrun every rank runs its own replica (images are independent, so
the work partitions with no collective); rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from ragged_attention_token_gb300 import workloads as W  # noqa: E402

METRIC = "ragged attend µs @BS1-4 (host-timed); pack-attend-unpack tokens/s; % roofline"
UNIT = "tokens/s"
SCALE = 0.125
L2_BYTES = 129 * 1024 * 1024


# ----------------------------------------------------------------- workloads

def make_case(name: str, pruning: float | None = None):
    if name == "batched" and pruning is not None:
        return W.make_batched(pruning), f"batched DeiT-B: B=64, N=197, H=12, d=64, bf16, {int(pruning * 100)}% pruned +-10%"
    if name == "hires" and pruning is not None:
        return W.make_hires(pruning), f"high-res DeiT-B 384px: B=32, N=577, H=12, d=64, bf16, {int(pruning * 100)}% pruned +-10%"
    if name == "serving":
        return W.make_serving(4), "serving DeiT-S: B=4, N=197, H=6, d=64, bf16, 80% pruned (39+-4 tokens/image)"
    if name == "tiny":
        return W.make_tiny(), "tiny DeiT-T: B=2, N=197, H=3, d=64, fp16, keep rate ~U[0.2,1]"
    if name == "batched":
        return W.make_batched(0.8), "batched DeiT-B: B=64, N=197, H=12, d=64, bf16, 80% pruned +-10%"
    if name == "hires":
        return W.make_hires(0.5), "high-res DeiT-B 384px: B=32, N=577, H=12, d=64, bf16, 50% pruned +-10%"
    raise ValueError(name)


def case_bytes(case, out_bytes_per_el=None):
    """Algorithmic bytes per launch (attend, index pass, pack with copy, fused minimum) and FLOPs."""
    B, N, H, d = case.B, case.N, case.H, case.d
    s = case.q.element_size()
    so = out_bytes_per_el or s
    T = case.kept_tokens
    return dict(
        attend=3 * T * H * d * s + T * H * d * so,
        index=B * N + (B * N - T) * H * d * so + 4 * (B + 1) + 4 * B * N + 4 * T,
        pack=B * N + 2 * 3 * T * H * d * s + (B * N - T) * H * d * so + 4 * (B + 1) + 4 * B * N + 4 * T,
        fused_min=B * N + 3 * T * H * d * s + B * N * H * d * so,   # the fused kernel writes no indices
        flops=4 * H * d * sum(n * n for n in case.lengths),
    )


# ------------------------------------------------------------------ peaks

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.t_start = self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        self.t_start = time.time()

    def stop(self):
        self.t_stop = time.time()
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "window_s": round(self.t_stop - self.t_start, 2)}


# -------------------------------------------------------------- GPU helpers

class InputSets:
    """R device copies of one seeded input set (rotated to defeat L2 reuse)."""

    def __init__(self, case, device, rra, out_dtype, R=None):
        B, N, H, d = case.B, case.N, case.H, case.d
        base = [x.to(device) for x in (case.keep, case.q, case.k, case.v)]
        ws_bytes = rra.workspace_bytes(B, N, H, d, case.dtype)
        per_set = sum(x.numel() * x.element_size() for x in base) + ws_bytes + \
            B * N * H * d * torch.empty((), dtype=out_dtype).element_size()
        if R is None:
            R = max(2, min(512, math.ceil(2 * L2_BYTES / per_set)))
        self.R = R
        self.per_set = per_set
        self.sets = []
        for _ in range(R):
            keep, q, k, v = (x.clone() for x in base)
            out = torch.empty((B, N, H, d), dtype=out_dtype, device=device)
            ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
            self.sets.append((keep, q, k, v, out, ws))


def capture(fn_list, stream):
    """A CUDA graph of the launches in fn_list, captured on `stream` (after one eager pass)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for fn in fn_list:
            fn()
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for fn in fn_list:
                fn()
    stream.synchronize()
    return g


SLEEP_CYCLES = 200_000      # ~0.1 ms at the GB300's 2.07 GHz


def graph_time_per_launch(fn_list, stream, reps=5):
    """Median device µs per launch of a CUDA graph of back-to-back launches.

    The graph is replayed on the same stream the events are recorded on."""
    g = capture(fn_list, stream)
    times = []
    with torch.cuda.stream(stream):
        g.replay()
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3 / len(fn_list))
    del g
    return statistics.median(times)


def kernel_times(case, sets, rra, stream, n_launch=None, packed=False):
    """Per-launch device µs on cold inputs (graphs of back-to-back launches).

    fused_us: rra_pipeline under the current kernel selection -- ONE launch
    (mask scan, gather, attention, every output row written).  With
    packed=True also: fused_tc_us (the warp-specialised tcgen05 kernel
    forced), the two-launch packed path (pack_copy_us: rra_pack with the row
    copy and zero fill; attend_packed_us: rra_attend on the packed buffers
    with the mma.sync kernel; attend_packed_tc_us: the same with the
    warp-specialised tcgen05 kernel) and, for N <= 256, the small-grid
    tcgen05 kernel (attend_packed_tcl_us, fused_tcl_us)."""
    B, N, H, d = case.B, case.N, case.H, case.d
    R = sets.R
    n_launch = n_launch or max(R, 64)
    views = [rra.workspace_views(s[5], B, N, H, d, case.dtype) for s in sets.sets]

    def fused_fn(i):
        keep, q, k, v, out, ws = sets.sets[i % R]
        return lambda: rra.pipeline(keep, q, k, v, out, ws, scale=SCALE, stream=stream)

    # fused_us: rra_pipeline under the current kernel selection (what the
    # timed steps run); the rest force one kernel each.
    res = {"fused_us": graph_time_per_launch([fused_fn(i) for i in range(n_launch)], stream)}
    prev = rra.set_attend_kernel(rra.ATTEND_TCGEN05)
    try:
        if packed:
            res["fused_tc_us"] = graph_time_per_launch([fused_fn(i) for i in range(n_launch)], stream)
            def pack_fn(i):
                keep, q, k, v, out, ws = sets.sets[i % R]
                cu, dst, src, qp, kp, vp = views[i % R]
                return lambda: rra.pack(keep, q, k, v, cu, dst, src, qp, kp, vp, out, stream=stream)

            def attend_fn(i):
                keep, q, k, v, out, ws = sets.sets[i % R]
                cu, dst, src, qp, kp, vp = views[i % R]
                return lambda: rra.attend(qp, kp, vp, cu, B, N, out, scale=SCALE, src_idx=src, N=N,
                                          stream=stream)

            res["pack_copy_us"] = graph_time_per_launch([pack_fn(i) for i in range(n_launch)], stream)
            res["attend_packed_tc_us"] = graph_time_per_launch([attend_fn(i) for i in range(n_launch)], stream)
            if N <= 256:
                rra.set_attend_kernel(rra.ATTEND_TCGEN05_LATENCY)
                res["attend_packed_tcl_us"] = graph_time_per_launch([attend_fn(i) for i in range(n_launch)], stream)
                res["fused_tcl_us"] = graph_time_per_launch([fused_fn(i) for i in range(n_launch)], stream)
            rra.set_attend_kernel(rra.ATTEND_MMA_SYNC)
            res["attend_packed_us"] = graph_time_per_launch([attend_fn(i) for i in range(n_launch)], stream)
    finally:
        rra.set_attend_kernel(prev)
    return res


# DRAM bytes (read + write) per launch of the kernel rra_pipeline runs on a workload,
# each from one ncu capture of the same launches (dram__bytes_read.sum +
# dram__bytes_write.sum): (kernel source, the SHA-256 prefix of that source and the
# headers it includes when it was captured, bytes).  Once any of them changes, the
# traffic is reported as null until it is captured again.
KERNEL_HEADERS = ("common.cuh", "tc_ptx.cuh", "softmax_tc.cuh")
TRAFFIC = {"serving_B4": ("attend_small.cu", "9aa3be4f30069e31", 421376),
           "batched_b64_p80": ("attend_tc.cu", "be714d8c0419632c", 11919360)}


def kernel_source_sha(name):
    """SHA-256 of a kernel source followed by the headers it includes."""
    h = hashlib.sha256()
    for f in (name,) + KERNEL_HEADERS:
        with open(os.path.join(ROOT, "ragged_attention_token_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def pipeline_kernel_name(case, n_sms):
    """The kernel rra_pipeline launches for this workload under the automatic choice."""
    units = case.B * case.H * ((case.N + 127) // 128)
    if units <= 4 * n_sms and case.N <= 256:
        return "attend_small_kernel (fused pipeline, small-grid form: mask scan, gather, attention, zero fill)"
    return "attend_tc_kernel (fused pipeline: mask scan, gather, attention, zero fill)"


def measured_traffic(key):
    if key not in TRAFFIC:
        return None
    name, sha, nbytes = TRAFFIC[key]
    try:
        ok = kernel_source_sha(name).startswith(sha)
    except OSError:
        ok = False
    return nbytes if ok else None


def packed_qkvo_frac(case, us, peaks):
    """Fraction of the attention roofline as stated for this problem: the slower of
    the packed Q/K/V/O bytes (4*T*H*d*s) at the HBM peak and 4*H*d*sum(n_b^2)
    FLOPs at the bf16 peak, over the measured time.  Smaller than the pipeline's
    own byte count (which also writes every padded output row), so a pipeline
    kernel reads lower against it."""
    s = case.q.element_size()
    t_bytes = 4 * case.kept_tokens * case.H * case.d * s / (peaks["hbm_gbs"] * 1e9)
    t_flops = 4 * case.H * case.d * sum(n * n for n in case.lengths) / (peaks["bf16_tflops"] * 1e12)
    return round(max(t_bytes, t_flops) * 1e6 / us, 4)


def roofline_obj(bytes_alg, flops, us, peaks):
    t = us * 1e-6
    bw = bytes_alg / t / 1e9
    tf = flops / t / 1e12
    hbm_frac = bw / peaks["hbm_gbs"]
    ten_frac = tf / peaks["bf16_tflops"]
    if ten_frac > hbm_frac:
        return {"bound": "tensor", "achieved": round(tf, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(ten_frac, 4), "traffic": None}
    return {"bound": "hbm", "achieved": round(bw, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(hbm_frac, 4), "traffic": None}


def percentile(samples, q):
    """The q-quantile of the samples (nearest rank, no interpolation)."""
    s = sorted(samples)
    return s[min(len(s) - 1, int(q * len(s)))]


def host_latency(rra, B, stream, reps=1000, warmup=100):
    """Host-timed µs of one rra_attend at serving batch B (median; p90 for the two C-timed
    forms): + stream sync, and as rra_attend_wait."""
    case = W.make_serving(B)
    keep, q, k, v = (x.cuda() for x in (case.keep, case.q, case.k, case.v))
    out = torch.empty_like(q)
    ws = rra.alloc_workspace(B, case.N, case.H, case.d, case.dtype)
    cu, dst, src, qp, kp, vp = rra.workspace_views(ws, B, case.N, case.H, case.d, case.dtype)
    rra.pack(keep, q, k, v, cu, dst, src, qp, kp, vp, out_zero_fill=out)      # the packed inputs rra_attend reads
    torch.cuda.synchronize()
    rra.get_device_error(clear=True)
    c_samples = rra.time_attend_host(qp, kp, vp, cu, B, case.N, out, warmup=warmup, reps=reps, src_idx=src,
                                     N=case.N, stream=stream)
    w_samples = rra.time_attend_wait_host(qp, kp, vp, cu, B, case.N, out, warmup=warmup, reps=reps, src_idx=src,
                                          N=case.N, stream=stream)
    py = []
    for i in range(warmup + reps):
        t0 = time.perf_counter()
        rra.attend(qp, kp, vp, cu, B, case.N, out, scale=SCALE, src_idx=src, N=case.N, stream=stream)
        stream.synchronize()
        t1 = time.perf_counter()
        if i >= warmup:
            py.append((t1 - t0) * 1e6)
    plan = rra.Plan(keep, q, k, v, out, ws, scale=SCALE)
    g_samples = plan.time_host(warmup, reps, stream=stream)
    plan.close()
    null = rra.time_null_host(warmup, reps, stream=stream)
    torch.cuda.synchronize()
    if rra.get_device_error() != 0:
        raise RuntimeError("host_latency: a kernel recorded a device-side error")
    return {"attend_c": round(statistics.median(c_samples), 2),
            "attend_c_p90": round(percentile(c_samples, 0.9), 2),
            "attend_wait_c": round(statistics.median(w_samples), 2),
            "attend_wait_c_p90": round(percentile(w_samples, 0.9), 2),
            "attend_python": round(statistics.median(py), 2),
            "pipeline_graph_c": round(statistics.median(g_samples), 2),
            "null_kernel_c": round(statistics.median(null), 2)}


# ----------------------------------------------------------------- CPU side

def oracle_legs(case, budget_s=10.0):
    """The CPU oracle (as it stands) on the workload, on this host: kept tokens/s
    on one thread (in this process, BLAS pinned to one thread above) and on every
    core of the affinity mask (one worker process per core, each repeating full
    steps of the same inputs; oracle/timing.py)."""
    import oracle
    from oracle import timing as OT
    keep = case.keep.numpy()
    q, k, v = (x.double().numpy() for x in (case.q, case.k, case.v))
    T = case.kept_tokens
    steps = 0
    t0 = time.perf_counter()
    while True:
        oracle.pipeline(keep, q, k, v, SCALE)
        steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    one = {"value": round(T * steps / el, 1), "threads": 1, "steps": steps, "seconds": round(el, 2)}
    cores = OT.host_cores()
    allc = OT.time_pipeline(keep, q, k, v, SCALE, budget_s, cores)
    every = {"value": round(allc["tokens_per_s"], 1), "threads": cores, "steps": allc["steps"],
             "seconds": round(allc["window_s"], 2)}
    return one, every, cores


def cpu_baseline_obj(case, budget_s=10.0):
    one, every, cores = oracle_legs(case, budget_s)
    return {"value": every["value"], "unit": UNIT, "cores": cores, "threads": every["threads"], "kind": "oracle",
            "sample": (f"full steps of the same workload for ~{budget_s:.0f} s per leg: {every['steps']} steps on "
                       f"{every['threads']} worker processes (one per core, fp64 numpy, BLAS 1 thread each) and "
                       f"{one['steps']} steps on 1 thread"),
            "legs": {"all_cores": every, "one_thread": one}}


# -------------------------------------------------------------------- main

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "rra" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def image_shard(B: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous image range [start, end) of `rank` when B images split over `world` ranks.

    Images are independent (attention never crosses images), so any split
    needs no exchange; the first B % world ranks take one extra image."""
    base, extra = divmod(B, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_config(case, desc, world):
    """The `config` object of both arms' JSON lines (identical for the same workload)."""
    return {"workload": desc, "B": case.B, "N": case.N, "H": case.H, "d": case.d,
            "kept_tokens_per_step": case.kept_tokens,
            "path": "CUDA graphs of rra_pipeline steps on rotating input sets, replayed back to back",
            "l2": "rotating input sets larger than 2x L2 in total: every step reads cold inputs",
            "parallelism": f"replicas x{world}"}


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle, as it stands, on this host's cores.

    One worker process per core repeats full steps of the workload (images and
    steps are independent, as on the GPU side) for about --cpu-budget seconds
    (at least ceil(steps / cores) steps each, bounded to about two minutes)."""
    if rank != 0:
        return 0
    case, desc = make_case(args.workload)
    import oracle
    from oracle import timing as OT
    keep = case.keep.numpy()
    q, k, v = (x.double().numpy() for x in (case.q, case.k, case.v))
    T = case.kept_tokens
    t0 = time.perf_counter()
    oracle.pipeline(keep, q, k, v, SCALE)
    t_one = time.perf_counter() - t0
    cores = OT.host_cores()
    per_worker = max(1, math.ceil(args.steps / cores))
    budget = min(120.0, max(args.cpu_budget, per_worker * t_one))
    warm = max(0, min(args.warmup, int(60.0 / max(t_one, 1e-6)) + 1))
    for _ in range(warm):
        oracle.pipeline(keep, q, k, v, SCALE)
    r = OT.time_pipeline(keep, q, k, v, SCALE, budget, cores)
    value = r["tokens_per_s"]
    steps = r["steps"]
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": args.gpus,
        "steps": steps, "warmup": warm, "ms_per_step": round(T / value * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(case, desc, world),
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": cores, "threads": cores, "kind": "oracle",
                         "sample": f"{steps} full steps of the workload on {cores} worker processes (one per core, "
                                   f"fp64 numpy, BLAS 1 thread each) in {r['window_s']:.1f} s"},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_rra(args, world, rank, local):
    from ragged_attention_token_gb300 import build as _build
    if not _build.up_to_date():
        if rank == 0:
            _build.build()
        barrier(world)
    from ragged_attention_token_gb300 import rra
    rra.set_attend_kernel({"auto": rra.ATTEND_AUTO, "tcgen05": rra.ATTEND_TCGEN05,
                           "mma_sync": rra.ATTEND_MMA_SYNC}[args.attend_kernel])

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    rra.lib()
    stream = torch.cuda.Stream(device=device)
    peaks = measured_peaks()
    case, desc = make_case(args.workload, args.pruning)
    B, N, H, d = case.B, case.N, case.H, case.d
    T = case.kept_tokens
    sets = InputSets(case, device, rra, case.dtype)
    plans = [rra.Plan(*s, scale=SCALE) for s in sets.sets]

    # The timed steps replay CUDA graphs that each hold R consecutive steps
    # (one per rotating input set): the host dispatches once per R steps.
    def step_fn(s):
        return lambda: rra.pipeline(*s[:5], s[5], scale=SCALE, stream=stream)
    q_full, rem = divmod(args.steps, sets.R)
    n_cap0 = rra.launch_count()
    g_full = capture([step_fn(s) for s in sets.sets], stream)
    per_full = (rra.launch_count() - n_cap0) // 2            # eager pass + capture each count once
    launches_per_step = per_full // sets.R
    g_rem, per_rem = None, 0
    if rem:
        n_cap0 = rra.launch_count()
        g_rem = capture([step_fn(s) for s in sets.sets[:rem]], stream)
        per_rem = (rra.launch_count() - n_cap0) // 2

    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            plans[i % sets.R].launch(stream)
        stream.synchronize()
        # identical load for a while so the clock samples describe the timed region
        t_end = time.time() + args.clock_window
        while time.time() < t_end:
            for _ in range(8):
                g_full.replay()
            stream.synchronize()

        barrier(world)
        torch.cuda.synchronize(device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        # A ~0.1 ms device sleep ahead of the start event: the host submits the
        # first graph while the GPU sleeps, so the events time the steps on the
        # device and not the first submission (which a short --steps run would
        # otherwise spread over few steps).
        torch.cuda._sleep(SLEEP_CYCLES)
        e0.record(stream)
        for _ in range(q_full):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        e1.record(stream)
        e1.synchronize()
        torch.cuda.synchronize(device)
        barrier(world)
        launches = q_full * per_full + per_rem

        # the same steps dispatched one call at a time (one graph launch per step)
        e4 = torch.cuda.Event(enable_timing=True)
        e5 = torch.cuda.Event(enable_timing=True)
        e4.record(stream)
        for i in range(args.steps):
            plans[i % sets.R].launch(stream)
        e5.record(stream)
        e5.synchronize()
    clocks = sampler.stop()
    el_ms = max_over_ranks(e0.elapsed_time(e1), world, device)
    value = T * args.steps * world / (el_ms * 1e-3)
    per_call_ms = max_over_ranks(e4.elapsed_time(e5), world, device)
    per_call_value = T * args.steps * world / (per_call_ms * 1e-3)

    # e2e: pinned host inputs -> GPU -> path -> pinned host output, every step.
    # Headline: rra_pipeline_mapped, whose kernels read the mask and the kept
    # rows over the CPU-GPU link and write the output into host memory.
    # Beside it: rra_pipeline_host (copy engines move the whole padded
    # tensors in, the output back).
    keep_h, q_h, k_h, v_h = (x.contiguous().pin_memory() for x in (case.keep, case.q, case.k, case.v))
    out_h = torch.empty((B, N, H, d), dtype=case.dtype).pin_memory()
    keep_d, q_d, k_d, v_d, out_d, ws_d = sets.sets[0]
    elem = case.q.element_size()
    d2h = out_h.numel() * out_h.element_size()

    def e2e_time(step):
        with torch.cuda.stream(stream):
            for _ in range(max(3, args.warmup)):
                step()
            stream.synchronize()
            barrier(world)
            ea = torch.cuda.Event(enable_timing=True)
            eb = torch.cuda.Event(enable_timing=True)
            ea.record(stream)
            for _ in range(args.steps):
                step()
            eb.record(stream)
            eb.synchronize()
        return max_over_ranks(ea.elapsed_time(eb), world, device)

    e2e_ms = e2e_time(lambda: rra.pipeline_mapped(keep_h, q_h, k_h, v_h, out_h, ws_d, SCALE, stream))
    e2e_value = T * args.steps * world / (e2e_ms * 1e-3)
    h2d = keep_h.numel() + 3 * T * H * d * elem            # the mask and the kept rows cross the link
    copy_ms = e2e_time(lambda: rra.pipeline_host(keep_h, q_h, k_h, v_h, out_h, keep_d, q_d, k_d, v_d, out_d, ws_d,
                                                 SCALE, stream))
    e2e_copy = {"value": round(T * args.steps * world / (copy_ms * 1e-3), 1), "unit": UNIT,
                "ms_per_step": round(copy_ms / args.steps, 5),
                "h2d_bytes_per_step": sum(x.numel() * x.element_size() for x in (keep_h, q_h, k_h, v_h)),
                "d2h_bytes_per_step": d2h,
                "path": "rra_pipeline_host (cudaMemcpyAsync of the padded keep/q/k/v in, the fused kernel, the "
                        "output out)"}

    # per-kernel device time (graph of back-to-back launches on cold inputs)
    n_sms = torch.cuda.get_device_properties(device).multi_processor_count
    fused = args.attend_kernel != "mma_sync"     # rra_pipeline: fused tcgen05 unless mma.sync is forced
    kt = kernel_times(case, sets, rra, stream, packed=not fused)
    by = case_bytes(case)
    if fused:
        kern = {"fused_us": round(kt["fused_us"], 3)}
        roof = roofline_obj(by["fused_min"], by["flops"], kt["fused_us"], peaks)
        roof["traffic"] = measured_traffic(case.name)
        roof["kernel"] = pipeline_kernel_name(case, n_sms)
    else:
        kern = {"pack_copy_us": round(kt["pack_copy_us"], 3), "attend_packed_us": round(kt["attend_packed_us"], 3),
                "fused_tcgen05_us": round(kt["fused_tc_us"], 3)}
        if kt["attend_packed_us"] >= kt["pack_copy_us"]:
            roof = roofline_obj(by["attend"], by["flops"], kt["attend_packed_us"], peaks)
            roof["kernel"] = "attend_mma_kernel (packed)"
        else:
            roof = roofline_obj(by["pack"], 0, kt["pack_copy_us"], peaks)
            roof["kernel"] = "pack_kernel (row copy + indices + zero fill)"
    roof["peak_source"] = peaks["source"]

    extra = {}
    if rank == 0 and not args.quick:
        extra["host_us"] = {f"bs{b}": host_latency(rra, b, stream) for b in W.SERVING_BATCHES}
        big, big_desc = make_case("batched")
        big_sets = InputSets(big, device, rra, big.dtype)
        bk = kernel_times(big, big_sets, rra, stream)
        bb = case_bytes(big)
        extra["batched_b64_p80"] = {"workload": big_desc, "fused_us": round(bk["fused_us"], 3),
                                    "roofline": {**roofline_obj(bb["fused_min"], bb["flops"], bk["fused_us"], peaks),
                                                 "traffic": measured_traffic("batched_b64_p80")},
                                    "packed_qkvo_frac": packed_qkvo_frac(big, bk["fused_us"], peaks),
                                    "pipeline_tokens_per_s": round(big.kept_tokens / (bk["fused_us"] * 1e-6), 1)}
        del big_sets

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline_obj(case, budget_s=args.cpu_budget)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": round(el_ms / args.steps, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if case.dtype == torch.bfloat16 else "f16",
            "data": "synthetic (seeded N(0,1) Q/K/V, seeded keep masks)",
            "config": workload_config(case, desc, world),
            "timing": {"graph": f"CUDA graphs of {sets.R} rra_pipeline steps, replayed back to back",
                       "l2": f"{sets.R} rotating input sets of {sets.per_set / 2**20:.1f} MiB "
                             f"({sets.R * sets.per_set / 2**20:.0f} MiB > L2)",
                       "start": "a ~0.1 ms device sleep is queued before the start event, so the events time "
                                "the steps on the device and not the first graph's host submission"},
            "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(e2e_ms / args.steps, 5),
                    "path": "rra_pipeline_mapped (inputs and output in pinned host memory; the kernel (at serving "
                            "sizes one fused launch, else pack + attend) reads the mask and the kept rows over the "
                            "CPU-GPU link and writes the output into host memory)"},
            "e2e_copy": e2e_copy,
            "roofline": roof,
            "kernels": kern,
            "attend_kernel": args.attend_kernel,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "gpu_launches": int(launches) * world,
            "launches_per_step": launches_per_step,
            "per_call_dispatch": {"value": round(per_call_value, 1), "unit": UNIT,
                                  "ms_per_step": round(per_call_ms / args.steps, 5),
                                  "path": f"one rra_plan_launch (a graph of {launches_per_step} kernel launch"
                                          f"{'es' if launches_per_step != 1 else ''}) per step from Python"},
        }
        line.update(extra)
        print(json.dumps(line), flush=True)
    for p in plans:
        p.close()
    return 0


def progressive_chain_times(rra, stream, peaks, B=256, reps=10):
    """The 12-layer progressive workload at batch B, one CUDA graph per pass, four ways.

    Every layer after the first receives its Q/K/V in the previous layer's
    packed layout (as projections of packed features would).
    chain (in place): at layer 1 and at each pruning layer an index pass
    (rra_pack_index) and attention reading the layer's input rows where they
    are (rra_attend_rows, packed output); rra_attend at the other layers; one
    unpack after the last layer.  No Q/K/V row is copied.
    chain_copy: layer 1 packs its padded Q/K/V (rra_pack) and each pruning
    layer re-packs them (rra_repack) before rra_attend.
    chain_device: the in-place chain with the three pruning decisions made on
    the device from the attention's class-token side output (rra_prune_index).
    per_layer: rra_pipeline (padded in, padded out) for every layer."""
    dev = torch.device("cuda", 0)
    masks, cases = W.make_progressive_chain(B)
    N, H, d = cases[0].N, cases[0].H, cases[0].d
    L = len(cases)
    keeps = [m.to(dev) for m in masks]
    padded = [tuple(x.to(dev) for x in (c.q, c.k, c.v)) for c in cases]

    def index_bufs():
        return (torch.empty(B + 1, dtype=torch.int32, device=dev), torch.empty(B * N, dtype=torch.int32, device=dev),
                torch.empty(B * N, dtype=torch.int32, device=dev))

    def packed_bufs():
        return [torch.empty((B * N, H, d), dtype=torch.bfloat16, device=dev) for _ in range(3)]

    inputs = [padded[0]]
    for l in range(1, L):
        pb = packed_bufs()
        rra.pack(keeps[l - 1], *padded[l], *index_bufs(), *pb, stream=stream)
        inputs.append(tuple(pb))
    stream.synchronize()
    event = [l > 0 and not torch.equal(masks[l], masks[l - 1]) for l in range(L)]
    idx = []
    for l in range(L):
        idx.append(index_bufs() if (l == 0 or event[l]) else idx[l - 1])
    packed = [packed_bufs() if (l == 0 or event[l]) else None for l in range(L)]
    outs = [torch.empty((B * N, H, d), dtype=torch.bfloat16, device=dev) for _ in range(L)]
    final = torch.empty((B, N, H, d), dtype=torch.bfloat16, device=dev)

    def chain():
        rra.pack(keeps[0], *inputs[0], *idx[0], *packed[0], stream=stream)
        for l in range(L):
            src = packed[0] if l == 0 else inputs[l]
            if l > 0 and event[l]:
                rra.repack(keeps[l], idx[l - 1][1], *inputs[l], *idx[l], *packed[l], stream=stream)
                src = packed[l]
            rra.attend(*src, idx[l][0], B, N, outs[l], scale=SCALE, stream=stream)
        rra.unpack(outs[L - 1], idx[L - 1][1], B, N, final, stream=stream)

    rows = [torch.empty(B * N, dtype=torch.int32, device=dev) if (l == 0 or event[l]) else None for l in range(L)]
    flat = [tuple(x.view(-1, H, d) for x in inputs[l]) for l in range(L)]

    def chain_in_place():
        for l in range(L):
            if l == 0 or event[l]:
                rra.pack_index(keeps[l], *idx[l], rows[l], dst_prev=None if l == 0 else idx[l - 1][1], stream=stream)
                rra.attend_rows(*flat[l], rows[l], idx[l][0], B, N, outs[l], scale=SCALE, stream=stream)
            else:
                rra.attend(*inputs[l], idx[l][0], B, N, outs[l], scale=SCALE, stream=stream)
        rra.unpack(outs[L - 1], idx[L - 1][1], B, N, final, stream=stream)

    # chain_device: the same chain with every pruning decision made on the
    # device -- the layer before an event writes the class-token side output
    # (rra_attend_cls / rra_attend_rows) and one rra_prune_index launch gives
    # the next layer's indices (the workload's keep fraction, so the kept
    # counts equal the fixed masks').
    stride = (N + 15) // 16 * 16
    cls_bufs = {l - 1: torch.empty((B, H, stride), dtype=torch.float32, device=dev)
                for l in range(1, L) if event[l]}
    idx_d = [index_bufs() if (l == 0 or event[l]) else None for l in range(L)]
    for l in range(L):
        idx_d[l] = idx_d[l] if idx_d[l] is not None else idx_d[l - 1]
    rows_d = [torch.empty(B * N, dtype=torch.int32, device=dev) if (l == 0 or event[l]) else None for l in range(L)]
    num, den = round(W.PROGRESSIVE_KEEP * 10), 10

    def chain_device():
        rra.pack_index(keeps[0], *idx_d[0], rows_d[0], stream=stream)
        for l in range(L):
            cls = cls_bufs.get(l)
            if l == 0 or event[l]:
                rra.attend_rows(*flat[l], rows_d[l], idx_d[l][0], B, N, outs[l], scale=SCALE, cls=cls, stream=stream)
            elif cls is not None:
                rra.attend_cls(*inputs[l], idx_d[l][0], B, N, outs[l], cls, scale=SCALE, stream=stream)
            else:
                rra.attend(*inputs[l], idx_d[l][0], B, N, outs[l], scale=SCALE, stream=stream)
            if cls is not None:
                rra.prune_index(cls, idx_d[l][0], idx_d[l][2], N, num, den, *idx_d[l + 1], rows_d[l + 1],
                                stream=stream)
        rra.unpack(outs[L - 1], idx_d[L - 1][1], B, N, final, stream=stream)

    ws = rra.alloc_workspace(B, N, H, d, torch.bfloat16)
    outs_pl = [torch.empty_like(padded[l][0]) for l in range(L)]

    def per_layer():
        for l in range(L):
            rra.pipeline(keeps[l], *padded[l], outs_pl[l], ws, scale=SCALE, stream=stream)

    t_copy = graph_time_per_launch([chain], stream, reps)
    t_chain = graph_time_per_launch([chain_in_place], stream, reps)
    t_device = graph_time_per_launch([chain_device], stream, reps)
    same_counts = all(torch.equal(idx_d[l][0], idx[l][0]) for l in range(L))
    t_layer = graph_time_per_launch([per_layer], stream, reps)
    kept = [int((m != 0).sum()) for m in masks]
    row = H * d * 2
    # Algorithmic bytes of the in-place chain: per index pass the mask, the
    # previous dst (pruning layers), dst/src/rows/cu written; per layer Q, K,
    # V read and O written; the final unpack (packed rows in, padded out).
    chain_bytes = B * N * row + kept[-1] * row
    for l in range(L):
        chain_bytes += 4 * kept[l] * row
        if l == 0 or event[l]:
            chain_bytes += B * N + (4 * B * N if l > 0 else 0) + 4 * B * N + 8 * kept[l] + 4 * (B + 1)
    t_min = chain_bytes / (peaks["hbm_gbs"] * 1e9) * 1e6
    events = sum(event)
    line = {"case": f"progressive_chain_B{B}", "B": B, "N": N, "H": H, "layers": L, "kept_tokens_all_layers": sum(kept),
            "chain_us": round(t_chain, 2), "chain_copy_us": round(t_copy, 2), "per_layer_fused_us": round(t_layer, 2),
            "chain_device_decisions_us": round(t_device, 2), "device_decisions_same_lengths": bool(same_counts),
            "per_device_decision_us": round((t_device - t_chain) / max(1, sum(event)), 2),
            "chain_speedup": round(t_layer / t_chain, 3),
            "chain_tokens_per_s": round(sum(kept) / (t_chain * 1e-6), 1),
            "chain_min_us": round(t_min, 2), "chain_frac": round(t_min / t_chain, 4),
            "launches_chain": 2 * (1 + events) + (L - 1 - events) + 1,
            "launches_chain_copy": 1 + L + events + 1, "launches_per_layer": L}
    del padded, inputs, packed, outs, outs_pl, final, ws, rows, flat, cls_bufs, idx_d, rows_d
    torch.cuda.empty_cache()
    return line


def device_pruning_times(rra, stream, B=256, reps=10):
    """One pruning step of the progressive workload on the device (layer 3 -> 4 at batch B):
    class-token scores from layer 3's packed Q/K, then the 70% top-k keep decision."""
    dev = torch.device("cuda", 0)
    masks, cases = W.make_progressive_chain(B)
    c = cases[2]
    keep, q, k, v = (x.to(dev) for x in (c.keep, c.q, c.k, c.v))
    N, H, d = c.N, c.H, c.d
    cu = torch.empty(B + 1, dtype=torch.int32, device=dev)
    dst = torch.empty(B * N, dtype=torch.int32, device=dev)
    src = torch.empty(B * N, dtype=torch.int32, device=dev)
    qp, kp, vp = (torch.empty((B * N, H, d), dtype=c.dtype, device=dev) for _ in range(3))
    rra.pack(keep, q, k, v, cu, dst, src, qp, kp, vp, stream=stream)
    scores = torch.empty((B, N), dtype=torch.float32, device=dev)
    keep_new = torch.empty_like(keep)
    # graphs of 20 back-to-back launches (the inputs stay in L2 between them)
    t_scores = graph_time_per_launch([lambda: rra.cls_scores(qp, kp, cu, src, B, N, scores, scale=SCALE,
                                                             stream=stream)] * 20, stream, reps)
    t_topk = graph_time_per_launch([lambda: rra.topk_keep(scores, keep, 7, 10, keep_new, stream=stream)] * 20,
                                   stream, reps)
    # The same step from the attention's class-token side output: the layer's
    # attention with the side output plus one decision launch, against the
    # plain attention (tcgen05 kernel both).
    o = torch.empty((B * N, H, d), dtype=c.dtype, device=dev)
    cls = torch.empty((B, H, (N + 15) // 16 * 16), dtype=torch.float32, device=dev)
    keep_cls = torch.empty_like(keep)
    prev = rra.set_attend_kernel(rra.ATTEND_TCGEN05)
    try:
        t_attend = graph_time_per_launch([lambda: rra.attend(qp, kp, vp, cu, B, N, o, scale=SCALE, stream=stream)] * 10,
                                         stream, reps)
        t_attend_cls = graph_time_per_launch(
            [lambda: rra.attend_cls(qp, kp, vp, cu, B, N, o, cls, scale=SCALE, stream=stream)] * 10, stream, reps)
        t_step = graph_time_per_launch(
            [lambda: rra.attend_cls(qp, kp, vp, cu, B, N, o, cls, scale=SCALE, stream=stream),
             lambda: rra.topk_keep_cls(cls, cu, src, N, 7, 10, keep_cls, stream=stream)] * 10, stream, reps) * 2
    finally:
        rra.set_attend_kernel(prev)
    t_topk_cls = graph_time_per_launch([lambda: rra.topk_keep_cls(cls, cu, src, N, 7, 10, keep_cls, stream=stream)]
                                       * 20, stream, reps)
    return {"case": f"device_pruning_B{B}", "B": B, "N": N, "H": H, "kept_before": int((c.keep != 0).sum()),
            "kept_after": int((keep_new != 0).sum()), "cls_scores_us": round(t_scores, 2),
            "topk_keep_us": round(t_topk, 2),
            "side_output": {"attend_us": round(t_attend, 2), "attend_cls_us": round(t_attend_cls, 2),
                            "topk_keep_cls_us": round(t_topk_cls, 2), "attend_cls_and_topk_us": round(t_step, 2),
                            "pruning_over_attention_us": round(t_step - t_attend, 2),
                            "same_keep": bool(torch.equal(keep_cls, keep_new))}}


def linear_times(rra, stream, peaks, reps=10):
    """Packed QKV projection of the batched DeiT-B workload (K=768 -> N=2304) with
    rra_linear_packed: over the kept rows only (T from cu_seqlens on the device)
    at 80% and 0% pruning, and over every padded row; torch's cuBLAS GEMM on the
    same rows for context."""
    dev = torch.device("cuda", 0)
    K, Nout = 768, 2304
    g = torch.Generator().manual_seed(2024)
    w = (torch.randn((Nout, K), generator=g) / math.sqrt(K)).to(torch.bfloat16).to(dev)
    bias = torch.randn((Nout,), generator=g).to(dev)
    lines = []
    for rate in (0.8, 0.0):
        case = W.make_batched(rate)
        cap = case.B * case.N
        T = case.kept_tokens
        a = torch.randn((cap, K), generator=g).to(torch.bfloat16).to(dev)
        c = torch.empty((cap, Nout), dtype=torch.bfloat16, device=dev)
        cu_kept = torch.tensor([0, T], dtype=torch.int32, device=dev)
        cu_all = torch.tensor([0, cap], dtype=torch.int32, device=dev)
        t_kept = graph_time_per_launch([lambda: rra.linear_packed(a, w, cu_kept, 1, c, bias=bias, stream=stream)] * 10,
                                       stream, reps)
        t_all = graph_time_per_launch([lambda: rra.linear_packed(a, w, cu_all, 1, c, bias=bias, stream=stream)] * 10,
                                      stream, reps)
        a_t = a[:T]
        bias_lp = bias.to(torch.bfloat16)

        def cublas():
            with torch.cuda.stream(stream):
                torch.nn.functional.linear(a_t, w, bias_lp)
        t_cublas = graph_time_per_launch([cublas] * 10, stream, reps)
        flops = 2.0 * T * K * Nout
        peak = peaks.get("bf16_tflops")
        lines.append({"case": f"linear_packed_qkv_b64_p{int(rate * 100)}", "T": T, "rows_padded": cap, "K": K,
                      "N": Nout, "packed_us": round(t_kept, 2), "padded_rows_us": round(t_all, 2),
                      "cublas_packed_us": round(t_cublas, 2),
                      "tflops": round(flops / (t_kept * 1e-6) / 1e12, 1), "peak_tflops": peak,
                      "frac": round(flops / (t_kept * 1e-6) / 1e12 / peak, 4) if peak else None})
        del a, c
    return lines


def run_sweep(args):
    """Every workload: device µs per kernel, path tokens/s, roofline (one JSON line each)."""
    from ragged_attention_token_gb300 import build as _build
    _build.build()
    from ragged_attention_token_gb300 import rra
    rra.set_attend_kernel({"auto": rra.ATTEND_AUTO, "tcgen05": rra.ATTEND_TCGEN05,
                           "mma_sync": rra.ATTEND_MMA_SYNC}[args.attend_kernel])
    device = torch.device("cuda", 0)
    n_sms = torch.cuda.get_device_properties(device).multi_processor_count
    stream = torch.cuda.Stream(device=device)
    peaks = measured_peaks()
    parts = set(args.sweep_parts.split(","))
    cases = []
    if "kernels" in parts:
        cases = [W.make_tiny()] + [W.make_serving(b) for b in W.SERVING_BATCHES] + \
                [W.make_batched(p) for p in W.BATCHED_RATES] + [W.make_hires(p) for p in W.HIRES_RATES]
        masks = W.progressive_masks()
        cases += [W.make_progressive_layer(L, masks) for L in (1, 4, 7, 10)]
    for case in cases:
        sets = InputSets(case, device, rra, case.dtype)
        kt = kernel_times(case, sets, rra, stream, packed=True)
        by = case_bytes(case)
        fused_min_t = by["fused_min"] / (peaks["hbm_gbs"] * 1e9) * 1e6
        two = kt["pack_copy_us"] + kt["attend_packed_us"]
        line = {"case": case.name, "B": case.B, "N": case.N, "H": case.H, "T": case.kept_tokens,
                **{k: round(v, 3) for k, v in kt.items()},
                "fused_min_us": round(fused_min_t, 3), "fused_frac": round(fused_min_t / kt["fused_us"], 4),
                "packed_qkvo_frac": {"fused": packed_qkvo_frac(case, kt["fused_us"], peaks),
                                     "attend_packed_tc": packed_qkvo_frac(case, kt["attend_packed_tc_us"], peaks)},
                "fused": roofline_obj(by["fused_min"], by["flops"], kt["fused_us"], peaks),
                "two_launch_mma_us": round(two, 3),
                "fused_tokens_per_s": round(case.kept_tokens / (kt["fused_us"] * 1e-6), 1)}
        print(json.dumps(line), flush=True)
        del sets
    if "chain" in parts:
        print(json.dumps(progressive_chain_times(rra, stream, peaks)), flush=True)
    if "pruning" in parts:
        print(json.dumps(device_pruning_times(rra, stream)), flush=True)
    if "linear" in parts:
        for line in linear_times(rra, stream, peaks):
            print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("rra", "reference"), default="rra")
    ap.add_argument("--workload", default="serving", choices=("serving", "tiny", "batched", "hires"))
    ap.add_argument("--sweep", action="store_true", help="per-workload kernel timings, one line each")
    ap.add_argument("--sweep-parts", default="kernels,chain,pruning,linear",
                    help="comma-separated parts of --sweep: kernels, chain, pruning, linear")
    ap.add_argument("--quick", action="store_true", help="skip host-latency and B=64 extras")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of CPU oracle work")
    ap.add_argument("--clock-window", type=float, default=1.5, help="seconds of load before the timed region")
    ap.add_argument("--pruning", type=float, default=None,
                    help="pruning rate for the batched / hires workloads (their sweep values)")
    ap.add_argument("--attend-kernel", choices=("auto", "tcgen05", "mma_sync"), default="auto",
                    help="attention kernel behind rra_attend / rra_pipeline")
    args = ap.parse_args(argv)
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        rc = run_reference(args, world, rank)
    elif args.sweep:
        rc = run_sweep(args) if rank == 0 else 0
    else:
        rc = run_rra(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
