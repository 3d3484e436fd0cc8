"""Benchmark of the sm_103a pipelined tiled fp16 GEMM.

One step = one GEMM C = A @ B (fp16 in, fp32 accumulate) over one batch of
synthetic input.  The default workload is the compute-bound 8192^3 fp16-out
product; ``--workload`` picks another of the five shapes.

Prints ONE JSON line (rank 0):
  value      TFLOP/s = 2MNK x ranks / (max over ranks of the timed seconds / steps),
             inputs resident in HBM, rotated over 3 copies (each > L2)
  e2e        the same metric through the public API with host buffers: every
             step's H2D copy of A and B from pinned memory and D2H copy of C
             are inside the timed region; value: copies and GEMMs pipelined
             over three streams and two buffer sets; serial_value: all of it
             on one stream, in turn
  roofline   the GEMM kernel's achieved TFLOP/s (algorithmic flops / average
             launch time from CUDA events) against the measured dense peak
  cpu_baseline  the CPU oracle timed on a bounded sample of the same workload
  clocks     SM clocks and throttle reasons sampled during the timed region
  configs    after the headline, every one of the five workloads (256^3,
             4096^3, 8192^3, the M = 128 skinny product, long K with fp32 out)
             timed on its own: inputs rotated past L2, at least 20 launches
             back to back, eager and replayed from a CUDA graph; per config
             the milliseconds per launch, TFLOP/s, GB/s, its roofline (the
             tensor peak or the HBM copy rate, whichever binds) and its plan;
             then <workload>_sustained for 8192^3, long K and 4096^3: each
             back to back for a few seconds, at the power cap, with its
             clocks.  Beside each,
             `cublas`: torch.mm (cuBLAS, fp16 out) on the same operands, timed
             the same way, for comparison only

``--impl reference`` times the CPU oracle instead (the reference arm): each
step computes a bounded sample of rows of the same product on the host cores.

Multi-GPU (torchrun, one rank per GPU): replicas only -- every rank runs the
same full GEMM on its own GPU; there is no data-path collective.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (fp16 in, fp32 acc) at 8192³; % of GB300 dense FP16 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["tensor_core_tiled_02_gb300/csrc/add_kernel.cuh", "tensor_core_tiled_02_gb300/csrc/bounds.cuh",
                  "tensor_core_tiled_02_gb300/csrc/gemm_common.cuh", "tensor_core_tiled_02_gb300/csrc/gemm_kernel.cuh",
                  "tensor_core_tiled_02_gb300/csrc/gemm_pair_kernel.cuh", "tensor_core_tiled_02_gb300/csrc/ptx.cuh",
                  "tensor_core_tiled_02_gb300/csrc/gemm_small_kernel.cuh",
                  "tensor_core_tiled_02_gb300/csrc/gemm_f16.cu"]


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gemm_8192")
    ap.add_argument("--e2e-steps", type=int, default=30, help="0 skips the end-to-end leg")
    ap.add_argument("--copies", type=int, default=3, help="rotated input copies (each larger than L2)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU baseline sample budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--configs", default="all",
                    help="per-config leg after the headline: 'all', 'none' or a comma list of workloads")
    ap.add_argument("--config-ms", type=float, default=30.0, help="timed milliseconds per config (at least 20 launches)")
    ap.add_argument("--no-cublas", action="store_true", help="skip the cuBLAS comparison in the config leg")
    ap.add_argument("--sustained-s", type=float, default=3.0,
                    help="seconds of back-to-back launches at the power cap per sustained workload (0 skips)")
    ap.add_argument("--sustained", default="gemm_8192,long_k,gemm_4096",
                    help="comma list of workloads timed at the power cap")
    return ap.parse_args(argv)


# ---- distributed plumbing (replicas only) -------------------------------------


class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend: str):
        if self.world > 1:
            import torch.distributed as dist

            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float, device=None) -> float:
        if self.pg is None:
            return x
        import torch

        t = torch.tensor([x], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def aggregate(per_rank_seconds: list[float], flops_per_step: float, steps: int) -> dict:
    """Whole-job throughput from every rank's timed seconds: all ranks' work
    over the slowest rank's time (replicas: each rank ran `steps` GEMMs)."""
    t = max(per_rank_seconds)
    n = len(per_rank_seconds)
    return {"seconds": t, "ms_per_step": 1e3 * t / steps, "tflops": n * flops_per_step * steps / t / 1e12}


# ---- peaks, clocks, profiles -------------------------------------------------------


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, enabled: bool = True):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None
        self.enabled = enabled

    def start(self):
        if not self.enabled:
            return
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        return summarize_clocks(rows)


def summarize_clocks(rows) -> dict | None:
    def num(s):
        try:
            return float(s)
        except ValueError:
            return None

    if not rows:
        return None
    sm = [num(r[1]) for r in rows if num(r[1]) is not None]
    mx = [num(r[2]) for r in rows if num(r[2]) is not None]
    pw = [num(r[3]) for r in rows if num(r[3]) is not None]
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = set()
    for r in rows:
        for name, v in zip(names, r[5:9]):
            if v.strip().lower() in ("active", "1", "yes"):
                reasons.add(name)
    # samples under load: the upper part of the clock range (idle samples at the
    # edges of the window are dropped by taking the samples with power near max)
    loaded = sm
    if pw and len(pw) == len(sm):
        pmax = max(pw)
        loaded = [s for s, p in zip(sm, pw) if p >= 0.6 * pmax] or sm
    return {"sm_mhz": statistics.median(loaded) if loaded else None,
            "sm_max_mhz": max(mx) if mx else None,
            "power_w_max": max(pw) if pw else None,
            "samples": len(rows),
            "reasons": sorted(reasons)}


def kernel_source_hash() -> str:
    """Hash of the kernel and host sources with comments and blank space
    removed, so that recorded ncu counters stay valid across comment edits
    and go stale on any code change."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = re.sub(r"\s+", " ", text)
        h.update(text.encode())
    return h.hexdigest()[:16]


def kernel_family(plan: dict) -> str:
    if plan.get("kind") == "add":
        return "add_f32_kernel"
    if plan.get("cta_group") == 1 and plan.get("tile_m", 128) < 128:
        return "gemm_f16_small_kernel"
    return "gemm_f16_pair_kernel" if plan.get("cta_group") == 2 else "gemm_f16_kernel"


def recorded_traffic(workload: str, plan: dict) -> int | None:
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, if it was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel_family(plan)}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    m_traffic = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    if not (m_hash and m_traffic) or m_hash.group(1) != kernel_source_hash():
        return None
    return int(m_traffic.group(1))


# ---- the CPU oracle (baseline and reference arm) -----------------------------------


def cpu_oracle_sample(a, b, w, budget_s: float, rows_per_call: int | None = None):
    """Time the oracle on whole rows of the product; return (value TFLOP/s,
    rows, seconds, threads).  B is decoded once before timing (inputs
    resident), then rows are computed until about `budget_s` has passed."""
    import numpy as np

    import oracle

    threads = os.cpu_count() or 1
    dec = oracle.DecodedB(b.numpy())
    a_np = a.numpy()
    rng = np.random.default_rng(0)
    per_call = rows_per_call or threads
    # calibration call (also faults in pages), not counted
    dec.gemm_rows(a_np, rng.integers(0, w.M, per_call), w.out_dtype, nthreads=threads)
    done_rows = 0
    t0 = time.perf_counter()
    while True:
        rows = rng.integers(0, w.M, per_call)
        dec.gemm_rows(a_np, rows, w.out_dtype, nthreads=threads)
        done_rows += per_call
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    flops = 2.0 * done_rows * w.N * w.K
    return flops / el / 1e12, done_rows, el, threads


def run_reference(args, w, dist: Dist):
    """The reference arm: the CPU oracle, each step a bounded sample of rows."""
    import numpy as np

    import oracle
    from tensor_core_tiled_02_gb300.synthetic import workload_inputs

    if dist.rank != 0:
        return 0
    if w.kind == "add":
        return run_reference_add(args, w)
    threads = os.cpu_count() or 1
    a, b = workload_inputs(w)
    dec = oracle.DecodedB(b.numpy())
    a_np = a.numpy()
    rng = np.random.default_rng(0)
    rows_per_step = threads  # one whole row per thread per step
    for _ in range(args.warmup):
        dec.gemm_rows(a_np, rng.integers(0, w.M, rows_per_step), w.out_dtype, nthreads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        dec.gemm_rows(a_np, rng.integers(0, w.M, rows_per_step), w.out_dtype, nthreads=threads)
    el = time.perf_counter() - t0
    flops = 2.0 * rows_per_step * w.N * w.K * args.steps
    value = flops / el / 1e12
    sample = (f"{rows_per_step} whole rows of the {w.M}x{w.N}x{w.K} product per step "
              f"({rows_per_step}*{w.N} of {w.M * w.N} outputs), B decoded to fp64 once before timing")
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": workload_config(w, None),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference_add(args, w):
    """Reference arm of the blocked add: the oracle, one whole addition per step."""
    import oracle
    from tensor_core_tiled_02_gb300.synthetic import add_inputs

    x, y = add_inputs(w.M, w.N)
    xn, yn = x.numpy(), y.numpy()
    for _ in range(args.warmup):
        oracle.add_f32(xn, yn)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.add_f32(xn, yn)
    el = time.perf_counter() - t0
    value = float(w.bytes_moved) * args.steps / el / 1e9
    line = {
        "metric": ADD_METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "impl": "reference",
        "config": {"workload": w.name, "M": w.M, "N": w.N},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"one whole {w.M}x{w.N} addition per step (one thread)"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def gemm_roofline(w, launch_s: float) -> dict:
    """The GEMM's roofline: the tensor peak or the HBM copy rate, whichever
    takes longer to do the launch's algorithmic work (2MNK flops; A, B and C
    each moved once).  The other fraction is reported beside it."""
    peaks, src = load_peaks()
    tflops = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    tflops_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    gbs = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    ach_t = w.flops / launch_s / 1e12
    ach_b = w.bytes_moved / launch_s / 1e9
    tensor = {"bound": "tensor", "achieved": ach_t, "peak": tflops, "unit": "TFLOP/s", "frac": ach_t / tflops,
              "peak_source": f"bf16_tflops (burst) of {src}; fp16 dense rate equals bf16 on this part",
              "frac_of_sustained": ach_t / tflops_sus}
    hbm = {"bound": "hbm", "achieved": ach_b, "peak": gbs, "unit": "GB/s", "frac": ach_b / gbs,
           "peak_source": f"hbm_gbs of {src}"}
    if w.flops / (tflops * 1e12) >= w.bytes_moved / (gbs * 1e9):
        tensor["hbm_frac"] = hbm["frac"]
        return tensor
    hbm["tensor_frac"] = tensor["frac"]
    return hbm


CONFIG_WORKLOADS = ["gemm_256", "gemm_4096", "gemm_8192", "skinny", "long_k"]
PLAN_KEYS = ("cta_group", "tile_m", "tile_n", "tile_k", "stages", "release", "slots", "split", "grid",
             "raster_group", "num_tiles", "k_steps", "dp_tiles", "sk_tiles", "sk_pairs", "sk_split", "sk_helper_tiles",
             "workspace_bytes")


def rotation_copies(set_bytes: int, l2_bytes: int) -> int:
    """Input sets to rotate over so that a launch's operands were last touched
    at least twice the L2 capacity of other data ago (at least 3 sets)."""
    return max(3, math.ceil(2 * l2_bytes / max(set_bytes, 1)))


def kernel_name(w, plan, sms: int = 152) -> str:
    """The kernel instance the plan launches (the library's dispatch rule)."""
    if plan["cta_group"] == 2:
        # small pair launches (128 x 128 tiles filling at most half the pairs, no
        # shared tile) take the instance that prefetches its operands into L2
        pf = int(plan["tile_m"] == 128 and plan["sk_tiles"] == 0 and plan["k_steps"] > 0
                 and plan["num_tiles"] <= plan["grid"] // 2 and 2 * plan["grid"] <= sms)
        return f"gemm_f16_pair_kernel<{w.out_dtype},{plan['tile_k']},{plan['tile_m']},{plan['tile_n']},{pf}>"
    if plan["tile_m"] < 128:
        return f"gemm_f16_small_kernel<{w.out_dtype},{plan['tile_m']}>"
    return f"gemm_f16_kernel<{plan['tile_n']},{w.out_dtype}>"


def time_cublas(A, B, copies: int, n: int, reps: int, dev, out_dtype: int) -> float:
    """Seconds per launch of cuBLAS's fp16 GEMM (torch.mm, fp16 output) on the
    same rotated operands, n launches captured in a CUDA graph and replayed
    `reps` times after a 0.2 s idle spell, as our graph leg is timed.  For
    comparison only: our arm never calls it."""
    import torch

    C = torch.empty((copies, A.shape[1], B.shape[2]), dtype=torch.float16, device=dev)
    cur = torch.cuda.current_stream(dev)
    for i in range(3):
        torch.mm(A[i % copies], B[i % copies], out=C[i % copies])
    side = torch.cuda.Stream(dev)
    side.wait_stream(cur)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for i in range(n):
            torch.mm(A[i % copies], B[i % copies], out=C[i % copies])
    cur.wait_stream(side)
    g.replay()
    torch.cuda.synchronize(dev)
    time.sleep(0.2)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for _ in range(reps):
        g.replay()
    e1.record(cur)
    torch.cuda.synchronize(dev)
    del g, C
    return e0.elapsed_time(e1) / 1e3 / (n * reps)


def time_one_config(w, dev, a_cpu, b_cpu, target_s: float, l2_bytes: int, compare: bool = True) -> dict:
    """Time the GEMM of one workload on the device.  Inputs and outputs are
    rotated over enough copies that each launch reads operands evicted from
    L2.  Two timings, each with CUDA events on the launching stream around at
    least 20 back-to-back launches: `eager` (one ctypes call per launch, so
    host overhead shows for launches of a few microseconds) and `graph` (the
    same launches captured once in a CUDA graph and replayed: the kernels'
    own time).  `ms_per_launch`, and the roofline, take the shorter of the
    two."""
    import torch

    import tensor_core_tiled_02_gb300 as tc

    out_t = torch.float16 if w.out_dtype == 0 else torch.float32
    copies = rotation_copies(w.bytes_moved, l2_bytes)
    A = torch.empty((copies, w.M, w.K), dtype=torch.float16, device=dev)
    B = torch.empty((copies, w.K, w.N), dtype=torch.float16, device=dev)
    C = torch.empty((copies, w.M, w.N), dtype=out_t, device=dev)
    A.copy_(a_cpu.to(dev).unsqueeze(0).expand_as(A))
    B.copy_(b_cpu.to(dev).unsqueeze(0).expand_as(B))
    ws = tc.workspace(w.M, w.N, w.K, w.out_dtype, device=dev)
    plan = tc.gemm_f16_plan(w.M, w.N, w.K, w.out_dtype, with_workspace=ws is not None)
    ws_ptr = ws.data_ptr() if ws is not None else 0
    ws_bytes = ws.numel() if ws is not None else 0
    ptrs = [(A[j].data_ptr(), B[j].data_ptr(), C[j].data_ptr()) for j in range(copies)]

    def launch(i, handle):
        a, b, c = ptrs[i % copies]
        rc = tc.gemm_f16_ws(a, b, c, w.M, w.N, w.K, w.out_dtype, ws_ptr, ws_bytes, handle)
        if rc != 0:
            raise tc.GemmError(rc)

    def timed(fn, stream):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / 1e3

    cur = torch.cuda.current_stream(dev)
    h = cur.cuda_stream
    for i in range(5):
        launch(i, h)
    est = timed(lambda: [launch(i, h) for i in range(10)], cur) / 10
    n = int(min(2000, max(20, math.ceil(target_s / max(est, 1e-7)))))
    # each timed leg starts after a short idle spell, so that both begin in the
    # same power state (a leg started right after another runs nearer the cap)
    time.sleep(0.2)
    eager_s = timed(lambda: [launch(i, h) for i in range(n)], cur)

    side = torch.cuda.Stream(dev)
    side.wait_stream(cur)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for i in range(n):
            launch(i, side.cuda_stream)
    cur.wait_stream(side)
    g.replay()
    reps = int(max(1, math.ceil(target_s / max(n * est, 1e-7))))
    time.sleep(0.2)
    graph_s = timed(lambda: [g.replay() for _ in range(reps)], cur)
    rc, site = tc.gemm_f16_device_status(reset=True)
    if rc != 0:
        raise RuntimeError(f"{w.name}: device wait gave up (site {site})")
    # the kernel's duration: the graph replay when it is shorter (it carries
    # no host launch cost), else the eager launches
    launch_s = min(graph_s / (n * reps), eager_s / n)
    cublas_s = time_cublas(A, B, copies, n, reps, dev, w.out_dtype) if compare else None
    roof = gemm_roofline(w, launch_s)
    roof["traffic"] = recorded_traffic(w.name, plan)
    roof["kernel"] = kernel_name(w, plan, torch.cuda.get_device_properties(dev).multi_processor_count)
    entry = {"M": w.M, "N": w.N, "K": w.K, "out_dtype": "f16" if w.out_dtype == 0 else "f32",
             "ms_per_launch": launch_s * 1e3, "eager_ms_per_launch": eager_s / n * 1e3,
             "graph_ms_per_launch": graph_s / (n * reps) * 1e3,
             "launches": n * reps + n, "tflops": w.flops / launch_s / 1e12,
             "gbs": w.bytes_moved / launch_s / 1e9, "roofline": roof,
             "inputs": f"A ~ {w.a_dist[0]}({w.a_dist[1]:g}), B ~ {w.b_dist[0]}({w.b_dist[1]:g}), fp16, seeds 0/1",
             "l2": f"rotated over {copies} copies of A, B and C, {w.bytes_moved / 1e6:.1f} MB each, "
                   f"{copies * w.bytes_moved / 1e6:.0f} MB in all (> 2x L2)",
             "plan": {k: plan[k] for k in PLAN_KEYS}}
    if cublas_s is not None:
        entry["cublas"] = {"ms_per_launch": cublas_s * 1e3, "ours_over_cublas_speed": cublas_s / launch_s,
                           "what": "torch.mm, fp16 out, same operands, timed as the graph leg"
                                   + (" (ours writes fp32)" if w.out_dtype == 1 else "")}
    if roof["frac"] < 0.2:
        entry["regime"] = ("launch latency: the roofline time is a small part of the launch, which is "
                           "fixed prologue, pipeline fill and drain")
    del A, B, C, ws, g
    return entry


def time_sustained(w, dev, a_cpu, b_cpu, seconds: float, l2_bytes: int, sample_clocks: bool,
                   compare: bool = True) -> dict:
    """A workload back to back for `seconds` (eager launches, inputs rotated
    past L2), long enough for the GPU to settle at its power cap; clocks
    sampled during the run.  Its fraction is against both the burst and the
    sustained measured peak."""
    import torch

    import tensor_core_tiled_02_gb300 as tc

    out_t = torch.float16 if w.out_dtype == 0 else torch.float32
    copies = rotation_copies(w.bytes_moved, l2_bytes)
    As = [a_cpu.to(dev) for _ in range(copies)]
    Bs = [b_cpu.to(dev) for _ in range(copies)]
    Cs = [torch.empty((w.M, w.N), dtype=out_t, device=dev) for _ in range(copies)]
    ws = tc.workspace(w.M, w.N, w.K, w.out_dtype, device=dev)
    ws_ptr = ws.data_ptr() if ws is not None else 0
    ws_bytes = ws.numel() if ws is not None else 0
    cur = torch.cuda.current_stream(dev)

    def launch(i):
        j = i % copies
        rc = tc.gemm_f16_ws(As[j].data_ptr(), Bs[j].data_ptr(), Cs[j].data_ptr(), w.M, w.N, w.K, w.out_dtype,
                            ws_ptr, ws_bytes, cur.cuda_stream)
        if rc != 0:
            raise tc.GemmError(rc)

    for i in range(3):
        launch(i)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(5):
        launch(i)
    torch.cuda.synchronize(dev)
    est = (time.perf_counter() - t0) / 5
    n = max(20, int(seconds / max(est, 1e-6)))
    clocks = ClockSampler(dev.index or 0, enabled=sample_clocks)
    clocks.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for i in range(n):
        launch(i)
    e1.record(cur)
    torch.cuda.synchronize(dev)
    summary = clocks.stop()
    rc, site = tc.gemm_f16_device_status(reset=True)
    if rc != 0:
        raise RuntimeError(f"sustained {w.name}: device wait gave up (site {site})")
    launch_s = e0.elapsed_time(e1) / 1e3 / n
    peaks, src = load_peaks()
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    tflops = w.flops / launch_s / 1e12
    out = {"workload": w.name, "seconds": launch_s * n, "launches": n, "ms_per_launch": launch_s * 1e3,
           "tflops": tflops, "frac_of_burst": tflops / burst, "frac_of_sustained": tflops / sus,
           "peak_source": f"bf16_tflops and bf16_tflops_sustained of {src}", "clocks": summary}
    if compare:
        # cuBLAS's fp16 GEMM the same way, after the GPU has cooled for a second
        Cb = Cs if w.out_dtype == 0 else [torch.empty((w.M, w.N), dtype=torch.float16, device=dev)
                                          for _ in range(copies)]
        time.sleep(1.0)
        clocks = ClockSampler(dev.index or 0, enabled=sample_clocks)
        clocks.start()
        e0.record(cur)
        for i in range(n):
            j = i % copies
            torch.mm(As[j], Bs[j], out=Cb[j])
        e1.record(cur)
        torch.cuda.synchronize(dev)
        cb_s = e0.elapsed_time(e1) / 1e3 / n
        out["cublas"] = {"ms_per_launch": cb_s * 1e3, "tflops": w.flops / cb_s / 1e12,
                         "ours_over_cublas_speed": cb_s / launch_s, "clocks": clocks.stop(),
                         "what": "torch.mm, fp16 out, same operands, back to back for as long"
                                 + (" (ours writes fp32)" if w.out_dtype == 1 else "")}
    return out


def run_configs(args, dev, l2_bytes: int, cached_inputs: dict) -> dict:
    """The per-config leg: every workload of the five, one after another."""
    import torch

    from tensor_core_tiled_02_gb300.synthetic import WORKLOADS, workload_inputs

    names = CONFIG_WORKLOADS if args.configs == "all" else [n for n in args.configs.split(",") if n]
    out = {}
    clocks = ClockSampler(dev.index or 0, enabled=not args.no_clocks)
    clocks.start()
    for name in names:
        w = WORKLOADS[name]
        a_cpu, b_cpu = cached_inputs.get(name) or workload_inputs(w)
        out[name] = time_one_config(w, dev, a_cpu, b_cpu, args.config_ms / 1e3, l2_bytes, not args.no_cublas)
        torch.cuda.empty_cache()
    summary = clocks.stop()
    if summary is not None:
        out["clocks"] = summary
    for name in ([n for n in args.sustained.split(",") if n] if args.sustained_s > 0 else []):
        w = WORKLOADS[name]
        a_cpu, b_cpu = cached_inputs.get(w.name) or workload_inputs(w)
        time.sleep(0.5)
        out[f"{name}_sustained"] = time_sustained(w, dev, a_cpu, b_cpu, args.sustained_s, l2_bytes,
                                                  not args.no_clocks, not args.no_cublas)
        torch.cuda.empty_cache()
    return out


def workload_config(w, plan, copies: int | None = None) -> dict:
    cfg = {"workload": w.name, "M": w.M, "N": w.N, "K": w.K,
           "out_dtype": "f16" if w.out_dtype == 0 else "f32",
           "inputs": f"A ~ {w.a_dist[0]}({w.a_dist[1]:g}), B ~ {w.b_dist[0]}({w.b_dist[1]:g}), fp16, seeds 0/1"}
    if copies is not None:
        per = (w.M * w.K + w.K * w.N) * 2 + w.M * w.N * (2 if w.out_dtype == 0 else 4)
        cfg["l2"] = (f"inputs rotated over {copies} copies of A, B and C, {per / 1e6:.0f} MB each"
                     + (" (> L2)" if per > 126e6 else " (each set fits in L2: time includes no flush)"))
    if plan is not None:
        cfg["plan"] = {k: plan[k] for k in PLAN_KEYS}
    return cfg


# ---- our arm -----------------------------------------------------------------------


def run_ours(args, w, dist: Dist):
    import torch

    import tensor_core_tiled_02_gb300 as tc
    from tensor_core_tiled_02_gb300.synthetic import workload_inputs

    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    dist.init("nccl")
    out_t = torch.float16 if w.out_dtype == 0 else torch.float32
    a_cpu, b_cpu = workload_inputs(w)
    n_copies = max(1, args.copies)
    As = [a_cpu.to(dev) for _ in range(n_copies)]
    Bs = [b_cpu.to(dev) for _ in range(n_copies)]
    Cs = [torch.empty((w.M, w.N), dtype=out_t, device=dev) for _ in range(n_copies)]
    # stream-K workspace (zero-filled once, outside the timed region), when the
    # plan for this problem uses one
    ws = tc.workspace(w.M, w.N, w.K, w.out_dtype, device=dev)
    plan = tc.gemm_f16_plan(w.M, w.N, w.K, w.out_dtype, with_workspace=ws is not None)
    stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream
    ws_ptr = ws.data_ptr() if ws is not None else 0
    ws_bytes = ws.numel() if ws is not None else 0

    def step(i):
        j = i % n_copies
        rc = tc.gemm_f16_ws(As[j].data_ptr(), Bs[j].data_ptr(), Cs[j].data_ptr(), w.M, w.N, w.K, w.out_dtype,
                            ws_ptr, ws_bytes, handle)
        if rc != 0:
            raise tc.GemmError(rc)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize(dev)
    rc, site = tc.gemm_f16_device_status(reset=True)
    if rc != 0:
        raise RuntimeError(f"device wait gave up during warm-up (site {site})")

    # timed region: one launch per step, back to back on one stream (events only
    # at the two ends, so consecutive launches may overlap prologue and tail)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dist.local_rank, enabled=not args.no_clocks)
    clocks.start()
    dist.barrier()
    torch.cuda.synchronize(dev)
    start.record(stream)
    for i in range(args.steps):
        step(i)
    end.record(stream)
    torch.cuda.synchronize(dev)
    dist.barrier()
    clock_summary = clocks.stop()
    seconds = start.elapsed_time(end) / 1e3
    # the GEMM kernel is the only launch in a step: its average duration is the
    # timed region over the launches (an upper bound: gaps count against it)
    avg_launch_s = seconds / args.steps
    rc, site = tc.gemm_f16_device_status(reset=True)
    if rc != 0:
        raise RuntimeError(f"device wait gave up in the timed region (site {site})")

    t_max = dist.max(seconds, device=dev)
    flops = float(w.flops)
    value = aggregate([t_max] * dist.world, flops, args.steps)["tflops"]

    e2e = None
    if args.e2e_steps > 0:
        e2e = run_e2e(args, w, dist, dev, stream, a_cpu, b_cpu, out_t, ws)

    configs = None
    if args.configs != "none":
        del As, Bs, Cs
        torch.cuda.empty_cache()
        l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129 * 2 ** 20)
        configs = run_configs(args, dev, l2, {w.name: (a_cpu, b_cpu)})

    if dist.rank == 0:
        roofline = gemm_roofline(w, avg_launch_s)
        roofline["traffic"] = recorded_traffic(w.name, plan)
        roofline["kernel"] = kernel_name(w, plan, torch.cuda.get_device_properties(dev).multi_processor_count)
        roofline["avg_launch_ms"] = avg_launch_s * 1e3
        cpu = None
        if not args.no_cpu_baseline and dist.world == 1:
            v, rows, el, thr = cpu_oracle_sample(a_cpu, b_cpu, w, args.cpu_seconds)
            cpu = {"value": v, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                   "sample": f"{rows} whole rows (drawn at random, with repeats) of the {w.M}x{w.N}x{w.K} "
                             f"product, {rows * w.N} outputs in {el:.1f} s, B decoded to fp64 once before timing"}
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": dist.world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * t_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": workload_config(w, plan, n_copies),
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps,
            "clocks": clock_summary,
        }
        if configs is not None:
            line["configs"] = configs
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


def time_e2e(dev, steps: int, h_in, d_sets, h_outs, compute):
    """Seconds for `steps` end-to-end steps, each copying its inputs `h_in`
    (pinned) into a device buffer set, computing, and copying the result back
    to a pinned host buffer.  Two ways, both timed with events on the device:
      serial     one stream: H2D, compute, D2H, step after step;
      pipelined  three streams and two buffer sets: step i+1's H2D overlaps
                 step i's compute and step i-1's D2H (the streaming pattern a
                 user would write); a set is refilled only once the compute
                 that read it is done, and recomputed only once its result
                 has been copied out.
    d_sets: two lists [inputs..., output]; h_outs: two pinned host outputs.
    Returns (serial_s, pipelined_s)."""
    import torch

    cur = torch.cuda.current_stream(dev)
    s_in, s_c, s_out = (torch.cuda.Stream(dev) for _ in range(3))

    def serial(n):
        ins, out = d_sets[0][:-1], d_sets[0][-1]
        for _ in range(n):
            for d, h in zip(ins, h_in):
                d.copy_(h, non_blocking=True)
            compute(ins, out, cur)
            h_outs[0].copy_(out, non_blocking=True)

    def pipelined(n):
        for st in (s_in, s_c, s_out):
            st.wait_stream(cur)
        done_c, done_out = [None, None], [None, None]
        for i in range(n):
            k = i % 2
            ins, out = d_sets[k][:-1], d_sets[k][-1]
            with torch.cuda.stream(s_in):
                if done_c[k] is not None:
                    s_in.wait_event(done_c[k])
                for d, h in zip(ins, h_in):
                    d.copy_(h, non_blocking=True)
                e_in = torch.cuda.Event()
                e_in.record(s_in)
            with torch.cuda.stream(s_c):
                s_c.wait_event(e_in)
                if done_out[k] is not None:
                    s_c.wait_event(done_out[k])
                compute(ins, out, s_c)
                done_c[k] = torch.cuda.Event()
                done_c[k].record(s_c)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done_c[k])
                h_outs[k].copy_(out, non_blocking=True)
                done_out[k] = torch.cuda.Event()
                done_out[k].record(s_out)
        for st in (s_in, s_c, s_out):
            cur.wait_stream(st)

    result = []
    for fn in (serial, pipelined):
        fn(3)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        fn(steps)
        e1.record(cur)
        torch.cuda.synchronize(dev)
        result.append(e0.elapsed_time(e1) / 1e3)
    return result[0], result[1]


E2E_PIPELINE = "H2D, compute and D2H on three streams over two buffer sets; serial_value: one stream, in turn"


def run_e2e(args, w, dist, dev, stream, a_cpu, b_cpu, out_t, ws):
    """The same metric through the public API (tc.matmul) with host buffers:
    each step copies A and B in from pinned memory and C back out."""
    import torch

    import tensor_core_tiled_02_gb300 as tc

    h_in = [a_cpu.pin_memory(), b_cpu.pin_memory()]
    h_outs = [torch.empty((w.M, w.N), dtype=out_t).pin_memory() for _ in range(2)]
    d_sets = [[torch.empty_like(a_cpu, device=dev), torch.empty_like(b_cpu, device=dev),
               torch.empty((w.M, w.N), dtype=out_t, device=dev)] for _ in range(2)]

    def compute(ins, out, st):
        tc.matmul(ins[0], ins[1], out_dtype=out_t, out=out, workspace=ws, stream=st)

    dist.barrier()
    serial_s, pipe_s = time_e2e(dev, args.e2e_steps, h_in, d_sets, h_outs, compute)
    serial_s, pipe_s = dist.max(serial_s, device=dev), dist.max(pipe_s, device=dev)
    work = dist.world * float(w.flops) * args.e2e_steps
    return {"value": work / pipe_s / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in h_in),
            "d2h_bytes_per_step": h_outs[0].numel() * h_outs[0].element_size(), "steps": args.e2e_steps,
            "pipeline": E2E_PIPELINE, "serial_value": work / serial_s / 1e12}


ADD_METRIC = "blocked add GB/s (f32 Z = X + Y, each array moved once)"


def run_ours_add(args, w, dist: Dist):
    """The second workload: the pipelined blocked add, HBM-bound, in GB/s."""
    import torch

    import tensor_core_tiled_02_gb300 as tc
    from tensor_core_tiled_02_gb300.synthetic import add_inputs

    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    dist.init("nccl")
    x_cpu, y_cpu = add_inputs(w.M, w.N)
    n_copies = max(1, args.copies)
    Xs = [x_cpu.to(dev) for _ in range(n_copies)]
    Ys = [y_cpu.to(dev) for _ in range(n_copies)]
    Zs = [torch.empty_like(Xs[0]) for _ in range(n_copies)]
    stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream
    lib = tc.load_library()

    def step(i):
        j = i % n_copies
        rc = lib.add_matrices_f32(Xs[j].data_ptr(), Ys[j].data_ptr(), Zs[j].data_ptr(), w.M, w.N, handle)
        if rc != 0:
            raise tc.GemmError(rc, "add_matrices_f32")

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize(dev)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dist.local_rank, enabled=not args.no_clocks)
    clocks.start()
    dist.barrier()
    torch.cuda.synchronize(dev)
    start.record(stream)
    for i in range(args.steps):
        step(i)
    end.record(stream)
    torch.cuda.synchronize(dev)
    dist.barrier()
    clock_summary = clocks.stop()
    seconds = start.elapsed_time(end) / 1e3
    rc, site = tc.gemm_f16_device_status(reset=True)
    if rc != 0:
        raise RuntimeError(f"device wait gave up in the timed region (site {site})")
    t_max = dist.max(seconds, device=dev)
    nbytes = float(w.bytes_moved)
    value = dist.world * nbytes * args.steps / t_max / 1e9

    e2e = None
    if args.e2e_steps > 0:
        h_in = [x_cpu.pin_memory(), y_cpu.pin_memory()]
        h_outs = [torch.empty_like(x_cpu).pin_memory() for _ in range(2)]
        d_sets = [[torch.empty_like(x_cpu, device=dev) for _ in range(3)] for _ in range(2)]

        def compute(ins, out, st):
            tc.add_matrices(ins[0], ins[1], out=out, stream=st)

        dist.barrier()
        serial_s, pipe_s = time_e2e(dev, args.e2e_steps, h_in, d_sets, h_outs, compute)
        serial_s, pipe_s = dist.max(serial_s, device=dev), dist.max(pipe_s, device=dev)
        work = dist.world * nbytes * args.e2e_steps
        e2e = {"value": work / pipe_s / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": 2 * x_cpu.numel() * 4, "d2h_bytes_per_step": x_cpu.numel() * 4,
               "steps": args.e2e_steps, "pipeline": E2E_PIPELINE, "serial_value": work / serial_s / 1e9}

    if dist.rank == 0:
        peaks, peak_src = load_peaks()
        peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        achieved = nbytes / (seconds / args.steps) / 1e9
        cpu = None
        if not args.no_cpu_baseline and dist.world == 1:
            import oracle

            xn, yn = x_cpu.numpy(), y_cpu.numpy()
            oracle.add_f32(xn, yn)
            reps, t0 = 0, time.perf_counter()
            while time.perf_counter() - t0 < args.cpu_seconds:
                oracle.add_f32(xn, yn)
                reps += 1
            el = time.perf_counter() - t0
            cpu = {"value": nbytes * reps / el / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                   "sample": f"{reps} whole {w.M}x{w.N} additions in {el:.1f} s (one thread)"}
        line = {
            "metric": ADD_METRIC, "value": value, "unit": "GB/s", "n_gpus": dist.world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * t_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "M": w.M, "N": w.N, "inputs": "X, Y ~ U[0, 1) f32, seeds 0/1",
                       "l2": f"inputs rotated over {n_copies} copies of X, Y and Z, {3 * w.M * w.N * 4 / 1e6:.0f} MB each (> L2)",
                       "tile": "32 x 256, 3-slot ring"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": recorded_traffic(w.name, {"kind": "add"}),
                         "peak_source": f"hbm_gbs of {peak_src}", "kernel": "add_f32_kernel",
                         "avg_launch_ms": 1e3 * seconds / args.steps},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": args.steps, "clocks": clock_summary,
        }
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


def main(argv=None):
    args = parse_args(argv)
    from tensor_core_tiled_02_gb300.synthetic import WORKLOADS

    w = WORKLOADS[args.workload]
    dist = Dist()
    if args.impl == "reference":
        return run_reference(args, w, dist)
    if w.kind == "add":
        return run_ours_add(args, w, dist)
    return run_ours(args, w, dist)


if __name__ == "__main__":
    sys.exit(main())
