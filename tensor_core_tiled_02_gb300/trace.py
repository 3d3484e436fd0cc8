"""Timelines of the GEMM kernels from the trace build (libtcgemm_trace.so).

The trace build is the same library compiled with -DTCGEMM_TRACE: lane 0 of
each role of every CTA (0 producer, 1 MMA issuer, 2..5 epilogue warps) stamps
%globaltimer and the SM clock at fixed points of the pipeline (kernel entry,
set-up done, dependency wait, every K step's loads and landing, every unit's
last MMA, the epilogue's accumulator, split-K exchange, stores, exit) into a
buffer it is handed (include/gemm_f16_trace.h).  This module runs a workload
back to back through that library, reads the stamps and summarises them as
the time of each point after the end of the previous launch in the stream.

    python -m tensor_core_tiled_02_gb300.trace --workload skinny --launches 32 --graph
    python -m tensor_core_tiled_02_gb300.trace --shape 1024,8192,8192 --config cta_group=2,stream_k=2

builds the trace library if needed, runs the workload or shape (inputs
rotated past L2, as the bench does; a shape takes U[-1,1] operands and fp16
output unless a fourth field says 1, fp32) under the given tuning config and
prints the table.  Only the trace library is used
in this process: run it on its own, not inside a process that has loaded the
product library.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import sys
import warnings

import numpy as np

from . import build as tcbuild

ROLES = ["producer", "mma", "epilogue0", "epilogue1", "epilogue2", "epilogue3"]
EVENTS = {1: "entry", 2: "setup", 3: "dep_wait", 4: "load", 5: "full", 6: "tile_done", 7: "acc_ready",
          8: "pushed", 9: "partner", 10: "flags", 11: "stored", 12: "store_read", 13: "exit", 14: "parked"}
CODE = {v: k for k, v in EVENTS.items()}


def load_trace_library():
    """Load libtcgemm_trace.so as the binding's library (building it first if
    it is missing or older than its sources) and declare its trace entry
    point.  Must come before any other call into the binding."""
    import ctypes

    import tensor_core_tiled_02_gb300 as tc

    path = tcbuild.variant_lib("trace")
    if not os.path.exists(path) or os.path.getmtime(path) < newest_source():
        tcbuild.build(variant="trace")
    lib = tc.load_library(path)
    if not hasattr(lib, "gemm_f16_trace_buffer"):
        raise RuntimeError("the binding already holds the product library; run the trace in its own process")
    lib.gemm_f16_trace_buffer.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int]
    lib.gemm_f16_trace_buffer.restype = ctypes.c_int
    return lib


def newest_source() -> float:
    files = [os.path.join(tcbuild.CSRC, f) for f in os.listdir(tcbuild.CSRC)]
    files += [os.path.join(tcbuild.INCLUDE, f) for f in os.listdir(tcbuild.INCLUDE)]
    return max(os.path.getmtime(f) for f in files)


def events_for(plan: dict) -> int:
    """Records per role enough for every K step a CTA of this plan runs."""
    clusters = max(1, plan["grid"] // max(plan["cta_group"], plan["split"]))
    units = math.ceil(max(plan["dp_tiles"], 1) / clusters) + (2 if plan["sk_tiles"] else 0)
    return min(8192, units * plan["k_steps"] + 32)


def capture(M, N, K, out_dtype=0, launches=8, graph=False, copies=1, a_dist=("uniform", 1.0),
            b_dist=("uniform", 1.0), seed_a=0, seed_b=1, config=None):
    """Run `launches` GEMMs back to back through the trace library; return
    (records [launches, ctas, 6, events, 2] uint64, plan, A, B, C of the last
    launch on the host).  Inputs from the seeded generator, rotated over
    `copies` device copies; with `graph`, the launches are captured once in
    a CUDA graph and replayed."""
    import torch

    import tensor_core_tiled_02_gb300 as tc
    from tensor_core_tiled_02_gb300.synthetic import make_inputs

    lib = load_trace_library()
    tc.gemm_f16_set_config(**(config or {}))
    try:
        a, b = make_inputs(M, N, K, a_dist, b_dist, seed_a=seed_a, seed_b=seed_b)
        out_t = torch.float16 if out_dtype == 0 else torch.float32
        As = [a.cuda() for _ in range(copies)]
        Bs = [b.cuda() for _ in range(copies)]
        Cs = [torch.empty((M, N), dtype=out_t, device="cuda") for _ in range(copies)]
        ws = tc.workspace(M, N, K, out_dtype)
        plan = tc.gemm_f16_plan(M, N, K, out_dtype, with_workspace=ws is not None)
        ws_ptr, ws_bytes = (ws.data_ptr(), ws.numel()) if ws is not None else (0, 0)
        events = events_for(plan)
        ctas = plan["grid"]
        buf = torch.zeros(launches * ctas * len(ROLES) * events * 2, dtype=torch.int64, device="cuda")

        def launch(i, stream):
            j = i % copies
            rc = tc.gemm_f16_ws(As[j].data_ptr(), Bs[j].data_ptr(), Cs[j].data_ptr(), M, N, K, out_dtype, ws_ptr,
                                ws_bytes, stream)
            if rc != 0:
                raise tc.GemmError(rc)

        cur = torch.cuda.current_stream()
        launch(0, cur.cuda_stream)  # one-time set-up, untraced
        torch.cuda.synchronize()
        rc = lib.gemm_f16_trace_buffer(buf.data_ptr(), buf.numel() * 8, launches, ctas, events)
        if rc != 0:
            raise tc.GemmError(rc, "gemm_f16_trace_buffer")
        if graph:
            side = torch.cuda.Stream()
            side.wait_stream(cur)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for i in range(launches):
                    launch(i, side.cuda_stream)
            cur.wait_stream(side)
            g.replay()
        else:
            for i in range(launches):
                launch(i, cur.cuda_stream)
        torch.cuda.synchronize()
        lib.gemm_f16_trace_buffer(None, 0, 0, 0, 0)
        rc, site = tc.gemm_f16_device_status(reset=True)
        if rc != 0:
            raise RuntimeError(f"a device wait gave up (site {site})")
        rec = buf.cpu().numpy().view(np.uint64).reshape(launches, ctas, len(ROLES), events, 2)
        c_last = Cs[(launches - 1) % copies].cpu()
        return rec, plan, a, b, c_last
    finally:
        tc.gemm_f16_set_config()


def decode(rec: np.ndarray):
    """(t_ns float64, clk int64, code int64, arg int64) arrays of the records'
    shape without the last axis.  t_ns places every event in GPU time, in
    nanoseconds from the first entry stamp: its SM clock mapped linearly onto
    the global timer between its CTA's entry (earliest of its roles) and exit
    (latest); NaN where nothing was recorded."""
    clk = rec[..., 0].astype(np.int64)
    w1 = rec[..., 1]
    code = ((w1 >> np.uint64(56)) & np.uint64(0xFF)).astype(np.int64)
    arg = ((w1 >> np.uint64(32)) & np.uint64(0xFFFFFF)).astype(np.int64)
    gt32 = (w1 & np.uint64(0xFFFFFFFF)).astype(np.int64)
    empty = (rec[..., 0] == 0) & (w1 == 0)
    t = np.full(clk.shape, np.nan)
    is_entry, is_exit = code == CODE["entry"], code == CODE["exit"]
    if not is_entry.any():
        return t, clk, code, arg
    ref = gt32[is_entry].flat[0]
    gt = ((gt32 - ref + (1 << 31)) % (1 << 32)) - (1 << 31)  # signed ns from the reference, unwrapped
    L, C = clk.shape[:2]
    anchors = {}
    for i in range(L):
        for c in range(C):
            en, ex = is_entry[i, c], is_exit[i, c]
            if not en.any() or not ex.any():
                continue
            ce, cx = clk[i, c][en], clk[i, c][ex]
            je, jx = np.argmin(ce), np.argmax(cx)
            anchors[i, c] = (ce[je], gt[i, c][en][je], cx[jx], gt[i, c][ex][jx])
    rates = [(cx - ce) / (gx - ge) for ce, ge, cx, gx in anchors.values() if gx - ge >= 2000 and cx > ce]
    f_med = float(np.median(rates)) if rates else 1.9  # SM cycles per nanosecond
    for (i, c), (ce, ge, cx, gx) in anchors.items():
        f = (cx - ce) / (gx - ge) if gx - ge >= 2000 and cx > ce else f_med
        t[i, c] = ge + (clk[i, c] - ce) / f
    t[empty] = np.nan
    return t, clk, code, arg


def event_times(t, code, name, role=None, which="first"):
    """[launch, cta] time of the first (or last) event `name`, over the given
    roles (default: all); NaN where a CTA has none."""
    roles = range(t.shape[2]) if role is None else ([role] if isinstance(role, int) else role)
    sel = np.full(t.shape[:2], np.nan)
    for r in roles:
        tt = np.where(code[:, :, r, :] == CODE[name], t[:, :, r, :], np.nan)
        with warnings.catch_warnings():
            warnings.simplefilter("ignore", RuntimeWarning)  # CTAs without the event: NaN
            v = np.nanmin(tt, axis=-1) if which == "first" else np.nanmax(tt, axis=-1)
        sel = np.where(np.isnan(sel), v, np.fmin(sel, v) if which == "first" else np.fmax(sel, v))
    return sel


ROWS = [
    ("first CTA enters", "entry", None, "first", "min"),
    ("set-up done (barriers, TMEM, cluster)", "setup", 0, "first", "median"),
    ("dependency wait returns (producer)", "dep_wait", 0, "first", "median"),
    ("first step's loads issued", "load", 0, "first", "median"),
    ("first step's operands landed", "full", 1, "first", "median"),
    ("last step's loads issued", "load", 0, "last", "median"),
    ("last step's operands landed", "full", 1, "last", "median"),
    ("last unit's MMAs committed", "tile_done", 1, "last", "median"),
    ("accumulator ready in the epilogue", "acc_ready", [2, 3, 4, 5], "last", "median"),
    ("split-K partials sent", "pushed", [2, 3, 4, 5], "last", "median"),
    ("split-K partials received", "partner", [2, 3, 4, 5], "last", "median"),
    ("stream-K flags seen", "flags", [2, 3, 4, 5], "last", "median"),
    ("last chunk store issued", "stored", [2, 3, 4, 5], "last", "median"),
    ("stores have read the staging", "store_read", [2, 3, 4, 5], "last", "median"),
    ("CTA exits", "exit", None, "last", "median"),
    ("last CTA exits", "exit", None, "last", "max"),
]


def summarise(rec: np.ndarray, skip: int = 2) -> dict:
    """Medians over launches skip..end of each point's time after the end of
    the previous launch (the last exit of any of its CTAs), microseconds; per
    point the statistic over CTAs named in ROWS (median, min or max)."""
    t, _, code, _ = decode(rec)
    ends = event_times(t, code, "exit", None, "last")
    prev_end = np.nanmax(ends, axis=1)  # [launch]
    out = {}
    for label, name, role, which, stat in ROWS:
        v = event_times(t, code, name, role, which)  # [launch, cta]
        per_launch = []
        for i in range(max(skip, 1), t.shape[0]):
            row = v[i]
            row = row[~np.isnan(row)]
            if row.size == 0:
                continue
            s = {"median": np.median, "min": np.min, "max": np.max}[stat](row)
            per_launch.append((s - prev_end[i - 1]) / 1e3)
        if per_launch:
            out[label] = float(np.median(per_launch))
    periods = np.diff(prev_end)[max(skip, 1) - 1:] / 1e3
    out["launch period (end to end)"] = float(np.median(periods)) if periods.size else float("nan")
    return out


def check_records(rec: np.ndarray, plan: dict) -> list[str]:
    """Consistency of a trace: every role's stamps run forward in time, every
    traced CTA entered and left, and each producer issued one load event per
    K step it owns (at least one unit's worth).  Returns the problems found."""
    t, clk, code, _ = decode(rec)
    bad = []
    L, C, R, E = t.shape
    roles = min(R, max(1, plan.get("threads", 32 * R) // 32))  # the small kernel has four warps
    for i in range(L):
        for c in range(C):
            for r in range(roles):
                tt = t[i, c, r]
                tt = tt[~np.isnan(tt)]
                if tt.size and np.any(np.diff(tt) < 0):
                    bad.append(f"launch {i} cta {c} role {r}: timestamps go backwards")
                if not (code[i, c, r] == CODE["entry"]).any():
                    bad.append(f"launch {i} cta {c} role {r}: no entry")
                if not (code[i, c, r] == CODE["exit"]).any():
                    bad.append(f"launch {i} cta {c} role {r}: no exit")
            if plan["k_steps"] > 0:
                loads = int((code[i, c, 0] == CODE["load"]).sum())
                ks, split = plan["k_steps"], plan["split"]
                if split > 1:  # its rank's share of the one tile of its cluster
                    r = c % split
                    ok = loads == ks * (r + 1) // split - ks * r // split
                elif plan["sk_tiles"] == 0:  # whole tiles only
                    ok = loads > 0 and loads % ks == 0
                else:
                    ok = loads > 0
                if not ok:
                    bad.append(f"launch {i} cta {c}: {loads} load events")
    return bad


def format_table(summary: dict, title: str) -> str:
    lines = [f"| {title} | us after the previous launch ends |", "|---|---|"]
    for k, v in summary.items():
        lines.append(f"| {k} | {v:.2f} |")
    return "\n".join(lines)


def parse_shape(text: str):
    """'M,N,K' or 'M,N,K,out_dtype' -> (M, N, K, out_dtype)."""
    parts = [int(x) for x in text.split(",")]
    if len(parts) not in (3, 4) or min(parts[:3]) < 0 or (len(parts) == 4 and parts[3] not in (0, 1)):
        raise ValueError(f"shape must be M,N,K or M,N,K,out_dtype (0 fp16, 1 fp32), got {text!r}")
    return (*parts[:3], parts[3] if len(parts) == 4 else 0)


def parse_config(text: str) -> dict:
    """'key=value,...' (the fields of gemm_config) -> keyword arguments of
    gemm_f16_set_config."""
    cfg = {}
    for item in filter(None, text.split(",")):
        key, sep, value = item.partition("=")
        if not sep:
            raise ValueError(f"config items are key=value, got {item!r}")
        cfg[key.strip()] = int(value)
    return cfg


def main(argv=None):
    from tensor_core_tiled_02_gb300.synthetic import WORKLOADS, Workload

    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workload", default="skinny", choices=[n for n, w in WORKLOADS.items() if w.kind == "gemm"])
    ap.add_argument("--shape", default="", help="M,N,K[,out_dtype] instead of a workload")
    ap.add_argument("--config", default="", help="tuning config, e.g. cta_group=2,stream_k=2")
    ap.add_argument("--launches", type=int, default=32)
    ap.add_argument("--graph", action="store_true", help="capture the launches in a CUDA graph and replay it")
    ap.add_argument("--copies", type=int, default=0, help="input copies to rotate over (0: past L2, as the bench)")
    ap.add_argument("--json", default="", help="also write the summary here")
    ap.add_argument("--npz", default="", help="also write the raw records and the plan here")
    args = ap.parse_args(argv)
    if args.shape:
        M, N, K, dt = parse_shape(args.shape)
        w = Workload(f"{M}x{N}x{K}", M, N, K, ("uniform", 1.0), ("uniform", 1.0), dt)
    else:
        w = WORKLOADS[args.workload]
    cfg = parse_config(args.config)
    copies = args.copies or max(3, math.ceil(2 * 129 * 2 ** 20 / w.bytes_moved))
    copies = min(copies, args.launches)
    rec, plan, _, _, _ = capture(w.M, w.N, w.K, w.out_dtype, args.launches, args.graph, copies, w.a_dist, w.b_dist,
                                 config=cfg)
    problems = check_records(rec, plan)
    s = summarise(rec)
    title = (w.name if args.shape else f"{w.name} {w.M}x{w.N}x{w.K}") + (f" ({args.config})" if cfg else "") + \
        f", {'graph' if args.graph else 'eager'}, {args.launches} launches"
    print(format_table(s, title))
    print(f"plan: cta_group {plan['cta_group']}, tile {plan['tile_m']}x{plan['tile_n']}x{plan['tile_k']}, "
          f"split {plan['split']}, grid {plan['grid']}, stream-K tiles {plan['sk_tiles']}")
    if problems:
        print(f"{len(problems)} trace problems, first: {problems[0]}")
    if args.npz:
        np.savez_compressed(args.npz, records=rec, plan=json.dumps(plan))
    if args.json:
        with open(args.json, "w") as f:
            json.dump({"workload": w.name, "graph": args.graph, "launches": args.launches, "summary": s,
                       "plan": plan, "problems": problems[:20]}, f, indent=1)
    return 1 if problems else 0


if __name__ == "__main__":
    sys.exit(main())
