"""bench.py's host-side logic on the CPU: the max-over-ranks timing of the
replicas path under torch.distributed (gloo, world size 2), the whole-job
throughput, the clock-log summary, the recorded-traffic lookup and the
reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    d = bench.Dist()
    d.init("gloo")
    seconds = 1.0 + rank  # rank 1 is the slow one
    t = d.max(seconds)
    agg = bench.aggregate([t] * d.world, flops_per_step=1e12, steps=10)
    d.barrier()
    with open(os.path.join(outdir, f"r{rank}.json"), "w") as f:
        json.dump({"t": t, "agg": agg, "world": d.world}, f)
    d.close()


def test_replicas_take_the_max_over_ranks(tmp_path):
    import torch.multiprocessing as mp

    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    for r in range(2):
        d = json.load(open(tmp_path / f"r{r}.json"))
        assert d["world"] == 2
        assert d["t"] == 2.0                       # the slowest rank's time on every rank
        # 2 ranks x 10 steps x 1 TFLOP over 2 s
        assert d["agg"]["tflops"] == pytest.approx(10.0)
        assert d["agg"]["ms_per_step"] == pytest.approx(200.0)


def test_single_process_dist_is_a_noop():
    d = bench.Dist()
    assert d.world == int(os.environ.get("WORLD_SIZE", "1"))
    assert d.max(3.5) == 3.5
    assert bench.aggregate([2.0], 1e12, 4)["tflops"] == pytest.approx(2.0)


def test_clock_summary():
    rows = [
        ["0", "1500", "2070", "1350.1", "0x4", "Not Active", "Not Active", "Not Active", "Active"],
        ["0", "1600", "2070", "1390.0", "0x4", "Not Active", "Not Active", "Not Active", "Active"],
        ["0", "2070", "2070", "150.0", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"],
    ]
    s = bench.summarize_clocks(rows)
    assert s["sm_mhz"] == 1550.0          # idle sample (low power) left out
    assert s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert bench.summarize_clocks([]) is None


def test_recorded_traffic_follows_the_kernel_hash(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    src = tmp_path / "tensor_core_tiled_02_gb300" / "csrc"
    src.mkdir(parents=True)
    for rel in bench.KERNEL_SOURCES:
        (tmp_path / rel).write_text("int x; // comment\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash()
    (prof / "gemm_f16_kernel_w.md").write_text(f"kernel_source_sha256: {h}\ntraffic_bytes_per_launch: 1234\n")
    assert bench.recorded_traffic("w", {}) == 1234
    # a comment edit keeps it; a code edit makes it stale
    (tmp_path / bench.KERNEL_SOURCES[0]).write_text("int x;   /* other words */\n")
    assert bench.recorded_traffic("w", {}) == 1234
    (tmp_path / bench.KERNEL_SOURCES[0]).write_text("int y;\n")
    assert bench.recorded_traffic("w", {}) is None


@pytest.mark.slow
def test_reference_arm_prints_the_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "gemm_256", "--steps", "3", "--warmup", "1"],
                         capture_output=True, text=True, check=True, cwd=ROOT, timeout=600)
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["steps"] == 3 and d["warmup"] == 1 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "gemm_256"


def test_gemm_roofline_picks_the_binding_peak(monkeypatch):
    import bench
    from tensor_core_tiled_02_gb300.synthetic import WORKLOADS

    monkeypatch.setattr(bench, "load_peaks", lambda: ({"hbm_gbs": 6700.0, "bf16_tflops": 1900.0,
                                                       "bf16_tflops_sustained": 1700.0}, "measured"))
    by = WORKLOADS
    big = bench.gemm_roofline(by["gemm_8192"], 1e-3)
    assert big["bound"] == "tensor" and big["unit"] == "TFLOP/s"
    assert abs(big["achieved"] - 2 * 8192 ** 3 / 1e-3 / 1e12) < 1e-6
    # M = 128: 17 GFLOP but 138 MB, about 9 us of tensor time against 21 us of HBM time
    sk = bench.gemm_roofline(by["skinny"], 30e-6)
    assert sk["bound"] == "hbm" and sk["unit"] == "GB/s"
    nbytes = 2 * 128 * 8192 + 2 * 8192 * 8192 + 2 * 128 * 8192
    assert abs(sk["achieved"] - nbytes / 30e-6 / 1e9) < 1e-6
    assert abs(sk["frac"] - sk["achieved"] / 6700.0) < 1e-12 and 0 < sk["tensor_frac"] < sk["frac"]


def test_config_leg_covers_the_five_workloads_past_l2():
    from tensor_core_tiled_02_gb300.synthetic import WORKLOADS

    assert bench.parse_args([]).configs == "all"
    assert sorted(bench.CONFIG_WORKLOADS) == sorted(n for n, w in WORKLOADS.items() if w.kind == "gemm")
    l2 = 129 * 2 ** 20
    for name in bench.CONFIG_WORKLOADS:
        w = WORKLOADS[name]
        n = bench.rotation_copies(w.bytes_moved, l2)
        # each launch's operands were last touched at least two L2s of other data ago
        assert n >= 3 and (n - 1) * w.bytes_moved >= 2 * l2 - w.bytes_moved
    assert bench.rotation_copies(393216, l2) == 688  # 256^3: 0.39 MB a set
