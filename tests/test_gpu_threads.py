"""Several host threads making their first calls into the library at once.

The per-device facts the library caches (SM count, cluster capacity, each
kernel's raised shared-memory limit) are filled on first use.  A fresh
process starts six threads that wait on one barrier and then call, each on
its own CUDA stream, a different kernel: CTA-pair GEMMs of both tile sizes, a
split-K GEMM, a one-CTA GEMM, the small kernel and the blocked add.  Every result is checked against the
oracle (the add bit for bit).
"""
import os
import subprocess
import sys
import textwrap

import pytest

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent("""
    import sys, threading
    import numpy as np
    import torch
    sys.path[:0] = [{root!r}, {tests!r}]
    import oracle, parity
    import tensor_core_tiled_02_gb300 as tc
    from tensor_core_tiled_02_gb300.synthetic import make_inputs, add_inputs

    jobs = [("pair", 2048, 2048, 512, 0), ("split", 128, 1024, 4096, 1), ("one", 1280, 1024, 256, 0),
            ("pair128", 384, 640, 768, 0), ("small", 256, 256, 256, 1)]
    inputs = {{name: make_inputs(M, N, K, ("uniform", 1.0), ("uniform", 1.0), seed_a=i, seed_b=i + 10)
              for i, (name, M, N, K, _) in enumerate(jobs)}}
    x_cpu, y_cpu = add_inputs(256, 512)
    gate = threading.Barrier(len(jobs) + 1)
    results, errors = {{}}, []

    def gemm(name, M, N, K, dt):
        try:
            a, b = inputs[name]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                a_d, b_d = a.cuda(), b.cuda()
                gate.wait()
                c = tc.matmul(a_d, b_d, out_dtype=torch.float16 if dt == 0 else torch.float32, stream=s)
                s.synchronize()
            results[name] = (c.cpu(), a, b, K, dt)
        except Exception as e:
            errors.append(repr(e))

    def add():
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                x, y = x_cpu.cuda(), y_cpu.cuda()
                gate.wait()
                z = tc.add_matrices(x, y, stream=s)
                s.synchronize()
            results["add"] = z.cpu()
        except Exception as e:
            errors.append(repr(e))

    threads = [threading.Thread(target=gemm, args=j) for j in jobs] + [threading.Thread(target=add)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for name, (c, a, b, K, dt) in ((k, v) for k, v in results.items() if k != "add"):
        ref = oracle.as_values(oracle.gemm(a.numpy(), b.numpy(), dt), dt)
        parity.check(c.double().numpy(), ref, K, dt, name)
    want = oracle.add_f32(x_cpu.numpy(), y_cpu.numpy())
    assert np.array_equal(results["add"].numpy().view(np.uint32), want.view(np.uint32))
    rc, site = tc.gemm_f16_device_status(reset=True)
    assert rc == 0, site
    print("ok", sorted(results))
""")


def test_first_calls_from_several_threads():
    plan_names = {"pair": (2048, 2048, 512, 0), "split": (128, 1024, 4096, 1), "one": (1280, 1024, 256, 0),
                  "pair128": (384, 640, 768, 0), "small": (256, 256, 256, 1)}
    import tensor_core_tiled_02_gb300 as tc
    plans = {k: tc.gemm_f16_plan(*v) for k, v in plan_names.items()}
    # the five GEMMs really take five different paths
    assert plans["pair"]["cta_group"] == 2 and plans["pair"]["tile_m"] == 256
    assert plans["split"]["cta_group"] == 1 and plans["split"]["split"] > 1
    assert plans["one"]["cta_group"] == 1 and plans["one"]["split"] == 1
    assert plans["pair128"]["cta_group"] == 2 and plans["pair128"]["tile_m"] == 128
    assert plans["small"]["cta_group"] == 1 and plans["small"]["tile_m"] == 8
    code = SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stdout[-2000:] + out.stderr[-4000:]
    assert "ok" in out.stdout
