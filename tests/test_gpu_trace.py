"""The trace build (libtcgemm_trace.so, -DTCGEMM_TRACE) on the GPU: its
kernels still compute the product (checked against the oracle), every role's
stamps run forward in time, every CTA enters and leaves, each producer
stamps one load per K step it owns, and the timeline summary is finite.

The trace library runs in a child process: this process holds the product
library, and the binding keeps one library per process."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
import parity

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys
import numpy as np
sys.path.insert(0, {root!r})
from tensor_core_tiled_02_gb300 import trace
rec, plan, a, b, c = trace.capture({M}, {N}, {K}, {dt}, launches=4, graph={graph}, copies=2,
                                   a_dist=("normal", 1.0), b_dist=("normal", 1.0), seed_a=5, seed_b=6,
                                   config={cfg!r})
np.save({out!r} + "/a.npy", a.numpy().view(np.uint16))
np.save({out!r} + "/b.npy", b.numpy().view(np.uint16))
np.save({out!r} + "/c.npy", c.double().numpy())
json.dump({{"plan": plan, "problems": trace.check_records(rec, plan), "summary": trace.summarise(rec, skip=1)}},
          open({out!r} + "/r.json", "w"))
"""

CASES = [((700, 1096, 1000, 0), {}, False),                       # CTA pairs, ragged
         ((128, 2048, 4096, 0), {}, True),                        # split-K clusters of two, in a CUDA graph
         ((300, 1000, 3000, 1), dict(cta_group=1, stream_k=2), False),  # one-CTA stream-K, fp32 out
         ((1100, 1280, 2056, 0), dict(cta_group=2, stream_k=2), False)]  # pairs, every tile shared


@pytest.mark.parametrize("shape,cfg,graph", CASES, ids=["pairs", "split_k_graph", "stream_k_one_cta",
                                                        "stream_k_pairs"])
def test_trace_build_stamps_and_computes(shape, cfg, graph, tmp_path):
    M, N, K, dt = shape
    code = CHILD.format(root=ROOT, M=M, N=N, K=K, dt=dt, graph=graph, cfg=cfg, out=str(tmp_path))
    env = dict(os.environ)
    env.pop("TCGEMM_VARIANT", None)
    subprocess.run([sys.executable, "-c", code], check=True, cwd=ROOT, env=env, timeout=600)
    r = json.load(open(tmp_path / "r.json"))
    assert r["problems"] == [], r["problems"][:5]
    s = r["summary"]
    for key in ("first step's operands landed", "last unit's MMAs committed", "CTA exits"):
        assert np.isfinite(s[key]), (key, s)
    assert s["first step's operands landed"] <= s["last step's operands landed"]
    a = np.load(tmp_path / "a.npy").view(np.float16)
    b = np.load(tmp_path / "b.npy").view(np.float16)
    c = np.load(tmp_path / "c.npy")
    ref = oracle.as_values(oracle.gemm(a, b, dt), dt)
    parity.check(c, ref, K, dt, f"trace build {shape} {cfg}")
