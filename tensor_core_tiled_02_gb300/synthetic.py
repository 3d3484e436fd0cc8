"""Seeded synthetic inputs for the fp16 GEMM workloads.

This module only draws random numbers; it holds none of the GEMM's
arithmetic.  Both the CUDA path and the CPU oracle take their inputs from it,
and it imports neither.

The workloads are those of the matmul(a, b, out_dtype) statement of the
"Quickstart: GPU" page ("Pipelining: a matmul kernel":
fp16 operands, fp32 accumulator, fp16 or fp32 output), at five shapes:

  gemm_256     M=N=K=256,   A, B ~ U[-1, 1],            fp16 out
  gemm_4096    M=N=K=4096,  A, B ~ N(0, 1) / sqrt(K),   fp16 out
  gemm_8192    M=N=K=8192,  A, B ~ U[-1, 1],            fp16 out
  skinny       M=128, N=K=8192, A ~ N(0, 1), B ~ N(0, 0.02^2), fp16 out
  long_k       M=N=2048, K=32768, A, B ~ U[-1, 1],      fp32 out

and the second workload on the same pipeline machinery, the blocked add of
the "JAX Pallas 软件流水线 Software Pipelining 完全指南", section 6:

  add_4096     X, Y f32 [4096, 4096] ~ U[0, 1) (seeds 0, 1), Z = X + Y

Recipe: a CPU ``torch.Generator`` seeded with ``seed_a`` (A) or ``seed_b``
(B); U[-1, 1] is ``2 * rand - 1`` and N(0, s^2) is ``s * randn``, both drawn in
fp32, then rounded to fp16 with round-to-nearest-even (``.half()``).
"""
from __future__ import annotations

import dataclasses
import math

import torch

F16 = 0
F32 = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    a_dist: tuple  # ("uniform", half_width) or ("normal", sigma)
    b_dist: tuple
    out_dtype: int
    kind: str = "gemm"  # "gemm" or "add"

    @property
    def flops(self) -> int:
        if self.kind == "add":
            return self.M * self.N
        return 2 * self.M * self.N * self.K

    @property
    def bytes_moved(self) -> int:
        """Each matrix moved once: A and B (X and Y) read, C (Z) written."""
        if self.kind == "add":
            return 3 * 4 * self.M * self.N
        out_bytes = 2 if self.out_dtype == F16 else 4
        return 2 * self.M * self.K + 2 * self.K * self.N + out_bytes * self.M * self.N


WORKLOADS = {
    w.name: w
    for w in [
        Workload("gemm_256", 256, 256, 256, ("uniform", 1.0), ("uniform", 1.0), F16),
        Workload("gemm_4096", 4096, 4096, 4096, ("normal", 1.0 / math.sqrt(4096)),
                 ("normal", 1.0 / math.sqrt(4096)), F16),
        Workload("gemm_8192", 8192, 8192, 8192, ("uniform", 1.0), ("uniform", 1.0), F16),
        Workload("skinny", 128, 8192, 8192, ("normal", 1.0), ("normal", 0.02), F16),
        Workload("long_k", 2048, 2048, 32768, ("uniform", 1.0), ("uniform", 1.0), F32),
        Workload("add_4096", 4096, 4096, 0, ("unit", 1.0), ("unit", 1.0), F32, kind="add"),
    ]
}


def add_inputs(M: int, N: int, seed_x: int = 0, seed_y: int = 1):
    """(X, Y) f32 [M, N] CPU tensors ~ U[0, 1), as the blocked-add example draws them."""
    out = []
    for seed in (seed_x, seed_y):
        g = torch.Generator(device="cpu")
        g.manual_seed(int(seed))
        out.append(torch.rand((M, N), generator=g, dtype=torch.float32))
    return tuple(out)


def draw(shape, dist, seed: int) -> torch.Tensor:
    """fp16 CPU tensor of ``shape`` drawn from ``dist`` with ``seed``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    kind, scale = dist
    if kind == "uniform":
        x = torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
        x = x * float(scale)
    elif kind == "normal":
        x = torch.randn(shape, generator=g, dtype=torch.float32) * float(scale)
    elif kind == "ones":
        x = torch.ones(shape, dtype=torch.float32) * float(scale)
    elif kind == "int":
        # small integers in [-scale, scale]: exact in fp16, exact products
        x = torch.randint(-int(scale), int(scale) + 1, shape, generator=g).to(torch.float32)
    else:
        raise ValueError(f"unknown distribution {kind!r}")
    return x.half().contiguous()


def make_inputs(M: int, N: int, K: int, a_dist=("uniform", 1.0), b_dist=("uniform", 1.0),
                seed_a: int = 0, seed_b: int = 1):
    """(A [M, K], B [K, N]) as fp16 CPU tensors."""
    return draw((M, K), a_dist, seed_a), draw((K, N), b_dist, seed_b)


def workload_inputs(w: Workload, seed_a: int = 0, seed_b: int = 1):
    return make_inputs(w.M, w.N, w.K, w.a_dist, w.b_dist, seed_a, seed_b)
