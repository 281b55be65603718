"""Named synthetic workloads and their seeded input generator.

This module holds no attention arithmetic: it only draws the inputs, so both
the CUDA library's callers and the CPU oracle's callers can use it.

Recipe (the pages name no dataset; the cuTile FMHA example of "Add Fused
Multi-Head Attention example" draws q, k, v with ``randn``):
    g = torch.Generator('cpu').manual_seed(seed)
    q = randn(B, H, Nq, d); k = randn(B, H, Nk, d); v = randn(B, H, Nk, d)
drawn in that order, float32, iid N(0, 1).  A workload with ``k_mult`` scales
k by that factor in float32 before any cast.  bf16 workloads then round each
tensor to bf16 (round-to-nearest-even); the oracle reads those rounded values.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

DTYPE_BF16 = 0      # bf16 in/out, tcgen05 kind::f16
DTYPE_F32 = 1       # fp32 in/out, tcgen05 kind::tf32
DTYPE_F32_SIMT = 2  # fp32 in/out, plain fp32 FMA kernel (no tensor cores)
DTYPE_F16 = 3       # fp16 in/out, tcgen05 kind::f16

DTYPE_NAMES = {DTYPE_BF16: "bf16", DTYPE_F32: "f32", DTYPE_F32_SIMT: "f32_simt",
               DTYPE_F16: "f16"}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    dtype: int
    causal: tuple = (True,)
    k_mult: float = 1.0
    seed: int = 0
    note: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        return {DTYPE_BF16: torch.bfloat16, DTYPE_F16: torch.float16}.get(self.dtype,
                                                                         torch.float32)

    def flops(self, causal: bool) -> float:
        """Metric FLOPs: 4*B*H*Nq*Nk*d, halved for causal."""
        f = 4.0 * self.B * self.H * self.Nq * self.Nk * self.d
        return f / 2 if causal else f


WORKLOADS = {
    "b1h1n256d64-f32-simt": Workload(
        "b1h1n256d64-f32-simt", 1, 1, 256, 256, 64, DTYPE_F32_SIMT,
        causal=(False, True), seed=57000,
        note="tiny fp32 case, plain fp32 kernel, non-causal and causal"),
    "b2h4n1024d64-bf16-causal": Workload(
        "b2h4n1024d64-bf16-causal", 2, 4, 1024, 1024, 64, DTYPE_BF16,
        causal=(True,), seed=57001),
    "b4h4n4096d64-f32-tf32": Workload(
        "b4h4n4096d64-f32-tf32", 4, 4, 4096, 4096, 64, DTYPE_F32,
        causal=(False,), seed=57002,
        note="fp32 in/out, TF32 tensor-core compute, non-causal"),
    "b2h8n3001d128-bf16-causal-k3": Workload(
        "b2h8n3001d128-bf16-causal-k3", 2, 8, 3001, 3001, 128, DTYPE_BF16,
        causal=(True,), k_mult=3.0, seed=57003,
        note="ragged length, K scaled by 3"),
    "b8h32n8192d128-bf16-causal": Workload(
        "b8h32n8192d128-bf16-causal", 8, 32, 8192, 8192, 128, DTYPE_BF16,
        causal=(True,), seed=57004,
        note="large causal case, 256 heads"),
}

# The workload the benchmark times at one GPU.
BENCH_WORKLOAD = "b8h32n8192d128-bf16-causal"

# Same shape per head as the benchmark with 1/8 of the heads (inputs still
# larger than L2): the case the detailed profiler captures are taken on.
PROFILE_WORKLOADS = {
    "b2h16n8192d128-bf16-causal": Workload(
        "b2h16n8192d128-bf16-causal", 2, 16, 8192, 8192, 128, DTYPE_BF16,
        causal=(True,), seed=57005, note="profiling case, 1/8 of the benchmark's heads"),
    # Short queries against long keys: 8 query tiles in all, far fewer CTAs
    # than SMs unless the key range is split.
    "b1h8nq128nk65536d128-bf16": Workload(
        "b1h8nq128nk65536d128-bf16", 1, 8, 128, 65536, 128, DTYPE_BF16,
        causal=(False,), seed=57006, note="decode-like: one query tile per head"),
    # Head dim 256 at the benchmark's per-head FLOPs (half the heads).
    "b4h16n8192d256-bf16-causal": Workload(
        "b4h16n8192d256-bf16-causal", 4, 16, 8192, 8192, 256, DTYPE_BF16,
        causal=(True,), seed=57007, note="head dim 256"),
    "b4h4n4096d128-f32-tf32": Workload(
        "b4h4n4096d128-f32-tf32", 4, 4, 4096, 4096, 128, DTYPE_F32,
        causal=(False,), seed=57009, note="fp32 at head dim 128 (TF32 tensor cores)"),
    "b4h16n8192d32-bf16-causal": Workload(
        "b4h16n8192d32-bf16-causal", 4, 16, 8192, 8192, 32, DTYPE_BF16,
        causal=(True,), seed=57010, note="head dim 32 (runs zero-padded on the d = 64 kernel)"),
    "b4h16n8192d64-bf16-causal": Workload(
        "b4h16n8192d64-bf16-causal", 4, 16, 8192, 8192, 64, DTYPE_BF16,
        causal=(True,), seed=57008, note="head dim 64"),
    "b4h16n8192d128-bf16": Workload(
        "b4h16n8192d128-bf16", 4, 16, 8192, 8192, 128, DTYPE_BF16,
        causal=(False,), seed=57011, note="no mask"),
    "b4h16n8192d128-f16-causal": Workload(
        "b4h16n8192d128-f16-causal", 4, 16, 8192, 8192, 128, DTYPE_F16,
        causal=(True,), seed=57012, note="fp16 inputs"),
}


def make_inputs(B: int, H: int, Nq: int, Nk: int, d: int, dtype: int,
                seed: int, k_mult: float = 1.0):
    """Seeded q, k, v on the CPU, in the I/O dtype of ``dtype``."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    q = torch.randn(B, H, Nq, d, generator=g, dtype=torch.float32)
    k = torch.randn(B, H, Nk, d, generator=g, dtype=torch.float32)
    v = torch.randn(B, H, Nk, d, generator=g, dtype=torch.float32)
    if k_mult != 1.0:
        k.mul_(float(k_mult))
    if dtype == DTYPE_BF16:
        q, k, v = q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)
    elif dtype == DTYPE_F16:
        q, k, v = q.to(torch.float16), k.to(torch.float16), v.to(torch.float16)
    return q, k, v


def make_dout(B: int, H: int, Nq: int, d: int, dtype: int, seed: int):
    """Seeded upstream gradient dO [B, H, Nq, d] on the CPU, N(0, 1) values in
    the I/O dtype of ``dtype`` (the gradient of sum(O * dO))."""
    g = torch.Generator("cpu").manual_seed(int(seed) + 7919)
    do = torch.randn(B, H, Nq, d, generator=g, dtype=torch.float32)
    if dtype == DTYPE_BF16:
        do = do.to(torch.bfloat16)
    elif dtype == DTYPE_F16:
        do = do.to(torch.float16)
    return do


def workload_inputs(w: Workload):
    return make_inputs(w.B, w.H, w.Nq, w.Nk, w.d, w.dtype, w.seed, w.k_mult)
