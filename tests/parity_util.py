"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same inputs, and compare with the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from exact_attention_57_gb300 import fa
from exact_attention_57_gb300.workloads import DTYPE_BF16, DTYPE_F16, DTYPE_F32, DTYPE_F32_SIMT

# Tolerances on |O_gpu - O_oracle| and |LSE_gpu - LSE_oracle| (the oracle
# reads the same bf16/fp32 input values the GPU reads).
TOL = {
    DTYPE_BF16: dict(max_o=2e-2, mean_o=2e-3, max_lse=1e-3),
    DTYPE_F32: dict(max_o=5e-3, mean_o=None, max_lse=1e-3),
    DTYPE_F32_SIMT: dict(max_o=1e-4, mean_o=None, max_lse=1e-3),
    # fp16 I/O (no stated figure): P and O are rounded to fp16 (relative error
    # <= 2^-11 each), so |dO| <= 2 * 2^-11 * max|v| ~ 5e-3 for N(0,1) values.
    DTYPE_F16: dict(max_o=5e-3, mean_o=5e-4, max_lse=1e-3),
}

IMPL = {DTYPE_BF16: "tc", DTYPE_F32: "tc", DTYPE_F32_SIMT: "simt", DTYPE_F16: "tc"}


def run_gpu(q, k, v, scale, causal, dtype, poison=True):
    """Inputs are CPU tensors in the I/O dtype; returns numpy float64 O, LSE."""
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty(q.shape[:3], device=dev, dtype=torch.float32)
    if poison:
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
    fa.attention(qd, kd, vd, scale=scale, causal=causal, impl=IMPL[dtype], out=o, lse=lse)
    st, word = fa.fa_fwd_status(torch.cuda.current_stream(dev).cuda_stream)
    assert st == fa.FA_OK, f"device status word {word}"
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def run_oracle(q, k, v, scale, causal):
    return oracle.attn_fwd(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                           scale, causal)


def compare(o, lse, ro, rl, dtype, tag="", tol=None):
    tol = dict(TOL[dtype], **(tol or {}))
    assert np.isfinite(o).all(), f"{tag}: non-finite O (unwritten rows?)"
    assert np.isfinite(lse).all(), f"{tag}: non-finite LSE (unwritten rows?)"
    eo = np.abs(o - ro)
    el = np.abs(lse - rl)
    stats = dict(max_o=float(eo.max()), mean_o=float(eo.mean()), max_lse=float(el.max()))
    assert stats["max_o"] <= tol["max_o"], f"{tag}: max|dO| {stats}"
    if tol["mean_o"] is not None:
        assert stats["mean_o"] <= tol["mean_o"], f"{tag}: mean|dO| {stats}"
    assert stats["max_lse"] <= tol["max_lse"], f"{tag}: max|dLSE| {stats}"
    return stats
