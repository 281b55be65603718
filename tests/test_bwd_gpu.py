"""fa_bwd (tensor-core backward) against the float64 oracle gradients on the
same inputs: the forward's o and lse come from fa_fwd, the expected dq, dk,
dv from oracle.attn_bwd (needs a GB300)."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_57_gb300 import fa
from exact_attention_57_gb300.workloads import (DTYPE_BF16, DTYPE_F16, DTYPE_F32, make_dout,
                                                make_inputs)

pytestmark = pytest.mark.gpu

# Normwise tolerances on each gradient X: max|dX| <= max_rel * max|X| and
# mean|dX| <= mean_rel * mean|X|.  The products accumulate in fp32; what moves
# the result is the rounding to the 16-bit input type (unit roundoff u = 2^-9
# for bf16, 2^-12 for fp16) of P (the A operand of dV), of dS (the A operand
# of dQ and dK), of the forward's O (through D), and of the outputs.  Each
# term of every sum carries a relative error of about u, so the typical
# error is about u of the typical gradient: mean_rel = 2.5u, max_rel = 8u.
U = {DTYPE_BF16: 2.0 ** -9, DTYPE_F16: 2.0 ** -12}
TOL = {dt: dict(max_rel=8 * u, mean_rel=2.5 * u) for dt, u in U.items()}
# fp32 (CUDA-core backward after the plain fp32 forward): every step is fp32
# arithmetic, so each gradient is a sum of N products each within a few units
# of u = 2^-24 (expf within 2 ulp, P from the forward's fp32 LSE); sums of N
# such terms drift by about sqrt(N) u in the mean and N u at worst.  Bound
# with N = 1024 (the longest key range tested): mean 32u, max 1024u of the
# gradient's size.
TOL[DTYPE_F32] = dict(max_rel=1024 * 2.0 ** -24, mean_rel=32 * 2.0 ** -24)

CASES = [
    # B, H, Nq, Nk, d, causal, dtype, scale (None = 1/sqrt(d))
    (1, 2, 128, 128, 64, False, DTYPE_BF16, None),
    (1, 2, 128, 128, 128, True, DTYPE_BF16, None),
    (2, 2, 300, 300, 128, True, DTYPE_BF16, None),
    (1, 2, 200, 457, 64, False, DTYPE_BF16, None),
    (1, 2, 457, 200, 128, True, DTYPE_BF16, None),
    (1, 2, 100, 400, 128, True, DTYPE_BF16, None),   # keys past the last query
    (1, 3, 1, 1, 64, False, DTYPE_BF16, None),
    (1, 2, 384, 256, 64, True, DTYPE_F16, None),
    (2, 1, 333, 517, 128, False, DTYPE_F16, None),
    (1, 2, 256, 256, 128, True, DTYPE_BF16, -0.2),
    (1, 2, 256, 300, 64, False, DTYPE_BF16, 0.0),
    (1, 4, 1024, 1024, 128, True, DTYPE_BF16, None),
    (1, 4, 1024, 1024, 64, False, DTYPE_BF16, None),
    (2, 2, 300, 300, 32, True, DTYPE_BF16, None),     # runs zero-padded on the d = 64 kernel
    (1, 3, 200, 457, 32, False, DTYPE_F16, None),
    # fp32: the CUDA-core backward (any head dim up to 128)
    (1, 2, 128, 128, 64, False, DTYPE_F32, None),
    (2, 2, 300, 300, 128, True, DTYPE_F32, None),
    (1, 2, 200, 457, 64, False, DTYPE_F32, None),
    (1, 2, 457, 200, 128, True, DTYPE_F32, None),
    (1, 2, 100, 400, 128, True, DTYPE_F32, None),    # keys past the last query
    (1, 3, 1, 1, 64, False, DTYPE_F32, None),
    (2, 2, 150, 150, 33, True, DTYPE_F32, None),
    (1, 2, 256, 256, 128, True, DTYPE_F32, -0.2),
    (1, 2, 256, 300, 96, False, DTYPE_F32, 0.0),
    (1, 2, 1024, 1024, 128, True, DTYPE_F32, None),
]


def run_bwd(q, k, v, do, scale, causal):
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    # fp32: the forward's o and lse from the plain fp32 kernel, so that the
    # gradients are fp32 arithmetic throughout
    impl = "simt" if q.dtype == torch.float32 else "tc"
    o, lse = fa.attention(qd, kd, vd, scale=scale, causal=causal, impl=impl)
    grads = [torch.full_like(t, float("nan")) for t in (qd, kd, vd)]
    fa.attention_backward(qd, kd, vd, o, lse, dod, scale=scale, causal=causal,
                          dq=grads[0], dk=grads[1], dv=grads[2])
    st, word = fa.fa_fwd_status(torch.cuda.current_stream(dev).cuda_stream)
    assert st == fa.FA_OK, f"device status word {word}"
    return [g.double().cpu().numpy() for g in grads]


def fp32_floor(q, k, v, do, scale):
    """Absolute error floors of (dq, dk, dv) from fp32 arithmetic alone, for
    gradients that cancel to (near) zero, e.g. a row with one key (P = 1, so
    dS = dP - D = 0 exactly).  dP = dO.v and D = dO.O are fp32 dot products of
    length d, each within gamma_d * sum|dO||v| of exact (gamma_d =
    d 2^-24 / (1 - d 2^-24), the standard bound), so |dS| <= 2 gamma_d
    max sum|dO||v| and |dQ| <= |scale| |dS| max|k| (|dK| the same with q)."""
    q, k, v, do = (np.abs(np.asarray(t, dtype=np.float64)) for t in (q, k, v, do))
    d = q.shape[-1]
    g = d * 2.0 ** -24 / (1 - d * 2.0 ** -24)
    dov = float(np.max(do @ np.swapaxes(v, -1, -2)))  # max_ij sum_x |dO_ix| |v_jx|
    ds = 2 * g * dov
    return abs(scale) * ds * float(k.max()), abs(scale) * ds * float(q.max()), 0.0


def check(got, ref, dtype, what, floors=(0.0, 0.0, 0.0), d=128):
    """Normwise bounds per gradient; floors (fp32_floor) are added to the max
    bound as they stand and to the mean bound divided by sqrt(d) (the size of
    a sum of d random-sign rounding errors)."""
    tol = TOL[dtype]
    for name, a, b, fl in zip(("dq", "dk", "dv"), got, ref, floors):
        assert np.all(np.isfinite(a)), f"{what} {name}: non-finite values"
        err = np.abs(a - b)
        mx, mn = float(err.max()), float(err.mean())
        ref_max, ref_mean = float(np.abs(b).max()), float(np.abs(b).mean())
        print(f"{what} {name}: max {mx:.3e} ({mx / max(ref_max, 1e-30):.2e} of max) "
              f"mean {mn:.3e} ({mn / max(ref_mean, 1e-30):.2e} of mean)")
        assert mx <= tol["max_rel"] * ref_max + fl + 1e-6, f"{what} {name}: max |err| {mx:.3e}"
        assert mn <= tol["mean_rel"] * ref_mean + fl / math.sqrt(d) + 1e-7, \
            f"{what} {name}: mean |err| {mn:.3e}"


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,dtype,scale", CASES)
def test_bwd_matches_oracle(B, H, Nq, Nk, d, causal, dtype, scale):
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    seed = 3 * Nq + Nk + d
    q, k, v = make_inputs(B, H, Nq, Nk, d, dtype, seed=seed)
    do = make_dout(B, H, Nq, d, dtype, seed=seed)
    got = run_bwd(q, k, v, do, scale, causal)
    ref = oracle.attn_bwd(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                          do.float().numpy(), scale, causal)
    check(got, ref, dtype, f"{B,H,Nq,Nk,d} causal={causal} scale={scale:.3g}",
          floors=fp32_floor(q.float(), k.float(), v.float(), do.float(), scale), d=d)
    if causal and Nk > Nq:
        # keys no query sees: exactly zero gradients
        assert np.all(got[1][:, :, Nq:] == 0) and np.all(got[2][:, :, Nq:] == 0)


def test_bwd_rejects_bad_arguments():
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_inputs(1, 1, 128, 128, 64, DTYPE_BF16, seed=1))
    o, lse = fa.attention(q, k, v)
    do = torch.randn_like(q)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    need = fa.fa_bwd_workspace(1, 1, 128, 64)
    ws = torch.empty(fa.fa_bwd_workspace(1, 1, 128, 128) + 512, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream(dev).cuda_stream
    args = [q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
            do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), 1, 1, 128, 128, 64,
            0.125, 0, fa.FA_DTYPE_BF16]
    assert fa.fa_bwd(*args, ws.data_ptr(), need - 1, s) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd(*args, ws.data_ptr() + 16, need, s) == fa.FA_ERR_INVALID_ARG
    bad = list(args)
    bad[6] = q.data_ptr()   # dq over q
    assert fa.fa_bwd(*bad, ws.data_ptr(), need, s) == fa.FA_ERR_INVALID_ARG
    bad = list(args)
    bad[13] = 48   # head dim outside the compiled set (extents within the buffers)
    assert fa.fa_bwd(*bad, ws.data_ptr(), fa.fa_bwd_workspace(1, 1, 128, 48),
                     s) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_bwd(*args, ws.data_ptr(), need, s) == fa.FA_OK
    assert fa.fa_fwd_status(s)[0] == fa.FA_OK
