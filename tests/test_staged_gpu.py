"""fa_fwd_staged (fp32 inputs: K split into bf16 halves and V rounded and
transposed once per call by a pre-pass, scores as three bf16 products)
against the float64 oracle, and against fa_fwd on the same inputs (needs a
GB300)."""
import math

import pytest
import torch

from exact_attention_57_gb300 import fa
from exact_attention_57_gb300.workloads import (DTYPE_BF16, DTYPE_F32, WORKLOADS, make_inputs,
                                                workload_inputs)
from parity_util import compare, run_oracle

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, Nq, Nk, d
    (2, 3, 700, 700, 64),
    (1, 2, 300, 457, 128),
    (1, 2, 129, 1, 64),
    (2, 2, 257, 200, 32),
    (1, 1, 1, 1000, 128),
]


def run_staged(q, k, v, scale, causal):
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), device=dev, dtype=torch.float32)
    fa.attention(qd, kd, vd, scale=scale, causal=causal, out=o, lse=lse, staged=True)
    st, word = fa.fa_fwd_status(torch.cuda.current_stream(dev).cuda_stream)
    assert st == fa.FA_OK, word
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


@pytest.mark.parametrize("B,H,Nq,Nk,d", CASES)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("big_scale", [False, True])
def test_staged_matches_oracle(B, H, Nq, Nk, d, causal, big_scale):
    """Scale 1/sqrt(d), and 0.5, where an error in the score products moves
    the LSE most (one tf32 product put it off by 5e-3 there)."""
    q, k, v = make_inputs(B, H, Nq, Nk, d, DTYPE_F32, seed=Nq + 3 * Nk + d)
    scale = 0.5 if big_scale else 1.0 / math.sqrt(d)
    o, lse = run_staged(q, k, v, scale, causal)
    ro, rl = run_oracle(q, k, v, scale, causal)
    st = compare(o, lse, ro, rl, DTYPE_F32, f"staged {B,H,Nq,Nk,d} causal={causal}")
    print(f"staged {B,H,Nq,Nk,d} causal={causal} scale={scale:.3f}: {st}")


@pytest.mark.parametrize("scale", [-0.3, 0.0])
def test_staged_negative_and_zero_scale(scale):
    """A negative scale runs as S = (-Q) K^T with |scale| (the negate bit of
    the bf16 products' descriptor); scale 0 gives uniform weights."""
    q, k, v = make_inputs(1, 2, 300, 500, 64, DTYPE_F32, seed=77)
    for causal in (False, True):
        o, lse = run_staged(q, k, v, scale, causal)
        ro, rl = run_oracle(q, k, v, scale, causal)
        compare(o, lse, ro, rl, DTYPE_F32, f"staged scale={scale} causal={causal}")


def test_staged_fp32_workload_full():
    """The fp32 workload b4h4n4096d64 (non-causal) through the path its
    benchmark times, every element against the oracle."""
    w = WORKLOADS["b4h4n4096d64-f32-tf32"]
    q, k, v = workload_inputs(w)
    for causal in w.causal:
        o, lse = run_staged(q, k, v, w.scale, causal)
        ro, rl = run_oracle(q, k, v, w.scale, causal)
        st = compare(o, lse, ro, rl, DTYPE_F32, f"staged {w.name} causal={causal}")
        print(f"staged {w.name} causal={causal}: {st}")


def test_staged_other_dtypes_run_fa_fwd():
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_inputs(1, 2, 256, 256, 64, DTYPE_BF16, seed=4))
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 256, device=dev)
    s = torch.cuda.current_stream(dev).cuda_stream
    st = fa.fa_fwd_staged(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                          1, 2, 256, 256, 64, 0.125, 1, fa.FA_DTYPE_BF16, None, 0, s)
    assert st == fa.FA_OK
    o2, l2 = fa.attention(q, k, v, scale=0.125, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, l2)
