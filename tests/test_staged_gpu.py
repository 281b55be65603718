"""fa_fwd_staged (fp32 inputs: K rounded to tf32 and V transposed once per call
by a pre-pass) against the float64 oracle, and against fa_fwd on the same
inputs (needs a GB300)."""
import math

import pytest
import torch

from exact_attention_57_gb300 import fa
from exact_attention_57_gb300.workloads import DTYPE_BF16, DTYPE_F32, make_inputs
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
def test_staged_matches_oracle(B, H, Nq, Nk, d, causal):
    q, k, v = make_inputs(B, H, Nq, Nk, d, DTYPE_F32, seed=Nq + 3 * Nk + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_staged(q, k, v, scale, causal)
    ro, rl = run_oracle(q, k, v, scale, causal)
    compare(o, lse, ro, rl, DTYPE_F32, f"staged {B,H,Nq,Nk,d} causal={causal}")


def test_staged_equals_fa_fwd():
    """The same roundings, applied once instead of per query tile: the same
    result as fa_fwd up to fp32 accumulation order (identical here)."""
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_inputs(2, 4, 1000, 1300, 64, DTYPE_F32, seed=8))
    o1, l1 = fa.attention(q, k, v, causal=True)
    o2, l2 = fa.attention(q, k, v, causal=True, staged=True)
    torch.cuda.synchronize()
    assert (o1 - o2).abs().max().item() <= 1e-6
    assert (l1 - l2).abs().max().item() <= 1e-6


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
