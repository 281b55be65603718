"""fa_fwd_splitkv (key range split into chunks, merged by log-sum-exp) against
the float64 oracle, including chunk counts above the number of key tiles
(empty chunks) and the automatic choice (needs a GB300)."""
import math

import pytest
import torch

from exact_attention_57_gb300 import fa
from exact_attention_57_gb300.workloads import DTYPE_BF16, DTYPE_F16, DTYPE_F32, make_inputs
from parity_util import compare, run_oracle

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, Nq, Nk, d, dtype
    (1, 8, 1, 5000, 128, DTYPE_BF16),
    (2, 2, 130, 3001, 64, DTYPE_F16),
    (1, 4, 256, 1024, 64, DTYPE_F32),
    (1, 3, 300, 900, 128, DTYPE_F16),
    (2, 4, 128, 4096, 64, DTYPE_BF16),
    (1, 2, 200, 2000, 256, DTYPE_BF16),
    (1, 2, 130, 1500, 128, DTYPE_F32),
    (2, 2, 100, 1100, 32, DTYPE_BF16),
]


def run_split(q, k, v, scale, causal, num_splits):
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), device=dev, dtype=torch.float32)
    fa.attention(qd, kd, vd, scale=scale, causal=causal, out=o, lse=lse, num_splits=num_splits)
    st, word = fa.fa_fwd_status(torch.cuda.current_stream(dev).cuda_stream)
    assert st == fa.FA_OK, word
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


@pytest.mark.parametrize("B,H,Nq,Nk,d,dtype", CASES)
@pytest.mark.parametrize("num_splits", [0, 2, 5, 64])
@pytest.mark.parametrize("causal", [False, True])
def test_splitkv_matches_oracle(B, H, Nq, Nk, d, dtype, num_splits, causal):
    q, k, v = make_inputs(B, H, Nq, Nk, d, dtype, seed=Nq + Nk + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_split(q, k, v, scale, causal, num_splits)
    ro, rl = run_oracle(q, k, v, scale, causal)
    compare(o, lse, ro, rl, dtype, f"split={num_splits} {B,H,Nq,Nk,d} causal={causal}")


def test_splitkv_agrees_with_fa_fwd():
    """Same inputs through fa_fwd and through 7 chunks: the merged result
    differs from the single pass only by fp32 rounding and the bf16 output."""
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_inputs(1, 8, 128, 8192, 128, DTYPE_BF16, seed=3))
    o1, l1 = fa.attention(q, k, v, causal=False)
    o2, l2 = fa.attention(q, k, v, causal=False, num_splits=7)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert (l1 - l2).abs().max().item() <= 1e-4
