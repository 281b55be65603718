"""The persistent grid of the 16-bit forward (needs a GB300).

A CTA runs the query tiles the schedule deals it, of any heads, one after
another through one pipeline; which CTA computes a tile, and after which
other tile, must not change the tile's arithmetic.  Grids of 1, 2, 3, 7 CTAs
and the automatic size are checked bit for bit against one CTA per query
tile, which is checked against the float64 oracle, on ragged and unequal
lengths, causal and not, for every 16-bit head dim.
"""
import math

import numpy as np
import pytest
import torch

from exact_attention_57_gb300 import fa
from exact_attention_57_gb300.workloads import DTYPE_BF16, DTYPE_F16, make_inputs
from parity_util import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def automatic_grid_afterwards():
    yield
    assert fa.fa_set_fwd_schedule(0, 0, 0) == fa.FA_OK


ONE_PER_TILE = 1 << 30  # clamped to the number of query tiles: one tile per CTA


CASES = [
    (DTYPE_BF16, 128, 700, 700),    # 6 query tiles, ragged last tile
    (DTYPE_BF16, 128, 1000, 1000),  # 8 query tiles
    (DTYPE_BF16, 64, 1000, 1000),   # Q in tensor memory
    (DTYPE_BF16, 256, 700, 700),    # one K and one V stage
    (DTYPE_BF16, 32, 700, 700),     # zero-padded to the d = 64 kernel
    (DTYPE_F16, 128, 1000, 1000),
    (DTYPE_BF16, 128, 129, 129),    # two tiles, the second one row
    (DTYPE_BF16, 128, 1, 1),        # fewer tiles than CTAs
    (DTYPE_BF16, 128, 900, 300),    # Nq > Nk
    (DTYPE_BF16, 128, 300, 900),    # Nq < Nk
]


def _id(c):
    dt, d, nq, nk = c
    return f"{'bf16' if dt == DTYPE_BF16 else 'f16'}-d{d}-{nq}x{nk}"


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", CASES, ids=[_id(c) for c in CASES])
def test_grid_size_same_results(case, causal):
    dtype, d, Nq, Nk = case
    q, k, v = make_inputs(2, 3, Nq, Nk, d, dtype, seed=500 + d + Nq + 3 * Nk)
    scale = 1.0 / math.sqrt(d)
    assert fa.fa_set_fwd_schedule(ONE_PER_TILE, 0, 0) == fa.FA_OK
    o1, l1 = run_gpu(q, k, v, scale, causal, dtype)
    ro, rl = run_oracle(q, k, v, scale, causal)
    compare(o1, l1, ro, rl, dtype, f"{_id(case)} causal={causal} one tile per CTA")
    for ctas, groups, block in ((1, 0, 0), (2, 1, 0), (3, 0, 0), (7, 2, 0), (0, 1, 0),
                                (0, 0, 0), (0, 0, 1), (0, 0, 2), (0, 0, 3), (0, 0, 4)):
        assert fa.fa_set_fwd_schedule(ctas, groups, block) == fa.FA_OK
        o, lse = run_gpu(q, k, v, scale, causal, dtype)
        tag = f"ctas={ctas} groups={groups} block={block}"
        assert np.array_equal(o, o1), f"{tag}: O differs"
        assert np.array_equal(lse, l1), f"{tag}: LSE differs"


def test_grid_size_many_heads_and_groups():
    """More planes than one L2 group (groups of 12 at N = 8192, d = 128) and
    several rounds per CTA: the automatic grid against one tile per CTA."""
    B, H, N, d = 1, 14, 8192, 128
    q, k, v = make_inputs(B, H, N, N, d, DTYPE_BF16, seed=91)
    assert fa.fa_fwd_schedule(B, H, N, N, d, True, DTYPE_BF16, 152)[2] < H
    outs = []
    for ctas, groups, block in ((ONE_PER_TILE, 0, 0), (0, 0, 0), (5, 0, 0), (0, 3, 0),
                                (0, 0, 4)):
        assert fa.fa_set_fwd_schedule(ctas, groups, block) == fa.FA_OK
        outs.append(run_gpu(q, k, v, 1.0 / math.sqrt(d), True, DTYPE_BF16))
    for o, lse in outs[1:]:
        assert np.array_equal(o, outs[0][0]) and np.array_equal(lse, outs[0][1])


def test_noalloc_with_grid_size():
    """fa_fwd_noalloc takes the same persistent schedule."""
    dev = torch.device("cuda:0")
    B, H, N, d = 2, 3, 1000, 128
    q, k, v = (t.to(dev) for t in make_inputs(B, H, N, N, d, DTYPE_BF16, seed=77))
    stream = torch.cuda.current_stream(dev).cuda_stream
    outs = []
    for ctas, block in ((ONE_PER_TILE, 0), (4, 0), (0, 2)):
        assert fa.fa_set_fwd_schedule(ctas, 0, block) == fa.FA_OK
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, N), float("nan"), device=dev, dtype=torch.float32)
        st, word = fa.fa_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), B, H, N, N, d, 1.0 / math.sqrt(d), 1,
                                     DTYPE_BF16, stream, wait=True)
        assert (st, word) == (fa.FA_OK, 0)
        outs.append((o.cpu(), lse.cpu()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
