"""Stream order under programmatic dependent launch (needs a GB300).

The forward kernels may start their set-up while the previous kernel on the
stream still runs, and wait for it before their first global access.  A
chain of calls in which each call reads what the previous one wrote (its O
as the next query, key or value) must therefore give exactly what the same
calls give one at a time with the stream synchronised in between.
"""
import math

import pytest
import torch

from exact_attention_57_gb300 import fa
from exact_attention_57_gb300.workloads import make_inputs, DTYPE_BF16, DTYPE_F16, DTYPE_F32

pytestmark = pytest.mark.gpu


def _chain(q, k, v, impl, causal, sync):
    outs = []
    a, b, c = q, k, v
    for step in range(6):
        o, lse = fa.attention(a, b, c, causal=causal, impl=impl)
        if sync:
            torch.cuda.synchronize()
        outs.append((o, lse))
        # the next call reads this one's output in a different role each time
        a, b, c = [(o, b, c), (a, o, c), (a, b, o)][step % 3]
    torch.cuda.synchronize()
    return outs


@pytest.mark.parametrize("dtype,d,impl,shape", [
    (DTYPE_BF16, 128, "tc", (2, 4, 1024)),    # small grid: one CTA per query tile
    (DTYPE_BF16, 64, "tc", (1, 2, 300)),      # ragged
    (DTYPE_F16, 128, "tc", (8, 16, 2048)),    # blocked schedule, several waves
    (DTYPE_F32, 64, "tc", (2, 2, 512)),       # fp32 tensor-core path
    (DTYPE_F32, 64, "simt", (1, 1, 256)),     # the SIMT kernel
])
@pytest.mark.parametrize("causal", [False, True])
def test_dependent_chain_matches_synchronised_calls(dtype, d, impl, shape, causal):
    dev = torch.device("cuda:0")
    B, H, N = shape
    q, k, v = (t.to(dev) for t in make_inputs(B, H, N, N, d, dtype, seed=N + d))
    ref = _chain(q, k, v, impl, causal, sync=True)
    for _ in range(3):
        got = _chain(q, k, v, impl, causal, sync=False)
        for step, ((o, l), (ro, rl)) in enumerate(zip(got, ref)):
            assert torch.equal(o, ro) and torch.equal(l, rl), f"step {step} differs"
    st, word = fa.fa_fwd_status(torch.cuda.current_stream(dev).cuda_stream)
    assert (st, word) == (fa.FA_OK, 0)
