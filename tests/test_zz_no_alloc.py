"""fa_fwd_noalloc, the entry point that allocates no device memory, against
fa_fwd on the same inputs.

Callers that cannot let a library allocate device memory (a server that
reserves the whole GPU for its own pool at start-up, a latency-critical loop
that cannot pay the synchronisation of cudaMalloc, a framework that accounts
for every device allocation) use fa_fwd_noalloc; it has to return what fa_fwd
returns, call after call, although every call reuses one fixed scratch array.
This file sorts last so a run that stops at the first failure has already run
every other test.
"""
import numpy as np
import pytest
import torch

from exact_attention_57_gb300 import fa
from exact_attention_57_gb300.workloads import DTYPE_BF16, DTYPE_F32_SIMT, make_inputs
from parity_util import TOL

pytestmark = pytest.mark.gpu


def _close(o, lse, o_ref, lse_ref, dtype):
    tol = TOL[dtype]
    eo = (o.double() - o_ref.double()).abs()
    el = (lse.double() - lse_ref.double()).abs()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    assert eo.max().item() <= tol["max_o"], eo.max().item()
    if tol["mean_o"] is not None:
        assert eo.mean().item() <= tol["mean_o"], eo.mean().item()
    assert el.max().item() <= tol["max_lse"], el.max().item()


@pytest.mark.parametrize("dtype,d,causal", [(DTYPE_BF16, 128, True), (DTYPE_BF16, 64, False),
                                            (DTYPE_F32_SIMT, 64, True)])
def test_noalloc_matches_fa_fwd_on_two_calls(dtype, d, causal):
    dev = torch.device("cuda:0")
    B, H, N = 2, 4, 1000
    q, k, v = (t.to(dev) for t in make_inputs(B, H, N, N, d, dtype, seed=31 + d))
    scale = 1.0 / d ** 0.5
    stream = torch.cuda.current_stream(dev).cuda_stream
    o_ref = torch.empty_like(q)
    lse_ref = torch.empty(B, H, N, device=dev, dtype=torch.float32)
    assert fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o_ref.data_ptr(),
                     lse_ref.data_ptr(), B, H, N, N, d, scale, int(causal), dtype,
                     stream) == fa.FA_OK
    assert fa.fa_fwd_status(stream) == (fa.FA_OK, 0)
    for _ in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, N), float("nan"), device=dev, dtype=torch.float32)
        st, word = fa.fa_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), B, H, N, N, d, scale, int(causal), dtype,
                                     stream, wait=True)
        assert (st, word) == (fa.FA_OK, 0)
        _close(o, lse, o_ref, lse_ref, dtype)


def test_noalloc_enqueue_only_and_argument_checks():
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_inputs(1, 2, 300, 300, 128, DTYPE_BF16, seed=5))
    o_ref, lse_ref = fa.attention(q, k, v, causal=True)
    o, lse = torch.empty_like(o_ref), torch.empty_like(lse_ref)
    stream = torch.cuda.current_stream(dev).cuda_stream
    st, word = fa.fa_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), 1, 2, 300, 300, 128, 128 ** -0.5, 1,
                                 DTYPE_BF16, stream, wait=False)
    assert st == fa.FA_OK and word is None
    torch.cuda.synchronize()
    _close(o, lse, o_ref, lse_ref, DTYPE_BF16)
    # the same host-side validation as fa_fwd
    st, _ = fa.fa_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), q.data_ptr(),
                              lse.data_ptr(), 1, 2, 300, 300, 128, 0.1, 1, DTYPE_BF16, stream)
    assert st == fa.FA_ERR_INVALID_ARG
    st, _ = fa.fa_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), 1, 2, 300, 300, 96, 0.1, 1, DTYPE_BF16, stream)
    assert st == fa.FA_ERR_UNSUPPORTED
