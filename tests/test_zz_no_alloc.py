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
import pytest
import torch

from exact_attention_57_gb300 import fa
from exact_attention_57_gb300.workloads import DTYPE_BF16, DTYPE_F32_SIMT, make_inputs

pytestmark = pytest.mark.gpu


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
        # the same kernels on the same inputs: bit for bit
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


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
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    # the same host-side validation as fa_fwd
    st, _ = fa.fa_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), q.data_ptr(),
                              lse.data_ptr(), 1, 2, 300, 300, 128, 0.1, 1, DTYPE_BF16, stream)
    assert st == fa.FA_ERR_INVALID_ARG
    st, _ = fa.fa_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), 1, 2, 300, 300, 96, 0.1, 1, DTYPE_BF16, stream)
    assert st == fa.FA_ERR_UNSUPPORTED


def test_noalloc_reports_a_timeout_then_starts_clean():
    """A kernel that gives up waiting records it in the array's status word,
    the waiting form reports it, and the next call starts from a cleared word.
    The failure is made on the host (a test hook that skips one V-tile load
    and shortens the wait limit), never by faulting the GPU."""
    dev = torch.device("cuda:0")
    B, H, N, d = 1, 2, 512, 128
    q, k, v = (t.to(dev) for t in make_inputs(B, H, N, N, d, DTYPE_BF16, seed=3))
    o_ref, lse_ref = fa.attention(q, k, v, causal=False)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev).cuda_stream
    o = torch.empty_like(o_ref)
    lse = torch.empty_like(lse_ref)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, N,
            d, d ** -0.5, 0, DTYPE_BF16, stream)
    try:
        fa.fa_set_test_hooks(skip_v_load=1, wait_limit_ns=200_000_000)  # 0.2 s
        st, word = fa.fa_fwd_noalloc(*args, wait=True)
    finally:
        fa.fa_set_test_hooks(0, 0)
    assert st == fa.FA_ERR_DEVICE_TIMEOUT
    assert word & 8, word   # the injected skip was recorded
    assert word & 2, word   # the UMMA issuer gave up waiting for V
    # fa_fwd's own word is untouched by the no-allocation path
    assert fa.fa_fwd_status(stream) == (fa.FA_OK, 0)
    st, word = fa.fa_fwd_noalloc(*args, wait=True)
    assert (st, word) == (fa.FA_OK, 0)
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
