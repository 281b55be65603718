"""Bounded waits: a starved kernel gives up, reports through the status word,
and leaves the context usable.  The failure is made on the host (a test hook
that skips one V-tile load), never by faulting or trapping the GPU."""
import math

import pytest
import torch

from exact_attention_57_gb300 import fa
from exact_attention_57_gb300.workloads import DTYPE_BF16, DTYPE_F32, make_inputs
from parity_util import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [128, 64])  # the one-tile and the two-tile kernel
def test_starved_kernel_times_out_and_recovers(d):
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_inputs(1, 2, 512, 512, d, DTYPE_BF16, seed=3))
    stream = torch.cuda.current_stream(dev).cuda_stream
    assert fa.fa_fwd_status(stream)[0] == fa.FA_OK
    try:
        fa.fa_set_test_hooks(skip_v_load=1, wait_limit_ns=200_000_000)  # 0.2 s
        fa.attention(q, k, v, causal=False)
        st, word = fa.fa_fwd_status(stream)
    finally:
        fa.fa_set_test_hooks(0, 0)
    assert st == fa.FA_ERR_DEVICE_TIMEOUT
    assert word & 8, word          # the injected skip was recorded
    assert word & 2, word          # the UMMA issuer gave up waiting for V
    # the status word was cleared by the read, and the context still works
    assert fa.fa_fwd_status(stream) == (fa.FA_OK, 0)
    qc, kc, vc = (t.cpu() for t in (q, k, v))
    o, lse = run_gpu(qc, kc, vc, 1 / math.sqrt(d), False, DTYPE_BF16)
    ro, rl = run_oracle(qc, kc, vc, 1 / math.sqrt(d), False)
    compare(o, lse, ro, rl, DTYPE_BF16, "after timeout")


@pytest.mark.parametrize("d", [64, 128])
def test_starved_staged_fp32_kernel_times_out_and_recovers(d):
    """The staged fp32 kernel (bf16 split scores) under the same hook: its
    producer skips the first V^T tile, the P V issuer gives up waiting, and
    the next call runs clean."""
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_inputs(1, 2, 300, 400, d, DTYPE_F32, seed=4))
    stream = torch.cuda.current_stream(dev).cuda_stream
    assert fa.fa_fwd_status(stream)[0] == fa.FA_OK
    try:
        fa.fa_set_test_hooks(skip_v_load=1, wait_limit_ns=200_000_000)  # 0.2 s
        fa.attention(q, k, v, causal=True, staged=True)
        st, word = fa.fa_fwd_status(stream)
    finally:
        fa.fa_set_test_hooks(0, 0)
    assert st == fa.FA_ERR_DEVICE_TIMEOUT
    assert word & 8 and word & 2, word
    assert fa.fa_fwd_status(stream) == (fa.FA_OK, 0)
    o, lse = fa.attention(q, k, v, causal=True, staged=True)
    torch.cuda.synchronize()
    ro, rl = run_oracle(q.cpu(), k.cpu(), v.cpu(), 1 / math.sqrt(d), True)
    compare(o.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, DTYPE_F32,
            "staged after timeout")
