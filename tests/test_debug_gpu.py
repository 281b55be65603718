"""The debug build (libfa_debug.so, compiled with FA_DEBUG; needs a GB300).

Its kernels check the index of every plain global load and store against the
buffer's extent and report a failed check in the status word (bit 32)
instead of making the access.  On valid calls the checks must never fire and
must not change a single bit of the results; a test aid that understates the
LSE extent shows a check firing, with the skipped stores and nothing else
missing, and no access outside a buffer at any point.
"""
import ctypes

import numpy as np
import pytest
import torch

from exact_attention_57_gb300 import build, fa
from exact_attention_57_gb300.workloads import (DTYPE_BF16, DTYPE_F16, DTYPE_F32, DTYPE_F32_SIMT,
                                                make_dout, make_inputs)

pytestmark = pytest.mark.gpu

BOUNDS = 32  # status bit of a failed index check


@pytest.fixture(scope="module")
def dbg():
    """The debug library, built on first use (its objects live apart from the
    release build's)."""
    lib = fa.load(build.build_library(debug=True))
    assert lib.fa_debug_build() == 1
    assert fa.load().fa_debug_build() == 0
    return lib


def _status(lib, stream):
    word = ctypes.c_int(0)
    st = lib.fa_fwd_status(stream, ctypes.byref(word))
    return st, word.value


def _fwd(lib, q, k, v, scale, causal, dtype, stream):
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, Nq), float("nan"), device=q.device, dtype=torch.float32)
    st = lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H,
                    Nq, Nk, d, scale, int(causal), dtype, stream)
    assert st == fa.FA_OK
    return o, lse


@pytest.mark.parametrize("dtype,d,N,causal", [
    (DTYPE_BF16, 128, 700, True), (DTYPE_BF16, 64, 1000, False), (DTYPE_F16, 256, 333, True),
    (DTYPE_BF16, 32, 129, True), (DTYPE_F32, 64, 300, True), (DTYPE_F32, 128, 257, False),
    (DTYPE_F32_SIMT, 100, 200, True),
])
def test_debug_forward_same_bits_no_check_fires(dbg, dtype, d, N, causal):
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_inputs(2, 3, N, N, d, dtype, seed=N + d))
    stream = torch.cuda.current_stream(dev).cuda_stream
    rel = fa.load()
    o1, l1 = _fwd(rel, q, k, v, d ** -0.5, causal, dtype, stream)
    o2, l2 = _fwd(dbg, q, k, v, d ** -0.5, causal, dtype, stream)
    assert _status(dbg, stream) == (fa.FA_OK, 0)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("d,N", [(64, 300), (128, 257), (32, 129)])
def test_debug_staged_same_bits_no_check_fires(dbg, d, N):
    """fa_fwd_staged (fp32, bf16 split scores): the kernel's Q rows are plain
    loads checked against Q's extent."""
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev).cuda_stream
    q, k, v = (t.to(dev) for t in make_inputs(2, 3, N, N, d, DTYPE_F32, seed=N + 5 * d))
    outs = []
    for lib in (fa.load(), dbg):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((2, 3, N), float("nan"), device=dev, dtype=torch.float32)
        wsb = lib.fa_fwd_staged_workspace(2, 3, N, d, DTYPE_F32)
        ws = torch.empty(wsb, device=dev, dtype=torch.uint8)
        assert lib.fa_fwd_staged(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), 2, 3, N, N, d, d ** -0.5, 1, DTYPE_F32,
                                 ws.data_ptr(), wsb, stream) == fa.FA_OK
        assert _status(lib, stream) == (fa.FA_OK, 0)
        outs.append((o, lse))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_debug_splitkv_varlen_backward_no_check_fires(dbg):
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev).cuda_stream
    # split-KV: one query tile against a long key range
    q, k, v = (t.to(dev) for t in make_inputs(1, 2, 100, 3000, 128, DTYPE_BF16, seed=3))
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 100, device=dev)
    ws_bytes = dbg.fa_fwd_splitkv_workspace(1, 2, 100, 128, 8)
    ws = torch.empty(ws_bytes, device=dev, dtype=torch.uint8)
    assert dbg.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), 1, 2, 100, 3000, 128, 128 ** -0.5, 0, DTYPE_BF16, 8,
                              ws.data_ptr(), ws_bytes, stream) == fa.FA_OK
    assert _status(dbg, stream) == (fa.FA_OK, 0)
    o_ref, l_ref = fa.attention(q, k, v, causal=False)
    torch.cuda.synchronize()
    assert (o.float() - o_ref.float()).abs().max().item() <= 2e-2
    # variable lengths (rows written one by one, sequences without keys)
    lens_q, lens_k, H, d = [5, 130, 0, 40], [300, 0, 7, 40], 2, 64
    tq, tk = sum(lens_q), sum(lens_k)
    qp = torch.randn(tq, H, d, device=dev).to(torch.bfloat16)
    kp = torch.randn(tk, H, d, device=dev).to(torch.bfloat16)
    vp = torch.randn(tk, H, d, device=dev).to(torch.bfloat16)
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32, device=dev)
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32, device=dev)
    o = torch.empty_like(qp)
    lse = torch.empty(H, tq, device=dev)
    assert dbg.fa_fwd_varlen(qp.data_ptr(), kp.data_ptr(), vp.data_ptr(), o.data_ptr(),
                             lse.data_ptr(), cu_q.data_ptr(), cu_k.data_ptr(), 4, H, tq, tk,
                             max(lens_q), d, 0.125, 1, DTYPE_BF16, stream) == fa.FA_OK
    assert _status(dbg, stream) == (fa.FA_OK, 0)
    # backward, fixed and variable lengths
    B, H, N, d = 1, 2, 300, 128
    q, k, v = (t.to(dev) for t in make_inputs(B, H, N, N, d, DTYPE_BF16, seed=8))
    o, lse = fa.attention(q, k, v, causal=True)
    do = make_dout(B, H, N, d, DTYPE_BF16, seed=8).to(dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wsb = dbg.fa_bwd_workspace(B, H, N, d)
    ws = torch.empty(wsb, device=dev, dtype=torch.uint8)
    assert dbg.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, N, d,
                      d ** -0.5, 1, DTYPE_BF16, ws.data_ptr(), wsb, stream) == fa.FA_OK
    assert _status(dbg, stream) == (fa.FA_OK, 0)
    rq, rk, rv = fa.attention_backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(dq, rq) and torch.equal(dk, rk) and torch.equal(dv, rv)


def test_debug_check_fires_and_skips_only_that_store(dbg):
    """With the LSE extent understated by 5 entries, the last 5 LSE stores
    fail their check: bit 32 is reported, those entries keep their poison,
    and every other output is the release build's."""
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev).cuda_stream
    B, H, N, d = 1, 2, 256, 128
    q, k, v = (t.to(dev) for t in make_inputs(B, H, N, N, d, DTYPE_BF16, seed=21))
    o1, l1 = _fwd(fa.load(), q, k, v, 0.1, True, DTYPE_BF16, stream)
    assert fa.load().fa_set_debug_lse_shrink(5) == fa.FA_ERR_UNSUPPORTED  # release build
    try:
        assert dbg.fa_set_debug_lse_shrink(5) == fa.FA_OK
        o2, l2 = _fwd(dbg, q, k, v, 0.1, True, DTYPE_BF16, stream)
        st, word = _status(dbg, stream)
    finally:
        assert dbg.fa_set_debug_lse_shrink(0) == fa.FA_OK
    assert st == fa.FA_ERR_DEVICE_TIMEOUT and word == BOUNDS, word
    assert torch.equal(o1, o2)
    flat1, flat2 = l1.reshape(-1), l2.reshape(-1)
    assert torch.isnan(flat2[-5:]).all()
    assert torch.equal(flat1[:-5], flat2[:-5])
    # the next call is clean again
    o3, l3 = _fwd(dbg, q, k, v, 0.1, True, DTYPE_BF16, stream)
    assert _status(dbg, stream) == (fa.FA_OK, 0)
    assert torch.equal(l1, l3)
