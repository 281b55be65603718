"""fa_fwd_host (host buffers; above 64 MB of input the planes are pipelined
in chunks through host->device copies, kernels and device->host copies)
against fa_fwd on device buffers: the same bits (needs a GB300)."""
import pytest
import torch

from exact_attention_57_gb300 import fa
from exact_attention_57_gb300.workloads import (DTYPE_BF16, DTYPE_F16, DTYPE_F32, DTYPE_F32_SIMT,
                                                make_inputs)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,N,d,dtype,causal", [
    (3, 5, 700, 128, DTYPE_BF16, True),    # 15 planes: uneven chunks
    (1, 1, 300, 64, DTYPE_BF16, False),    # one plane, one chunk
    (2, 8, 1024, 64, DTYPE_F32, False),
    (2, 3, 257, 128, DTYPE_F16, True),
    (1, 20, 129, 32, DTYPE_BF16, True),
    (1, 2, 200, 64, DTYPE_F32_SIMT, True),
    (4, 16, 4096, 128, DTYPE_BF16, True),   # 201 MB in: three uneven chunks of 64 planes
    (3, 20, 4096, 128, DTYPE_F16, False),   # 189 MB in: two chunks
])
def test_host_matches_device(B, H, N, d, dtype, causal):
    dev = torch.device("cuda:0")
    q, k, v = make_inputs(B, H, N, N, d, dtype, seed=1200 + B * H + d)
    scale = d ** -0.5
    stream = torch.cuda.current_stream(dev).cuda_stream
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o_ref = torch.empty_like(qd)
    lse_ref = torch.empty(B, H, N, device=dev, dtype=torch.float32)
    assert fa.fa_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o_ref.data_ptr(),
                     lse_ref.data_ptr(), B, H, N, N, d, scale, int(causal), dtype,
                     stream) == fa.FA_OK
    assert fa.fa_fwd_status(stream) == (fa.FA_OK, 0)
    qh, kh, vh = (t.contiguous().pin_memory() for t in (q, k, v))
    # fresh device staging buffers and pinned outputs, two calls in a row
    q2, k2, v2 = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    o2 = torch.empty_like(qd)
    l2 = torch.empty(B, H, N, device=dev, dtype=torch.float32)
    for _ in range(2):
        oh = torch.full(q.shape, float("nan"), dtype=q.dtype).pin_memory()
        lh = torch.full((B, H, N), float("nan"), dtype=torch.float32).pin_memory()
        assert fa.fa_fwd_host(qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), oh.data_ptr(),
                              lh.data_ptr(), q2.data_ptr(), k2.data_ptr(), v2.data_ptr(),
                              o2.data_ptr(), l2.data_ptr(), B, H, N, N, d, scale, int(causal),
                              dtype, stream) == fa.FA_OK
        assert fa.fa_fwd_status(stream) == (fa.FA_OK, 0)
        assert torch.equal(oh, o_ref.cpu()), "o differs from the device-buffer forward"
        assert torch.equal(lh, lse_ref.cpu()), "lse differs from the device-buffer forward"
