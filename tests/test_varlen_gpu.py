"""fa_fwd_varlen (packed sequences of different lengths, token-major
[total, H, d]) against the float64 oracle run on each sequence alone
(needs a GB300)."""
import math
import time

import numpy as np
import pytest
import torch

from exact_attention_57_gb300 import fa
from exact_attention_57_gb300.workloads import DTYPE_BF16, DTYPE_F16, DTYPE_F32, make_inputs
from parity_util import compare, run_oracle

pytestmark = pytest.mark.gpu

CASES = [
    # query lengths, key lengths, H, d, dtype
    ([1, 127, 128, 129, 300], [1, 127, 128, 129, 300], 3, 128, DTYPE_BF16),
    ([5, 0, 260, 40], [300, 7, 0, 40], 2, 64, DTYPE_F16),
    ([200, 33], [64, 500], 2, 64, DTYPE_F32),
    ([1000, 1, 513], [1000, 2048, 513], 4, 128, DTYPE_BF16),
    ([130, 257], [300, 129], 2, 256, DTYPE_BF16),
    ([77, 200], [300, 64], 2, 128, DTYPE_F32),
    ([140, 3, 260], [140, 500, 0], 3, 32, DTYPE_F16),
]


def pack(parts):
    """[1, H, L, d] tensors -> token-major [sum L, H, d]."""
    return torch.cat([t[0].transpose(0, 1) for t in parts], dim=0).contiguous()


@pytest.mark.parametrize("lens_q,lens_k,H,d,dtype", CASES)
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_matches_oracle(lens_q, lens_k, H, d, dtype, causal):
    dev = torch.device("cuda:0")
    seqs = [make_inputs(1, H, max(lq, 1), max(lk, 1), d, dtype, seed=100 * i + lq + lk)
            for i, (lq, lk) in enumerate(zip(lens_q, lens_k))]
    seqs = [(q[:, :, :lq], k[:, :, :lk], v[:, :, :lk]) for (q, k, v), lq, lk in
            zip(seqs, lens_q, lens_k)]
    qp = pack([s[0] for s in seqs]).to(dev)
    kp = pack([s[1] for s in seqs]).to(dev)
    vp = pack([s[2] for s in seqs]).to(dev)
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32, device=dev)
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32, device=dev)
    scale = 1.0 / math.sqrt(d)
    o = torch.full_like(qp, float("nan"))
    lse = torch.full((H, qp.shape[0]), float("nan"), device=dev)
    fa.attention_varlen(qp, kp, vp, cu_q, cu_k, max(lens_q), scale=scale, causal=causal,
                        out=o, lse=lse)
    st, word = fa.fa_fwd_status(torch.cuda.current_stream(dev).cuda_stream)
    assert st == fa.FA_OK, word
    o = o.double().cpu()
    lse = lse.double().cpu()
    start = 0
    for (q, k, v), lq, lk in zip(seqs, lens_q, lens_k):
        rows = slice(start, start + lq)
        start += lq
        if lq == 0:
            continue
        go = o[rows].transpose(0, 1).unsqueeze(0).numpy()     # [1, H, lq, d]
        gl = lse[:, rows].unsqueeze(0).numpy()                 # [1, H, lq]
        if lk == 0:
            assert np.all(go == 0.0) and np.all(np.isneginf(gl)), "no keys: O = 0, LSE = -inf"
            continue
        ro, rl = run_oracle(q, k, v, scale, causal)
        compare(go, gl, ro, rl, dtype, f"seq lq={lq} lk={lk} causal={causal}")


@pytest.mark.parametrize("d,dtype", [(128, DTYPE_BF16), (64, DTYPE_BF16), (64, DTYPE_F16),
                                     (32, DTYPE_BF16)])
def test_varlen_equals_fixed_length(d, dtype):
    """Equal lengths: the packed call matches fa_fwd on [B, H, N, d] bit for
    bit (the same kernel, run with sequence offsets instead of planes)."""
    dev = torch.device("cuda:0")
    B, H, N = 3, 2, 384
    q, k, v = (t.to(dev) for t in make_inputs(B, H, N, N, d, dtype, seed=9))
    o_ref, l_ref = fa.attention(q, k, v, causal=True)
    tok = lambda t: t.permute(0, 2, 1, 3).reshape(B * N, H, d).contiguous()
    cu = torch.arange(0, (B + 1) * N, N, dtype=torch.int32, device=dev)
    o, lse = fa.attention_varlen(tok(q), tok(k), tok(v), cu, cu, N, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o, tok(o_ref))
    assert torch.equal(lse, l_ref.permute(1, 0, 2).reshape(H, B * N))


@pytest.mark.parametrize("cu_k_vals", [[0, 100, 2**31 - 1], [-50, 100, 10**9]])
def test_varlen_key_offsets_past_total_are_clamped(cu_k_vals):
    """Key offsets outside [0, total_k] (read on the device, not checked on
    the host) are clamped there: the call returns promptly, writes nothing
    outside O and LSE, and each sequence sees the keys that exist."""
    dev = torch.device("cuda:0")
    H, d, total_q, total_k = 2, 128, 160, 150
    q, k, v = make_inputs(1, H, total_q, total_k, d, DTYPE_BF16, seed=41)
    tok = lambda t: t[0].transpose(0, 1).contiguous()
    qp, kp, vp = tok(q).to(dev), tok(k).to(dev), tok(v).to(dev)
    cu_q = torch.tensor([0, 100, total_q], dtype=torch.int32, device=dev)
    cu_k = torch.tensor(cu_k_vals, dtype=torch.int32, device=dev)
    guard = 4096
    n_o, n_l = total_q * H * d, H * total_q
    obuf = torch.full((n_o + 2 * guard,), 7.0, device=dev, dtype=torch.bfloat16)
    lbuf = torch.full((n_l + 2 * guard,), 7.0, device=dev, dtype=torch.float32)
    o = obuf[guard:guard + n_o].view(total_q, H, d)
    lse = lbuf[guard:guard + n_l].view(H, total_q)
    scale = 1.0 / math.sqrt(d)
    # warm-up with valid offsets (module load, kernel attributes)
    good_k = torch.tensor([0, 100, total_k], dtype=torch.int32, device=dev)
    fa.attention_varlen(qp, kp, vp, cu_q, good_k, 100, scale=scale, causal=False)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    fa.attention_varlen(qp, kp, vp, cu_q, cu_k, 100, scale=scale, causal=False, out=o, lse=lse)
    st, word = fa.fa_fwd_status(torch.cuda.current_stream(dev).cuda_stream)
    elapsed = time.perf_counter() - t0
    assert st == fa.FA_OK, word
    assert elapsed < 1.0, f"{elapsed:.2f} s: the key range was not clamped"
    assert torch.all(obuf[:guard] == 7.0) and torch.all(obuf[guard + n_o:] == 7.0)
    assert torch.all(lbuf[:guard] == 7.0) and torch.all(lbuf[guard + n_l:] == 7.0)
    o, lse = o.double().cpu(), lse.double().cpu()
    # sequence 0: queries [0, 100), keys [0, 100); sequence 1: queries
    # [100, 160), keys [100, total_k)
    for (q0, q1), (k0, k1) in [((0, 100), (0, 100)), ((100, total_q), (100, total_k))]:
        ro, rl = run_oracle(q[:, :, q0:q1], k[:, :, k0:k1], v[:, :, k0:k1], scale, False)
        go = o[q0:q1].transpose(0, 1).unsqueeze(0).numpy()
        gl = lse[:, q0:q1].unsqueeze(0).numpy()
        compare(go, gl, ro, rl, DTYPE_BF16, f"clamped keys [{k0}, {k1})")
