"""fa_bwd_varlen (packed sequences of different lengths) against the float64
oracle gradients of each sequence on its own (needs a GB300)."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_57_gb300 import fa
from exact_attention_57_gb300.workloads import DTYPE_BF16, DTYPE_F16, make_dout, make_inputs
from test_bwd_gpu import check, fp32_floor

pytestmark = pytest.mark.gpu

CASES = [
    # query lengths, key lengths, H, d, dtype
    ([1, 127, 128, 129, 300], [1, 127, 128, 129, 300], 2, 128, DTYPE_BF16),
    ([200, 33, 0, 64], [64, 500, 70, 0], 2, 64, DTYPE_F16),
    ([257, 90], [100, 300], 3, 32, DTYPE_BF16),
    ([640, 1], [640, 513], 2, 128, DTYPE_BF16),
]


def pack(parts):
    """[1, H, L, d] tensors -> token-major [sum L, H, d]."""
    return torch.cat([t[0].transpose(0, 1) for t in parts], dim=0).contiguous()


def unpack(t, start, length):
    """token-major rows [start, start+length) -> [1, H, length, d] numpy."""
    return t[start:start + length].transpose(0, 1).unsqueeze(0).double().cpu().numpy()


@pytest.mark.parametrize("lens_q,lens_k,H,d,dtype", CASES)
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_varlen_matches_oracle(lens_q, lens_k, H, d, dtype, causal):
    dev = torch.device("cuda:0")
    seqs = []
    for i, (lq, lk) in enumerate(zip(lens_q, lens_k)):
        q, k, v = make_inputs(1, H, max(lq, 1), max(lk, 1), d, dtype, seed=300 + 10 * i + lq + lk)
        do = make_dout(1, H, max(lq, 1), d, dtype, seed=400 + i + lq)
        seqs.append((q[:, :, :lq], k[:, :, :lk], v[:, :, :lk], do[:, :, :lq]))
    qp, kp, vp, dop = (pack([s[j] for s in seqs]).to(dev) for j in range(4))
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32, device=dev)
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32, device=dev)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attention_varlen(qp, kp, vp, cu_q, cu_k, max(lens_q), scale=scale, causal=causal)
    dq, dk, dv = fa.attention_backward_varlen(qp, kp, vp, o, lse, dop, cu_q, cu_k, max(lens_q),
                                              max(lens_k), scale=scale, causal=causal)
    st, word = fa.fa_fwd_status(torch.cuda.current_stream(dev).cuda_stream)
    assert st == fa.FA_OK, word
    sq = sk = 0
    for (q, k, v, do), lq, lk in zip(seqs, lens_q, lens_k):
        gq, gk, gv = unpack(dq, sq, lq), unpack(dk, sk, lk), unpack(dv, sk, lk)
        sq += lq
        sk += lk
        if lq == 0:   # no query sees these keys: zero gradients
            assert np.all(gk == 0) and np.all(gv == 0)
            continue
        if lk == 0:   # O = 0 whatever q is
            assert np.all(gq == 0)
            continue
        ref = oracle.attn_bwd(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                              do.float().numpy(), scale, causal)
        check([gq, gk, gv], ref, dtype, f"seq lq={lq} lk={lk} causal={causal}",
              floors=fp32_floor(q.float(), k.float(), v.float(), do.float(), scale), d=d)


def test_bwd_varlen_equals_fixed_length():
    """One sequence packed alone gives the fixed-length backward's gradients."""
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_inputs(1, 4, 700, 700, 128, DTYPE_BF16, seed=21))
    do = make_dout(1, 4, 700, 128, DTYPE_BF16, seed=21).to(dev)
    o, lse = fa.attention(q, k, v, causal=True)
    g1 = fa.attention_backward(q, k, v, o, lse, do, causal=True)
    tok = lambda t: t[0].transpose(0, 1).contiguous()
    cu = torch.tensor([0, 700], dtype=torch.int32, device=dev)
    ov, lv = fa.attention_varlen(tok(q), tok(k), tok(v), cu, cu, 700, causal=True)
    g2 = fa.attention_backward_varlen(tok(q), tok(k), tok(v), ov, lv, tok(do), cu, cu, 700, 700,
                                      causal=True)
    torch.cuda.synchronize()
    for a, b in zip(g1, g2):
        # fp32 atomic adds into dq may land in a different order
        assert (tok(a).float() - b.float()).abs().max().item() <= 2e-2
