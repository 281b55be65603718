"""CUDA path vs the float64 CPU oracle, element by element (needs a GB300)."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_57_gb300 import fa
from exact_attention_57_gb300.workloads import (DTYPE_BF16, DTYPE_F16, DTYPE_F32, DTYPE_F32_SIMT,
                                                WORKLOADS, make_inputs, workload_inputs)
from parity_util import TOL, compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

FULL_WORKLOADS = [n for n in WORKLOADS if n != "b8h32n8192d128-bf16-causal"]


@pytest.mark.parametrize("name", FULL_WORKLOADS)
def test_named_workload_full(name):
    w = WORKLOADS[name]
    q, k, v = workload_inputs(w)
    for causal in w.causal:
        o, lse = run_gpu(q, k, v, w.scale, causal, w.dtype)
        ro, rl = run_oracle(q, k, v, w.scale, causal)
        compare(o, lse, ro, rl, w.dtype, f"{name} causal={causal}")


DT_NAME = {DTYPE_BF16: "bf16", DTYPE_F32: "f32tc", DTYPE_F32_SIMT: "simt", DTYPE_F16: "f16"}


def _dd(pairs):
    return [pytest.param(dt, d, id=f"{DT_NAME[dt]}-d{d}") for dt, d in pairs]


@pytest.mark.parametrize("dtype,d", _dd([(DTYPE_BF16, 64), (DTYPE_BF16, 128), (DTYPE_F32, 64),
                                         (DTYPE_F32_SIMT, 64), (DTYPE_F16, 64),
                                         (DTYPE_F16, 128), (DTYPE_BF16, 256), (DTYPE_F16, 256),
                                         (DTYPE_F32, 128), (DTYPE_BF16, 32), (DTYPE_F16, 32),
                                         (DTYPE_F32, 32)]))
@pytest.mark.parametrize("causal", [False, True])
def test_other_mask_per_dtype(dtype, d, causal):
    """Every kernel variant, causal and not, on a several-tile ragged case."""
    q, k, v = make_inputs(2, 3, 700, 700, d, dtype, seed=11 + d + 7 * dtype)
    o, lse = run_gpu(q, k, v, 1.0 / math.sqrt(d), causal, dtype)
    ro, rl = run_oracle(q, k, v, 1.0 / math.sqrt(d), causal)
    compare(o, lse, ro, rl, dtype, f"N=700 d={d} causal={causal}")


EDGE_N = [1, 2, 127, 128, 129, 255, 256, 257]


@pytest.mark.parametrize("N", EDGE_N)
@pytest.mark.parametrize("dtype,d", _dd([(DTYPE_BF16, 64), (DTYPE_BF16, 128), (DTYPE_F32, 64),
                                         (DTYPE_F32_SIMT, 64), (DTYPE_F16, 128), (DTYPE_BF16, 256),
                                         (DTYPE_F32, 128), (DTYPE_BF16, 32)]))
def test_edge_lengths(N, dtype, d):
    q, k, v = make_inputs(1, 2, N, N, d, dtype, seed=100 + N)
    for causal in (False, True):
        o, lse = run_gpu(q, k, v, 1.0 / math.sqrt(d), causal, dtype)
        ro, rl = run_oracle(q, k, v, 1.0 / math.sqrt(d), causal)
        compare(o, lse, ro, rl, dtype, f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("Nq,Nk", [(200, 77), (77, 200), (1, 1000), (1000, 1), (129, 384),
                                   (384, 129)])
@pytest.mark.parametrize("dtype,d", _dd([(DTYPE_BF16, 128), (DTYPE_F32, 64), (DTYPE_F32_SIMT, 64),
                                         (DTYPE_F16, 64), (DTYPE_F16, 256), (DTYPE_F32, 128),
                                         (DTYPE_F16, 32)]))
def test_unequal_lengths(Nq, Nk, dtype, d):
    """Nq != Nk, causal top-left aligned (key j allowed iff j <= i)."""
    q, k, v = make_inputs(2, 1, Nq, Nk, d, dtype, seed=Nq * 7 + Nk)
    for causal in (False, True):
        o, lse = run_gpu(q, k, v, 0.1, causal, dtype)
        ro, rl = run_oracle(q, k, v, 0.1, causal)
        compare(o, lse, ro, rl, dtype, f"Nq={Nq} Nk={Nk} causal={causal}")


@pytest.mark.parametrize("scale", [0.0, -0.125, 0.5, 1e-3])
@pytest.mark.parametrize("dtype,d", _dd([(DTYPE_BF16, 128), (DTYPE_F32, 64), (DTYPE_F32_SIMT, 32),
                                         (DTYPE_F16, 128), (DTYPE_BF16, 256)]))
def test_scales(scale, dtype, d):
    """Zero and negative scales are valid: scale multiplies q.k before the max."""
    q, k, v = make_inputs(1, 2, 300, 300, d, dtype, seed=5)
    for causal in (False, True):
        o, lse = run_gpu(q, k, v, scale, causal, dtype)
        ro, rl = run_oracle(q, k, v, scale, causal)
        compare(o, lse, ro, rl, dtype, f"scale={scale} causal={causal}")


def test_large_score_range():
    """Scores spanning many binades force the running max to move (rescale path)."""
    q, k, v = make_inputs(1, 2, 1024, 1024, 128, DTYPE_BF16, seed=9, k_mult=6.0)
    # increasing key magnitude along the sequence makes later tiles' maxima larger
    ramp = torch.linspace(0.2, 3.0, 1024).view(1, 1, 1024, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    for causal in (False, True):
        o, lse = run_gpu(q, k, v, 1.0 / math.sqrt(128), causal, DTYPE_BF16)
        ro, rl = run_oracle(q, k, v, 1.0 / math.sqrt(128), causal)
        compare(o, lse, ro, rl, DTYPE_BF16, f"ramped keys causal={causal}")


@pytest.mark.parametrize("H,Nq,Nk,causal", [(1, 1, 131072, False), (2, 300, 131072, False),
                                            (4, 8192, 8192, True)])
@pytest.mark.parametrize("dtype,d", _dd([(DTYPE_BF16, 128), (DTYPE_F16, 64), (DTYPE_F32, 64)]))
def test_long_sequences(H, Nq, Nk, causal, dtype, d):
    """Long key ranges: 1 024 key tiles through one query tile's pipeline (the
    running offset, the row sum and O carried across all of them), and
    8 192-token causal heads whose query tiles run 1 to 64 key tiles."""
    q, k, v = make_inputs(1, H, Nq, Nk, d, dtype, seed=Nq + Nk + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_gpu(q, k, v, scale, causal, dtype)
    ro, rl = run_oracle(q, k, v, scale, causal)
    compare(o, lse, ro, rl, dtype, f"Nq={Nq} Nk={Nk} causal={causal}")


@pytest.mark.parametrize("d", [1, 8, 17, 33, 100, 128])
def test_simt_head_dims(d):
    q, k, v = make_inputs(2, 1, 150, 150, d, DTYPE_F32_SIMT, seed=d)
    for causal in (False, True):
        o, lse = run_gpu(q, k, v, 1.0 / math.sqrt(d), causal, DTYPE_F32_SIMT)
        ro, rl = run_oracle(q, k, v, 1.0 / math.sqrt(d), causal)
        compare(o, lse, ro, rl, DTYPE_F32_SIMT, f"simt d={d} causal={causal}")


def test_constant_v_rows():
    """Constant value rows: every output row equals that row (bf16-exact v)."""
    q, k, _ = make_inputs(1, 2, 500, 500, 128, DTYPE_BF16, seed=3)
    c = torch.randn(128).to(torch.bfloat16)
    v = c.view(1, 1, 1, 128).expand(1, 2, 500, 128).contiguous()
    for causal in (False, True):
        o, _ = run_gpu(q, k, v, 0.09, causal, DTYPE_BF16)
        want = np.broadcast_to(c.double().numpy(), o.shape)
        assert np.abs(o - want).max() <= 2e-2 * max(1.0, float(np.abs(want).max()))


def test_outputs_stay_in_bounds():
    """Writes land only inside O and LSE: guard regions around them keep their
    sentinel values (ragged length so the last tile is partial)."""
    dev = torch.device("cuda:0")
    B, H, N, d = 1, 3, 333, 128
    q, k, v = make_inputs(B, H, N, N, d, DTYPE_BF16, seed=77)
    n_o, n_l, guard = B * H * N * d, B * H * N, 4096
    obuf = torch.full((n_o + 2 * guard,), 7.0, device=dev, dtype=torch.bfloat16)
    lbuf = torch.full((n_l + 2 * guard,), 7.0, device=dev, dtype=torch.float32)
    o = obuf[guard:guard + n_o].view(B, H, N, d)
    lse = lbuf[guard:guard + n_l].view(B, H, N)
    fa.attention(q.to(dev), k.to(dev), v.to(dev), causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(obuf[:guard] == 7.0) and torch.all(obuf[guard + n_o:] == 7.0)
    assert torch.all(lbuf[:guard] == 7.0) and torch.all(lbuf[guard + n_l:] == 7.0)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_deterministic_and_stream():
    """Bit-identical results across runs, on the default and a side stream."""
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_inputs(2, 4, 1024, 1024, 128, DTYPE_BF16, seed=1))
    o1, l1 = fa.attention(q, k, v, causal=True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o2, l2 = fa.attention(q, k, v, causal=True)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_large_workload_sampled_rows():
    """The 256-head N=8192 causal workload at full size, in the launch the
    benchmark times: sampled rows against the oracle, plus properties that
    hold at any size (finite, LSE >= the causal row's self-score bound)."""
    w = WORKLOADS["b8h32n8192d128-bf16-causal"]
    q, k, v = workload_inputs(w)
    o, lse = run_gpu(q, k, v, w.scale, True, w.dtype, poison=True)
    B, H, N, d = w.B, w.H, w.Nq, w.d
    rng = np.random.default_rng(2024)
    # rows: tile edges and the ends of the sequence, plus random ones
    picks = [0, 1, 127, 128, 129, 4095, 4096, 8063, 8064, 8190, 8191]
    heads = rng.integers(0, B * H, size=40)
    rows = [int(hh) * N + int(i) for hh in heads for i in picks]
    rows += list(rng.integers(0, B * H * N, size=600))
    rows = np.unique(np.array(rows, dtype=np.int64))
    ro, rl = oracle.attn_rows(q.float().numpy(), k.float().numpy(), v.float().numpy(), rows,
                              w.scale, True)
    go = o.reshape(-1, d)[rows]
    gl = lse.reshape(-1)[rows]
    eo, el = np.abs(go - ro), np.abs(gl - rl)
    tol = TOL[w.dtype]
    assert eo.max() <= tol["max_o"] and eo.mean() <= tol["mean_o"], (eo.max(), eo.mean())
    assert el.max() <= tol["max_lse"], el.max()
    # any-size property: LSE >= the score of the row's own diagonal key
    qs = q.view(-1, d)[torch.from_numpy(rows)].float()
    ks = k.view(-1, d)[torch.from_numpy(rows)].float()
    self_score = (qs * ks).sum(-1).double().numpy() * w.scale
    assert np.all(gl >= self_score - 1e-2)


def test_large_workload_every_row():
    """The 256-head N=8192 causal workload at full size, in the launch the
    benchmark times (fa_fwd, tiles per CTA chosen as in the benchmark), against
    the oracle on every element of O and LSE.  The oracle runs one batch (32
    heads) at a time to bound host memory; the statistics are over the whole
    output."""
    w = WORKLOADS["b8h32n8192d128-bf16-causal"]
    q, k, v = workload_inputs(w)
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), device=dev, dtype=torch.float32)
    fa.attention(qd, kd, vd, scale=w.scale, causal=True, out=o, lse=lse)
    st, word = fa.fa_fwd_status(torch.cuda.current_stream(dev).cuda_stream)
    assert st == fa.FA_OK, f"device status word {word}"
    o, lse = o.cpu(), lse.cpu()
    del qd, kd, vd
    max_o = sum_o = max_lse = 0.0
    for b in range(w.B):
        ro, rl = oracle.attn_fwd(q[b:b + 1].float().numpy(), k[b:b + 1].float().numpy(),
                                 v[b:b + 1].float().numpy(), w.scale, True)
        go = o[b:b + 1].double().numpy()
        gl = lse[b:b + 1].double().numpy()
        assert np.isfinite(go).all() and np.isfinite(gl).all(), f"batch {b}: unwritten rows"
        eo = np.abs(go - ro)
        max_o = max(max_o, float(eo.max()))
        sum_o += float(eo.sum())
        max_lse = max(max_lse, float(np.abs(gl - rl).max()))
    mean_o = sum_o / o.numel()
    print(f"\nb8h32n8192d128 causal, every row: max|dO| {max_o:.3e} mean|dO| {mean_o:.3e} "
          f"max|dLSE| {max_lse:.3e}")
    tol = TOL[w.dtype]
    assert max_o <= tol["max_o"], max_o
    assert mean_o <= tol["mean_o"], mean_o
    assert max_lse <= tol["max_lse"], max_lse
