"""The C-ABI library loads and exports what include/fa.h declares; host-side
argument checks (no GPU needed: these calls return before any CUDA work)."""
import os
import re

import pytest

from exact_attention_57_gb300 import fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    txt = open(os.path.join(ROOT, "include", "fa.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?(?:\w+\s+)*\w+\s*\*?\s*(fa_\w+)\s*\(", txt,
                                 flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(fa.LIB_PATH):
        from exact_attention_57_gb300 import build
        build.build_library()
    return fa.load()


def test_header_declares_the_entry_points():
    names = header_functions()
    assert set(names) == set(fa.EXPORTED), names


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), f"libfa.so does not export {name}"


def test_only_the_header_functions_are_exported(lib):
    """The library is built with hidden visibility: internal functions (here
    the launchers of the SIMT forward and of a tensor-core instantiation) are
    not in its dynamic symbol table, so a second build loaded in the same
    process (the debug library) cannot share their statics or symbols."""
    for internal in ("_ZN2fa11launch_simtERKNS_10SimtParamsEiP11CUstream_st",
                     "_ZN2fa19launch_tc_bf16_d128ERK14CUtensorMap_stS2_S2_S2_S2_RKNS_8TcParamsEiiP11CUstream_st"):
        with pytest.raises(AttributeError):
            getattr(lib, internal)


def test_version_and_strings(lib):
    assert fa.fa_version() == 10000
    assert fa.fa_status_string(0) == "FA_OK"
    assert fa.fa_status_string(1) == "FA_ERR_INVALID_ARG"
    assert fa.fa_status_string(2) == "FA_ERR_UNSUPPORTED"
    assert fa.fa_status_string(4) == "FA_ERR_DEVICE_TIMEOUT"
    assert fa.fa_status_string(99) == "FA_ERR_UNKNOWN"


# Fake, never-dereferenced device addresses (16-byte aligned, disjoint).
Q, K, V, O, L = 0x100000, 0x200000, 0x300000, 0x400000, 0x500000


def call(**kw):
    a = dict(q=Q, k=K, v=V, o=O, lse=L, B=1, H=1, Nq=16, Nk=16, d=64, scale=0.125,
             causal=0, dtype=fa.FA_DTYPE_BF16, stream=None)
    a.update(kw)
    return fa.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"], a["Nk"],
                     a["d"], a["scale"], a["causal"], a["dtype"], a["stream"])


@pytest.mark.parametrize("kw", [
    dict(q=None), dict(k=None), dict(v=None), dict(o=None), dict(lse=None),
    dict(B=0), dict(H=0), dict(Nq=0), dict(Nk=0), dict(d=0), dict(B=-3),
    dict(B=70000), dict(H=70000),
    dict(scale=float("nan")), dict(scale=float("inf")),
    dict(causal=2), dict(causal=-1), dict(dtype=4), dict(dtype=-1),
    dict(q=Q + 8), dict(o=O + 4), dict(lse=L + 2),
    dict(o=Q), dict(o=Q + 1024), dict(lse=O + 16), dict(lse=K + 64),
], ids=lambda kw: ",".join(f"{k}={v}" for k, v in kw.items()))
def test_invalid_arguments(lib, kw):
    assert call(**kw) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("B,H", [(65535, 65535), (65535, 32769), (32769, 65535)])
def test_plane_count_above_int32_is_refused(lib, B, H):
    """B * H above 2^31 - 1 planes is refused (the kernels index planes with
    32-bit ints).  The buffers are spaced 2^44 bytes apart so that only the
    plane count, not an overlap, can reject the call."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("host-only check: fake device addresses")
    far = [(i + 1) << 44 for i in range(5)]
    r = fa.fa_fwd(*far, B, H, 1, 1, 64, 0.125, 0, fa.FA_DTYPE_BF16, None)
    assert r == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [
    dict(dtype=fa.FA_DTYPE_BF16, d=16), dict(dtype=fa.FA_DTYPE_BF16, d=96),
    dict(dtype=fa.FA_DTYPE_BF16, d=512), dict(dtype=fa.FA_DTYPE_F32, d=256),
    dict(dtype=fa.FA_DTYPE_F32, d=48), dict(dtype=fa.FA_DTYPE_F32_SIMT, d=129),
    dict(dtype=fa.FA_DTYPE_F16, d=96), dict(dtype=fa.FA_DTYPE_F16, d=192),
], ids=lambda kw: ",".join(f"{k}={v}" for k, v in kw.items()))
def test_unsupported_problems(lib, kw):
    """Valid problems outside the compiled set are refused, not attempted."""
    assert call(**kw) == fa.FA_ERR_UNSUPPORTED


def test_host_variant_rejects_null_host_buffers(lib):
    r = fa.fa_fwd_host(None, 0x10, 0x20, 0x30, 0x40, Q, K, V, O, L, 1, 1, 16, 16, 64, 0.1, 0,
                       fa.FA_DTYPE_BF16, None)
    assert r == fa.FA_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError):
        fa.load(str(tmp_path / "missing.so"))


def test_splitkv_workspace_size(lib):
    """num_splits * B * H * Nq * (d + 1) floats, each part rounded up to 256 B."""
    def want(B, H, Nq, d, s):
        r = s * B * H * Nq
        up = lambda n: (n + 255) // 256 * 256
        return up(r * d * 4) + up(r * 4)
    for args in [(1, 1, 1, 64, 1), (2, 8, 3001, 128, 7), (1, 32, 128, 64, 64)]:
        assert fa.fa_fwd_splitkv_workspace(*args) == want(*args)
    for bad in [(0, 1, 1, 64, 2), (1, 1, 1, 64, 0), (1, 1, 1, 64, 65), (1, 1, 0, 64, 2)]:
        assert fa.fa_fwd_splitkv_workspace(*bad) == 0


@pytest.mark.parametrize("kw", [
    dict(num_splits=-1), dict(num_splits=65),
    dict(num_splits=4, ws=None), dict(num_splits=4, ws=0x600010),
    dict(num_splits=4, ws_bytes=100), dict(num_splits=4, ws=Q),
], ids=lambda kw: ",".join(f"{k}={v}" for k, v in kw.items()))
def test_splitkv_invalid_arguments(lib, kw):
    """Bad split counts and missing, misaligned, short or overlapping
    workspaces are refused before any device work."""
    ns = kw.get("num_splits", 4)
    need = fa.fa_fwd_splitkv_workspace(1, 1, 16, 64, max(1, min(ns, 64)))
    ws = kw.get("ws", 0x600000)
    wsb = kw.get("ws_bytes", need)
    r = fa.fa_fwd_splitkv(Q, K, V, O, L, 1, 1, 16, 16, 64, 0.125, 0, fa.FA_DTYPE_BF16, ns,
                          ws, wsb, None)
    assert r == fa.FA_ERR_INVALID_ARG


def test_splitkv_refuses_simt(lib):
    r = fa.fa_fwd_splitkv(Q, K, V, O, L, 1, 1, 16, 16, 64, 0.125, 0, fa.FA_DTYPE_F32_SIMT, 4,
                          0x600000, 1 << 20, None)
    assert r == fa.FA_ERR_UNSUPPORTED


CUQ, CUK = 0x700000, 0x700100


@pytest.mark.parametrize("kw", [
    dict(cu_q=None), dict(cu_k=None), dict(cu_q=CUQ + 2), dict(B=0), dict(max_q=0),
    dict(max_q=17), dict(total_q=0), dict(d=0), dict(o=Q),
], ids=lambda kw: ",".join(f"{k}={v}" for k, v in kw.items()))
def test_varlen_invalid_arguments(lib, kw):
    a = dict(cu_q=CUQ, cu_k=CUK, B=2, max_q=8, total_q=16, total_k=16, d=64, o=O)
    a.update(kw)
    r = fa.fa_fwd_varlen(Q, K, V, a["o"], L, a["cu_q"], a["cu_k"], a["B"], 2, a["total_q"],
                         a["total_k"], a["max_q"], a["d"], 0.125, 1, fa.FA_DTYPE_BF16, None)
    assert r == fa.FA_ERR_INVALID_ARG


def test_varlen_refuses_simt_and_unsupported_dims(lib):
    r = fa.fa_fwd_varlen(Q, K, V, O, L, CUQ, CUK, 2, 2, 16, 16, 8, 64, 0.125, 1,
                         fa.FA_DTYPE_F32_SIMT, None)
    assert r == fa.FA_ERR_UNSUPPORTED
    r = fa.fa_fwd_varlen(Q, K, V, O, L, CUQ, CUK, 2, 2, 16, 16, 8, 96, 0.125, 1,
                         fa.FA_DTYPE_BF16, None)
    assert r == fa.FA_ERR_UNSUPPORTED


DO, DQ, DK, DV, WS = 0x800000, 0x900000, 0xA00000, 0xB00000, 0xC00000


@pytest.mark.parametrize("shape,causal,dtype,want", [
    # persistent (up to 16 waves of query tiles): one CTA per SM while there
    # are more query tiles than SMs; planes per group: 48 MB of K and V
    # (2 * Nk * d * element size per plane)
    ((2, 8, 3001, 3001, 128), True, fa.FA_DTYPE_BF16, (152, 16, 0)),
    ((2, 16, 8192, 8192, 128), True, fa.FA_DTYPE_BF16, (152, 12, 0)),
    ((2, 4, 1024, 1024, 64), True, fa.FA_DTYPE_BF16, (64, 8, 0)),      # 64 query tiles
    ((1, 1, 128, 128, 128), False, fa.FA_DTYPE_F16, (1, 1, 0)),
    # blocked (more than 16 waves): the makespan model's query tiles per CTA
    ((8, 32, 8192, 8192, 128), True, fa.FA_DTYPE_BF16, (4096, 1, 4)),
    ((4, 16, 8192, 8192, 128), False, fa.FA_DTYPE_F16, (1024, 1, 4)),
    ((8, 32, 8192, 8192, 64), True, fa.FA_DTYPE_BF16, (4096, 1, 4)),
    # one CTA per query tile for the fp32 dtypes
    ((4, 4, 4096, 4096, 64), False, fa.FA_DTYPE_F32, (0, 1, 0)),
    ((4, 4, 4096, 4096, 64), False, fa.FA_DTYPE_F32_SIMT, (0, 1, 0)),
])
def test_fwd_schedule_choice(lib, shape, causal, dtype, want):
    """The schedule of fa_fwd's 16-bit forward (host logic only)."""
    B, H, Nq, Nk, d = shape
    assert fa.fa_fwd_schedule(B, H, Nq, Nk, d, causal, dtype, 152) == (fa.FA_OK,) + want


def test_fwd_schedule_edges(lib):
    bf = fa.FA_DTYPE_BF16
    assert fa.fa_fwd_schedule(0, 1, 128, 128, 64, 0, bf, 152)[0] == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_schedule(1, 1, 128, 128, 64, 0, bf, 0)[0] == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_schedule(1, 1, 128, 128, 128, 1, bf, 1) == (fa.FA_OK, 1, 1, 0)


@pytest.mark.parametrize("planes,n,ctas,group_heads,block", [
    (256, 64, 152, 12, 0), (16, 24, 152, 16, 0), (8, 8, 64, 8, 0), (1, 1, 1, 1, 0),
    (7, 5, 3, 2, 0), (5, 3, 15, 5, 0), (12, 9, 100, 5, 0), (3, 100, 7, 1, 0), (300, 2, 151, 17, 0),
    (1, 1000, 152, 1, 0),
    (256, 64, 4096, 1, 4), (16, 24, 192, 1, 2), (7, 5, 14, 1, 3), (3, 9, 27, 1, 1),
    (2, 7, 4, 1, 4), (5, 1, 5, 1, 2),
])
def test_fwd_schedule_deals_every_item_once(lib, planes, n, ctas, group_heads, block):
    """Every item goes to exactly one CTA, whatever the grid, group and block
    sizes (the mapping the kernels themselves use, evaluated on the host)."""
    assert fa.fa_fwd_schedule_covers(planes, n, ctas, group_heads, block)


def test_fwd_schedule_covers_rejects_bad_sizes(lib):
    for args in [(0, 1, 1, 1, 0), (1, 0, 1, 1, 0), (1, 1, 0, 1, 0), (1, 1, 1, 0, 0),
                 (2, 2, 5, 1, 0), (4, 8, 7, 1, 4), (1, 1, 1, 1, -1)]:
        assert not fa.fa_fwd_schedule_covers(*args)


def test_fwd_schedule_hook_range(lib):
    """The testing aid takes 0 (automatic) or positive counts."""
    for args in [(-1, 0, 0), (0, -1, 0), (0, 0, -3)]:
        assert fa.fa_set_fwd_schedule(*args) == fa.FA_ERR_INVALID_ARG
    try:
        assert fa.fa_set_fwd_schedule(0, 0, 2) == fa.FA_OK
        assert fa.fa_fwd_schedule(2, 8, 3001, 3001, 128, 1, fa.FA_DTYPE_BF16, 152)[1:] == (
            16 * 12, 1, 2)
        assert fa.fa_set_fwd_schedule(7, 3, 0) == fa.FA_OK
        assert fa.fa_fwd_schedule(8, 32, 8192, 8192, 128, 1, fa.FA_DTYPE_BF16, 152)[1:] == (
            7, 3, 0)
    finally:
        assert fa.fa_set_fwd_schedule(0, 0, 0) == fa.FA_OK
    st, ctas, groups, block = fa.fa_fwd_schedule(8, 32, 8192, 8192, 128, 1, fa.FA_DTYPE_BF16, 152)
    assert (st, ctas, groups, block) == (fa.FA_OK, 4096, 1, 4)


def test_bwd_workspace_size(lib):
    """B*H*Nq*max(d, 64) floats (dq accumulator rows of the gradient kernel's
    head dim) plus two floats per padded query row, parts rounded up to 256
    bytes."""
    up = lambda n: (n + 255) // 256 * 256
    for B, H, Nq, d in [(1, 1, 1, 64), (2, 16, 8192, 128), (1, 3, 300, 64), (2, 3, 300, 32)]:
        pad = (Nq + 127) // 128 * 128
        assert (fa.fa_bwd_workspace(B, H, Nq, d)
                == up(B * H * Nq * max(d, 64) * 4) + 2 * up(B * H * pad * 4))
    for bad in [(0, 1, 1, 64), (1, 0, 1, 64), (1, 1, 0, 64), (1, 1, 1, 0)]:
        assert fa.fa_bwd_workspace(*bad) == 0


def call_bwd(**kw):
    a = dict(q=Q, k=K, v=V, o=O, lse=L, do=DO, dq=DQ, dk=DK, dv=DV, B=1, H=1, Nq=16, Nk=16, d=64,
             scale=0.125, causal=0, dtype=fa.FA_DTYPE_BF16, ws=WS, ws_bytes=None)
    a.update(kw)
    if a["ws_bytes"] is None:
        a["ws_bytes"] = fa.fa_bwd_workspace(a["B"], a["H"], max(a["Nq"], 1), max(a["d"], 1))
    return fa.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"],
                     a["dv"], a["B"], a["H"], a["Nq"], a["Nk"], a["d"], a["scale"], a["causal"],
                     a["dtype"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw", [
    dict(do=None), dict(dq=None), dict(dk=None), dict(dv=None), dict(ws=None),
    dict(q=None), dict(lse=None), dict(Nq=0), dict(Nk=0), dict(scale=float("nan")),
    dict(causal=3), dict(dtype=7),
    dict(do=DO + 8), dict(dq=DQ + 4), dict(dk=DK + 2), dict(ws=WS + 16), dict(ws_bytes=1000),
    dict(dq=Q), dict(dk=V + 64), dict(dv=DO), dict(dq=DK), dict(ws=DV), dict(dv=L),
], ids=lambda kw: ",".join(f"{k}={v}" for k, v in kw.items()))
def test_bwd_invalid_arguments(lib, kw):
    """Missing, misaligned, short or overlapping buffers are refused before
    any device work."""
    assert call_bwd(**kw) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [
    dict(dtype=fa.FA_DTYPE_F32, d=192), dict(dtype=fa.FA_DTYPE_F32_SIMT, d=256), dict(d=96),
    dict(dtype=fa.FA_DTYPE_F16, d=256), dict(d=256),
], ids=lambda kw: ",".join(f"{k}={v}" for k, v in kw.items()))
def test_bwd_unsupported_problems(lib, kw):
    assert call_bwd(**kw) == fa.FA_ERR_UNSUPPORTED


def test_staged_workspace_size(lib):
    """fp32: 2*B*H*Nk*d bf16 values (K_hi, K_lo) + B*H*d*ceil(Nk/128)*128
    floats (V^T), parts rounded up to 256 bytes; other dtypes stage nothing."""
    up = lambda n: (n + 255) // 256 * 256
    for B, H, Nk, d in [(1, 1, 1, 64), (4, 4, 4096, 64), (2, 3, 300, 128), (1, 2, 77, 32)]:
        pad = (Nk + 127) // 128 * 128
        assert (fa.fa_fwd_staged_workspace(B, H, Nk, d, fa.FA_DTYPE_F32)
                == 2 * up(B * H * Nk * d * 2) + up(B * H * d * pad * 4))
    for dt in (fa.FA_DTYPE_BF16, fa.FA_DTYPE_F16, fa.FA_DTYPE_F32_SIMT):
        assert fa.fa_fwd_staged_workspace(1, 1, 128, 64, dt) == 0
    assert fa.fa_fwd_staged_workspace(0, 1, 128, 64, fa.FA_DTYPE_F32) == 0


@pytest.mark.parametrize("kw", [
    dict(ws=None), dict(ws=WS + 16), dict(ws_bytes=1000), dict(ws=Q), dict(ws=O - 64),
    dict(q=None), dict(Nk=0), dict(d=0),
], ids=lambda kw: ",".join(f"{k}={v}" for k, v in kw.items()))
def test_staged_invalid_arguments(lib, kw):
    """fp32 staging refuses a missing, misaligned, short or overlapping
    workspace before any device work."""
    a = dict(q=Q, ws=WS, ws_bytes=None, Nk=16, d=64)
    a.update(kw)
    wsb = a["ws_bytes"]
    if wsb is None:
        wsb = fa.fa_fwd_staged_workspace(1, 1, max(a["Nk"], 1), max(a["d"], 1), fa.FA_DTYPE_F32)
    r = fa.fa_fwd_staged(a["q"], K, V, O, L, 1, 1, 16, a["Nk"], a["d"], 0.125, 0,
                         fa.FA_DTYPE_F32, a["ws"], wsb, None)
    assert r == fa.FA_ERR_INVALID_ARG


def test_bwd_varlen_workspace_size(lib):
    up = lambda n: (n + 255) // 256 * 256
    for B, H, tq, mq, d in [(1, 1, 1, 1, 64), (3, 4, 1000, 700, 128), (2, 2, 300, 129, 32)]:
        pad = (mq + 127) // 128 * 128
        assert (fa.fa_bwd_varlen_workspace(B, H, tq, mq, d)
                == up(tq * H * max(d, 64) * 4) + 2 * up(H * B * pad * 4))
    assert fa.fa_bwd_varlen_workspace(0, 1, 10, 10, 64) == 0


@pytest.mark.parametrize("kw", [
    dict(cu_q=None), dict(cu_k=CUK + 2), dict(B=0), dict(max_q=0), dict(max_q=17), dict(max_k=17),
    dict(ws=None), dict(ws=WS + 16), dict(ws_bytes=64), dict(dq=Q), dict(dv=DO + 16),
], ids=lambda kw: ",".join(f"{k}={v}" for k, v in kw.items()))
def test_bwd_varlen_invalid_arguments(lib, kw):
    a = dict(cu_q=CUQ, cu_k=CUK, B=2, max_q=8, max_k=8, ws=WS, ws_bytes=None, dq=DQ, dv=DV)
    a.update(kw)
    wsb = a["ws_bytes"]
    if wsb is None:
        wsb = fa.fa_bwd_varlen_workspace(2, 2, 16, 8, 64)
    r = fa.fa_bwd_varlen(Q, K, V, O, L, DO, a["dq"], DK, a["dv"], a["cu_q"], a["cu_k"], a["B"], 2,
                         16, 16, a["max_q"], a["max_k"], 64, 0.125, 1, fa.FA_DTYPE_BF16, a["ws"],
                         wsb, None)
    assert r == fa.FA_ERR_INVALID_ARG
