"""ctypes binding of ``libfa.so`` (the C ABI in include/fa.h).

The ``fa_*`` functions mirror the C entry points one to one and only marshal
arguments.  ``attention``, ``attention_varlen`` and ``attention_backward`` are
convenience wrappers for torch tensors: they allocate outputs and workspaces
with torch (device memory is the only thing torch provides here) and call the
C entry points.

There is no fallback: if the library is missing or its call fails, these
functions raise.
"""
from __future__ import annotations

import ctypes
import math
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_DEVICE_TIMEOUT = 4

FA_DTYPE_BF16 = 0
FA_DTYPE_F32 = 1
FA_DTYPE_F32_SIMT = 2
FA_DTYPE_F16 = 3

EXPORTED = ("fa_fwd", "fa_fwd_host", "fa_fwd_status", "fa_status_string", "fa_version",
            "fa_set_test_hooks", "fa_debug_build", "fa_set_debug_lse_shrink",
            "fa_set_fwd_schedule", "fa_fwd_schedule", "fa_fwd_schedule_covers",
            "fa_fwd_noalloc",
            "fa_fwd_splitkv", "fa_fwd_splitkv_workspace",
            "fa_fwd_varlen", "fa_bwd", "fa_bwd_workspace", "fa_fwd_staged",
            "fa_fwd_staged_workspace", "fa_bwd_varlen", "fa_bwd_varlen_workspace")

_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fa_status_string(status)} ({status})")


def load(path: str | None = None):
    """Load libfa.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with exact_attention_57_gb300.build")
    lib = ctypes.CDLL(p)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
    lib.fa_fwd.restype = i
    lib.fa_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp,
                                   ctypes.POINTER(i)]
    lib.fa_fwd_noalloc.restype = i
    lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, i, vp,
                                   ctypes.c_ulonglong, vp]
    lib.fa_fwd_splitkv.restype = i
    lib.fa_fwd_splitkv_workspace.argtypes = [i, i, i, i, i]
    lib.fa_fwd_splitkv_workspace.restype = ctypes.c_ulonglong
    lib.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp]
    lib.fa_fwd_varlen.restype = i
    lib.fa_fwd_staged.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp,
                                  ctypes.c_ulonglong, vp]
    lib.fa_fwd_staged.restype = i
    lib.fa_fwd_staged_workspace.argtypes = [i, i, i, i, i]
    lib.fa_fwd_staged_workspace.restype = ctypes.c_ulonglong
    lib.fa_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i,
                                  f, i, i, vp, ctypes.c_ulonglong, vp]
    lib.fa_bwd_varlen.restype = i
    lib.fa_bwd_varlen_workspace.argtypes = [i, i, i, i, i]
    lib.fa_bwd_varlen_workspace.restype = ctypes.c_ulonglong
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp,
                           ctypes.c_ulonglong, vp]
    lib.fa_bwd.restype = i
    lib.fa_bwd_workspace.argtypes = [i, i, i, i]
    lib.fa_bwd_workspace.restype = ctypes.c_ulonglong
    lib.fa_fwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                i, i, i, i, i, f, i, i, vp]
    lib.fa_fwd_host.restype = i
    lib.fa_fwd_status.argtypes = [vp, ctypes.POINTER(i)]
    lib.fa_fwd_status.restype = i
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_version.argtypes = []
    lib.fa_version.restype = i
    lib.fa_set_test_hooks.argtypes = [i, ctypes.c_ulonglong]
    lib.fa_set_test_hooks.restype = i
    lib.fa_debug_build.argtypes = []
    lib.fa_debug_build.restype = i
    lib.fa_set_debug_lse_shrink.argtypes = [ctypes.c_longlong]
    lib.fa_set_debug_lse_shrink.restype = i
    lib.fa_set_fwd_schedule.argtypes = [i, i, i]
    lib.fa_set_fwd_schedule.restype = i
    lib.fa_fwd_schedule.argtypes = [i] * 8 + [ctypes.POINTER(i)] * 3
    lib.fa_fwd_schedule.restype = i
    lib.fa_fwd_schedule_covers.argtypes = [i] * 5
    lib.fa_fwd_schedule_covers.restype = i
    if path is None:
        _lib = lib
    return lib


def fa_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype, stream) -> int:
    """Raw C call; pointers and stream are integers (0 = NULL)."""
    return load().fa_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, float(scale), int(causal),
                         int(dtype), stream)


def fa_fwd_noalloc(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype, stream,
                   wait: bool = True):
    """Raw C call of the entry point that allocates no device memory.

    With wait=True the call synchronises the stream and returns
    (status, raw status word); with wait=False it only enqueues and returns
    (status, None)."""
    word = ctypes.c_int(0)
    st = load().fa_fwd_noalloc(q, k, v, o, lse, B, H, Nq, Nk, d, float(scale), int(causal),
                               int(dtype), stream, ctypes.byref(word) if wait else None)
    return st, (word.value if wait else None)


def fa_fwd_splitkv(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype, num_splits,
                   workspace, workspace_bytes, stream) -> int:
    return load().fa_fwd_splitkv(q, k, v, o, lse, B, H, Nq, Nk, d, float(scale), int(causal),
                                 int(dtype), int(num_splits), workspace, int(workspace_bytes),
                                 stream)


def fa_fwd_splitkv_workspace(B, H, Nq, d, num_splits) -> int:
    return load().fa_fwd_splitkv_workspace(B, H, Nq, d, num_splits)


def fa_fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, H, total_q, total_k,
                  max_seqlen_q, d, scale, causal, dtype, stream) -> int:
    return load().fa_fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, H, total_q,
                                total_k, max_seqlen_q, d, float(scale), int(causal), int(dtype),
                                stream)


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                     scale: float | None = None, causal: bool = False, out=None, lse=None,
                     stream=None):
    """Packed sequences: q [total_q, H, d], k/v [total_k, H, d], cu_seqlens
    int32 CUDA tensors of B+1 offsets.  Returns (o [total_q, H, d],
    lse [H, total_q])."""
    import torch
    total_q, H, d = q.shape
    total_k = k.shape[0]
    if k.shape[1:] != (H, d) or v.shape != k.shape:
        raise ValueError("q [total_q,H,d], k and v [total_k,H,d] expected")
    if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_k.dtype != torch.int32:
        raise ValueError("cu_seqlens must be int32")
    B = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != B + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k need the same batch size")
    code = _dtype_code(q, "tc")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((H, total_q), device=q.device, dtype=torch.float32)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    with torch.cuda.device(q.device):
        st = fa_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                           lse.data_ptr(), cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), B,
                           H, total_q, total_k, max_seqlen_q, d, scale, int(bool(causal)), code,
                           stream)
    if st != FA_OK:
        raise FaError(st, "fa_fwd_varlen")
    return out, lse


def fa_fwd_staged(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype, workspace,
                  workspace_bytes, stream) -> int:
    return load().fa_fwd_staged(q, k, v, o, lse, B, H, Nq, Nk, d, float(scale), int(causal),
                                int(dtype), workspace, int(workspace_bytes), stream)


def fa_fwd_staged_workspace(B, H, Nk, d, dtype) -> int:
    return load().fa_fwd_staged_workspace(B, H, Nk, d, dtype)


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, scale, causal, dtype,
           workspace, workspace_bytes, stream) -> int:
    return load().fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, float(scale),
                         int(causal), int(dtype), workspace, int(workspace_bytes), stream)


def fa_bwd_workspace(B, H, Nq, d) -> int:
    return load().fa_bwd_workspace(B, H, Nq, d)


def attention_backward(q, k, v, out, lse, dout, scale: float | None = None,
                       causal: bool = False, dq=None, dk=None, dv=None, workspace=None,
                       stream=None):
    """Gradients (dq, dk, dv) of attention() for the upstream gradient dout.

    q, k, v, dout, out: contiguous bf16 / fp16 / fp32 CUDA tensors as for
    attention() (fp32 runs the CUDA-core backward, head dim up to 128);
    out and lse are that forward's outputs.  The workspace (fa_bwd_workspace
    bytes) is allocated with torch unless given.  Raises FaError on failure."""
    import torch
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    for t in (k, v, out, dout):
        if t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError("q, k, v, out, dout: contiguous tensors of one dtype")
    if out.shape != q.shape or dout.shape != q.shape or v.shape != k.shape:
        raise ValueError("shape mismatch")
    # fp32 gradients come from the CUDA-core backward whichever fp32 forward
    # ran; its dtype code admits every head dim up to 128
    code = _dtype_code(q, "simt" if q.dtype == torch.float32 else "tc")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws_bytes = fa_bwd_workspace(B, H, Nq, d)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    with torch.cuda.device(q.device):
        st = fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                    dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Nq, Nk,
                    d, scale, int(bool(causal)), code, workspace.data_ptr(),
                    workspace.numel() * workspace.element_size(), stream)
    if st != FA_OK:
        raise FaError(st, "fa_bwd")
    return dq, dk, dv


def fa_bwd_varlen(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, B, H, total_q,
                  total_k, max_seqlen_q, max_seqlen_k, d, scale, causal, dtype, workspace,
                  workspace_bytes, stream) -> int:
    return load().fa_bwd_varlen(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, B,
                                H, total_q, total_k, max_seqlen_q, max_seqlen_k, d, float(scale),
                                int(causal), int(dtype), workspace, int(workspace_bytes), stream)


def fa_bwd_varlen_workspace(B, H, total_q, max_seqlen_q, d) -> int:
    return load().fa_bwd_varlen_workspace(B, H, total_q, max_seqlen_q, d)


def attention_backward_varlen(q, k, v, out, lse, dout, cu_seqlens_q, cu_seqlens_k,
                              max_seqlen_q: int, max_seqlen_k: int, scale: float | None = None,
                              causal: bool = False, stream=None):
    """Gradients (dq, dk, dv) of attention_varlen() for the upstream gradient
    dout (token-major [total_q, H, d]).  Raises FaError on failure."""
    import torch
    total_q, H, d = q.shape
    total_k = k.shape[0]
    B = cu_seqlens_q.numel() - 1
    code = _dtype_code(q, "tc")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = fa_bwd_varlen_workspace(B, H, total_q, max_seqlen_q, d)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    with torch.cuda.device(q.device):
        st = fa_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                           dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                           cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), B, H, total_q,
                           total_k, max_seqlen_q, max_seqlen_k, d, scale, int(bool(causal)), code,
                           ws.data_ptr(), ws_bytes, stream)
    if st != FA_OK:
        raise FaError(st, "fa_bwd_varlen")
    return dq, dk, dv


def fa_fwd_host(q_h, k_h, v_h, o_h, lse_h, q_d, k_d, v_d, o_d, lse_d,
                B, H, Nq, Nk, d, scale, causal, dtype, stream) -> int:
    return load().fa_fwd_host(q_h, k_h, v_h, o_h, lse_h, q_d, k_d, v_d, o_d, lse_d,
                              B, H, Nq, Nk, d, float(scale), int(causal), int(dtype), stream)


def fa_fwd_status(stream=None):
    """Returns (status, raw device status word)."""
    word = ctypes.c_int(0)
    st = load().fa_fwd_status(stream, ctypes.byref(word))
    return st, word.value


def fa_status_string(status: int) -> str:
    try:
        return load().fa_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def fa_version() -> int:
    return load().fa_version()


def fa_set_test_hooks(skip_v_load: int = 0, wait_limit_ns: int = 0) -> int:
    return load().fa_set_test_hooks(int(skip_v_load), int(wait_limit_ns))


def fa_set_fwd_schedule(ctas: int = 0, group_heads: int = 0, block_items: int = 0) -> int:
    """Testing aid: force the 16-bit forward's schedule (0 = automatic)."""
    return load().fa_set_fwd_schedule(int(ctas), int(group_heads), int(block_items))


def fa_fwd_schedule(B: int, H: int, Nq: int, Nk: int, d: int, causal: bool, dtype: int,
                    num_sms: int):
    """(status, CTAs, planes per group, items per CTA of the blocked schedule
    or 0) of fa_fwd's schedule on a GPU with num_sms SMs (host-only)."""
    c, g, b = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    st = load().fa_fwd_schedule(int(B), int(H), int(Nq), int(Nk), int(d), int(bool(causal)),
                                int(dtype), int(num_sms), ctypes.byref(c), ctypes.byref(g),
                                ctypes.byref(b))
    return st, c.value, g.value, b.value


def fa_fwd_schedule_covers(planes: int, n: int, ctas: int, group_heads: int,
                           block_items: int = 0) -> bool:
    """Host-only check that the schedule deals every item exactly once."""
    return bool(load().fa_fwd_schedule_covers(int(planes), int(n), int(ctas), int(group_heads),
                                              int(block_items)))


# --------------------------------------------------------------- torch helpers
def _dtype_code(t, impl: str) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        if impl != "tc":
            raise ValueError("bf16 inputs run on the tensor-core kernel only")
        return FA_DTYPE_BF16
    if t.dtype == torch.float16:
        if impl != "tc":
            raise ValueError("fp16 inputs run on the tensor-core kernel only")
        return FA_DTYPE_F16
    if t.dtype == torch.float32:
        return FA_DTYPE_F32 if impl == "tc" else FA_DTYPE_F32_SIMT
    raise ValueError(f"unsupported dtype {t.dtype}")


def attention(q, k, v, scale: float | None = None, causal: bool = False, impl: str = "tc",
              out=None, lse=None, stream=None, num_splits: int | None = None,
              staged: bool = False):
    """O, LSE for contiguous CUDA tensors q [B,H,Nq,d], k/v [B,H,Nk,d].

    impl "tc": bf16 / fp16 -> tcgen05 kind::f16, fp32 -> tcgen05 kind::tf32;
    impl "simt": fp32 only, plain fp32 kernel.  num_splits (tensor-core
    dtypes): split each query tile's key range into that many chunks (0 =
    automatic) through fa_fwd_splitkv, with a torch-allocated workspace.
    staged (fp32, impl "tc"): run fa_fwd_staged, converting K and V once per
    call into a torch-allocated workspace (scores as three bf16 products of
    split operands instead of fa_fwd's three tf32 ones).  Raises FaError on failure.
    """
    import torch
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("attention() needs CUDA tensors")
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("q [B,H,Nq,d], k and v [B,H,Nk,d] expected")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape[0] != B or k.shape[1] != H or k.shape[3] != d:
        raise ValueError("k/v shape does not match q")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("contiguous [B,H,N,d] tensors expected")
    code = _dtype_code(q, impl)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share a dtype")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), device=q.device, dtype=torch.float32)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    with torch.cuda.device(q.device):
        if staged and code == FA_DTYPE_F32:
            ws_bytes = fa_fwd_staged_workspace(B, H, Nk, d, code)
            ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
            st = fa_fwd_staged(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                               lse.data_ptr(), B, H, Nq, Nk, d, scale, int(bool(causal)), code,
                               ws.data_ptr(), ws_bytes, stream)
            where = "fa_fwd_staged"
        elif num_splits is None:
            st = fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                        lse.data_ptr(), B, H, Nq, Nk, d, scale, int(bool(causal)), code, stream)
            where = "fa_fwd"
        else:
            nws = num_splits if num_splits > 0 else 64
            ws_bytes = fa_fwd_splitkv_workspace(B, H, Nq, d, nws)
            ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
            st = fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                lse.data_ptr(), B, H, Nq, Nk, d, scale, int(bool(causal)), code,
                                num_splits, ws.data_ptr(), ws_bytes, stream)
            where = "fa_fwd_splitkv"
    if st != FA_OK:
        raise FaError(st, where)
    return out, lse
