"""Python binding of libfa.so: row softmax and fused attention forward on GB300.

This module only marshals arguments: it passes device pointers of torch
tensors, sizes and the current CUDA stream to the C-ABI entry points declared
in ``include/fa.h`` and raises on a non-zero return code.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback.  If the
compiled library is missing, importing the C functions fails loudly.

Raw C-ABI names (same names, same argument order, ints and pointers only):
``fa_softmax_rows``, ``fa_attention_fwd``, ``fa_attention_fwd_varlen``,
``fa_attention_fwd_splitkv``, ``fa_attention_fwd_splitkv_varlen``, ``fa_splitkv_num_splits``, ``fa_attention_fwd_splitkv_noalloc``,
``fa_attention_fwd_f32``, ``fa_attention_bwd``, ``fa_attention_bwd_varlen``,
``fa_attention_bwd_atomic``, ``fa_attention_bwd_atomic_workspace_bytes``,
``fa_attention_bwd_atomic_varlen``, ``fa_attention_bwd_atomic_varlen_workspace_bytes``,
``fa_attention_fwd_fp8``, ``fa_attention_fwd_fp8_varlen``,
``fa_attention_fp8_workspace_bytes``, ``fa_attention_fwd_host``,
``fa_attention_host_workspace_bytes``,
``fa_set_stream``, ``fa_get_stream``, ``fa_get_device_error``, ``fa_strerror``,
``fa_version``, ``fa_debug_expire_next_wait``.
Tensor-level helpers: :func:`softmax_rows`, :func:`attention_fwd`,
:func:`attention_fwd_splitkv`, :func:`attention_bwd`, :func:`attention_fwd_fp8`.
"""
from __future__ import annotations

import ctypes
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libfa.so")

FA_OK = 0
FA_ERR_NULL_POINTER = -1
FA_ERR_BAD_SIZE = -2
FA_ERR_UNSUPPORTED = -3
FA_ERR_MISALIGNED = -4
FA_ERR_CUDA = -5
FA_ERR_TOO_LARGE = -6
FA_ERR_NO_DEVICE = -7
FA_DEVERR_WAIT_TIMEOUT = 0x1
FA_DEVERR_BAD_SEQLENS = 0x2
FA_ERR_SCRATCH_LIMIT = -8
FA_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024   # static scratch of the _noalloc entry point

_lib = None


class FaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where} failed: {code} ({strerror(code)})")


def build(force: bool = False) -> str:
    """Compile the CUDA sources into _build/libfa.so (nvcc, sm_103a)."""
    from . import _build
    return _build.build(force=force)


def lib():
    """The loaded libfa.so (ctypes.CDLL).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libfa.so not built ({LIB_PATH} missing); run "
                              "online_softmax_06_gb300.build() first")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        L.fa_softmax_rows.argtypes = [vp, vp, i64, i64]
        L.fa_attention_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i32, vp]
        L.fa_attention_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i64, i32, f32,
                                              i32, vp]
        L.fa_attention_fwd_f32.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i32, vp]
        L.fa_attention_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32,
                                               i32, i32, vp, vp]
        L.fa_splitkv_num_splits.argtypes = [i32, i32, i32, i32, i32]
        L.fa_attention_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i32, vp,
                                           vp, i64]
        L.fa_attention_fp8_workspace_bytes.argtypes = [i32, i32, i32, i32]
        L.fa_attention_fp8_workspace_bytes.restype = i64
        L.fa_attention_fwd_host.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i32, vp,
                                            i64]
        L.fa_attention_host_workspace_bytes.argtypes = [i32, i32, i32, i32]
        L.fa_attention_host_workspace_bytes.restype = i64
        L.fa_attention_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                       i32, f32, i32]
        L.fa_attention_fwd_splitkv_varlen.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                      i64, i64, i32, f32, i32, i32, vp, vp, vp,
                                                      vp]
        L.fa_attention_fwd_fp8_varlen.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i64, i32, f32,
                                                  i32, vp, vp, vp, i64]
        L.fa_attention_fp8_varlen_workspace_bytes.argtypes = [i32, i32, i32, i64, i32]
        L.fa_attention_fp8_varlen_workspace_bytes.restype = i64
        L.fa_attention_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32,
                                              i32, i64, i32, f32, i32, vp]
        L.fa_attention_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                       i32, f32, i32, i32]
        L.fa_attention_bwd_atomic.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32,
                                              i32, i32, f32, i32, vp, i64]
        L.fa_attention_bwd_atomic_workspace_bytes.argtypes = [i32, i32, i32, i32]
        L.fa_attention_bwd_atomic_workspace_bytes.restype = i64
        L.fa_attention_bwd_atomic_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                                     i32, i32, i64, i32, f32, i32, vp, vp, i64]
        L.fa_attention_bwd_atomic_varlen_workspace_bytes.argtypes = [i32, i32, i32, i64, i32]
        L.fa_attention_bwd_atomic_varlen_workspace_bytes.restype = i64
        L.fa_set_stream.argtypes = [vp]
        L.fa_get_stream.argtypes = []
        L.fa_get_stream.restype = vp
        L.fa_get_device_error.argtypes = []
        L.fa_strerror.argtypes = [i32]
        L.fa_strerror.restype = ctypes.c_char_p
        L.fa_version.argtypes = []
        L.fa_debug_expire_next_wait.argtypes = [i64]
        for name in ("fa_softmax_rows", "fa_attention_fwd", "fa_attention_fwd_varlen",
                     "fa_attention_fwd_f32", "fa_attention_fwd_splitkv", "fa_splitkv_num_splits",
                     "fa_attention_fwd_splitkv_noalloc", "fa_attention_bwd",
                     "fa_attention_bwd_varlen", "fa_attention_bwd_atomic",
                     "fa_attention_bwd_atomic_varlen",
                     "fa_attention_fwd_splitkv_varlen",
                     "fa_attention_fwd_fp8", "fa_attention_fwd_fp8_varlen",
                     "fa_attention_fwd_host",
                     "fa_set_stream", "fa_get_device_error", "fa_version",
                     "fa_debug_expire_next_wait"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def strerror(code: int) -> str:
    try:
        return lib().fa_strerror(int(code)).decode()
    except ImportError:
        return "libfa.so not loaded"


def _check(rc: int, where: str) -> None:
    if rc != FA_OK:
        raise FaError(rc, where)


# ---- raw C-ABI wrappers (same names as include/fa.h) -------------------------

def fa_softmax_rows(x_ptr: int, y_ptr: int, rows: int, N: int) -> int:
    return lib().fa_softmax_rows(x_ptr, y_ptr, rows, N)


def fa_attention_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, cu_seqlens) -> int:
    return lib().fa_attention_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, cu_seqlens)


def fa_attention_fwd_varlen(q, k, v, o, lse, B, H, N, total, d, scale, causal,
                            cu_seqlens) -> int:
    return lib().fa_attention_fwd_varlen(q, k, v, o, lse, B, H, N, total, d, scale, causal,
                                         cu_seqlens)


def fa_attention_fwd_f32(q, k, v, o, lse, B, H, N, d, scale, causal, cu_seqlens) -> int:
    return lib().fa_attention_fwd_f32(q, k, v, o, lse, B, H, N, d, scale, causal, cu_seqlens)


def fa_attention_fwd_splitkv(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, num_splits,
                             o_accum, lse_accum) -> int:
    return lib().fa_attention_fwd_splitkv(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal,
                                          num_splits, o_accum, lse_accum)


def fa_attention_fwd_splitkv_varlen(q, k, v, o, lse, B, H, Nq, Nk, total_q, total_k, d, scale,
                                    causal, num_splits, cu_q, cu_k, o_accum, lse_accum) -> int:
    return lib().fa_attention_fwd_splitkv_varlen(q, k, v, o, lse, B, H, Nq, Nk, total_q,
                                                 total_k, d, scale, causal, num_splits, cu_q,
                                                 cu_k, o_accum, lse_accum)


def fa_splitkv_num_splits(B, H, Nq, Nk, d) -> int:
    return lib().fa_splitkv_num_splits(B, H, Nq, Nk, d)


def fa_attention_fwd_splitkv_noalloc(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal,
                                     num_splits) -> int:
    return lib().fa_attention_fwd_splitkv_noalloc(q, k, v, o, lse, B, H, Nq, Nk, d, scale,
                                                  causal, num_splits)


def fa_attention_fwd_fp8(q, k, v, o, lse, B, H, N, d, scale, causal, signs, workspace,
                         workspace_bytes) -> int:
    return lib().fa_attention_fwd_fp8(q, k, v, o, lse, B, H, N, d, scale, causal, signs,
                                      workspace, workspace_bytes)


def fa_attention_fp8_workspace_bytes(B, H, N, d) -> int:
    return lib().fa_attention_fp8_workspace_bytes(B, H, N, d)


def fa_attention_fwd_fp8_varlen(q, k, v, o, lse, B, H, N, total, d, scale, causal, cu_seqlens,
                                signs, workspace, workspace_bytes) -> int:
    return lib().fa_attention_fwd_fp8_varlen(q, k, v, o, lse, B, H, N, total, d, scale, causal,
                                             cu_seqlens, signs, workspace, workspace_bytes)


def fa_attention_fp8_varlen_workspace_bytes(B, H, N, total, d) -> int:
    return lib().fa_attention_fp8_varlen_workspace_bytes(B, H, N, total, d)


def fa_attention_fwd_host(q, k, v, o, lse, B, H, N, d, scale, causal, workspace,
                          workspace_bytes) -> int:
    return lib().fa_attention_fwd_host(q, k, v, o, lse, B, H, N, d, scale, causal, workspace,
                                       workspace_bytes)


def fa_attention_host_workspace_bytes(B, H, N, d) -> int:
    return lib().fa_attention_host_workspace_bytes(B, H, N, d)


def fa_attention_bwd(q, k, v, o, do, lse, dq, dk, dv, d_buf, B, H, N, d, scale, causal) -> int:
    return lib().fa_attention_bwd(q, k, v, o, do, lse, dq, dk, dv, d_buf, B, H, N, d, scale,
                                  causal)


def fa_attention_bwd_varlen(q, k, v, o, do, lse, dq, dk, dv, d_buf, B, H, N, total, d, scale,
                            causal, cu_seqlens) -> int:
    return lib().fa_attention_bwd_varlen(q, k, v, o, do, lse, dq, dk, dv, d_buf, B, H, N, total,
                                         d, scale, causal, cu_seqlens)


def fa_attention_bwd_atomic(q, k, v, o, do, lse, dq, dk, dv, d_buf, B, H, N, d, scale, causal,
                            workspace, workspace_bytes) -> int:
    return lib().fa_attention_bwd_atomic(q, k, v, o, do, lse, dq, dk, dv, d_buf, B, H, N, d,
                                         scale, causal, workspace, workspace_bytes)


def fa_attention_bwd_atomic_workspace_bytes(B, H, N, d) -> int:
    return lib().fa_attention_bwd_atomic_workspace_bytes(B, H, N, d)


def fa_attention_bwd_atomic_varlen(q, k, v, o, do, lse, dq, dk, dv, d_buf, B, H, N, total, d,
                                   scale, causal, cu_seqlens, workspace, workspace_bytes) -> int:
    return lib().fa_attention_bwd_atomic_varlen(q, k, v, o, do, lse, dq, dk, dv, d_buf, B, H, N,
                                                total, d, scale, causal, cu_seqlens, workspace,
                                                workspace_bytes)


def fa_attention_bwd_atomic_varlen_workspace_bytes(B, H, N, total, d) -> int:
    return lib().fa_attention_bwd_atomic_varlen_workspace_bytes(B, H, N, total, d)


def fa_set_stream(stream_ptr) -> int:
    return lib().fa_set_stream(stream_ptr)


def fa_get_stream():
    return lib().fa_get_stream()


def fa_get_device_error() -> int:
    return lib().fa_get_device_error()


def fa_version() -> int:
    return lib().fa_version()


def fa_debug_expire_next_wait(ns: int) -> int:
    return lib().fa_debug_expire_next_wait(ns)


# ---- tensor-level helpers -------------------------------------------------------

def _use_current_stream(device):
    import torch
    fa_set_stream(torch.cuda.current_stream(device).cuda_stream)


def _ptr(t) -> int | None:
    return t.data_ptr() if t is not None else None


def softmax_rows(x, out=None):
    """Row softmax of a contiguous fp32 CUDA tensor viewed as [rows, N] (last dim N).

    ``out`` may be ``x`` itself (in place).  Returns ``out``.
    """
    import torch
    if not (x.is_cuda and x.dtype == torch.float32 and x.is_contiguous()):
        raise ValueError("x must be a contiguous float32 CUDA tensor")
    if out is None:
        out = torch.empty_like(x)
    if out.shape != x.shape or not out.is_contiguous() or out.dtype != torch.float32:
        raise ValueError("out must match x")
    N = x.shape[-1] if x.dim() > 0 else 1
    rows = x.numel() // N if N > 0 else 0
    _use_current_stream(x.device)
    _check(fa_softmax_rows(_ptr(x), _ptr(out), rows, N), "fa_softmax_rows")
    return out


def attention_fwd(q, k, v, causal: bool = False, scale: float | None = None,
                  cu_seqlens=None, max_seqlen: int | None = None, total: int | None = None,
                  out=None, lse=None):
    """Exact attention forward through the C ABI.

    Dense: q, k, v [B, N, H, d] -> (O [B, N, H, d], lse [B, H, N] fp32).
    Packed: q, k, v [total, H, d] with ``cu_seqlens`` (int32 CUDA [B+1]) and
    ``max_seqlen`` -> (O [total, H, d], lse [H, total]).  ``total`` defaults to
    q.shape[0], which avoids the library's read-back of cu_seqlens[B].
    bf16 inputs run on the tensor cores (d = 64 or 128); fp32 inputs on the
    fp32 path (d <= 128).
    """
    import torch
    for t in (q, k, v):
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError("q, k, v must be contiguous CUDA tensors")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("q, k, v must all be bfloat16 or all float32")
    if not (q.shape == k.shape == v.shape):
        raise ValueError("q, k, v must have the same shape")
    d = q.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if cu_seqlens is None:
        B, N, H, _ = q.shape
        lse_shape = (B, H, N)
    else:
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
            raise ValueError("cu_seqlens must be an int32 CUDA tensor")
        tot, H, _ = q.shape
        B = cu_seqlens.numel() - 1
        N = int(max_seqlen) if max_seqlen is not None else tot
        total = tot if total is None else int(total)
        lse_shape = (H, tot)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(lse_shape, dtype=torch.float32, device=q.device)
    _use_current_stream(q.device)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse))
    cu = _ptr(cu_seqlens)
    if q.dtype == torch.float32:
        rc = fa_attention_fwd_f32(*args, B, H, N, d, float(scale), int(bool(causal)), cu)
        _check(rc, "fa_attention_fwd_f32")
    elif cu_seqlens is not None:
        rc = fa_attention_fwd_varlen(*args, B, H, N, total, d, float(scale), int(bool(causal)),
                                     cu)
        _check(rc, "fa_attention_fwd_varlen")
    else:
        rc = fa_attention_fwd(*args, B, H, N, d, float(scale), int(bool(causal)), None)
        _check(rc, "fa_attention_fwd")
    return out, lse


def attention_fwd_splitkv(q, k, v, causal: bool = False, scale: float | None = None,
                          num_splits: int = 0, out=None, lse=None):
    """Split-KV attention forward through the C ABI (bf16, dense).

    q: [B, Nq, H, d]; k, v: [B, Nk, H, d]; causal is bottom-right aligned
    (query i sees keys j <= i + Nk - Nq).  The fp32 split scratch is allocated
    here (torch) and passed in.  Returns (O [B, Nq, H, d], lse [B, H, Nq]).
    """
    import torch
    for t in (q, k, v):
        if not (t.is_cuda and t.is_contiguous() and t.dtype == torch.bfloat16):
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors")
    B, Nq, H, d = q.shape
    Nk = k.shape[1]
    if k.shape != (B, Nk, H, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Nk, H, d]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _use_current_stream(q.device)
    splits = num_splits if num_splits > 0 else fa_splitkv_num_splits(B, H, Nq, Nk, d)
    if splits < 0:
        raise FaError(splits, "fa_splitkv_num_splits")
    splits = min(splits, (Nk + 127) // 128)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    o_acc = l_acc = None
    if splits > 1:
        o_acc = torch.empty((splits, B, Nq, H, d), dtype=torch.float32, device=q.device)
        l_acc = torch.empty((splits, B, H, Nq), dtype=torch.float32, device=q.device)
    rc = fa_attention_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nq, Nk,
                                  d, float(scale), int(bool(causal)), splits, _ptr(o_acc),
                                  _ptr(l_acc))
    _check(rc, "fa_attention_fwd_splitkv")
    return out, lse


def attention_fwd_splitkv_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                                 max_seqlen_k: int, causal: bool = False,
                                 scale: float | None = None, num_splits: int = 0):
    """Split-KV attention forward on packed sequences through the C ABI (bf16).

    q: [total_q, H, d]; k, v: [total_k, H, d]; cu_seqlens_q / cu_seqlens_k:
    int32 CUDA [B+1].  causal is bottom-right aligned within each sequence.
    The fp32 split scratch is allocated here (torch).  Returns
    (O [total_q, H, d], lse [H, total_q]).
    """
    import torch
    for t in (q, k, v):
        if not (t.is_cuda and t.is_contiguous() and t.dtype == torch.bfloat16):
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors")
    for c in (cu_seqlens_q, cu_seqlens_k):
        if c.dtype != torch.int32 or not c.is_cuda:
            raise ValueError("cu_seqlens must be int32 CUDA tensors")
    total_q, H, d = q.shape
    total_k = k.shape[0]
    if k.shape != (total_k, H, d) or v.shape != k.shape:
        raise ValueError("k and v must be [total_k, H, d]")
    B = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != B + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have one length")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _use_current_stream(q.device)
    splits = num_splits if num_splits > 0 else fa_splitkv_num_splits(B, H, max_seqlen_q,
                                                                     max_seqlen_k, d)
    if splits < 0:
        raise FaError(splits, "fa_splitkv_num_splits")
    splits = min(splits, (max_seqlen_k + 127) // 128)
    out = torch.empty_like(q)
    lse = torch.empty((H, total_q), dtype=torch.float32, device=q.device)
    o_acc = l_acc = None
    if splits > 1:
        o_acc = torch.empty((splits, total_q, H, d), dtype=torch.float32, device=q.device)
        l_acc = torch.empty((splits, H, total_q), dtype=torch.float32, device=q.device)
    rc = fa_attention_fwd_splitkv_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H,
                                         int(max_seqlen_q), int(max_seqlen_k), total_q, total_k,
                                         d, float(scale), int(bool(causal)), splits,
                                         _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(o_acc),
                                         _ptr(l_acc))
    _check(rc, "fa_attention_fwd_splitkv_varlen")
    return out, lse


def attention_fwd_fp8(q, k, v, signs, causal: bool = False, scale: float | None = None,
                      workspace=None, cu_seqlens=None, max_seqlen: int | None = None):
    """FP8 attention forward through the C ABI (bf16 inputs, d = 128).

    Dense: q, k, v [B, N, H, d] -> (O [B, N, H, d], lse [B, H, N]).  Packed:
    [total, H, d] with ``cu_seqlens`` (int32 CUDA [B+1]) and ``max_seqlen`` ->
    (O [total, H, d], lse [H, total]).  ``signs``: float32 CUDA tensor [d] of
    +-1.  The workspace (uint8, sized by fa_attention_fp8_workspace_bytes or
    its packed counterpart) is allocated here unless given.  Returns
    (O, lse, workspace).
    """
    import torch
    for t in (q, k, v):
        if not (t.is_cuda and t.is_contiguous() and t.dtype == torch.bfloat16):
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors")
        if t.shape != q.shape:
            raise ValueError("q, k, v must have one shape")
    if cu_seqlens is None:
        B, N, H, d = q.shape
        nbytes = fa_attention_fp8_workspace_bytes(B, H, N, d)
        lse_shape = (B, H, N)
    else:
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
            raise ValueError("cu_seqlens must be an int32 CUDA tensor")
        tot, H, d = q.shape
        B = cu_seqlens.numel() - 1
        N = int(max_seqlen) if max_seqlen is not None else tot
        nbytes = fa_attention_fp8_varlen_workspace_bytes(B, H, N, tot, d)
        lse_shape = (H, tot)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if nbytes < 0:
        raise FaError(int(nbytes), "fa_attention_fp8_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=q.device)
    _use_current_stream(q.device)
    o = torch.empty_like(q)
    lse = torch.empty(lse_shape, dtype=torch.float32, device=q.device)
    if cu_seqlens is None:
        rc = fa_attention_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                                  float(scale), int(bool(causal)), _ptr(signs), _ptr(workspace),
                                  workspace.numel())
        _check(rc, "fa_attention_fwd_fp8")
    else:
        rc = fa_attention_fwd_fp8_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N,
                                         q.shape[0], d, float(scale), int(bool(causal)),
                                         _ptr(cu_seqlens), _ptr(signs), _ptr(workspace),
                                         workspace.numel())
        _check(rc, "fa_attention_fwd_fp8_varlen")
    return o, lse, workspace


def attention_fwd_host(q, k, v, causal: bool = False, scale: float | None = None,
                       workspace=None, device=None, out=None):
    """bf16 attention forward on HOST tensors through the C ABI (dense
    [B, N, H, d]); the library copies to and from the device itself, head
    group by head group, overlapping the copies with the kernels.

    ``q``, ``k``, ``v``: contiguous bf16 CPU tensors (pinned for overlap).
    The DEVICE workspace (uint8, fa_attention_host_workspace_bytes) is
    allocated here on ``device`` (default cuda:current) unless given; ``out``
    may pass preallocated (O, lse) CPU tensors.  The call returns after the
    library stream has been synchronised.  Returns (O, lse, workspace).
    """
    import torch
    for t in (q, k, v):
        if t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError("q, k, v must be contiguous bf16 CPU tensors")
        if t.shape != q.shape:
            raise ValueError("q, k, v must have one shape")
    B, N, H, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    nbytes = fa_attention_host_workspace_bytes(B, H, N, d)
    if nbytes < 0:
        raise FaError(int(nbytes), "fa_attention_host_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=dev)
    if out is None:
        pin = q.is_pinned()
        o = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pin)
        lse = torch.empty((B, H, N), dtype=torch.float32, pin_memory=pin)
    else:
        o, lse = out
    _use_current_stream(dev)
    rc = fa_attention_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                               float(scale), int(bool(causal)), _ptr(workspace),
                               workspace.numel())
    _check(rc, "fa_attention_fwd_host")
    torch.cuda.current_stream(dev).synchronize()
    return o, lse, workspace


def attention_bwd(q, k, v, o, do, lse, causal: bool = False, scale: float | None = None,
                  cu_seqlens=None, max_seqlen: int | None = None, deterministic: bool = True):
    """Attention backward through the C ABI (bf16).

    Dense: q, k, v, o, do [B, N, H, d], lse [B, H, N].  Packed: [total, H, d]
    with ``cu_seqlens`` (int32 CUDA [B+1]) and ``max_seqlen``, lse [H, total].
    ``o`` and ``lse`` are the forward's outputs for the same inputs.  The fp32
    D scratch (lse's shape) is allocated here (torch).  ``deterministic=False``
    calls the one-pass form with atomic dQ sums (``fa_attention_bwd_atomic`` /
    ``_varlen``; its workspace is allocated here).  Returns (dq, dk, dv).
    """
    import torch
    for t in (q, k, v, o, do):
        if not (t.is_cuda and t.is_contiguous() and t.dtype == torch.bfloat16):
            raise ValueError("q, k, v, o, do must be contiguous bf16 CUDA tensors")
        if t.shape != q.shape:
            raise ValueError("q, k, v, o, do must have one shape")
    if cu_seqlens is None:
        B, N, H, d = q.shape
        lse_shape = (B, H, N)
    else:
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
            raise ValueError("cu_seqlens must be an int32 CUDA tensor")
        tot, H, d = q.shape
        B = cu_seqlens.numel() - 1
        N = int(max_seqlen) if max_seqlen is not None else tot
        lse_shape = (H, tot)
    if not (lse.is_cuda and lse.dtype == torch.float32 and tuple(lse.shape) == lse_shape
            and lse.is_contiguous()):
        raise ValueError(f"lse must be a contiguous float32 CUDA tensor {list(lse_shape)}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _use_current_stream(q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    d_buf = torch.empty(lse_shape, dtype=torch.float32, device=q.device)
    ptrs = (_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
            _ptr(d_buf))
    if not deterministic and cu_seqlens is None:
        nbytes = fa_attention_bwd_atomic_workspace_bytes(B, H, N, d)
        _check(int(min(nbytes, 0)), "fa_attention_bwd_atomic_workspace_bytes")
        ws = torch.empty(max(nbytes // 4, 1), dtype=torch.float32, device=q.device)
        rc = fa_attention_bwd_atomic(*ptrs, B, H, N, d, float(scale), int(bool(causal)), _ptr(ws),
                                     nbytes)
        _check(rc, "fa_attention_bwd_atomic")
    elif not deterministic:
        nbytes = fa_attention_bwd_atomic_varlen_workspace_bytes(B, H, N, q.shape[0], d)
        _check(int(min(nbytes, 0)), "fa_attention_bwd_atomic_varlen_workspace_bytes")
        ws = torch.empty(max(nbytes // 4, 1), dtype=torch.float32, device=q.device)
        rc = fa_attention_bwd_atomic_varlen(*ptrs, B, H, N, q.shape[0], d, float(scale),
                                            int(bool(causal)), _ptr(cu_seqlens), _ptr(ws), nbytes)
        _check(rc, "fa_attention_bwd_atomic_varlen")
    elif cu_seqlens is None:
        rc = fa_attention_bwd(*ptrs, B, H, N, d, float(scale), int(bool(causal)))
        _check(rc, "fa_attention_bwd")
    else:
        rc = fa_attention_bwd_varlen(*ptrs, B, H, N, q.shape[0], d, float(scale),
                                     int(bool(causal)), _ptr(cu_seqlens))
        _check(rc, "fa_attention_bwd_varlen")
    return dq, dk, dv


__all__ = [
    "build", "lib", "strerror", "FaError", "softmax_rows", "attention_fwd",
    "attention_fwd_splitkv", "attention_fwd_splitkv_varlen", "fa_attention_fwd_splitkv",
    "fa_attention_fwd_splitkv_varlen",
    "fa_splitkv_num_splits",
    "fa_attention_fwd_splitkv_noalloc", "FA_ERR_SCRATCH_LIMIT", "FA_NOALLOC_SCRATCH_BYTES",
    "attention_bwd", "fa_attention_bwd", "fa_attention_bwd_varlen", "fa_attention_bwd_atomic",
    "fa_attention_bwd_atomic_workspace_bytes", "fa_attention_bwd_atomic_varlen",
    "fa_attention_bwd_atomic_varlen_workspace_bytes", "attention_fwd_fp8",
    "fa_attention_fwd_fp8", "fa_attention_fwd_fp8_varlen",
    "fa_attention_fp8_workspace_bytes",
    "fa_softmax_rows", "fa_attention_fwd", "fa_attention_fwd_varlen", "fa_attention_fwd_f32",
    "fa_set_stream", "fa_get_stream", "fa_get_device_error", "fa_version",
    "FA_DEVERR_WAIT_TIMEOUT", "FA_DEVERR_BAD_SEQLENS", "fa_debug_expire_next_wait",
]
