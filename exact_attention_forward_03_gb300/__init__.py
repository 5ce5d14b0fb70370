"""Exact attention forward for GB300 (sm_103a): a thin ctypes binding of libfa.so.

Every step of the computation runs in the library's CUDA kernels; this module
only checks tensors, allocates outputs with torch when the caller passes none,
and forwards raw pointers, sizes and the current CUDA stream to the C ABI
declared in ``include/fa.h``.  There is no fallback: if ``libfa.so`` is not
built or the tensors are not on a CUDA device, the calls raise.

Functions (same names as the C ABI without the ``fa_`` prefix):
    fwd(q, k, v, causal=False, scale=None, out=None, lse=None)            -> (o, lse)
    fwd_splitkv(q, k, v, causal=False, scale=None, num_splits=0, ...)     -> (o, lse)
    splitkv_combine(o_part, lse_part, out=None, lse=None, dtype=...)      -> (o, lse)
    bwd(q, k, v, o, dout, lse, causal=False, scale=None, ...)            -> (dq, dk, dv)
    attention(q, k, v, causal=False, scale=None)   differentiable: fwd, then bwd in backward
    fp8_quantize(x, transpose=False) -> (codes, scales);  fwd_fp8(q8, qs, k8, ks, v8t, vs, ...) -> (o, lse)
    fwd_fp8_from(q, k, v, causal=False) -> (o, lse)       quantize, then the FP8 forward
    splitkv_num_splits, splitkv_split_len, splitkv_workspace_bytes, bwd_workspace_bytes,
    get_device_status, status_string, version
Tensors are ``[B, H, N, d]`` contiguous fp16 or bf16 on one CUDA device;
``lse`` is ``[B, H, Nq]`` fp32.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfa.so")

FA_F16, FA_BF16 = 0, 1
FA_OK = 0
FA_ERR_INVALID_ARG = -1
FA_ERR_UNSUPPORTED = -2
FA_ERR_MISALIGNED = -3
FA_ERR_WORKSPACE = -4
FA_ERR_CUDA = -5
FA_ERR_DEVICE_TIMEOUT = -6
FA_ERR_SCRATCH_LIMIT = -7

EXPORTS = ("fa_fwd", "fa_fwd_splitkv", "fa_splitkv_combine", "fa_splitkv_workspace_bytes",
           "fa_splitkv_num_splits", "fa_splitkv_split_len", "fa_get_device_status", "fa_status_string",
           "fa_version", "fa_fwd_splitkv_noalloc", "fa_splitkv_noalloc_capacity_bytes", "fa_fwd_gqa",
           "fa_fwd_splitkv_gqa", "fa_fwd_varlen", "fa_bwd", "fa_bwd_workspace_bytes", "fa_last_error", "fa_fp8_quantize", "fa_fwd_fp8", "fa_selftest_timeout", "fa_bwd_gqa",
           "fa_bwd_varlen", "fa_bwd_varlen_workspace_bytes", "fa_fwd_host",
           "fa_fwd_host_workspace_bytes", "fa_fwd_varlen_ws", "fa_fwd_varlen_workspace_bytes")

_lock = threading.Lock()
_lib = None


class FaError(RuntimeError):
    def __init__(self, code: int, what: str):
        detail = ""
        if code == FA_ERR_CUDA:
            try:
                detail = " [" + load_library().fa_last_error().decode() + "]"
            except RuntimeError:
                pass
        super().__init__(f"{what}: {status_string(code)} ({code}){detail}")
        self.code = code


def load_library(path: str | None = None):
    """Load libfa.so (built by ``build.build()``) and declare its C signatures."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is not built; run exact_attention_forward_03_gb300.build.build()")
        lib = ctypes.CDLL(p)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
        lib.fa_fwd.restype = i
        lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp, sz, vp]
        lib.fa_fwd_splitkv.restype = i
        lib.fa_splitkv_combine.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, vp]
        lib.fa_splitkv_combine.restype = i
        lib.fa_splitkv_workspace_bytes.argtypes = [i, i, i, i, i, i]
        lib.fa_splitkv_workspace_bytes.restype = sz
        lib.fa_splitkv_num_splits.argtypes = [i, i, i, i, i]
        lib.fa_splitkv_num_splits.restype = i
        lib.fa_splitkv_split_len.argtypes = [i, i]
        lib.fa_splitkv_split_len.restype = i
        lib.fa_get_device_status.argtypes = [vp]
        lib.fa_get_device_status.restype = i
        lib.fa_status_string.argtypes = [i]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_version.argtypes = []
        lib.fa_version.restype = i
        lib.fa_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp]
        lib.fa_fwd_splitkv_noalloc.restype = i
        lib.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp]
        lib.fa_fwd_gqa.restype = i
        lib.fa_fwd_splitkv_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, i, vp, sz, vp]
        lib.fa_fwd_splitkv_gqa.restype = i
        lib.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp]
        lib.fa_fwd_varlen.restype = i
        lib.fa_fwd_varlen_ws.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp, sz, vp]
        lib.fa_fwd_varlen_ws.restype = i
        lib.fa_fwd_varlen_workspace_bytes.argtypes = [i, i]
        lib.fa_fwd_varlen_workspace_bytes.restype = sz
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, sz, vp]
        lib.fa_bwd.restype = i
        lib.fa_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp, sz, vp]
        lib.fa_bwd_gqa.restype = i
        lib.fa_bwd_workspace_bytes.argtypes = [i, i, i, i]
        lib.fa_bwd_workspace_bytes.restype = sz
        lib.fa_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp,
                                      sz, vp]
        lib.fa_bwd_varlen.restype = i
        lib.fa_bwd_varlen_workspace_bytes.argtypes = [i, i, i, i, i]
        lib.fa_bwd_varlen_workspace_bytes.restype = sz
        lib.fa_fwd_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, i, vp, sz, vp]
        lib.fa_fwd_host.restype = i
        lib.fa_fwd_host_workspace_bytes.argtypes = [i, i, i, i, i, i]
        lib.fa_fwd_host_workspace_bytes.restype = sz
        lib.fa_fp8_quantize.argtypes = [vp, vp, vp, i, i, i, i, i, vp]
        lib.fa_fp8_quantize.restype = i
        lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
        lib.fa_fwd_fp8.restype = i
        lib.fa_selftest_timeout.argtypes = [i, vp]
        lib.fa_selftest_timeout.restype = i
        lib.fa_last_error.argtypes = []
        lib.fa_last_error.restype = ctypes.c_char_p
        lib.fa_splitkv_noalloc_capacity_bytes.argtypes = []
        lib.fa_splitkv_noalloc_capacity_bytes.restype = sz
        if path is None:
            _lib = lib
        return lib


def status_string(code: int) -> str:
    try:
        return load_library().fa_status_string(int(code)).decode()
    except RuntimeError:
        return f"status {code}"


def version() -> int:
    return load_library().fa_version()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return FA_F16
    if t.dtype == torch.bfloat16:
        return FA_BF16
    raise TypeError(f"dtype {t.dtype} not supported (fp16 or bf16)")


def _stream_handle(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _check_qkv(q, k, v, allow_gqa=True):
    """(B, H, H_kv, Nq, Nk, d) of q [B, H, Nq, d] and k, v [B, H_kv, Nk, d] (H_kv divides H)."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, H, N, d] tensor")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k and v must share one dtype")
    B, H, Nq, d = q.shape
    H_kv = k.shape[1]
    ok_heads = H_kv == H or (allow_gqa and H_kv > 0 and H % H_kv == 0)
    if k.shape[0] != B or not ok_heads or v.shape != k.shape or k.shape[3] != d:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    return B, H, H_kv, Nq, k.shape[2], d


def _outputs(q, out, lse, B, H, Nq, want_lse=True):
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must match q")
    if lse is None and want_lse:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    elif lse is not None and (lse.shape != (B, H, Nq) or lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous fp32 [B, H, Nq] tensor")
    return out, lse


def fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None, want_lse: bool = True,
        stream=None):
    """Fused attention forward through ``fa_fwd`` (``fa_fwd_gqa`` when k and v have
    fewer heads than q: grouped-query attention).  Returns (o, lse)."""
    B, H, H_kv, Nq, Nk, d = _check_qkv(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out, lse = _outputs(q, out, lse, B, H, Nq, want_lse)
    lib = load_library()
    lse_p = lse.data_ptr() if lse is not None else None
    if H_kv == H:
        rc = lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_p, B, H, Nq, Nk, d,
                        int(bool(causal)), scale, _dtype_code(q), _stream_handle(stream))
    else:
        rc = lib.fa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_p, B, H, H_kv, Nq, Nk, d,
                            int(bool(causal)), scale, _dtype_code(q), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd" if H_kv == H else "fa_fwd_gqa")
    return out, lse


def fwd_host_workspace_bytes(B, H, H_kv, Nq, Nk, d) -> int:
    return int(load_library().fa_fwd_host_workspace_bytes(B, H, H_kv, Nq, Nk, d))


def fwd_host(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None, want_lse: bool = True,
             num_chunks: int = 0, workspace=None, stream=None, synchronize: bool = True):
    """Forward from and to host memory through ``fa_fwd_host``: q [B, H, Nq, d], k, v
    [B, H_kv, Nk, d] CPU tensors (page-locked for overlapped copies); returns (o, lse)
    as CPU tensors (page-locked when allocated here).  The copies and the kernels are
    queued on ``stream`` (the current stream by default); with ``synchronize`` the
    call waits for that stream before returning."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU [B, H, N, d] tensor")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k and v must share one dtype")
    B, H, Nq, d = q.shape
    H_kv, Nk = k.shape[1], k.shape[2]
    if k.shape[0] != B or v.shape != k.shape or k.shape[3] != d or H_kv <= 0 or H % H_kv != 0:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    elif out.is_cuda or out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous CPU tensor like q")
    if lse is None and want_lse:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, pin_memory=True)
    elif lse is not None and (lse.is_cuda or lse.shape != (B, H, Nq) or lse.dtype != torch.float32
                              or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous fp32 CPU [B, H, Nq] tensor")
    lib = load_library()
    need = fwd_host_workspace_bytes(B, H, H_kv, Nq, Nk, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    rc = lib.fa_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                         lse.data_ptr() if lse is not None else None, B, H, H_kv, Nq, Nk, d, int(bool(causal)), scale,
                         _dtype_code(q), int(num_chunks), workspace.data_ptr(),
                         workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_host")
    if synchronize:
        (stream if stream is not None else torch.cuda.current_stream()).synchronize()
    return out, lse


def bwd_workspace_bytes(B, H, Nq, d) -> int:
    return int(load_library().fa_bwd_workspace_bytes(B, H, Nq, d))


def bwd(q, k, v, o, dout, lse, causal: bool = False, scale: float | None = None, dq=None, dk=None, dv=None,
        workspace=None, stream=None):
    """Attention backward through ``fa_bwd`` (``fa_bwd_gqa`` when k and v have fewer
    heads than q): (dq, dk, dv) for the forward that gave (o, lse) from (q, k, v)
    with the same causal flag and scale."""
    B, H, H_kv, Nq, Nk, d = _check_qkv(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    for name, t, shape in (("o", o, q.shape), ("dout", dout, q.shape)):
        if not t.is_cuda or t.shape != shape or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous tensor like q")
    if lse.shape != (B, H, Nq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, Nq] tensor")
    outs = []
    for name, t, like in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if t is None:
            t = torch.empty_like(like)
        elif t.shape != like.shape or t.dtype != like.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must match its input")
        outs.append(t)
    dq, dk, dv = outs
    need = bwd_workspace_bytes(B, H, Nq, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    rc = load_library().fa_bwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                                   lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, H_kv, Nq, Nk, d,
                                   int(bool(causal)), scale, _dtype_code(q), workspace.data_ptr(),
                                   workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_gqa")
    return dq, dk, dv


class _Attention(torch.autograd.Function):
    """Forward through fa_fwd, backward through fa_bwd."""

    @staticmethod
    def forward(ctx, q, k, v, causal, scale):
        o, lse = fwd(q, k, v, causal=causal, scale=scale)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.causal, ctx.scale = causal, scale
        return o

    @staticmethod
    def backward(ctx, dout):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = bwd(q, k, v, o, dout.contiguous(), lse, causal=ctx.causal, scale=ctx.scale)
        return dq, dk, dv, None, None


def attention(q, k, v, causal: bool = False, scale: float | None = None):
    """Differentiable attention: fa_fwd in the forward pass, fa_bwd in the backward."""
    return _Attention.apply(q, k, v, bool(causal), scale)


def fp8_quantize(x, transpose: bool = False, out=None, scales=None, stream=None):
    """E4M3 codes (uint8) and per-128-row-block fp32 scales of x [B, H, N, 128] through
    ``fa_fp8_quantize``.  transpose=False: codes [B, H, N, 128]; transpose=True (the
    layout of V for fwd_fp8): codes [B, H, 128, ceil(N/128)*128]."""
    if not x.is_cuda or x.dim() != 4 or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA [B, H, N, d] tensor")
    B, H, N, d = x.shape
    nb = (N + 127) // 128
    shape = (B, H, d, nb * 128) if transpose else (B, H, N, d)
    if out is None:
        out = torch.empty(shape, dtype=torch.uint8, device=x.device)
    elif tuple(out.shape) != shape or out.dtype != torch.uint8 or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous uint8 {shape} tensor")
    if scales is None:
        scales = torch.empty((B * H, nb), dtype=torch.float32, device=x.device)
    elif tuple(scales.shape) != (B * H, nb) or scales.dtype != torch.float32 or not scales.is_contiguous():
        raise ValueError(f"scales must be a contiguous fp32 {(B * H, nb)} tensor")
    rc = load_library().fa_fp8_quantize(x.data_ptr(), out.data_ptr(), scales.data_ptr(), B * H, N, d,
                                        int(bool(transpose)), _dtype_code(x), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fp8_quantize")
    return out, scales


def fwd_fp8(q8, q_scale, k8, k_scale, v8t, v_scale, causal: bool = False, scale: float | None = None,
            out_dtype=torch.bfloat16, out=None, lse=None, want_lse: bool = True, stream=None):
    """FP8 attention forward through ``fa_fwd_fp8`` on codes and scales made by
    fp8_quantize (v8t from the transposed form).  Returns (o, lse)."""
    for name, t in (("q8", q8), ("k8", k8), ("v8t", v8t)):
        if not t.is_cuda or t.dtype != torch.uint8 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous uint8 CUDA tensor")
    B, H, Nq, d = q8.shape
    Nk = k8.shape[2]
    if k8.shape != (B, H, Nk, d) or v8t.shape != (B, H, d, (Nk + 127) // 128 * 128):
        raise ValueError(f"shape mismatch q8{tuple(q8.shape)} k8{tuple(k8.shape)} v8t{tuple(v8t.shape)}")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty((B, H, Nq, d), dtype=out_dtype, device=q8.device)
    if lse is None and want_lse:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q8.device)
    code = FA_BF16 if out.dtype == torch.bfloat16 else FA_F16
    rc = load_library().fa_fwd_fp8(q8.data_ptr(), q_scale.data_ptr(), k8.data_ptr(), k_scale.data_ptr(),
                                   v8t.data_ptr(), v_scale.data_ptr(), out.data_ptr(),
                                   lse.data_ptr() if lse is not None else None, B, H, Nq, Nk, d,
                                   int(bool(causal)), scale, code, _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_fp8")
    return out, lse


def fwd_fp8_from(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """Quantize 16-bit q, k, v (fa_fp8_quantize) and run fa_fwd_fp8; returns (o, lse)
    in q's dtype."""
    q8, qs = fp8_quantize(q, stream=stream)
    k8, ks = fp8_quantize(k, stream=stream)
    v8t, vs = fp8_quantize(v, transpose=True, stream=stream)
    return fwd_fp8(q8, qs, k8, ks, v8t, vs, causal=causal, scale=scale, out_dtype=q.dtype, stream=stream)


def fwd_varlen_workspace_bytes(num_seqs: int, total_q: int) -> int:
    return int(load_library().fa_fwd_varlen_workspace_bytes(num_seqs, total_q))


def fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int | None = None, causal: bool = False,
               scale: float | None = None, out=None, lse=None, want_lse: bool = True, stream=None,
               plan: bool = True, workspace=None):
    """Variable-length (packed) batch.

    q: [total_q, H, d], k, v: [total_k, H_kv, d] (H_kv divides H), cu_seqlens_q/k:
    int32 CUDA tensors of num_seqs + 1 offsets.  Returns (o [total_q, H, d],
    lse [H, total_q]).  With ``plan`` (the default) this is ``fa_fwd_varlen_ws``:
    a device-built work list in ``workspace`` (a uint8 CUDA tensor of at least
    ``fwd_varlen_workspace_bytes`` bytes, allocated here when None) sends CTAs only
    to row blocks that hold rows.  Without it, ``fa_fwd_varlen``: a grid sized by
    ``max_seqlen_q``, which must bound every sequence's query length.
    """
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or t.dim() != 3 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA [tokens, heads, d] tensor")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k and v must share one dtype")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if not t.is_cuda or t.dtype != torch.int32 or t.dim() != 1 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA vector")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both hold num_seqs + 1 offsets")
    total_q, H, d = q.shape
    total_k, H_kv = k.shape[0], k.shape[1]
    if v.shape != k.shape or k.shape[2] != d or H_kv <= 0 or H % H_kv != 0:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must match q")
    if lse is None and want_lse:
        lse = torch.empty((H, total_q), dtype=torch.float32, device=q.device)
    lib = load_library()
    num_seqs = cu_seqlens_q.numel() - 1
    if plan:
        need = fwd_varlen_workspace_bytes(num_seqs, total_q)
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        elif not workspace.is_cuda or workspace.dtype != torch.uint8 or workspace.numel() < need:
            raise ValueError(f"workspace must be a uint8 CUDA tensor of at least {need} bytes")
        rc = lib.fa_fwd_varlen_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  lse.data_ptr() if lse is not None else None, cu_seqlens_q.data_ptr(),
                                  cu_seqlens_k.data_ptr(), num_seqs, total_q, total_k, H, H_kv, d, int(bool(causal)),
                                  scale, _dtype_code(q), workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
        if rc != FA_OK:
            raise FaError(rc, "fa_fwd_varlen_ws")
        return out, lse
    if max_seqlen_q is None:
        raise ValueError("the unplanned grid needs max_seqlen_q")
    rc = lib.fa_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                           lse.data_ptr() if lse is not None else None, cu_seqlens_q.data_ptr(),
                           cu_seqlens_k.data_ptr(), num_seqs, int(max_seqlen_q), total_q, total_k, H,
                           H_kv, d, int(bool(causal)), scale, _dtype_code(q), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_varlen")
    return out, lse


def bwd_varlen_workspace_bytes(num_seqs, total_q, total_k, H, d) -> int:
    return int(load_library().fa_bwd_varlen_workspace_bytes(num_seqs, total_q, total_k, H, d))


def bwd_varlen(q, k, v, o, dout, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_k: int, causal: bool = False,
               scale: float | None = None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward of a variable-length (packed) batch through ``fa_bwd_varlen``:
    (dq [total_q, H, d], dk, dv [total_k, H_kv, d]) for the ``fwd_varlen`` call that
    gave (o, lse [H, total_q]).  ``max_seqlen_k`` must bound every sequence's key count."""
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        if not t.is_cuda or t.dim() != 3 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA [tokens, heads, d] tensor")
    if not (q.dtype == k.dtype == v.dtype == o.dtype == dout.dtype):
        raise TypeError("q, k, v, o and dout must share one dtype")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if not t.is_cuda or t.dtype != torch.int32 or t.dim() != 1 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA vector")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both hold num_seqs + 1 offsets")
    total_q, H, d = q.shape
    total_k, H_kv = k.shape[0], k.shape[1]
    if v.shape != k.shape or k.shape[2] != d or H_kv <= 0 or H % H_kv != 0:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if o.shape != q.shape or dout.shape != q.shape:
        raise ValueError("o and dout must have q's shape")
    if lse.shape != (H, total_q) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [H, total_q] tensor")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    outs = []
    for name, t, like in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if t is None:
            t = torch.empty_like(like)
        elif t.shape != like.shape or t.dtype != like.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must match its input")
        outs.append(t)
    dq, dk, dv = outs
    num_seqs = cu_seqlens_q.numel() - 1
    need = bwd_varlen_workspace_bytes(num_seqs, total_q, total_k, H, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    rc = load_library().fa_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                                      lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                      cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), num_seqs, int(max_seqlen_k),
                                      total_q, total_k, H, H_kv, d, int(bool(causal)), scale, _dtype_code(q),
                                      workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                      _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_varlen")
    return dq, dk, dv


class _AttentionVarlen(torch.autograd.Function):
    """Forward through fa_fwd_varlen, backward through fa_bwd_varlen."""

    @staticmethod
    def forward(ctx, q, k, v, cu_q, cu_k, max_q, max_k, causal, scale):
        o, lse = fwd_varlen(q, k, v, cu_q, cu_k, max_q, causal=causal, scale=scale)
        ctx.save_for_backward(q, k, v, o, lse, cu_q, cu_k)
        ctx.max_k, ctx.causal, ctx.scale = max_k, causal, scale
        return o

    @staticmethod
    def backward(ctx, dout):
        q, k, v, o, lse, cu_q, cu_k = ctx.saved_tensors
        dq, dk, dv = bwd_varlen(q, k, v, o, dout.contiguous(), lse, cu_q, cu_k, ctx.max_k, causal=ctx.causal,
                                scale=ctx.scale)
        return dq, dk, dv, None, None, None, None, None, None


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                     causal: bool = False, scale: float | None = None):
    """Differentiable attention of a packed variable-length batch: fa_fwd_varlen in
    the forward pass, fa_bwd_varlen in the backward (layouts as ``fwd_varlen``)."""
    return _AttentionVarlen.apply(q, k, v, cu_seqlens_q, cu_seqlens_k, int(max_seqlen_q), int(max_seqlen_k), causal,
                                  scale)


def splitkv_num_splits(B, H, Nq, Nk, d) -> int:
    return load_library().fa_splitkv_num_splits(B, H, Nq, Nk, d)


def splitkv_split_len(Nk, num_splits) -> int:
    return load_library().fa_splitkv_split_len(Nk, num_splits)


def splitkv_workspace_bytes(B, H, Nq, Nk, d, num_splits=0) -> int:
    return load_library().fa_splitkv_workspace_bytes(B, H, Nq, Nk, d, num_splits)


def splitkv_workspace(q, k, num_splits=0):
    """Allocate a workspace tensor for ``fwd_splitkv`` (torch allocator, 256-byte aligned)."""
    B, H, Nq, d = q.shape
    nbytes = splitkv_workspace_bytes(B, H, Nq, k.shape[2], d, num_splits)
    if nbytes == 0:
        raise ValueError("invalid sizes for a split-KV workspace")
    return torch.empty(nbytes, dtype=torch.uint8, device=q.device)


def fwd_splitkv(q, k, v, causal: bool = False, scale: float | None = None, num_splits: int = 0, workspace=None,
                out=None, lse=None, want_lse: bool = True, stream=None):
    """Split-KV forward (partials + combine) through ``fa_fwd_splitkv`` (``fa_fwd_splitkv_gqa``
    when k and v have fewer heads than q).  Returns (o, lse)."""
    B, H, H_kv, Nq, Nk, d = _check_qkv(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out, lse = _outputs(q, out, lse, B, H, Nq, want_lse)
    if num_splits <= 0:
        num_splits = splitkv_num_splits(B, H, Nq, Nk, d)
    if workspace is None:
        workspace = splitkv_workspace(q, k, num_splits)
    lib = load_library()
    lse_p = lse.data_ptr() if lse is not None else None
    ws_bytes = workspace.numel() * workspace.element_size()
    if H_kv == H:
        rc = lib.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_p, B, H, Nq, Nk, d,
                                int(bool(causal)), scale, _dtype_code(q), int(num_splits), workspace.data_ptr(),
                                ws_bytes, _stream_handle(stream))
    else:
        rc = lib.fa_fwd_splitkv_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_p, B, H, H_kv, Nq,
                                    Nk, d, int(bool(causal)), scale, _dtype_code(q), int(num_splits),
                                    workspace.data_ptr(), ws_bytes, _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_splitkv" if H_kv == H else "fa_fwd_splitkv_gqa")
    return out, lse


def fwd_splitkv_noalloc(q, k, v, causal: bool = False, scale: float | None = None, num_splits: int = 0, out=None,
                        lse=None, want_lse: bool = True, stream=None):
    """Split-KV forward through ``fa_fwd_splitkv_noalloc``: the partials use the
    library's built-in scratch, so no workspace is passed.  Returns (o, lse)."""
    B, H, _, Nq, Nk, d = _check_qkv(q, k, v, allow_gqa=False)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out, lse = _outputs(q, out, lse, B, H, Nq, want_lse)
    lib = load_library()
    rc = lib.fa_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                    lse.data_ptr() if lse is not None else None, B, H, Nq, Nk, d,
                                    int(bool(causal)), scale, _dtype_code(q), int(num_splits), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_splitkv_noalloc")
    return out, lse


def workspace_views(workspace, B, H, Nq, d, num_splits):
    """The (o_part [S, B, H, Nq, d], lse_part [S, B, H, Nq]) fp32 views of a split-KV workspace."""
    rows = B * H * Nq
    o_bytes = (num_splits * rows * d * 4 + 255) // 256 * 256
    o_part = workspace[: num_splits * rows * d * 4].view(torch.float32).view(num_splits, B, H, Nq, d)
    lse_part = workspace[o_bytes: o_bytes + num_splits * rows * 4].view(torch.float32).view(num_splits, B, H, Nq)
    return o_part, lse_part


def splitkv_combine(o_part, lse_part, dtype=torch.bfloat16, out=None, lse=None, stream=None):
    """LSE-weighted merge of fp32 partials through ``fa_splitkv_combine``.  Returns (o, lse)."""
    if o_part.dim() != 5 or lse_part.dim() != 4 or not o_part.is_contiguous() or not lse_part.is_contiguous():
        raise ValueError("o_part must be [S, B, H, Nq, d] and lse_part [S, B, H, Nq], contiguous")
    S, B, H, Nq, d = o_part.shape
    if out is None:
        out = torch.empty((B, H, Nq, d), dtype=dtype, device=o_part.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=o_part.device)
    lib = load_library()
    rc = lib.fa_splitkv_combine(o_part.data_ptr(), lse_part.data_ptr(), out.data_ptr(), lse.data_ptr(), S, B, H, Nq,
                                d, _dtype_code(out), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_splitkv_combine")
    return out, lse


def selftest_timeout(limit_ms: int = 50, stream=None) -> None:
    """Launch the timeout self-test kernel (fa_selftest_timeout); read the result
    with get_device_status()."""
    rc = load_library().fa_selftest_timeout(int(limit_ms), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_selftest_timeout")


def get_device_status(stream=None) -> int:
    """Synchronise the stream and return the library's device status (FA_OK, FA_ERR_DEVICE_TIMEOUT, ...)."""
    return load_library().fa_get_device_status(_stream_handle(stream))
