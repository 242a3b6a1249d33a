"""GB300 (sm_103a) fused scaled-dot-product-attention forward.

Thin Python binding over the C ABI in ``include/sdpa.h`` (library
``libsdpa_gb300.so``, built in-tree by ``flash_attention_forward_gb300.build``).
The binding only marshals arguments: it reads shapes, strides and data pointers of
torch tensors, allocates outputs and scratch with torch when the caller does not
pass them, and calls the library on the current CUDA stream.  Every step of the
computation runs in the library's kernels; there is no fallback.

Entry points (same names as the C ABI):
    sdpa_fwd(q, k, v, ...)                     fp16 / bf16 prefill
    sdpa_fwd_fp8(q, k, v, dq, dk, dv, ...)     e4m3 prefill with per-tensor scales
    sdpa_fwd_varlen(q, k, v, cu_q, cu_k, max_seqlen_q, ...)   prefill of packed sequences
    sdpa_fwd_varlen_fp8(q, k, v, cu_q, cu_k, max_seqlen_q, dq, dk, dv, ...)   the same in e4m3
    sdpa_fwd_int8(q, k, v, q_scale, k_scale, v_scale, ...)   int8 Q/K codes with per-block scales
    sdpa_fwd_host(q, k, v, ...)                 sdpa_fwd on pinned host tensors, copies overlapped
    sdpa_decode(q, k_cache, v_cache, kv_len, ...)   two-phase split-KV decode
    sdpa_decode_paged(q, k_pool, v_pool, page_table, kv_len, ...)   the same over a paged cache
    sdpa_decode_noalloc(q, k_cache, v_cache, kv_len, ...)   the same with library-owned scratch
    sdpa_fwd_workspace_size, sdpa_fwd_varlen_workspace_size, sdpa_fwd_int8_workspace_size,
    sdpa_fwd_host_workspace_size,
    sdpa_decode_workspace_size,
    sdpa_check_device_status,
    sdpa_status_string, sdpa_version
"""
from __future__ import annotations

import ctypes
import math
import os
import re
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsdpa_gb300.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "sdpa.h")

SDPA_OK, SDPA_ERR_INVALID, SDPA_ERR_UNSUPPORTED, SDPA_ERR_CUDA, SDPA_ERR_TIMEOUT = range(5)
SDPA_F16, SDPA_BF16, SDPA_E4M3, SDPA_I8 = range(4)
_DT = {torch.float16: SDPA_F16, torch.bfloat16: SDPA_BF16, torch.float8_e4m3fn: SDPA_E4M3, torch.int8: SDPA_I8}

_lock = threading.Lock()
_lib = None


class SdpaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {sdpa_status_string(status)} ({status})")


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m flash_attention_forward_gb300.build` "
                               f"(or __graft_entry__.build())")
        lib = ctypes.CDLL(LIB_PATH)
        p, i, i64, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        lib.sdpa_fwd_workspace_size.argtypes = [i, i, i, i, i, i, i]
        lib.sdpa_fwd_workspace_size.restype = sz
        lib.sdpa_fwd.argtypes = [p, p, p, p, p, i, i, i, i, i, i, i, p, f, i, p, p, p, sz, i, i, p]
        lib.sdpa_fwd.restype = i
        lib.sdpa_fwd_fp8.argtypes = [p, p, p, p, p, i, i, i, i, i, i, i, p, f, i, p, p, p, sz, f, f, f, i, p]
        lib.sdpa_fwd_fp8.restype = i
        lib.sdpa_fwd_varlen_workspace_size.argtypes = [i]
        lib.sdpa_fwd_varlen_workspace_size.restype = sz
        lib.sdpa_fwd_varlen.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, i, i, i, p, f, i, p, sz, i, i, p]
        lib.sdpa_fwd_varlen.restype = i
        lib.sdpa_fwd_varlen_fp8.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, i, i, i, p, f, i, p, sz, f, f, f, i,
                                            p]
        lib.sdpa_fwd_varlen_fp8.restype = i
        lib.sdpa_fwd_int8_workspace_size.argtypes = [i, i, i, i, i, i, i, i]
        lib.sdpa_fwd_int8_workspace_size.restype = sz
        lib.sdpa_fwd_int8.argtypes = [p, p, p, p, p, i, i, i, i, i, i, p, p, p, p, f, i, p, sz, i, i, p]
        lib.sdpa_fwd_int8.restype = i
        lib.sdpa_fwd_host_workspace_size.argtypes = [i, i, i, i, i, i, i, i]
        lib.sdpa_fwd_host_workspace_size.restype = sz
        lib.sdpa_fwd_host.argtypes = [p, p, p, p, p, i, i, i, i, i, i, i, f, i, p, sz, i, i, p]
        lib.sdpa_fwd_host.restype = i
        lib.sdpa_decode_workspace_size.argtypes = [i, i, i, i]
        lib.sdpa_decode_workspace_size.restype = sz
        lib.sdpa_decode.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, p, f, p, sz, i, p]
        lib.sdpa_decode.restype = i
        lib.sdpa_check_device_status.argtypes = [p]
        lib.sdpa_check_device_status.restype = i
        lib.sdpa_status_string.argtypes = [i]
        lib.sdpa_status_string.restype = ctypes.c_char_p
        lib.sdpa_version.argtypes = []
        lib.sdpa_version.restype = i
        _lib = lib
        return lib


def library():
    """The loaded ctypes library (raises if it has not been built)."""
    return _load()


def declared_functions():
    """Names of the functions include/sdpa.h declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(sdpa_\w+)\s*\(", text, flags=re.M)))


def sdpa_status_string(status: int) -> str:
    return _load().sdpa_status_string(int(status)).decode()


def sdpa_version() -> int:
    return _load().sdpa_version()


def _stream_ptr(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(name, rc):
    if rc != SDPA_OK:
        raise SdpaError(name, rc)


def _i64(vals):
    arr = (ctypes.c_int64 * len(vals))(*[int(x) for x in vals])
    return arr


def _on_device(**tensors):
    """Every given tensor (None skipped) must be a CUDA tensor on the current device with a unit
    innermost stride: the library takes raw device pointers for the current device's stream."""
    dev = torch.cuda.current_device() if torch.cuda.is_available() else None
    for name, t in tensors.items():
        if t is None:
            continue
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
        if t.device.index != dev:
            raise ValueError(f"{name} is on {t.device}, not on the current device cuda:{dev}")
        if t.dim() > 0 and t.stride(-1) != 1:
            raise ValueError(f"{name} must have a unit innermost stride")


def _int32_vector(name, t, n=None):
    if t.dtype != torch.int32 or t.dim() != 1 or (n is not None and t.numel() != n):
        raise ValueError(f"{name} must be an int32 vector" + ("" if n is None else f" of {n} entries"))


def _check_decode(q, k, v, kv_len, out, lse, cache_dims=4):
    if q.dim() != 3 or k.dim() != cache_dims or v.dim() != cache_dims:
        raise ValueError("q must be [B, Hq, D] and the caches [*, rows, Hkv, D|Dv]")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q and the caches must share one dtype")
    _on_device(q=q, k_cache=k, v_cache=v, kv_len=kv_len, out=out, lse=lse)
    _int32_vector("kv_len", kv_len, q.shape[0])
    B, Hq, _ = q.shape
    Dv = v.shape[-1]
    if out is not None and (tuple(out.shape) != (B, Hq, Dv) or out.dtype != q.dtype):
        raise ValueError(f"out must be a {q.dtype} tensor of shape {(B, Hq, Dv)}")
    if lse is not None and (tuple(lse.shape) != (B, Hq) or lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise ValueError(f"lse must be a contiguous fp32 tensor of shape {(B, Hq)}")


def sdpa_fwd_workspace_size(B: int, Hq: int, Sq: int, Sk: int, Dv: int, causal: bool, has_mask: bool) -> int:
    """Bytes of prefill workspace for the current device: the condensed mask (required with a
    mask) followed by the partials of the split last round of work tiles (optional)."""
    return int(_load().sdpa_fwd_workspace_size(B, Hq, Sq, Sk, Dv, int(bool(causal)), int(bool(has_mask))))


def sdpa_decode_workspace_size(B: int, Hq: int, max_kv: int, Dv: int) -> int:
    return int(_load().sdpa_decode_workspace_size(B, Hq, max_kv, Dv))


def _fwd_args(q, k, v, out, lse, mask, workspace, out_dtype, return_lse, causal):
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, S, H, D]")
    B, Sq, Hq, D = q.shape
    _, Sk, Hkv, _ = k.shape
    Dv = v.shape[-1]
    _on_device(q=q, k=k, v=v, out=out, lse=lse, mask=mask, workspace=workspace)
    if out is None:
        out = torch.empty((B, Sq, Hq, Dv), dtype=out_dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    if lse is not None and (tuple(lse.shape) != (B, Hq, Sq) or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous fp32 [B, Hq, Sq] tensor")
    strides = _i64([*q.stride()[:3], *k.stride()[:3], *v.stride()[:3], *out.stride()[:3]])
    mstr = None
    if mask is not None:
        if mask.dtype != torch.float16 or mask.dim() != 3 or mask.stride(-1) != 1:
            raise ValueError("mask must be an fp16 [B, Sq, Sk] tensor with unit innermost stride")
        mstr = _i64([mask.stride(0), mask.stride(1)])
    if workspace is None:
        need = sdpa_fwd_workspace_size(B, Hq, Sq, Sk, Dv, causal, mask is not None)
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return B, Sq, Hq, Hkv, Sk, D, Dv, out, lse, strides, mstr, workspace, ws_bytes


def sdpa_fwd(q, k, v, *, scale: float | None = None, causal: bool = False, mask=None, out=None, lse=None,
             return_lse: bool = True, workspace=None, stream=None):
    """O = softmax(scale * Q K^T + mask) V for fp16/bf16 q [B,Sq,Hq,D], k [B,Sk,Hkv,D], v [B,Sk,Hkv,Dv].

    Returns (o [B,Sq,Hq,Dv] in the input dtype, lse [B,Hq,Sq] fp32 or None)."""
    if q.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("sdpa_fwd takes fp16 or bf16 inputs (use sdpa_fwd_fp8 for e4m3)")
    scale = 1.0 / math.sqrt(q.shape[-1]) if scale is None else float(scale)
    B, Sq, Hq, Hkv, Sk, D, Dv, out, lse, strides, mstr, workspace, ws_bytes = _fwd_args(
        q, k, v, out, lse, mask, workspace, q.dtype, return_lse, causal)
    rc = _load().sdpa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Sk, D, Dv, strides,
                          scale, int(bool(causal)), _ptr(mask), mstr, _ptr(workspace), ws_bytes, _DT[q.dtype],
                          _DT[out.dtype], _stream_ptr(stream))
    _check("sdpa_fwd", rc)
    return out, lse


def sdpa_fwd_fp8(q, k, v, descale_q: float, descale_k: float, descale_v: float, *, scale: float | None = None,
                 causal: bool = False, mask=None, out=None, lse=None, return_lse: bool = True, workspace=None,
                 stream=None):
    """e4m3 prefill: Q = q * descale_q (likewise K, V).  Returns (o bf16, lse fp32 or None)."""
    if q.dtype != torch.float8_e4m3fn:
        raise ValueError("sdpa_fwd_fp8 takes float8_e4m3fn inputs")
    scale = 1.0 / math.sqrt(q.shape[-1]) if scale is None else float(scale)
    B, Sq, Hq, Hkv, Sk, D, Dv, out, lse, strides, mstr, workspace, ws_bytes = _fwd_args(
        q, k, v, out, lse, mask, workspace, torch.bfloat16, return_lse, causal)
    rc = _load().sdpa_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Sk, D, Dv, strides,
                              scale, int(bool(causal)), _ptr(mask), mstr, _ptr(workspace), ws_bytes,
                              float(descale_q), float(descale_k), float(descale_v), _DT[out.dtype],
                              _stream_ptr(stream))
    _check("sdpa_fwd_fp8", rc)
    return out, lse


def sdpa_fwd_varlen_workspace_size(B: int) -> int:
    """Bytes of workspace a packed prefill of B sequences needs (the per-sequence tile prefix)."""
    return int(_load().sdpa_fwd_varlen_workspace_size(B))


def _varlen_args(q, k, v, cu_seqlens_q, cu_seqlens_k, out, lse, workspace, out_dtype, return_lse):
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise ValueError("q, k, v must be packed [total, H, D]")
    total_q, Hq, D = q.shape
    total_k, Hkv, _ = k.shape
    Dv = v.shape[-1]
    _on_device(q=q, k=k, v=v, cu_seqlens_q=cu_seqlens_q, cu_seqlens_k=cu_seqlens_k, out=out, lse=lse,
               workspace=workspace)
    for t, name in ((cu_seqlens_q, "cu_seqlens_q"), (cu_seqlens_k, "cu_seqlens_k")):
        _int32_vector(name, t)
    B = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != B + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both hold B + 1 offsets")
    if out is None:
        out = torch.empty((total_q, Hq, Dv), dtype=out_dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
    if lse is not None and (tuple(lse.shape) != (Hq, total_q) or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous fp32 [Hq, total_q] tensor")
    if workspace is None:
        workspace = torch.empty(max(16, sdpa_fwd_varlen_workspace_size(B)), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    strides = _i64([*q.stride()[:2], *k.stride()[:2], *v.stride()[:2], *out.stride()[:2]])
    return B, total_q, total_k, Hq, Hkv, D, Dv, out, lse, strides, workspace, ws_bytes


def sdpa_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, *, scale: float | None = None,
                    causal: bool = False, out=None, lse=None, return_lse: bool = True, workspace=None, stream=None):
    """Prefill of B sequences packed back to back: q [total_q,Hq,D], k [total_k,Hkv,D], v [total_k,Hkv,Dv]
    (fp16/bf16); sequence b owns rows cu_seqlens_q[b]..cu_seqlens_q[b+1]-1 (keys likewise), both
    int32 [B+1] on the device; max_seqlen_q bounds every query length.  Causal masking is top-left
    within each sequence.  Returns (o [total_q,Hq,Dv], lse [Hq,total_q] fp32 or None)."""
    if q.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("sdpa_fwd_varlen takes fp16 or bf16 inputs (use sdpa_fwd_varlen_fp8 for e4m3)")
    scale = 1.0 / math.sqrt(q.shape[-1]) if scale is None else float(scale)
    B, total_q, total_k, Hq, Hkv, D, Dv, out, lse, strides, workspace, ws_bytes = _varlen_args(
        q, k, v, cu_seqlens_q, cu_seqlens_k, out, lse, workspace, q.dtype, return_lse)
    rc = _load().sdpa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q),
                                 _ptr(cu_seqlens_k), B, Hq, Hkv, total_q, total_k, int(max_seqlen_q), D, Dv, strides,
                                 scale, int(bool(causal)), _ptr(workspace), ws_bytes, _DT[q.dtype], _DT[out.dtype],
                                 _stream_ptr(stream))
    _check("sdpa_fwd_varlen", rc)
    return out, lse


def sdpa_fwd_varlen_fp8(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, descale_q: float,
                        descale_k: float, descale_v: float, *, scale: float | None = None, causal: bool = False,
                        out=None, lse=None, return_lse: bool = True, workspace=None, stream=None):
    """sdpa_fwd_varlen with e4m3 codes and per-tensor scales.  Returns (o bf16, lse fp32 or None)."""
    if q.dtype != torch.float8_e4m3fn:
        raise ValueError("sdpa_fwd_varlen_fp8 takes float8_e4m3fn inputs")
    scale = 1.0 / math.sqrt(q.shape[-1]) if scale is None else float(scale)
    B, total_q, total_k, Hq, Hkv, D, Dv, out, lse, strides, workspace, ws_bytes = _varlen_args(
        q, k, v, cu_seqlens_q, cu_seqlens_k, out, lse, workspace, torch.bfloat16, return_lse)
    rc = _load().sdpa_fwd_varlen_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q),
                                     _ptr(cu_seqlens_k), B, Hq, Hkv, total_q, total_k, int(max_seqlen_q), D, Dv,
                                     strides, scale, int(bool(causal)), _ptr(workspace), ws_bytes, float(descale_q),
                                     float(descale_k), float(descale_v), _DT[out.dtype], _stream_ptr(stream))
    _check("sdpa_fwd_varlen_fp8", rc)
    return out, lse


def sdpa_fwd_int8_workspace_size(B: int, Hq: int, Hkv: int, Sq: int, Sk: int, D: int, v_int8: bool,
                                 causal: bool) -> int:
    """Bytes of workspace for sdpa_fwd_int8: 16-bit copies of the int8 operands, then the optional
    split partials."""
    return int(_load().sdpa_fwd_int8_workspace_size(B, Hq, Hkv, Sq, Sk, D, int(bool(v_int8)), int(bool(causal))))


def sdpa_fwd_int8(q, k, v, q_scale, k_scale, v_scale=None, *, scale: float | None = None, causal: bool = False,
                  out_dtype=torch.float16, out=None, lse=None, return_lse: bool = True, workspace=None,
                  stream=None):
    """Prefill with int8 codes: q [B,Sq,Hq,D], k [B,Sk,Hkv,D] int8 with fp32 scales q_scale
    [B,Hq,ceil(Sq/128)], k_scale [B,Hkv,ceil(Sk/128)] (one per 128-row block); v either out_dtype values
    or int8 codes with per-channel v_scale [B,Hkv,D].  Returns (o [B,Sq,Hq,D] out_dtype, lse or None)."""
    if q.dtype != torch.int8 or k.dtype != torch.int8:
        raise ValueError("sdpa_fwd_int8 takes int8 q and k codes")
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, S, H, D]")
    B, Sq, Hq, D = q.shape
    _, Sk, Hkv, _ = k.shape
    _on_device(q=q, k=k, v=v, q_scale=q_scale, k_scale=k_scale, v_scale=v_scale, out=out, lse=lse,
               workspace=workspace)
    nqb, nkb = (Sq + 127) // 128, (Sk + 127) // 128
    checks = [(q_scale, (B, Hq, nqb), "q_scale"), (k_scale, (B, Hkv, nkb), "k_scale")]
    if v_scale is not None:
        checks.append((v_scale, (B, Hkv, D), "v_scale"))
    for t, shape, name in checks:
        if t.dtype != torch.float32 or not t.is_cuda or tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor of shape {shape}")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty((B, Sq, Hq, D), dtype=out_dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    if lse is not None and (tuple(lse.shape) != (B, Hq, Sq) or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous fp32 [B, Hq, Sq] tensor")
    if workspace is None:
        workspace = torch.empty(max(16, sdpa_fwd_int8_workspace_size(B, Hq, Hkv, Sq, Sk, D, v.dtype == torch.int8,
                                                                     causal)), dtype=torch.uint8, device=q.device)
    strides = _i64([*q.stride()[:3], *k.stride()[:3], *v.stride()[:3], *out.stride()[:3]])
    rc = _load().sdpa_fwd_int8(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Sk, D, strides,
                               _ptr(q_scale), _ptr(k_scale), _ptr(v_scale), scale, int(bool(causal)),
                               _ptr(workspace), workspace.numel() * workspace.element_size(), _DT[v.dtype],
                               _DT[out.dtype], _stream_ptr(stream))
    _check("sdpa_fwd_int8", rc)
    return out, lse


def sdpa_fwd_host_workspace_size(B: int, Hq: int, Hkv: int, Sq: int, Sk: int, D: int, Dv: int,
                                 causal: bool) -> int:
    """Bytes of device workspace for sdpa_fwd_host (device copies of Q, K, V, O, LSE + split partials)."""
    return int(_load().sdpa_fwd_host_workspace_size(B, Hq, Hkv, Sq, Sk, D, Dv, int(bool(causal))))


def sdpa_fwd_host(q, k, v, *, scale: float | None = None, causal: bool = False, out=None, lse=None,
                  return_lse: bool = True, workspace=None, device=None, stream=None):
    """sdpa_fwd on CPU tensors (pinned for overlap): copies up, computes and copies back in chunks of
    query rows, overlapping the three.  q [B,Sq,Hq,D], k [B,Sk,Hkv,D], v [B,Sk,Hkv,Dv] contiguous
    fp16/bf16 CPU tensors.  Returns (o, lse) CPU tensors, valid once the stream is synchronized."""
    for t in (q, k, v):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("sdpa_fwd_host takes contiguous CPU tensors")
    if q.dtype not in (torch.float16, torch.bfloat16) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("sdpa_fwd_host takes fp16 or bf16 inputs of one type")
    B, Sq, Hq, D = q.shape
    _, Sk, Hkv, _ = k.shape
    Dv = v.shape[-1]
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty((B, Sq, Hq, Dv), dtype=q.dtype).pin_memory()
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32).pin_memory()
    for t, shape in ((out, (B, Sq, Hq, Dv)), (lse, (B, Hq, Sq))):
        if t is not None and (t.is_cuda or not t.is_contiguous() or tuple(t.shape) != shape):
            raise ValueError(f"outputs must be contiguous CPU tensors of shape {shape}")
    if workspace is None:
        workspace = torch.empty(sdpa_fwd_host_workspace_size(B, Hq, Hkv, Sq, Sk, D, Dv, causal), dtype=torch.uint8,
                                device=dev)
    rc = _load().sdpa_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Sk, D, Dv, scale,
                               int(bool(causal)), _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _DT[q.dtype], _DT[out.dtype], _stream_ptr(stream))
    _check("sdpa_fwd_host", rc)
    return out, lse


def sdpa_decode(q, k_cache, v_cache, kv_len, *, scale: float | None = None, out=None, lse=None,
                return_lse: bool = True, workspace=None, stream=None):
    """Decode: q [B,Hq,D], caches [B,max_kv,Hkv,D|Dv], kv_len int32 [B] (device).  Returns (o, lse)."""
    _check_decode(q, k_cache, v_cache, kv_len, out, lse)
    _on_device(workspace=workspace)
    B, Hq, D = q.shape
    _, max_kv, Hkv, _ = k_cache.shape
    Dv = v_cache.shape[-1]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty((B, Hq, Dv), dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    need = sdpa_decode_workspace_size(B, Hq, max_kv, Dv)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    strides = _i64([*q.stride()[:2], *k_cache.stride()[:3], *v_cache.stride()[:3], *out.stride()[:2]])
    rc = _load().sdpa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), _ptr(out), _ptr(lse), B, Hq,
                             Hkv, max_kv, D, Dv, strides, scale, _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _DT[q.dtype], _stream_ptr(stream))
    _check("sdpa_decode", rc)
    return out, lse


def sdpa_decode_paged(q, k_pool, v_pool, page_table, kv_len, *, scale: float | None = None, out=None, lse=None,
                      return_lse: bool = True, workspace=None, stream=None):
    """Decode over a paged cache: q [B,Hq,D], pools [n_pages,page_size,Hkv,D|Dv], page_table int32
    [B, max_pages] (device; logical page -> physical page), kv_len int32 [B] (device)."""
    _check_decode(q, k_pool, v_pool, kv_len, out, lse)
    _on_device(page_table=page_table, workspace=workspace)
    if page_table.dim() != 2 or page_table.dtype != torch.int32 or page_table.shape[0] != q.shape[0]:
        raise ValueError("page_table must be an int32 [B, max_pages] tensor")
    B, Hq, D = q.shape
    n_pages, page_size, Hkv, _ = k_pool.shape
    Dv = v_pool.shape[-1]
    max_pages = page_table.shape[1]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty((B, Hq, Dv), dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(sdpa_decode_workspace_size(B, Hq, max_pages * page_size, Dv), dtype=torch.uint8,
                                device=q.device)
    strides = _i64([*q.stride()[:2], *k_pool.stride()[:3], *v_pool.stride()[:3], *out.stride()[:2],
                    page_table.stride(0)])
    lib = _load()
    fn = lib.sdpa_decode_paged
    p, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, i, i, i, p, f, p, ctypes.c_size_t, i, p]
    fn.restype = i
    rc = fn(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), _ptr(kv_len), _ptr(out), _ptr(lse), B, Hq, Hkv,
            page_size, max_pages, n_pages, D, Dv, strides, scale, _ptr(workspace),
            workspace.numel() * workspace.element_size(), _DT[q.dtype], _stream_ptr(stream))
    _check("sdpa_decode_paged", rc)
    return out, lse


def sdpa_check_device_status(stream=None) -> int:
    """Synchronizes the stream and returns (and clears) the device status (SDPA_OK if clean)."""
    return int(_load().sdpa_check_device_status(_stream_ptr(stream)))


def sdpa_decode_noalloc(q, k_cache, v_cache, kv_len, *, scale: float | None = None, out=None, lse=None,
                        return_lse: bool = True, stream=None):
    """sdpa_decode without a workspace: the per-split partials go to a fixed 32 MiB array inside
    the library, for callers that cannot allocate device memory (an allocator-free runtime, a host
    that hands out device memory only through its own pool, a hot path that must not call cudaMalloc).

    Such callers pass ``out`` (and ``lse``) themselves; this wrapper only allocates them when they
    are omitted.  The first call on a device resolves the array's address and should precede any
    stream capture; calls that overlap on the GPU share the array and race."""
    _check_decode(q, k_cache, v_cache, kv_len, out, lse)
    lib = _load()
    fn = lib.sdpa_decode_noalloc
    p, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, p, f, i, p]
    fn.restype = i
    B, Hq, D = q.shape
    _, max_kv, Hkv, _ = k_cache.shape
    Dv = v_cache.shape[-1]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty((B, Hq, Dv), dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    strides = _i64([*q.stride()[:2], *k_cache.stride()[:3], *v_cache.stride()[:3], *out.stride()[:2]])
    rc = fn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len), _ptr(out), _ptr(lse), B, Hq, Hkv, max_kv, D, Dv,
            strides, scale, _DT[q.dtype], _stream_ptr(stream))
    _check("sdpa_decode_noalloc", rc)
    return out, lse
