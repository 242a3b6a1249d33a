"""fp64 CPU oracle for scaled-dot-product attention forward.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The library under
``flash_attention_forward_gb300`` never imports it and shares no code with it.

The arithmetic lives in ``oracle.cpp`` (plain two-pass fp64 softmax, one query
row at a time).  This wrapper only converts tensors to fp64 exactly as the GPU
sees them (fp16/bf16 values as stored; e4m3 codes times their per-tensor scale,
through torch's own float8 cast) and calls the C entry points.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_OUT = os.path.join(_HERE, "_obj", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.cpp into oracle/_obj/liboracle.so (plain g++, no fast-math)."""
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    if not force and os.path.exists(_OUT) and os.path.getmtime(_OUT) >= os.path.getmtime(_SRC):
        return _OUT
    tmp = _OUT + f".{os.getpid()}.tmp"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-fno-fast-math", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _OUT)
    return _OUT


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            d, i64, p = ctypes.c_double, ctypes.c_int64, ctypes.c_void_p
            lib.oracle_sdpa_fwd.argtypes = [p, p, p, p, p, p, i64, i64, i64, i64, i64, i64, i64, d, ctypes.c_int,
                                            p, i64, ctypes.c_int]
            lib.oracle_sdpa_fwd.restype = ctypes.c_int
            lib.oracle_sdpa_decode.argtypes = [p, p, p, p, p, p, i64, i64, i64, i64, i64, i64, d, ctypes.c_int]
            lib.oracle_sdpa_decode.restype = ctypes.c_int
            _lib = lib
    return _lib


def threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def as_f64(t, scale: float = 1.0) -> np.ndarray:
    """Exact fp64 view of stored values (times a per-tensor scale for e4m3 codes)."""
    if isinstance(t, np.ndarray):
        a = t.astype(np.float64, copy=False)
    else:
        a = t.detach().to("cpu").to(torch.float64).numpy()
    if scale != 1.0:
        a = a * float(scale)
    return np.ascontiguousarray(a)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def sdpa_fwd(q, k, v, mask=None, *, scale: float, causal: bool = False, rows=None, descale=(1.0, 1.0, 1.0),
             nthreads: int | None = None):
    """O and LSE of softmax(scale * Q K^T + mask) V in fp64.

    q [B,Sq,Hq,D], k [B,Sk,Hkv,D], v [B,Sk,Hkv,Dv], mask [B,Sq,Sk] or None.
    rows: optional int array [n, 3] of (b, h, i); then O is [n, Dv] and LSE [n].
    Otherwise O is [B,Sq,Hq,Dv] and LSE [B,Hq,Sq]."""
    qd, kd, vd = as_f64(q, descale[0]), as_f64(k, descale[1]), as_f64(v, descale[2])
    md = None if mask is None else as_f64(mask)
    B, Sq, Hq, D = qd.shape
    _, Sk, Hkv, _ = kd.shape
    Dv = vd.shape[-1]
    if md is not None:
        assert md.shape == (B, Sq, Sk), md.shape
    if rows is not None:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
        n = r.shape[0]
        o = np.empty((n, Dv), dtype=np.float64)
        lse = np.empty((n,), dtype=np.float64)
    else:
        r, n = None, 0
        o = np.empty((B, Sq, Hq, Dv), dtype=np.float64)
        lse = np.empty((B, Hq, Sq), dtype=np.float64)
    rc = _load().oracle_sdpa_fwd(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(md), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Sk, D,
                                 Dv, float(scale), int(bool(causal)), _ptr(r), n, nthreads or threads())
    if rc != 0:
        raise ValueError("oracle_sdpa_fwd: invalid arguments")
    return o, lse


def dequantize_int8(codes, scales, block: int | None):
    """fp64 values of int8 codes [B, S, H, D]: code * scale with scales [B, H, ceil(S / block)]
    (one per block of rows) or, for block=None, [B, H, D] (one per channel)."""
    c = as_f64(codes)
    sc = as_f64(scales)
    if block is None:
        return c * sc[:, None, :, :]
    rows = np.arange(c.shape[1]) // block  # block of each row
    return c * sc[:, :, rows].transpose(0, 2, 1)[..., None]


def sdpa_fwd_int8(q, k, v, q_scale, k_scale, v_scale=None, *, scale: float, causal: bool = False, rows=None,
                  block: int = 128, nthreads: int | None = None):
    """O and LSE of attention over int8 codes in fp64: Q = q_code * q_scale[b, h, i / block],
    K = k_code * k_scale[b, kvh, j / block], V = v values or v_code * v_scale[b, kvh, c] (page "Xe SDPA
    Forward Mainloop", section "SageV1 concrete instance": Q/K dtype, P.V dtype and scale pointers).
    The dequantised operands go through sdpa_fwd, so s = scale * q_scale * k_scale * (integer dot
    product), exactly up to fp64 rounding."""
    qd = dequantize_int8(q, q_scale, block)
    kd = dequantize_int8(k, k_scale, block)
    vd = as_f64(v) if v_scale is None else dequantize_int8(v, v_scale, None)
    return sdpa_fwd(qd, kd, vd, scale=scale, causal=causal, rows=rows, nthreads=nthreads)


def _offsets(cu):
    return [int(x) for x in (cu.tolist() if hasattr(cu, "tolist") else cu)]


def sdpa_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, *, scale: float, causal: bool = False, rows=None,
                    descale=(1.0, 1.0, 1.0), nthreads: int | None = None):
    """O and LSE of packed variable-length sequences in fp64.

    q [total_q,Hq,D], k [total_k,Hkv,D], v [total_k,Hkv,Dv]; sequence b owns query rows
    cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key rows cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1.
    Each sequence is its own attention problem (page "Xe SDPA Forward Mainloop", section "SageV1
    concrete instance": the variable-length variant of the same mainloop), computed by sdpa_fwd
    on its rows with causal masking counted from the sequence's first row.  A sequence with
    queries but no keys has every score masked: O = 0, LSE = -inf (the fully-masked-row
    convention of sdpa_fwd).

    rows: optional int array [n, 2] of (packed query row, query head), each row owned by some
    sequence; then O is [n, Dv] and LSE [n].  Otherwise O is [total_q, Hq, Dv] and LSE
    [Hq, total_q], NaN on rows no sequence owns."""
    cq, ck = _offsets(cu_seqlens_q), _offsets(cu_seqlens_k)
    assert len(cq) == len(ck) >= 2
    B = len(cq) - 1
    total_q, Hq, _ = q.shape
    Dv = v.shape[-1]

    def seq(b, sel=None):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        n = (q1 - q0) if sel is None else len(sel)
        if k1 <= k0:
            return np.zeros((n, Hq, Dv) if sel is None else (n, Dv)), np.full((Hq, n) if sel is None else (n,), -np.inf)
        r = None if sel is None else np.array([(0, h, i) for (i, h) in sel], dtype=np.int64)
        o, lse = sdpa_fwd(q[q0:q1][None], k[k0:k1][None], v[k0:k1][None], scale=scale, causal=causal, rows=r,
                          descale=descale, nthreads=nthreads)
        return (o[0], lse[0]) if sel is None else (o, lse)

    if rows is None:
        o = np.full((total_q, Hq, Dv), np.nan)
        lse = np.full((Hq, total_q), np.nan)
        for b in range(B):
            if cq[b + 1] > cq[b]:
                o[cq[b]:cq[b + 1]], lse[:, cq[b]:cq[b + 1]] = seq(b)
        return o, lse
    r = np.asarray(rows, dtype=np.int64).reshape(-1, 2)
    owner = np.searchsorted(np.asarray(cq), r[:, 0], side="right") - 1
    assert ((owner >= 0) & (owner < B)).all() and (r[:, 0] < cq[-1]).all(), "row owned by no sequence"
    o = np.empty((len(r), Dv))
    lse = np.empty((len(r),))
    for b in np.unique(owner):
        idx = np.nonzero(owner == b)[0]
        ob, lb = seq(int(b), [(int(r[n, 0]) - cq[b], int(r[n, 1])) for n in idx])
        o[idx], lse[idx] = ob, lb
    return o, lse


def sdpa_decode(q, k_cache, v_cache, kv_len, *, scale: float, batches=None, nthreads: int | None = None):
    """Decode oracle: q [B,Hq,D], caches [B,max_kv,Hkv,.], kv_len [B].

    Only the first kv_len[b] cache rows of each sequence are converted and read.  ``batches``
    restricts the work to a subset of sequences; the result then has len(batches) rows."""
    kvl = [int(x) for x in (kv_len.tolist() if hasattr(kv_len, "tolist") else kv_len)]
    B, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    Dv = v_cache.shape[-1]
    sel = list(range(B)) if batches is None else [int(b) for b in batches]
    o = np.empty((len(sel), Hq, Dv), dtype=np.float64)
    lse = np.empty((len(sel), Hq), dtype=np.float64)
    lib = _load()
    for n, b in enumerate(sel):
        L = kvl[b]
        qd = as_f64(q[b:b + 1])
        kd = as_f64(k_cache[b:b + 1, :L])
        vd = as_f64(v_cache[b:b + 1, :L])
        kl = np.array([L], dtype=np.int32)
        ob = np.empty((1, Hq, Dv), dtype=np.float64)
        lb = np.empty((1, Hq), dtype=np.float64)
        rc = lib.oracle_sdpa_decode(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(kl), _ptr(ob), _ptr(lb), 1, Hq, Hkv, L, D, Dv,
                                    float(scale), nthreads or threads())
        if rc != 0:
            raise ValueError("oracle_sdpa_decode: invalid arguments")
        o[n], lse[n] = ob[0], lb[0]
    return o, lse


def gather_pages(pool, page_table, kv_len):
    """Contiguous caches [B, max_pages * page_size, Hkv, .] from a paged pool: logical page i of
    sequence b is pool[page_table[b, i]].  Only pages holding rows below kv_len[b] are taken (the
    rest of each row stays zero), so table entries past a sequence's pages are never read.

    The reading of a paged cache (page "Xe SDPA Forward Mainloop", section "Arguments / params":
    a page table, a page size and pages per sequence): key row t of sequence b is row
    t % page_size of page page_table[b, t / page_size].  The gather is a plain index copy."""
    pool = torch.as_tensor(pool)
    table = torch.as_tensor(page_table).cpu().long()
    kvl = [int(x) for x in (kv_len.tolist() if hasattr(kv_len, "tolist") else kv_len)]
    n_pages, page_size = pool.shape[0], pool.shape[1]
    B, max_pages = table.shape
    out = torch.zeros((B, max_pages * page_size, *pool.shape[2:]), dtype=pool.dtype)
    for b in range(B):
        used = (min(kvl[b], max_pages * page_size) + page_size - 1) // page_size
        for i in range(used):
            out[b, i * page_size:(i + 1) * page_size] = pool[int(table[b, i])]
    return out


def sdpa_decode_paged(q, k_pool, v_pool, page_table, kv_len, *, scale: float, batches=None,
                      nthreads: int | None = None):
    """Decode oracle over a paged cache: the pages are gathered into contiguous caches and the
    contiguous decode oracle runs on them."""
    k = gather_pages(k_pool, page_table, kv_len)
    v = gather_pages(v_pool, page_table, kv_len)
    return sdpa_decode(q, k, v, kv_len, scale=scale, batches=batches, nthreads=nthreads)
