"""sdpa_decode_noalloc, the decode entry point that allocates nothing.  It serves callers that
cannot allocate device memory where they run attention: a runtime without a device allocator of
its own, a host whose pool hands out no memory to libraries, or a serving loop that must not call
cudaMalloc on its hot path.  Its partial results go to a fixed array
inside the library instead of a caller workspace.  Through the C ABI its results must equal
sdpa_decode's bit for bit (the same kernels on the same inputs), on two calls in a row that share
the fixed array, and match the fp64 oracle.

This file is collected last on purpose, so that a run stopping at the first failure has
already run every other test."""
import ctypes

import pytest
import torch

import flash_attention_forward_gb300 as fa
import oracle
import workloads
from parity import TOL_16BIT, TOL_LSE_BF16, TOL_LSE_F16, assert_close, assert_lse_close

pytestmark = pytest.mark.gpu

DEV = "cuda"
W = workloads.WORKLOADS["splitkv_decode_bf16_d128"]


def _noalloc_fn():
    fn = fa.library().sdpa_decode_noalloc
    p, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, p, f, i, p]
    fn.restype = i
    return fn


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _check(o, lse, ref, x, w, dtype):
    ref_o, ref_lse = ref
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse), "no-alloc and workspace decode differ"
    oo, ol = oracle.sdpa_decode(x["q"], x["k"], x["v"], x["kv_len"], scale=w.scale)
    assert_close(o.float().cpu().numpy(), oo, TOL_16BIT)
    assert_lse_close(lse.cpu().numpy(), ol, TOL_LSE_F16 if dtype == "f16" else TOL_LSE_BF16)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_noalloc_decode_matches_workspace_decode_on_two_calls(dtype):
    fn = _noalloc_fn()
    w = W.with_shape(B=8, Sk=6000, dtype=dtype)
    # the second call has shorter sequences, so stale partials of the first call stay in the
    # shared array past the splits the second call reads
    lengths = ([6000, 5999, 4097, 3000, 2048, 1025, 777, 6000], [1, 1024, 1500, 0, 300, 2049, 4096, 17])
    stream = torch.cuda.current_stream()
    code = fa.SDPA_BF16 if dtype == "bf16" else fa.SDPA_F16
    for call, lens in enumerate(lengths):
        x = workloads.decode_inputs(w, rotation=call, kv_len=lens)
        q, k, v, kvl = (x[n].to(DEV) for n in ("q", "k", "v", "kv_len"))
        ref = fa.sdpa_decode(q, k, v, kvl, scale=w.scale)
        o = torch.full((w.B, w.Hq, w.Dv), float("nan"), dtype=q.dtype, device=DEV)
        lse = torch.full((w.B, w.Hq), float("nan"), dtype=torch.float32, device=DEV)
        rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(kvl), _ptr(o), _ptr(lse), w.B, w.Hq, w.Hkv, w.Sk, w.D, w.Dv, None,
                w.scale, code, ctypes.c_void_p(stream.cuda_stream))
        assert rc == fa.SDPA_OK, fa.sdpa_status_string(rc)
        torch.cuda.synchronize()
        assert fa.sdpa_check_device_status() == fa.SDPA_OK
        _check(o, lse, ref, x, w, dtype)


def test_noalloc_decode_with_strided_caches():
    # caches that are slices of wider tensors (the K and V halves of one fused buffer) and an
    # output with padded rows: the strides go through the C ABI as given
    fn = _noalloc_fn()
    w = W.with_shape(B=4, Sk=3000)
    x = workloads.decode_inputs(w, kv_len=[3000, 1, 2048, 999])
    kv = torch.empty((w.B, w.Sk, w.Hkv, w.D + w.Dv), dtype=torch.bfloat16, device=DEV)
    kv[..., :w.D] = x["k"].to(DEV)
    kv[..., w.D:] = x["v"].to(DEV)
    k, v = kv[..., :w.D], kv[..., w.D:]
    q, kvl = x["q"].to(DEV), x["kv_len"].to(DEV)
    ref = fa.sdpa_decode(q, k, v, kvl, scale=w.scale)
    o_buf = torch.full((w.B, w.Hq, w.Dv + 64), float("nan"), dtype=torch.bfloat16, device=DEV)
    o = o_buf[..., :w.Dv]
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=DEV)
    st = [*q.stride()[:2], *k.stride()[:3], *v.stride()[:3], *o.stride()[:2]]
    strides = (ctypes.c_int64 * len(st))(*st)
    rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(kvl), _ptr(o), _ptr(lse), w.B, w.Hq, w.Hkv, w.Sk, w.D, w.Dv, strides,
            w.scale, fa.SDPA_BF16, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == fa.SDPA_OK, fa.sdpa_status_string(rc)
    torch.cuda.synchronize()
    assert fa.sdpa_check_device_status() == fa.SDPA_OK
    _check(o, lse, ref, x, w, "bf16")
    assert torch.isnan(o_buf[..., w.Dv:].float()).all()  # the padding of the output rows is untouched


def test_noalloc_rejects_more_than_its_scratch():
    fn = _noalloc_fn()
    q = torch.zeros((64, 32, 128), dtype=torch.bfloat16, device=DEV)
    kv = torch.zeros((1, 8, 8, 128), dtype=torch.bfloat16, device=DEV)  # never read: rejected first
    kvl = torch.zeros((64,), dtype=torch.int32, device=DEV)
    o = torch.zeros((64, 32, 128), dtype=torch.bfloat16, device=DEV)
    # 64 * 32 * ceil(131072 / 2048) * 130 * 4 bytes = 68 MB > 32 MiB
    rc = fn(_ptr(q), _ptr(kv), _ptr(kv), _ptr(kvl), _ptr(o), None, 64, 32, 8, 131072, 128, 128, None, 0.088,
            fa.SDPA_BF16, None)
    assert rc == fa.SDPA_ERR_UNSUPPORTED
