"""sdpa_decode_noalloc, the decode entry point that allocates nothing (for callers that cannot
allocate device memory, e.g. code running under CUDA graph capture): through the C ABI its
results must match sdpa_decode's, on two calls in a row that share its fixed scratch array.

This file is collected last on purpose, so that a run stopping at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import flash_attention_forward_gb300 as fa
import workloads
from parity import TOL_16BIT

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _noalloc_fn():
    fn = fa.library().sdpa_decode_noalloc
    p, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, p, f, i, p]
    fn.restype = i
    return fn


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_decode_matches_workspace_decode_on_two_calls():
    fn = _noalloc_fn()
    w = workloads.WORKLOADS["splitkv_decode_bf16_d128"].with_shape(B=8, Sk=6000)
    # the second call has shorter sequences, so stale partials of the first call stay in the
    # shared array past the splits the second call reads
    lengths = ([6000, 5999, 4097, 3000, 2048, 1025, 777, 6000], [1, 1024, 1500, 0, 300, 2049, 4096, 17])
    stream = torch.cuda.current_stream()
    for call, lens in enumerate(lengths):
        x = workloads.decode_inputs(w, rotation=call, kv_len=lens)
        q, k, v, kvl = (x[n].to(DEV) for n in ("q", "k", "v", "kv_len"))
        ref_o, ref_lse = fa.sdpa_decode(q, k, v, kvl, scale=w.scale)
        o = torch.full((w.B, w.Hq, w.Dv), float("nan"), dtype=torch.bfloat16, device=DEV)
        lse = torch.full((w.B, w.Hq), float("nan"), dtype=torch.float32, device=DEV)
        rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(kvl), _ptr(o), _ptr(lse), w.B, w.Hq, w.Hkv, w.Sk, w.D, w.Dv, None,
                w.scale, fa.SDPA_BF16, ctypes.c_void_p(stream.cuda_stream))
        assert rc == fa.SDPA_OK, fa.sdpa_status_string(rc)
        torch.cuda.synchronize()
        assert fa.sdpa_check_device_status() == fa.SDPA_OK
        got = o.float().cpu().numpy()
        assert np.isfinite(got).all(), f"call {call}: NaN/Inf in the no-alloc output"
        err = float(np.abs(got - ref_o.float().cpu().numpy()).max())
        assert err <= TOL_16BIT, f"call {call}: max abs difference {err}"
        ref_l, got_l = ref_lse.cpu().numpy(), lse.cpu().numpy()
        assert np.array_equal(np.isneginf(ref_l), np.isneginf(got_l))
        fin = np.isfinite(ref_l)
        assert np.abs(got_l[fin] - ref_l[fin]).max() <= 1e-3


def test_noalloc_rejects_more_than_its_scratch():
    fn = _noalloc_fn()
    q = torch.zeros((64, 32, 128), dtype=torch.bfloat16, device=DEV)
    kv = torch.zeros((1, 8, 8, 128), dtype=torch.bfloat16, device=DEV)  # never read: rejected first
    kvl = torch.zeros((64,), dtype=torch.int32, device=DEV)
    o = torch.zeros((64, 32, 128), dtype=torch.bfloat16, device=DEV)
    # 64 * 32 * ceil(65536 / 1024) * 130 * 4 bytes = 68 MB > 32 MiB
    rc = fn(_ptr(q), _ptr(kv), _ptr(kv), _ptr(kvl), _ptr(o), None, 64, 32, 8, 65536, 128, 128, None, 0.088,
            fa.SDPA_BF16, None)
    assert rc == fa.SDPA_ERR_UNSUPPORTED
