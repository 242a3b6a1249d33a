"""GPU parity of the FP8 e4m3 prefill against the fp64 oracle on codes x per-tensor scales."""
import numpy as np
import pytest
import torch

import flash_attention_forward_gb300 as fa
import oracle
import workloads
from parity import TOL_FP8, TOL_LSE_F16, assert_close, assert_lse_close, gather_rows, oracle_rows, sample_rows

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _run(x, scale, causal, use_mask=False):
    sq, sk, sv = x["descale"]
    m = x["mask"].to(DEV) if use_mask else None
    o, lse = fa.sdpa_fwd_fp8(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), sq, sk, sv, scale=scale,
                             causal=causal, mask=m)
    torch.cuda.synchronize()
    assert fa.sdpa_check_device_status() == fa.SDPA_OK
    return o, lse


@pytest.mark.parametrize("D", [128, 192])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 2, 2, 1, 1), (1, 2, 1, 129, 200), (2, 4, 4, 300, 300), (1, 2, 2, 513, 640)])
def test_small_shapes_match_oracle(shape, D, causal):
    B, Hq, Hkv, Sq, Sk = shape
    x = workloads.custom_prefill(B, Hq, Hkv, Sq, Sk, D, 128, dtype="e4m3", seed=Sq + Sk + D + causal)
    scale = 1.0 / np.sqrt(D)
    o, lse = _run(x, scale, causal)
    assert o.dtype == torch.bfloat16
    ref_o, ref_lse = oracle.sdpa_fwd(x["q"], x["k"], x["v"], scale=scale, causal=causal, descale=x["descale"])
    assert_close(o.float().cpu().numpy(), ref_o, TOL_FP8)
    assert_lse_close(lse.cpu().numpy(), ref_lse, TOL_LSE_F16)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 2, 1, 129, 200), (2, 4, 4, 300, 300)])
def test_d64_matches_oracle(shape, causal):
    B, Hq, Hkv, Sq, Sk = shape
    x = workloads.custom_prefill(B, Hq, Hkv, Sq, Sk, 64, 64, dtype="e4m3", seed=Sq + Sk + causal + 64)
    o, lse = _run(x, 0.125, causal)
    assert o.shape[-1] == 64
    ref_o, ref_lse = oracle.sdpa_fwd(x["q"], x["k"], x["v"], scale=0.125, causal=causal, descale=x["descale"])
    assert_close(o.float().cpu().numpy(), ref_o, TOL_FP8)
    assert_lse_close(lse.cpu().numpy(), ref_lse, TOL_LSE_F16)


def test_fp8_with_mask():
    x = workloads.custom_prefill(2, 2, 2, 300, 500, 192, 128, dtype="e4m3", seed=41, mask=True)
    o, lse = _run(x, 1 / np.sqrt(192), True, use_mask=True)
    ref_o, ref_lse = oracle.sdpa_fwd(x["q"], x["k"], x["v"], x["mask"], scale=1 / np.sqrt(192), causal=True,
                                     descale=x["descale"])
    assert_close(o.float().cpu().numpy(), ref_o, TOL_FP8)
    assert_lse_close(lse.cpu().numpy(), ref_lse, TOL_LSE_F16)


def test_mla_fp8_workload_sampled_rows():
    w = workloads.WORKLOADS["mla_fp8_causal_prefill_d192"]
    x = workloads.prefill_inputs(w)
    o, lse = _run(x, w.scale, True)
    rows = sample_rows(w.B, w.Hq, w.Sq, 160, seed=5, extra=[(0, 0, 0), (0, 127, 8191), (0, 64, 4096)])
    ref_o, ref_lse = oracle_rows(x["q"], x["k"], x["v"], None, rows, scale=w.scale, causal=True,
                                 descale=x["descale"])
    got_o, got_lse = gather_rows(o, lse, rows)
    assert_close(got_o, ref_o, TOL_FP8)
    assert_lse_close(got_lse, ref_lse, TOL_LSE_F16)
    assert torch.isfinite(o).all()


def test_strided_v():
    # a V whose rows are strided (a slice of a wider tensor): its raw e4m3 boxes come in by TMA with
    # the caller's row stride
    B, Hq, Hkv, Sq, Sk, D, Dv = 1, 2, 2, 200, 333, 128, 128
    x = workloads.custom_prefill(B, Hq, Hkv, Sq, Sk, D, Dv, dtype="e4m3", seed=77)
    wide = torch.zeros((B, Sk, Hkv, 2 * Dv), dtype=torch.uint8, device=DEV)
    wide[..., :Dv] = x["v"].view(torch.uint8).to(DEV)
    v = wide.view(torch.float8_e4m3fn)[..., :Dv]
    sq, sk, sv = x["descale"]
    o, lse = fa.sdpa_fwd_fp8(x["q"].to(DEV), x["k"].to(DEV), v, sq, sk, sv, scale=1 / np.sqrt(D), causal=True)
    torch.cuda.synchronize()
    assert fa.sdpa_check_device_status() == fa.SDPA_OK
    ref_o, ref_lse = oracle.sdpa_fwd(x["q"], x["k"], x["v"], scale=1 / np.sqrt(D), causal=True, descale=x["descale"])
    assert_close(o.float().cpu().numpy(), ref_o, TOL_FP8)
    assert_lse_close(lse.cpu().numpy(), ref_lse, TOL_LSE_F16)
