"""Whole-output parity at the workloads' full sizes: every element of O and LSE of the GQA causal
prefill (B=2, 32/8 heads, 4096 x 4096, D=128, bf16), the unaligned masked prefill (B=3, 28/4 heads,
1000 x 3001, fp16 additive mask), the MLA-shaped FP8 prefill (128 heads, 8192 x 8192, D=192,
Dv=128) and the split-KV decode (B=64, 32/8 heads, kv_len up to 16384) against the fp64 oracle on
the same seeded inputs, NaN/Inf counted before the maximum error (page "Xe2 ESIMD Flash
Attention - SDP Prefill & Decode", section "Correctness testing").  The oracle runs on all host
cores: about a minute for the FP8 workload, seconds for the others."""
import pytest
import torch

import flash_attention_forward_gb300 as fa
import oracle
import workloads
from parity import TOL_16BIT, TOL_FP8, TOL_LSE_BF16, TOL_LSE_FP32_SUM, assert_close, assert_lse_close

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _prefill(w):
    x = workloads.prefill_inputs(w)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    mask = x["mask"].to(DEV) if x["mask"] is not None else None
    if w.dtype == "e4m3":
        o, lse = fa.sdpa_fwd_fp8(q, k, v, *x["descale"], scale=w.scale, causal=w.causal, mask=mask)
    else:
        o, lse = fa.sdpa_fwd(q, k, v, scale=w.scale, causal=w.causal, mask=mask)
    torch.cuda.synchronize()
    assert fa.sdpa_check_device_status() == fa.SDPA_OK
    got_o, got_lse = o.float().cpu().numpy(), lse.cpu().numpy()
    del q, k, v, mask, o, lse
    torch.cuda.empty_cache()
    ref_o, ref_lse = oracle.sdpa_fwd(x["q"], x["k"], x["v"], x["mask"], scale=w.scale, causal=w.causal,
                                     descale=x["descale"])
    return got_o, got_lse, ref_o, ref_lse


@pytest.mark.parametrize("name", ["gqa_causal_prefill_bf16_d128", "unaligned_mask_prefill_bf16_d128"])
def test_bf16_prefill_workload_whole_output(name):
    got_o, got_lse, ref_o, ref_lse = _prefill(workloads.WORKLOADS[name])
    assert_close(got_o, ref_o, TOL_16BIT)
    assert_lse_close(got_lse, ref_lse, TOL_LSE_FP32_SUM)


def test_mla_fp8_workload_whole_output():
    got_o, got_lse, ref_o, ref_lse = _prefill(workloads.WORKLOADS["mla_fp8_causal_prefill_d192"])
    assert_close(got_o, ref_o, TOL_FP8)
    assert_lse_close(got_lse, ref_lse, TOL_LSE_FP32_SUM)


def test_decode_workload_whole_output():
    w = workloads.WORKLOADS["splitkv_decode_bf16_d128"]
    x = workloads.decode_inputs(w, pad_value=float("nan"))
    o, lse = fa.sdpa_decode(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), x["kv_len"].to(DEV), scale=w.scale)
    torch.cuda.synchronize()
    assert fa.sdpa_check_device_status() == fa.SDPA_OK
    ref_o, ref_lse = oracle.sdpa_decode(x["q"], x["k"], x["v"], x["kv_len"], scale=w.scale)
    assert_close(o.float().cpu().numpy(), ref_o, TOL_16BIT)
    assert_lse_close(lse.cpu().numpy(), ref_lse, TOL_LSE_BF16)
