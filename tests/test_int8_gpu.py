"""GPU parity of the int8-code prefill (sdpa_fwd_int8) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import flash_attention_forward_gb300 as fa
import oracle
import workloads
from parity import (TOL_16BIT, TOL_LSE_BF16, TOL_LSE_F16, assert_close, assert_lse_close, gather_rows,
                    oracle_rows, sample_rows)

pytestmark = pytest.mark.gpu

DEV = "cuda"
OUT = {"f16": torch.float16, "bf16": torch.bfloat16}

# (B, Hq, Hkv, Sq, Sk, D): ragged lengths around the 128-row scale blocks and tiles, GQA, and the
# page's SageV1 instance (head dim 128, 512 x 512)
SHAPES = [
    (1, 1, 1, 1, 1, 64),
    (2, 4, 2, 129, 300, 64),
    (1, 2, 1, 257, 255, 128),
    (1, 4, 4, 512, 512, 128),
    (2, 8, 2, 1000, 700, 128),
]
# (V storage, output type): 16-bit V values, or int8 V codes with per-channel scales
V_MODES = [("f16", "f16"), ("bf16", "bf16"), ("i8", "f16"), ("i8", "bf16")]


def _gpu(x):
    return {n: (None if t is None else t.to(DEV)) for n, t in x.items()}


def _run(x, scale, causal, out):
    g = _gpu(x)
    o, lse = fa.sdpa_fwd_int8(g["q"], g["k"], g["v"], g["q_scale"], g["k_scale"], g["v_scale"], scale=scale,
                              causal=causal, out_dtype=OUT[out])
    torch.cuda.synchronize()
    assert fa.sdpa_check_device_status() == fa.SDPA_OK
    return o, lse


@pytest.mark.parametrize("vmode", V_MODES)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_int8_matches_oracle(shape, causal, vmode):
    B, Hq, Hkv, Sq, Sk, D = shape
    v_store, out = vmode
    x = workloads.int8_prefill(B, Hq, Hkv, Sq, Sk, D, v=v_store, seed=sum(shape) + 3 * causal)
    scale = 1.0 / np.sqrt(D)
    o, lse = _run(x, scale, causal, out)
    ref_o, ref_lse = oracle.sdpa_fwd_int8(x["q"], x["k"], x["v"], x["q_scale"], x["k_scale"], x["v_scale"],
                                          scale=scale, causal=causal)
    assert_close(o.float().cpu().numpy(), ref_o, TOL_16BIT)
    assert_lse_close(lse.cpu().numpy(), ref_lse, TOL_LSE_F16 if out == "f16" else TOL_LSE_BF16)


def test_int8_scores_are_exact_integer_products():
    # codes of +-127 in every position give the largest integer dot products (D * 127^2 < 2^24): with
    # unit scales the LSE of a row over identical keys is exactly s + ln(Sk)
    B, Hq, Sq, Sk, D = 1, 1, 130, 300, 128
    q = torch.full((B, Sq, Hq, D), 127, dtype=torch.int8)
    k = torch.full((B, Sk, Hq, D), -127, dtype=torch.int8)
    v = torch.randn(B, Sk, Hq, D, generator=torch.Generator().manual_seed(3)).to(torch.float16)
    qs = torch.ones(B, Hq, 2)
    ks = torch.ones(B, Hq, 3)
    g = _gpu({"q": q, "k": k, "v": v, "qs": qs, "ks": ks})
    scale = 2.0 ** -14  # s = -127^2 * 128 * 2^-14 = -127^2 / 128 exactly
    o, lse = fa.sdpa_fwd_int8(g["q"], g["k"], g["v"], g["qs"], g["ks"], scale=scale)
    torch.cuda.synchronize()
    want = -127.0 ** 2 / 128.0 + np.log(Sk)
    assert np.abs(lse.cpu().numpy() - want).max() <= 1e-4 * abs(want)
    ref_o, _ = oracle.sdpa_fwd_int8(q, k, v, qs, ks, scale=scale)
    assert_close(o.float().cpu().numpy(), ref_o, TOL_16BIT)


def test_int8_validation():
    x = _gpu(workloads.int8_prefill(1, 2, 1, 64, 64, 64, v="i8", seed=9))
    with pytest.raises(fa.SdpaError) as e:  # int8 V needs its per-channel scales
        fa.sdpa_fwd_int8(x["q"], x["k"], x["v"], x["q_scale"], x["k_scale"], None)
    assert e.value.status == fa.SDPA_ERR_INVALID
    v16 = x["v"].to(torch.float16)
    with pytest.raises(fa.SdpaError) as e:  # 16-bit V takes no V scales
        fa.sdpa_fwd_int8(x["q"], x["k"], v16, x["q_scale"], x["k_scale"], x["v_scale"])
    assert e.value.status == fa.SDPA_ERR_INVALID
    with pytest.raises(fa.SdpaError) as e:  # V values must be in the output type
        fa.sdpa_fwd_int8(x["q"], x["k"], v16, x["q_scale"], x["k_scale"], out_dtype=torch.bfloat16)
    assert e.value.status == fa.SDPA_ERR_UNSUPPORTED
    with pytest.raises(fa.SdpaError) as e:  # head dims 64 and 128 only
        q = torch.zeros(1, 64, 2, 192, dtype=torch.int8, device=DEV)
        k = torch.zeros(1, 64, 1, 192, dtype=torch.int8, device=DEV)
        fa.sdpa_fwd_int8(q, k, torch.zeros(1, 64, 1, 192, dtype=torch.float16, device=DEV), x["q_scale"],
                         x["k_scale"])
    assert e.value.status == fa.SDPA_ERR_UNSUPPORTED
    assert fa.sdpa_check_device_status() == fa.SDPA_OK


def test_full_size_workload_sampled_rows():
    # the workload the benchmark times, on 400 sampled rows; no NaN/Inf anywhere in O
    w = workloads.WORKLOADS["int8_qk_causal_prefill_d128"]
    x = workloads.int8_inputs(w)
    o, lse = _run(x, w.scale, w.causal, w.out_dtype)
    assert not bool(torch.isnan(o).any()) and not bool(torch.isinf(o).any())
    rows = sample_rows(w.B, w.Hq, w.Sq, 400, seed=11)
    qd = oracle.dequantize_int8(x["q"], x["q_scale"], 128)
    kd = oracle.dequantize_int8(x["k"], x["k_scale"], 128)
    ref_o, ref_lse = oracle_rows(qd, kd, x["v"], None, rows, scale=w.scale, causal=w.causal)
    got_o, got_lse = gather_rows(o, lse, rows)
    assert_close(got_o, ref_o, TOL_16BIT)
    assert_lse_close(got_lse, ref_lse, TOL_LSE_F16)


def test_int8_strided_codes_match_contiguous():
    # q and int8 v as head-dim slices of wider rows: the widening reads them through their strides
    x = workloads.int8_prefill(2, 4, 2, 300, 260, 128, v="i8", seed=21)
    g = _gpu(x)
    wide_q = torch.zeros((2, 300, 4, 192), dtype=torch.int8, device=DEV)
    wide_q[..., 32:160] = g["q"]
    wide_v = torch.zeros((2, 260, 2, 192), dtype=torch.int8, device=DEV)
    wide_v[..., 64:192] = g["v"]
    args = (g["q_scale"], g["k_scale"], g["v_scale"])
    o1, l1 = fa.sdpa_fwd_int8(wide_q[..., 32:160], g["k"], wide_v[..., 64:192], *args, causal=True)
    o2, l2 = fa.sdpa_fwd_int8(g["q"], g["k"], g["v"], *args, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
