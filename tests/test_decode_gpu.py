"""GPU parity of the two-phase split-KV decode against the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import flash_attention_forward_gb300 as fa
import oracle
import workloads
from parity import TOL_16BIT, TOL_LSE_BF16, TOL_LSE_F16, assert_close, assert_lse_close

pytestmark = pytest.mark.gpu

DEV = "cuda"
W = workloads.WORKLOADS["splitkv_decode_bf16_d128"]


def _run(x, dtype_scale, **kw):
    o, lse = fa.sdpa_decode(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), x["kv_len"].to(DEV),
                            scale=dtype_scale, **kw)
    torch.cuda.synchronize()
    assert fa.sdpa_check_device_status() == fa.SDPA_OK
    return o, lse


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 8), (16, 2), (8, 1)])
def test_ragged_lengths_nan_padding(dtype, Hq, Hkv):
    # lengths around the 16-key step, the 256-key warp share and the 1024-key split, and 0;
    # padding rows are NaN, so reading any of them would poison the output
    lens = [0, 1, 15, 16, 17, 255, 256, 257, 1023, 1024, 1025, 2047, 2048, 2049, 3000, 4096]
    w = W.with_shape(B=len(lens), Hq=Hq, Hkv=Hkv, Sk=4096, dtype=dtype)
    x = workloads.decode_inputs(w, kv_len=lens)
    o, lse = _run(x, w.scale)
    ref_o, ref_lse = oracle.sdpa_decode(x["q"], x["k"], x["v"], x["kv_len"], scale=w.scale)
    assert_close(o.float().cpu().numpy(), ref_o, TOL_16BIT)
    assert_lse_close(lse.cpu().numpy(), ref_lse, TOL_LSE_F16 if dtype == "f16" else TOL_LSE_BF16)
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_decode_workload_sampled_sequences():
    x = workloads.decode_inputs(W, pad_value=float("nan"))
    o, lse = _run(x, W.scale)
    kv = x["kv_len"].numpy()
    pick = sorted({int(np.argmin(kv)), int(np.argmax(kv)), 0, 17, 40, W.B - 1})
    ref_o, ref_lse = oracle.sdpa_decode(x["q"], x["k"], x["v"], x["kv_len"], scale=W.scale, batches=pick)
    assert_close(o[pick].float().cpu().numpy(), ref_o, TOL_16BIT)
    assert_lse_close(lse[pick].cpu().numpy(), ref_lse)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


def test_decode_equals_prefill_with_one_query():
    # the split/combine result equals the unsplit prefill kernel on the same keys (Sq = 1)
    w = W.with_shape(B=2, Sk=5000)
    x = workloads.decode_inputs(w, kv_len=[5000, 3333], pad_value=0.0)
    o, _ = _run(x, w.scale)
    for b, L in enumerate([5000, 3333]):
        q = x["q"][b:b + 1, None].to(DEV)
        k = x["k"][b:b + 1, :L].to(DEV).contiguous()
        v = x["v"][b:b + 1, :L].to(DEV).contiguous()
        op, _ = fa.sdpa_fwd(q, k, v, scale=w.scale)
        torch.cuda.synchronize()
        assert (op[0, 0].float() - o[b].float()).abs().max().item() <= 2e-2


def test_out_of_range_lengths_are_clamped():
    w = W.with_shape(B=2, Sk=300)
    x = workloads.decode_inputs(w, kv_len=[300, 5], pad_value=0.0)
    x2 = dict(x)
    x2["kv_len"] = torch.tensor([100000, -3], dtype=torch.int32)  # clamped to [0, max_kv]
    o, lse = _run(x2, w.scale)
    ref_o, _ = oracle.sdpa_decode(x["q"], x["k"], x["v"], torch.tensor([300, 0]), scale=w.scale)
    assert_close(o.float().cpu().numpy(), ref_o, TOL_16BIT)
    assert torch.isneginf(lse[1]).all()


def test_decode_rejects_bad_workspace():
    w = W.with_shape(B=1, Sk=64)
    x = workloads.decode_inputs(w, kv_len=[64], pad_value=0.0)
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(fa.SdpaError) as e:
        fa.sdpa_decode(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), x["kv_len"].to(DEV), workspace=ws)
    assert e.value.status == fa.SDPA_ERR_INVALID
