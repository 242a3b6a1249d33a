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
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 8), (16, 2), (8, 1), (12, 1), (16, 1), (32, 2)])
@pytest.mark.parametrize("D", [128, 192])
def test_ragged_lengths_nan_padding(dtype, Hq, Hkv, D):
    # lengths around the 16-key step, the 64-key chunk, the 2048-key split (and the former
    # 1024-key one), and 0;
    # padding rows are NaN, so reading any of them would poison the output.  Groups of 9-16
    # query heads use the second half of the tensor-core tile's rows; D = 192 with Dv = 128 is
    # the MLA-shaped head of the "MlaMmaOp" page.
    lens = [0, 1, 15, 16, 17, 255, 256, 257, 1023, 1024, 1025, 2047, 2048, 2049, 3000, 4096]
    w = W.with_shape(B=len(lens), Hq=Hq, Hkv=Hkv, Sk=4096, dtype=dtype, D=D)
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


@pytest.mark.parametrize("D", [128, 192])
def test_decode_equals_prefill_with_one_query(D):
    # the split/combine result equals the unsplit prefill kernel on the same keys (Sq = 1)
    w = W.with_shape(B=2, Sk=5000, D=D)
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


def _paged(x, page_size, spare=5, garbage=True, seed=11):
    kp, vp, table = workloads.page_caches(x["k"], x["v"], page_size, seed=seed, spare_pages=spare)
    if garbage:
        # entries past each sequence's pages are never used for a visible key: make them wild
        for b, L in enumerate(x["kv_len"].tolist()):
            used = (int(L) + page_size - 1) // page_size
            table[b, used:] = torch.tensor([-7, 1 << 30, kp.shape[0], 3], dtype=torch.int32).repeat(64)[: table.shape[1] - used]
    return kp, vp, table


@pytest.mark.parametrize("page_size", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (8, 1, 128), (16, 1, 128), (16, 1, 192)])
def test_paged_decode_matches_oracle(page_size, Hq, Hkv, D):
    lens = [0, 1, 15, 16, 63, 64, 65, 1023, 1024, 1025, 3000]
    w = W.with_shape(B=len(lens), Hq=Hq, Hkv=Hkv, Sk=4096, D=D)
    x = workloads.decode_inputs(w, kv_len=lens)
    kp, vp, table = _paged(x, page_size)
    o, lse = fa.sdpa_decode_paged(x["q"].to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), x["kv_len"].to(DEV),
                                  scale=w.scale)
    torch.cuda.synchronize()
    assert fa.sdpa_check_device_status() == fa.SDPA_OK
    ref_o, ref_lse = oracle.sdpa_decode_paged(x["q"], kp, vp, table, x["kv_len"], scale=w.scale)
    assert_close(o.float().cpu().numpy(), ref_o, TOL_16BIT)
    assert_lse_close(lse.cpu().numpy(), ref_lse, TOL_LSE_BF16)
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))


@pytest.mark.parametrize("page_size", [16, 64, 512])
def test_paged_decode_equals_contiguous_decode(page_size):
    # paging changes only where the rows come from: chunk for chunk the same arithmetic
    w = W.with_shape(B=6, Sk=8192)
    x = workloads.decode_inputs(w, kv_len=[8192, 5000, 1, 4097, 1024, 777], pad_value=0.0)
    kp, vp, table = _paged(x, page_size, garbage=False)
    o_c, lse_c = _run(x, w.scale)
    o_p, lse_p = fa.sdpa_decode_paged(x["q"].to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), x["kv_len"].to(DEV),
                                      scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o_p, o_c) and torch.equal(lse_p, lse_c)


def test_paged_decode_workload_sampled_sequences():
    # the decode workload's caches in 64-row pages scattered over the pool
    x = workloads.decode_inputs(W, pad_value=float("nan"))
    dev_k, dev_v = x["k"].to(DEV), x["v"].to(DEV)
    kp, vp, table = workloads.page_caches(dev_k, dev_v, 64, seed=3, spare_pages=17)
    del dev_k, dev_v
    o, lse = fa.sdpa_decode_paged(x["q"].to(DEV), kp, vp, table, x["kv_len"].to(DEV), scale=W.scale)
    torch.cuda.synchronize()
    assert fa.sdpa_check_device_status() == fa.SDPA_OK
    kv = x["kv_len"].numpy()
    pick = sorted({int(np.argmin(kv)), int(np.argmax(kv)), 0, 33, W.B - 1})
    ref_o, ref_lse = oracle.sdpa_decode(x["q"], x["k"], x["v"], x["kv_len"], scale=W.scale, batches=pick)
    assert_close(o[pick].float().cpu().numpy(), ref_o, TOL_16BIT)
    assert_lse_close(lse[pick].cpu().numpy(), ref_lse)
    assert torch.isfinite(o).all()


def test_paged_decode_rejects_bad_arguments():
    w = W.with_shape(B=2, Sk=256)
    x = workloads.decode_inputs(w, kv_len=[10, 20], pad_value=0.0)
    kp, vp, table = _paged(x, 16, garbage=False)
    args = dict(q=x["q"].to(DEV), k_pool=kp.to(DEV), v_pool=vp.to(DEV), page_table=table.to(DEV),
                kv_len=x["kv_len"].to(DEV))
    with pytest.raises(fa.SdpaError):   # page_size 8: below the 16-row minimum
        kp8, vp8, t8 = _paged(x, 8, garbage=False)
        fa.sdpa_decode_paged(args["q"], kp8.to(DEV), vp8.to(DEV), t8.to(DEV), args["kv_len"], scale=w.scale)
    with pytest.raises(fa.SdpaError):   # page_size 48: not a power of two
        k48 = torch.zeros((12, 48, w.Hkv, 128), dtype=x["k"].dtype, device=DEV)
        fa.sdpa_decode_paged(args["q"], k48, k48, table[:, :6].contiguous().to(DEV), args["kv_len"], scale=w.scale)
    torch.cuda.synchronize()
    assert fa.sdpa_check_device_status() == fa.SDPA_OK
