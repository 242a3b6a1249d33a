"""GPU parity of the fp16/bf16 prefill kernel against the fp64 oracle (through the C ABI)."""
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


def _run(x, scale, causal, use_mask):
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    m = x["mask"].to(DEV) if use_mask else None
    o, lse = fa.sdpa_fwd(q, k, v, scale=scale, causal=causal, mask=m)
    torch.cuda.synchronize()
    assert fa.sdpa_check_device_status() == fa.SDPA_OK
    return o, lse


# (B, Hq, Hkv, Sq, Sk, D): ragged lengths around the 128-row/key tiles and 256-row CTAs,
# GQA groups 1, 2, 4, 8; the corner cases of the page "Xe2 ESIMD Flash Attention", section
# "Workflow" (q not 16-aligned, kv not chunk- or 8-aligned, kv shorter than a chunk).
SHAPES = [
    (1, 1, 1, 1, 1, 64),
    (1, 2, 1, 17, 2, 64),
    (2, 4, 2, 129, 127, 64),
    (1, 2, 2, 256, 128, 128),
    (1, 4, 1, 257, 129, 128),
    (2, 8, 1, 300, 1000, 128),
    (1, 2, 2, 513, 513, 128),
    (1, 3, 3, 100, 77, 128),
    (1, 4, 4, 640, 384, 64),
]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("use_mask", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_small_shapes_match_oracle(shape, dtype, causal, use_mask):
    B, Hq, Hkv, Sq, Sk, D = shape
    x = workloads.custom_prefill(B, Hq, Hkv, Sq, Sk, D, D, dtype=dtype, seed=hash(shape) % 1000 + 7 * causal,
                                 mask=use_mask, masked_frac=0.1, full_row_frac=0.05)
    scale = 1.0 / np.sqrt(D)
    o, lse = _run(x, scale, causal, use_mask)
    ref_o, ref_lse = oracle.sdpa_fwd(x["q"], x["k"], x["v"], x["mask"] if use_mask else None, scale=scale,
                                     causal=causal)
    assert_close(o.float().cpu().numpy(), ref_o, TOL_16BIT)
    assert_lse_close(lse.cpu().numpy(), ref_lse, TOL_LSE_F16 if dtype == "f16" else TOL_LSE_BF16)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("use_mask", [False, True])
@pytest.mark.parametrize("shape", [(1, 2, 1, 300, 500), (2, 4, 2, 257, 129), (1, 1, 1, 1, 1)])
def test_d192_dv128_matches_oracle(shape, dtype, causal, use_mask):
    # Dv != D on 16-bit inputs: the QK contraction runs over 192 dims, P.V produces 128
    B, Hq, Hkv, Sq, Sk = shape
    x = workloads.custom_prefill(B, Hq, Hkv, Sq, Sk, 192, 128, dtype=dtype, seed=Sq * 7 + Sk + causal + 2 * use_mask,
                                 mask=use_mask, masked_frac=0.1, full_row_frac=0.05)
    scale = 1.0 / np.sqrt(192)
    o, lse = _run(x, scale, causal, use_mask)
    assert o.shape[-1] == 128
    ref_o, ref_lse = oracle.sdpa_fwd(x["q"], x["k"], x["v"], x["mask"] if use_mask else None, scale=scale,
                                     causal=causal)
    assert_close(o.float().cpu().numpy(), ref_o, TOL_16BIT)
    assert_lse_close(lse.cpu().numpy(), ref_lse, TOL_LSE_F16 if dtype == "f16" else TOL_LSE_BF16)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_split_tail_agrees_with_unsplit_and_oracle(dtype):
    # 6 work tiles of 2 x 128 rows are far fewer than the SMs: each is split into 8 key ranges
    # (when the workspace holds the partials) and merged; with a workspace too small for the
    # partials the same call runs unsplit.  Both must match the oracle.
    B, Hq, Hkv, Sq, Sk, D = 1, 3, 1, 500, 2000, 128
    x = workloads.custom_prefill(B, Hq, Hkv, Sq, Sk, D, D, dtype=dtype, seed=913)
    scale = 1.0 / np.sqrt(D)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    need = fa.sdpa_fwd_workspace_size(B, Hq, Sq, Sk, D, False, False)
    assert need > 0
    o_split, lse_split = fa.sdpa_fwd(q, k, v, scale=scale, workspace=torch.empty(need, dtype=torch.uint8, device=DEV))
    o_whole, lse_whole = fa.sdpa_fwd(q, k, v, scale=scale, workspace=torch.empty(16, dtype=torch.uint8, device=DEV))
    torch.cuda.synchronize()
    assert fa.sdpa_check_device_status() == fa.SDPA_OK
    ref_o, ref_lse = oracle.sdpa_fwd(x["q"], x["k"], x["v"], scale=scale)
    tol_lse = TOL_LSE_F16 if dtype == "f16" else TOL_LSE_BF16
    for o, lse in ((o_split, lse_split), (o_whole, lse_whole)):
        assert_close(o.float().cpu().numpy(), ref_o, TOL_16BIT)
        assert_lse_close(lse.cpu().numpy(), ref_lse, tol_lse)
    # the causal path never splits: its workspace size is zero without a mask
    assert fa.sdpa_fwd_workspace_size(B, Hq, Sq, Sk, D, True, False) == 0


def test_split_with_key_ranges_fully_masked_for_some_rows():
    # rows whose visible keys fall in only some of the split key ranges: the other ranges
    # contribute max = -inf and sum = 0 to the merge; fully masked rows give O = 0, LSE = -inf
    B, Hq, Hkv, Sq, Sk, D = 1, 2, 2, 300, 1500, 64
    x = workloads.custom_prefill(B, Hq, Hkv, Sq, Sk, D, D, dtype="bf16", seed=57)
    mask = torch.zeros((B, Sq, Sk), dtype=torch.float16)
    mask[:, 0:100, :1000] = float("-inf")      # only the last ranges are visible
    mask[:, 100:150, 200:] = float("-inf")     # only the first ranges are visible
    mask[:, 150:160, :] = float("-inf")        # nothing visible
    mask[:, 160:170, 700:701] = 3.0            # a finite non-zero value inside one range
    x["mask"] = mask
    scale = 1.0 / np.sqrt(D)
    o, lse = _run(x, scale, False, True)
    ref_o, ref_lse = oracle.sdpa_fwd(x["q"], x["k"], x["v"], x["mask"], scale=scale)
    assert_close(o.float().cpu().numpy(), ref_o, TOL_16BIT)
    assert_lse_close(lse.cpu().numpy(), ref_lse, TOL_LSE_BF16)
    assert torch.all(o[:, 150:160] == 0) and torch.all(torch.isneginf(lse[:, :, 150:160]))


def test_tiny_workload_full_output():
    w = workloads.WORKLOADS["tiny_prefill_f16_d64"]
    x = workloads.prefill_inputs(w)
    o, lse = _run(x, w.scale, w.causal, False)
    ref_o, ref_lse = oracle.sdpa_fwd(x["q"], x["k"], x["v"], scale=w.scale, causal=w.causal)
    assert o.dtype == torch.float16
    assert_close(o.float().cpu().numpy(), ref_o, TOL_16BIT)
    assert_lse_close(lse.cpu().numpy(), ref_lse, TOL_LSE_F16)


def test_gqa_causal_workload_sampled_rows():
    w = workloads.WORKLOADS["gqa_causal_prefill_bf16_d128"]
    x = workloads.prefill_inputs(w)
    o, lse = _run(x, w.scale, w.causal, False)
    rows = sample_rows(w.B, w.Hq, w.Sq, 400, seed=2, extra=[(0, 0, 0), (1, 31, 4095), (0, 5, 3967)])
    ref_o, ref_lse = oracle_rows(x["q"], x["k"], x["v"], None, rows, scale=w.scale, causal=True)
    got_o, got_lse = gather_rows(o, lse, rows)
    assert_close(got_o, ref_o, TOL_16BIT)
    assert_lse_close(got_lse, ref_lse)
    # properties over the whole output: finite everywhere, row 0 of every head is V[0]
    assert torch.isfinite(o).all()
    v0 = x["v"][:, 0].to(DEV).repeat_interleave(w.Hq // w.Hkv, dim=1)
    assert torch.equal(o[:, 0], v0)


def test_unaligned_mask_workload_sampled_rows():
    w = workloads.WORKLOADS["unaligned_mask_prefill_bf16_d128"]
    x = workloads.prefill_inputs(w)
    o, lse = _run(x, w.scale, w.causal, True)
    full = torch.isinf(x["mask"]).all(dim=-1)  # [B, Sq] fully masked rows
    fb, fi = torch.nonzero(full, as_tuple=True)
    extra = [(int(fb[j]), j % w.Hq, int(fi[j])) for j in range(0, len(fb), 7)]
    rows = sample_rows(w.B, w.Hq, w.Sq, 400, seed=3, extra=extra + [(2, 27, 999)])
    ref_o, ref_lse = oracle_rows(x["q"], x["k"], x["v"], x["mask"], rows, scale=w.scale, causal=False)
    got_o, got_lse = gather_rows(o, lse, rows)
    assert_close(got_o, ref_o, TOL_16BIT)
    assert_lse_close(got_lse, ref_lse)
    # every fully masked row is exactly zero with LSE = -inf, in every head
    fm = full.to(DEV)
    assert torch.all(o.float().abs().sum(dim=-1)[fm] == 0)
    assert torch.all(torch.isneginf(lse.permute(0, 2, 1)[fm]))
    assert torch.isfinite(o).all()


def test_general_additive_mask_values():
    # finite non-zero mask entries take the rare path that adds them to the scores
    x = workloads.custom_prefill(2, 4, 2, 200, 300, 128, 128, dtype="bf16", seed=11, mask=True)
    g = torch.Generator().manual_seed(12)
    bias = (torch.rand((2, 200, 300), generator=g) * 4 - 2).to(torch.float16)
    bias[:, :50] = 0  # some block rows with only 0 / -inf
    m = torch.where(torch.isinf(x["mask"]), x["mask"], bias)
    x["mask"] = m
    o, lse = _run(x, 1 / np.sqrt(128), True, True)
    ref_o, ref_lse = oracle.sdpa_fwd(x["q"], x["k"], x["v"], m, scale=1 / np.sqrt(128), causal=True)
    assert_close(o.float().cpu().numpy(), ref_o, TOL_16BIT)
    assert_lse_close(lse.cpu().numpy(), ref_lse)


def test_strided_views_and_broadcast_mask():
    # q/k/v as views into a packed [B, S, 3, H, D] buffer; mask broadcast over batch (stride 0)
    B, S, H, D = 2, 300, 4, 128
    g = torch.Generator().manual_seed(21)
    qkv = torch.randn((B, S, 3, H, D), generator=g).to(torch.bfloat16)
    mask1 = torch.where(torch.rand((1, S, S), generator=g) < 0.2, float("-inf"), 0.0).to(torch.float16)
    mask1[:, :, 0] = 0
    d = qkv.to(DEV)
    q, k, v = d[:, :, 0], d[:, :, 1], d[:, :, 2]
    m = mask1.to(DEV).expand(B, S, S)
    o, lse = fa.sdpa_fwd(q, k, v, scale=0.1, causal=False, mask=m)
    torch.cuda.synchronize()
    ref_o, ref_lse = oracle.sdpa_fwd(qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2], mask1.expand(B, S, S), scale=0.1)
    assert_close(o.float().cpu().numpy(), ref_o, TOL_16BIT)
    assert_lse_close(lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("Sk,first", [(5, 3), (1100, 1), (2100, 7), (1031, 0)])
def test_mask_views_at_every_alignment(Sk, first):
    # the mask as a window of a wider buffer: rows start at every 2-byte offset from a 16-byte
    # boundary (row 0 too, when `first` is odd), so the condensing reads key by key at the row
    # edges and shifts the 16-byte chunks between them; Sk = 1100 and 2100 span several groups
    # of 1024 keys, and some rows hold finite non-zero values
    B, Sq, H = 2, 70, 2
    x = workloads.custom_prefill(B, H, H, Sq, Sk, 64, 64, dtype="f16", seed=Sk + first)
    g = torch.Generator().manual_seed(Sk)
    wide = torch.where(torch.rand((B, Sq, Sk + 13), generator=g) < 0.3, float("-inf"), 0.0).to(torch.float16)
    wide[:, :, first] = 0  # the first key of every row stays visible
    wide[:, 5:9, first + Sk // 2] = 1.5
    m = wide[:, :, first:first + Sk]
    x["mask"] = m.contiguous()
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = fa.sdpa_fwd(q, k, v, scale=0.125, causal=False, mask=wide.to(DEV)[:, :, first:first + Sk])
    torch.cuda.synchronize()
    assert fa.sdpa_check_device_status() == fa.SDPA_OK
    ref_o, ref_lse = oracle.sdpa_fwd(x["q"], x["k"], x["v"], x["mask"], scale=0.125)
    assert_close(o.float().cpu().numpy(), ref_o, TOL_16BIT)
    assert_lse_close(lse.cpu().numpy(), ref_lse, TOL_LSE_F16)


def test_output_canaries_untouched():
    # O written into the middle of a larger buffer: the padding around it must stay as it was
    B, Sq, Sk, H, D = 1, 130, 200, 2, 64
    x = workloads.custom_prefill(B, H, H, Sq, Sk, D, D, dtype="f16", seed=31)
    big = torch.full((B, Sq + 2, H, D + 64), 7.0, dtype=torch.float16, device=DEV)
    out = big[:, 1:Sq + 1, :, 32:32 + D]
    lse_big = torch.full((B * H * Sq + 64,), 5.0, device=DEV)
    lse = lse_big[32:32 + B * H * Sq].view(B, H, Sq)
    fa.sdpa_fwd(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), scale=0.125, out=out, lse=lse)
    torch.cuda.synchronize()
    ref_o, _ = oracle.sdpa_fwd(x["q"], x["k"], x["v"], scale=0.125)
    assert_close(out.float().cpu().numpy(), ref_o, TOL_16BIT)
    keep = torch.ones_like(big, dtype=torch.bool)
    keep[:, 1:Sq + 1, :, 32:32 + D] = False
    assert torch.all(big[keep] == 7.0)
    assert torch.all(lse_big[:32] == 5.0) and torch.all(lse_big[32 + B * H * Sq:] == 5.0)


def test_invalid_arguments_launch_nothing():
    q = torch.zeros((1, 8, 2, 64), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(fa.SdpaError) as e:
        fa.sdpa_fwd(q, q[:, :, :1].repeat(1, 1, 3, 1), q, scale=0.1)  # Hq % Hkv != 0
    assert e.value.status == fa.SDPA_ERR_INVALID
    with pytest.raises(fa.SdpaError) as e:
        fa.sdpa_fwd(q, q, q, scale=-1.0)
    assert e.value.status == fa.SDPA_ERR_INVALID
    q96 = torch.zeros((1, 8, 2, 96), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(fa.SdpaError) as e:
        fa.sdpa_fwd(q96, q96, q96, scale=0.1)
    assert e.value.status == fa.SDPA_ERR_UNSUPPORTED
