"""GPU parity of the packed variable-length prefill (sdpa_fwd_varlen / sdpa_fwd_varlen_fp8)
against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import flash_attention_forward_gb300 as fa
import oracle
import workloads
from parity import TOL_16BIT, TOL_FP8, TOL_LSE_BF16, TOL_LSE_F16, assert_close, assert_lse_close

pytestmark = pytest.mark.gpu

DEV = "cuda"
SENTINEL = 7.0

# (query lengths, key lengths, Hq, Hkv, D, Dv): lengths around the 128-row tiles and 256-row work
# tiles, a sequence without queries, one without keys, key lengths unlike query lengths, GQA.
CASES = [
    ([1], [1], 1, 1, 64, 64),
    ([300, 0, 129, 1, 256, 257], [300, 0, 129, 1, 256, 257], 4, 2, 128, 128),
    ([5, 700, 128], [900, 3, 0], 2, 1, 128, 128),
    ([513, 77, 1000], [513, 77, 1000], 8, 2, 64, 64),
    ([200, 333], [200, 333], 2, 2, 192, 128),
]


def _gpu(x):
    return [x[n].to(DEV) for n in ("q", "k", "v", "cu_q", "cu_k")]


def _run(x, max_q, scale, causal, fp8=False):
    q, k, v, cu_q, cu_k = _gpu(x)
    Hq, Dv = q.shape[1], v.shape[2]
    out_dtype = torch.bfloat16 if fp8 else q.dtype
    o = torch.full((q.shape[0], Hq, Dv), SENTINEL, dtype=out_dtype, device=DEV)
    lse = torch.full((Hq, q.shape[0]), SENTINEL, dtype=torch.float32, device=DEV)
    if fp8:
        fa.sdpa_fwd_varlen_fp8(q, k, v, cu_q, cu_k, max_q, *x["descale"], scale=scale, causal=causal, out=o, lse=lse)
    else:
        fa.sdpa_fwd_varlen(q, k, v, cu_q, cu_k, max_q, scale=scale, causal=causal, out=o, lse=lse)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _check(x, o, lse, scale, causal, tol, tol_lse, descale=(1.0, 1.0, 1.0)):
    assert fa.sdpa_check_device_status() == fa.SDPA_OK
    ref_o, ref_lse = oracle.sdpa_fwd_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], scale=scale,
                                            causal=causal, descale=descale)
    owned = int(x["cu_q"][-1])
    assert_close(o[:owned], ref_o[:owned], tol)
    assert_lse_close(lse[:, :owned], ref_lse[:, :owned], tol_lse)
    # rows that belong to no sequence are never written
    assert (o[owned:] == SENTINEL).all() and (lse[:, owned:] == SENTINEL).all()


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_varlen_matches_oracle(case, causal, dtype):
    seq_q, seq_k, Hq, Hkv, D, Dv = CASES[case]
    x = workloads.varlen_pack(seq_q, seq_k, Hq, Hkv, D, Dv, dtype=dtype, seed=40 + case, pad_q=3, pad_k=5)
    scale = 1.0 / np.sqrt(D)
    o, lse = _run(x, max(seq_q), scale, causal)
    _check(x, o, lse, scale, causal, TOL_16BIT, TOL_LSE_F16 if dtype == "f16" else TOL_LSE_BF16)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", [1, 2, 4])
def test_varlen_fp8_matches_oracle(case, causal):
    seq_q, seq_k, Hq, Hkv, D, Dv = CASES[case]
    x = workloads.varlen_pack(seq_q, seq_k, Hq, Hkv, D, Dv, dtype="e4m3", seed=60 + case, pad_q=2, pad_k=0)
    scale = 1.0 / np.sqrt(D)
    o, lse = _run(x, max(seq_q), scale, causal, fp8=True)
    _check(x, o, lse, scale, causal, TOL_FP8, TOL_LSE_F16, descale=x["descale"])


def test_varlen_equal_lengths_match_dense_call():
    # packing B equal-length sequences is a reshape of the dense batch: both entry points must agree
    B, S, Hq, Hkv, D = 3, 300, 4, 2, 128
    x = workloads.varlen_pack([S] * B, [S] * B, Hq, Hkv, D, D, dtype="bf16", seed=71)
    q, k, v, cu_q, cu_k = _gpu(x)
    o1, l1 = fa.sdpa_fwd_varlen(q, k, v, cu_q, cu_k, S, causal=True)
    o2, l2 = fa.sdpa_fwd(q.view(B, S, Hq, D), k.view(B, S, Hkv, D), v.view(B, S, Hkv, D), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(B, S, Hq, D), o2)
    assert torch.equal(l1.view(Hq, B, S).transpose(0, 1), l2)


def test_varlen_strided_views():
    # q and o as head-dim slices of wider rows: row and head strides from the views
    seq = [130, 260]
    Hq, Hkv, D = 4, 2, 128
    x = workloads.varlen_pack(seq, seq, Hq, Hkv, D, D, dtype="bf16", seed=72)
    q, k, v, cu_q, cu_k = _gpu(x)
    wide = torch.zeros((q.shape[0], Hq, D + 64), dtype=q.dtype, device=DEV)
    wide[:, :, 32:32 + D] = q
    qv = wide[:, :, 32:32 + D]
    obuf = torch.full((q.shape[0], Hq + 1, D), SENTINEL, dtype=q.dtype, device=DEV)
    ov = obuf[:, 1:]
    fa.sdpa_fwd_varlen(qv, k, v, cu_q, cu_k, max(seq), causal=True, out=ov)
    o_ref, _ = fa.sdpa_fwd_varlen(q, k, v, cu_q, cu_k, max(seq), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(ov, o_ref)
    assert (obuf[:, 0] == SENTINEL).all()


def test_bad_offsets_store_nothing_and_report_invalid():
    seq = [300, 100]
    x = workloads.varlen_pack(seq, seq, 2, 1, 64, 64, dtype="f16", seed=73)
    q, k, v, cu_q, cu_k = _gpu(x)
    o = torch.full((q.shape[0], 2, 64), SENTINEL, dtype=q.dtype, device=DEV)
    # decreasing offsets
    bad = torch.tensor([0, 300, 200], dtype=torch.int32, device=DEV)
    fa.sdpa_fwd_varlen(q, k, v, bad, cu_k, 300, out=o)
    assert fa.sdpa_check_device_status() == fa.SDPA_ERR_INVALID
    assert (o == SENTINEL).all()
    # a sequence longer than max_seqlen_q claims more work tiles than the launch has
    fa.sdpa_fwd_varlen(q, k, v, cu_q, cu_k, 100, out=o)
    assert fa.sdpa_check_device_status() == fa.SDPA_ERR_INVALID
    assert (o == SENTINEL).all()
    # the context stays usable and a good call still matches the oracle
    o, lse = _run(x, 300, 0.125, True)
    _check(x, o, lse, 0.125, True, TOL_16BIT, TOL_LSE_F16)


def test_host_validation_rejects_before_launch():
    x = workloads.varlen_pack([10, 20], [10, 20], 2, 2, 64, 64, dtype="bf16", seed=74)
    q, k, v, cu_q, cu_k = _gpu(x)
    with pytest.raises(fa.SdpaError) as e:
        fa.sdpa_fwd_varlen(q, k, v, cu_q, cu_k, 31)  # max_seqlen_q > total_q
    assert e.value.status == fa.SDPA_ERR_INVALID
    with pytest.raises(fa.SdpaError) as e:
        fa.sdpa_fwd_varlen(q, k, v, cu_q, cu_k, 20, workspace=torch.empty(8, dtype=torch.uint8, device=DEV))
    assert e.value.status == fa.SDPA_ERR_INVALID
    with pytest.raises(fa.SdpaError) as e:
        fa.sdpa_fwd_varlen(q[:, :, :48], k[:, :, :48], v[:, :, :48], cu_q, cu_k, 20)  # head dim 48 not built
    assert e.value.status == fa.SDPA_ERR_UNSUPPORTED
    assert fa.sdpa_check_device_status() == fa.SDPA_OK


def test_full_size_workload_sampled_rows():
    # the packed workload at the size the benchmark times, checked on sampled (row, head) pairs:
    # the first, second and last row of every sequence plus seeded random rows
    w = workloads.WORKLOADS["varlen_causal_prefill_bf16_d128"]
    x = workloads.varlen_inputs(w)
    q, k, v, cu_q, cu_k = _gpu(x)
    o, lse = fa.sdpa_fwd_varlen(q, k, v, cu_q, cu_k, max(x["lengths"]), scale=w.scale, causal=w.causal)
    torch.cuda.synchronize()
    assert fa.sdpa_check_device_status() == fa.SDPA_OK
    assert not bool(torch.isnan(o).any()) and not bool(torch.isnan(lse).any())
    cu = x["cu_q"].tolist()
    g = np.random.default_rng(5)
    rows = set()
    for b in range(w.B):
        for r in (cu[b], cu[b] + 1, cu[b + 1] - 1, int(g.integers(cu[b], cu[b + 1]))):
            rows.add((r, int(g.integers(w.Hq))))
    rows = sorted(rows)
    group = w.Hq // w.Hkv
    by_head = {}
    for n, (r, h) in enumerate(rows):
        by_head.setdefault(h, []).append((n, r))
    ref_o = np.empty((len(rows), w.Dv))
    ref_lse = np.empty((len(rows),))
    for h, items in by_head.items():
        kvh = h // group
        oo, ll = oracle.sdpa_fwd_varlen(x["q"][:, h:h + 1], x["k"][:, kvh:kvh + 1], x["v"][:, kvh:kvh + 1],
                                        x["cu_q"], x["cu_k"], scale=w.scale, causal=w.causal,
                                        rows=[[r, 0] for _, r in items])
        for j, (n, _) in enumerate(items):
            ref_o[n], ref_lse[n] = oo[j], ll[j]
    ri = torch.tensor([r for r, _ in rows], device=DEV)
    hi = torch.tensor([h for _, h in rows], device=DEV)
    assert_close(o[ri, hi].float().cpu().numpy(), ref_o, TOL_16BIT)
    assert_lse_close(lse[hi, ri].cpu().numpy(), ref_lse, TOL_LSE_BF16)
