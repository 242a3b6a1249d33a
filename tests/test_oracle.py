"""Pins for the fp64 oracle, independent of the oracle itself.

Each test checks the oracle against something the mathematics fixes: closed
forms, invariants, exhaustive tiny grids against torch's own fp64
scaled_dot_product_attention, and hand-derived values.  A plausible slip in the
oracle (a dropped mask or max term, a wrong GQA index, a causal off-by-one, a
transposed operand, a missing 1/l) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads

NEG_INF = float("-inf")


def _rand(shape, seed, lo=-1.0, hi=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.rand(shape, generator=g, dtype=torch.float64) * (hi - lo) + lo)


def _torch_sdpa(q, k, v, mask, scale, causal):
    """torch's fp64 reference on [B,S,H,D] tensors (GQA through enable_gqa)."""
    qt, kt, vt = (x.transpose(1, 2) for x in (q, k, v))
    am = None if mask is None else mask.unsqueeze(1)
    if am is not None and causal:
        Sq, Sk = q.shape[1], k.shape[1]
        keep = torch.ones(Sq, Sk, dtype=torch.bool).tril()
        am, causal = am.masked_fill(~keep, NEG_INF), False
    o = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=am, is_causal=causal, scale=scale,
                                       enable_gqa=q.shape[2] != k.shape[2])
    return o.transpose(1, 2)


def _torch_lse(q, k, mask, scale, causal):
    group = q.shape[2] // k.shape[2]
    kr = k.repeat_interleave(group, dim=2)
    s = torch.einsum("bihd,bjhd->bhij", q, kr) * scale
    if mask is not None:
        s = s + mask.unsqueeze(1)
    if causal:
        Sq, Sk = s.shape[-2:]
        keep = torch.ones(Sq, Sk, dtype=torch.bool).tril()
        s = s.masked_fill(~keep, NEG_INF)
    return torch.logsumexp(s, dim=-1)


def test_hand_worked_two_keys():
    # q = (1, 0), k0 = (2, 0), k1 = (0, 3), scale = 1/2  ->  s = (1, 0)
    q = torch.tensor([1.0, 0.0], dtype=torch.float64).view(1, 1, 1, 2)
    k = torch.tensor([[2.0, 0.0], [0.0, 3.0]], dtype=torch.float64).view(1, 2, 1, 2)
    v = torch.tensor([[1.0, -1.0], [3.0, 5.0]], dtype=torch.float64).view(1, 2, 1, 2)
    o, lse = oracle.sdpa_fwd(q, k, v, scale=0.5)
    e = math.e
    want = [(e * 1.0 + 3.0) / (e + 1.0), (e * -1.0 + 5.0) / (e + 1.0)]
    assert np.allclose(o.reshape(-1), want, rtol=0, atol=1e-15)
    assert abs(lse.item() - math.log(e + 1.0)) < 1e-15
    # causal: query 0 sees key 0 only
    o, lse = oracle.sdpa_fwd(q, k, v, scale=0.5, causal=True)
    assert np.allclose(o.reshape(-1), [1.0, -1.0], atol=0)
    assert lse.item() == pytest.approx(1.0, abs=1e-15)


def test_huge_scores_do_not_overflow():
    # scores 1000 and 999: a missing max subtraction overflows exp to inf -> nan
    q = torch.tensor([1.0], dtype=torch.float64).view(1, 1, 1, 1)
    k = torch.tensor([[1000.0], [999.0]], dtype=torch.float64).view(1, 2, 1, 1)
    v = torch.tensor([[0.0], [1.0]], dtype=torch.float64).view(1, 2, 1, 1)
    o, lse = oracle.sdpa_fwd(q, k, v, scale=1.0)
    w1 = math.exp(-1.0) / (1.0 + math.exp(-1.0))
    assert o.item() == pytest.approx(w1, abs=1e-15)
    assert lse.item() == pytest.approx(1000.0 + math.log1p(math.exp(-1.0)), abs=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_single_key_returns_v_row(causal):
    B, Sq, Hq, Hkv, D, Dv = 2, 5, 4, 2, 7, 3
    q, k, v = _rand((B, Sq, Hq, D), 1), _rand((B, 1, Hkv, D), 2), _rand((B, 1, Hkv, Dv), 3)
    mask = _rand((B, Sq, 1), 4)
    o, lse = oracle.sdpa_fwd(q, k, v, mask, scale=0.3, causal=causal)
    for b in range(B):
        for h in range(Hq):
            kvh = h // (Hq // Hkv)
            for i in range(Sq):
                assert np.array_equal(o[b, i, h], v[b, 0, kvh].numpy())
                want = 0.3 * float(q[b, i, h] @ k[b, 0, kvh]) + float(mask[b, i, 0])
                assert lse[b, h, i] == pytest.approx(want, abs=1e-14)


def test_constant_v_rows_give_that_row():
    B, Sq, Sk, Hq, Hkv, D, Dv = 1, 9, 13, 2, 1, 5, 6
    q, k = _rand((B, Sq, Hq, D), 5, -3, 3), _rand((B, Sk, Hkv, D), 6, -3, 3)
    row = _rand((Dv,), 7)
    v = row.view(1, 1, 1, Dv).expand(B, Sk, Hkv, Dv).contiguous()
    for causal in (False, True):
        o, _ = oracle.sdpa_fwd(q, k, v, scale=0.7, causal=causal)
        assert np.allclose(o, row.numpy().reshape(1, 1, 1, Dv), atol=1e-14, rtol=0)


@pytest.mark.parametrize("Sq,Sk", [(6, 6), (4, 9), (9, 4)])
def test_zero_query_is_mean_of_visible_rows(Sq, Sk):
    B, Hq, Hkv, D, Dv = 2, 3, 3, 4, 5
    q = torch.zeros((B, Sq, Hq, D), dtype=torch.float64)
    k, v = _rand((B, Sk, Hkv, D), 8), _rand((B, Sk, Hkv, Dv), 9)
    o, lse = oracle.sdpa_fwd(q, k, v, scale=1.0, causal=False)
    assert np.allclose(o, v.mean(dim=1, keepdim=True).numpy(), atol=1e-14)
    assert np.allclose(lse, math.log(Sk), atol=1e-14)
    o, lse = oracle.sdpa_fwd(q, k, v, scale=1.0, causal=True)
    for i in range(Sq):
        n = min(i + 1, Sk)  # top-left causal: key j visible iff j <= i
        assert np.allclose(o[:, i], v[:, :n].mean(dim=1).numpy(), atol=1e-14)
        assert np.allclose(lse[:, :, i], math.log(n), atol=1e-14)


def test_causal_first_row_is_first_v_row():
    B, Sq, Sk, Hq, Hkv, D, Dv = 2, 7, 7, 4, 2, 8, 8
    q, k, v = _rand((B, Sq, Hq, D), 10, -4, 4), _rand((B, Sk, Hkv, D), 11, -4, 4), _rand((B, Sk, Hkv, Dv), 12)
    o, _ = oracle.sdpa_fwd(q, k, v, scale=1.0, causal=True)
    for h in range(Hq):
        assert np.array_equal(o[:, 0, h], v[:, 0, h // 2].numpy())


@pytest.mark.parametrize("causal", [False, True])
def test_identity_v_exposes_probabilities(causal):
    # V = I (Dv = Sk) turns O into the probability matrix itself
    B, Sq, Sk, H, D = 1, 6, 8, 1, 4
    q, k = _rand((B, Sq, H, D), 13, -2, 2), _rand((B, Sk, H, D), 14, -2, 2)
    mask = _rand((B, Sq, Sk), 15)
    v = torch.eye(Sk, dtype=torch.float64).view(1, Sk, 1, Sk)
    o, _ = oracle.sdpa_fwd(q, k, v, mask, scale=0.9, causal=causal)
    P = o[0, :, 0, :]
    assert np.allclose(P.sum(axis=1), 1.0, atol=1e-14)
    s = 0.9 * (q[0, :, 0] @ k[0, :, 0].T) + mask[0]
    if causal:
        s = s.masked_fill(~torch.ones(Sq, Sk, dtype=torch.bool).tril(), NEG_INF)
        assert np.all(P[np.triu_indices(Sq, 1, Sk)] == 0.0)
    assert np.allclose(P, torch.softmax(s, dim=-1).numpy(), atol=1e-15)


def test_joint_permutation_of_keys_is_invariant():
    B, Sq, Sk, Hq, Hkv, D, Dv = 2, 5, 11, 4, 2, 6, 7
    q, k, v = _rand((B, Sq, Hq, D), 16), _rand((B, Sk, Hkv, D), 17), _rand((B, Sk, Hkv, Dv), 18)
    mask = _rand((B, Sq, Sk), 19)
    perm = torch.randperm(Sk, generator=torch.Generator().manual_seed(20))
    o1, l1 = oracle.sdpa_fwd(q, k, v, mask, scale=0.4)
    o2, l2 = oracle.sdpa_fwd(q, k[:, perm], v[:, perm], mask[:, :, perm], scale=0.4)
    assert np.allclose(o1, o2, atol=1e-14) and np.allclose(l1, l2, atol=1e-14)
    # a permutation of K alone (V not moved) must change the result
    o3, _ = oracle.sdpa_fwd(q, k[:, perm], v, mask, scale=0.4)
    assert not np.allclose(o1, o3, atol=1e-6)


def test_mask_shift_moves_lse_only():
    B, Sq, Sk, Hq, D, Dv = 1, 4, 9, 2, 5, 3
    q, k, v = _rand((B, Sq, Hq, D), 21), _rand((B, Sk, Hq, D), 22), _rand((B, Sk, Hq, Dv), 23)
    mask = _rand((B, Sq, Sk), 24)
    o1, l1 = oracle.sdpa_fwd(q, k, v, mask, scale=1.1, causal=True)
    o2, l2 = oracle.sdpa_fwd(q, k, v, mask + 2.5, scale=1.1, causal=True)
    assert np.allclose(o1, o2, atol=1e-14)
    assert np.allclose(l2, l1 + 2.5, atol=1e-13)


def test_fully_masked_rows_are_zero_without_nan():
    B, Sq, Sk, Hq, Hkv, D, Dv = 2, 6, 10, 4, 2, 8, 8
    q, k, v = _rand((B, Sq, Hq, D), 25), _rand((B, Sk, Hkv, D), 26), _rand((B, Sk, Hkv, Dv), 27)
    mask = torch.zeros((B, Sq, Sk), dtype=torch.float64)
    mask[0, 2, :] = NEG_INF
    mask[1, 5, :] = NEG_INF
    mask[1, 0, 3:] = NEG_INF  # partially masked row stays finite
    o, lse = oracle.sdpa_fwd(q, k, v, mask, scale=0.5)
    assert not np.isnan(o).any() and not np.isnan(lse).any()
    assert np.all(o[0, 2] == 0.0) and np.all(o[1, 5] == 0.0)
    assert np.all(lse[0, :, 2] == NEG_INF) and np.all(lse[1, :, 5] == NEG_INF)
    assert np.isfinite(lse[1, :, 0]).all()
    # with causal on top, row 0 of batch 1 sees key 0 only -> but key 0 is visible there
    mask2 = mask.clone()
    mask2[1, 0, 0] = NEG_INF
    o, lse = oracle.sdpa_fwd(q, k, v, mask2, scale=0.5, causal=True)
    assert np.all(o[1, 0] == 0.0) and np.all(lse[1, :, 0] == NEG_INF)


def test_gqa_equals_mha_with_repeated_heads():
    B, Sq, Sk, Hq, Hkv, D, Dv = 2, 7, 9, 6, 2, 5, 4
    q, k, v = _rand((B, Sq, Hq, D), 28), _rand((B, Sk, Hkv, D), 29), _rand((B, Sk, Hkv, Dv), 30)
    o1, l1 = oracle.sdpa_fwd(q, k, v, scale=0.8, causal=True)
    g = Hq // Hkv
    o2, l2 = oracle.sdpa_fwd(q, k.repeat_interleave(g, dim=2), v.repeat_interleave(g, dim=2), scale=0.8,
                             causal=True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # interleaved mapping (h % Hkv) would differ
    o3, _ = oracle.sdpa_fwd(q, k.repeat(1, 1, g, 1), v.repeat(1, 1, g, 1), scale=0.8, causal=True)
    assert not np.allclose(o1, o3, atol=1e-6)


@pytest.mark.parametrize("Sk", [1, 2, 127, 128, 129])
@pytest.mark.parametrize("Sq", [1, 15, 16, 17])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("use_mask", [False, True])
def test_matches_torch_sdpa_fp64(Sq, Sk, causal, use_mask):
    # the page "Xe2 ESIMD Flash Attention", section "Workflow", lists these corner cases:
    # q not 16-aligned, kv not chunk-aligned, kv not 8-aligned, kv shorter than a chunk
    B, Hq, Hkv, D, Dv = 2, 4, 2, 8, 6
    seed = 1000 * Sq + Sk + 7 * causal + 3 * use_mask
    q, k, v = _rand((B, Sq, Hq, D), seed, -2, 2), _rand((B, Sk, Hkv, D), seed + 1, -2, 2), \
        _rand((B, Sk, Hkv, Dv), seed + 2)
    mask = None
    if use_mask:
        g = torch.Generator().manual_seed(seed + 3)
        mask = torch.where(torch.rand((B, Sq, Sk), generator=g) < 0.2, NEG_INF, 0.0).to(torch.float64)
        mask[:, :, 0] = _rand((B, Sq), seed + 4)  # key 0 never -inf: no fully masked rows here
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.sdpa_fwd(q, k, v, mask, scale=scale, causal=causal)
    ref = _torch_sdpa(q, k, v, mask, scale, causal).numpy()
    assert np.abs(o - ref).max() <= 1e-12
    ref_lse = _torch_lse(q, k, mask, scale, causal).numpy()
    assert np.abs(lse - ref_lse).max() <= 1e-12


def test_row_subset_matches_full():
    B, Sq, Sk, Hq, Hkv, D, Dv = 2, 33, 40, 4, 1, 16, 8
    q, k, v = _rand((B, Sq, Hq, D), 31), _rand((B, Sk, Hkv, D), 32), _rand((B, Sk, Hkv, Dv), 33)
    o, lse = oracle.sdpa_fwd(q, k, v, scale=0.25, causal=True)
    rows = np.array([[0, 0, 0], [1, 3, 32], [0, 2, 17], [1, 1, 5]])
    os_, ls = oracle.sdpa_fwd(q, k, v, scale=0.25, causal=True, rows=rows)
    for n, (b, h, i) in enumerate(rows):
        assert np.array_equal(os_[n], o[b, i, h]) and ls[n] == lse[b, h, i]


def test_decode_matches_torch_per_sequence():
    B, Hq, Hkv, max_kv, D, Dv = 3, 8, 2, 50, 16, 16
    kv_len = torch.tensor([50, 1, 23], dtype=torch.int32)
    q = _rand((B, Hq, D), 34)
    k, v = _rand((B, max_kv, Hkv, D), 35), _rand((B, max_kv, Hkv, Dv), 36)
    k[1, 1:] = float("nan")  # padding must never be read
    v[2, 23:] = float("nan")
    o, lse = oracle.sdpa_decode(q, k, v, kv_len, scale=0.25)
    for b in range(B):
        L = int(kv_len[b])
        ref = _torch_sdpa(q[b:b + 1, None], k[b:b + 1, :L], v[b:b + 1, :L], None, 0.25, False)
        assert np.abs(o[b] - ref[0, 0].numpy()).max() <= 1e-12
        ref_lse = _torch_lse(q[b:b + 1, None], k[b:b + 1, :L], None, 0.25, False)
        assert np.abs(lse[b] - ref_lse[0, :, 0].numpy()).max() <= 1e-12
    o2, _ = oracle.sdpa_decode(q, k, v, kv_len, scale=0.25, batches=[2, 0])
    assert np.array_equal(o2[0], o[2]) and np.array_equal(o2[1], o[0])


@pytest.mark.parametrize("page_size", [16, 64])
def test_paged_decode_equals_contiguous_for_any_page_placement(page_size):
    # the paged oracle gathers pages through the table; any physical placement of the same rows,
    # garbage in spare pages and in table entries past a sequence's pages must not change the result
    w = workloads.WORKLOADS["splitkv_decode_bf16_d128"].with_shape(B=3, Hq=4, Hkv=2, Sk=256)
    x = workloads.decode_inputs(w, kv_len=[1, 100, 256], pad_value=float("nan"))
    kp, vp, table = workloads.page_caches(x["k"], x["v"], page_size, seed=5, spare_pages=7)
    used = [(int(L) + page_size - 1) // page_size for L in x["kv_len"]]
    for b, u in enumerate(used):
        table[b, u:] = -123456  # never read: past the sequence's pages
    ref_o, ref_lse = oracle.sdpa_decode(x["q"], x["k"], x["v"], x["kv_len"], scale=w.scale)
    o, lse = oracle.sdpa_decode_paged(x["q"], kp, vp, table, x["kv_len"], scale=w.scale)
    assert np.array_equal(o, ref_o) and np.array_equal(lse, ref_lse)
    # attention does not depend on key order, so swapping two fully used pages must not change a
    # row, while pointing a used entry at another sequence's page must
    t2 = table.clone()
    t2[2, 0], t2[2, 1] = table[2, 1], table[2, 0]
    o2, _ = oracle.sdpa_decode_paged(x["q"], kp, vp, t2, x["kv_len"], scale=w.scale)
    assert np.allclose(o2[2], ref_o[2], rtol=0, atol=1e-12)
    t3 = table.clone()
    t3[2, 0] = table[1, 0]
    o3, _ = oracle.sdpa_decode_paged(x["q"], kp, vp, t3, x["kv_len"], scale=w.scale)
    assert not np.allclose(o3[2], ref_o[2])


def test_e4m3_inputs_are_codes_times_scale():
    # the oracle reads e4m3 codes through torch's float8 cast, times the per-tensor scale
    x = torch.tensor([0.0, 1.0, -2.5, 448.0, 0.001953125, -0.875], dtype=torch.float32)
    codes = x.to(torch.float8_e4m3fn)
    got = oracle.as_f64(codes, 0.5)
    assert np.array_equal(got, np.array([0.0, 0.5, -1.25, 224.0, 0.0009765625, -0.4375]))


def test_workload_inputs_are_seeded_and_exact():
    w = workloads.WORKLOADS["tiny_prefill_f16_d64"]
    a, b = workloads.prefill_inputs(w), workloads.prefill_inputs(w)
    assert all(torch.equal(a[n], b[n]) for n in ("q", "k", "v"))
    assert a["q"].dtype == torch.float16 and a["q"].shape == (1, 512, 1, 64)
    assert float(a["q"].abs().max()) <= 1.0
    c = workloads.prefill_inputs(w, rotation=1)
    assert not torch.equal(a["q"], c["q"])
    m = workloads.make_mask(workloads.generator(3), 2, 100, 300, 0.1, 0.05)
    full = torch.isinf(m).all(dim=-1)
    assert int(full[0].sum()) >= 5 and int(full[1].sum()) >= 5
    frac = float(torch.isinf(m[~full]).float().mean())
    assert 0.08 < frac < 0.12


def _block_diagonal_mask(cq, ck, causal):
    """Additive [total_q, total_k] mask: 0 where query row i and key row j belong to the same
    sequence (and, when causal, j's position in it is at most i's), else -inf."""
    tq, tk = cq[-1], ck[-1]
    m = torch.full((tq, tk), NEG_INF, dtype=torch.float64)
    for b in range(len(cq) - 1):
        nq, nk = cq[b + 1] - cq[b], ck[b + 1] - ck[b]
        keep = torch.ones(nq, nk, dtype=torch.bool)
        if causal:
            keep = keep.tril()
        m[cq[b]:cq[b + 1], ck[b]:ck[b + 1]] = torch.where(keep, 0.0, NEG_INF)
    return m


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_equals_one_problem_with_block_diagonal_mask(causal):
    # packed sequences are one attention problem over all rows whose mask confines every query to
    # its own sequence's keys; torch's fp64 SDPA evaluates that problem independently of the oracle
    seq_q, seq_k = [5, 0, 17, 1, 9, 3], [7, 4, 17, 1, 2, 0]
    cq = [0, *np.cumsum(seq_q).tolist()]
    ck = [0, *np.cumsum(seq_k).tolist()]
    Hq, Hkv, D, Dv = 4, 2, 8, 6
    q, k, v = _rand((cq[-1], Hq, D), 41), _rand((ck[-1], Hkv, D), 42), _rand((ck[-1], Hkv, Dv), 43)
    o, lse = oracle.sdpa_fwd_varlen(q, k, v, cq, ck, scale=0.7, causal=causal)
    mask = _block_diagonal_mask(cq, ck, causal)
    ref = _torch_sdpa(q[None], k[None], v[None], mask[None], 0.7, False)[0].numpy()
    ref_lse = _torch_lse(q[None], k[None], mask[None], 0.7, False)[0].numpy()
    empty = np.isneginf(ref_lse[0])  # query rows of the sequence without keys
    assert empty.sum() == seq_q[5]
    assert np.abs(o[~empty] - ref[~empty]).max() <= 1e-12
    assert np.abs(lse[:, ~empty] - ref_lse[:, ~empty]).max() <= 1e-12
    assert (o[empty] == 0.0).all() and np.isneginf(lse[:, empty]).all()


def test_varlen_equal_lengths_is_the_dense_batch():
    B, S, Hq, Hkv, D, Dv = 3, 21, 4, 4, 16, 16
    q, k, v = _rand((B, S, Hq, D), 44), _rand((B, S, Hkv, D), 45), _rand((B, S, Hkv, Dv), 46)
    cu = [b * S for b in range(B + 1)]
    o, lse = oracle.sdpa_fwd_varlen(q.reshape(B * S, Hq, D), k.reshape(B * S, Hkv, D), v.reshape(B * S, Hkv, Dv),
                                    cu, cu, scale=0.5, causal=True)
    ref_o, ref_lse = oracle.sdpa_fwd(q, k, v, scale=0.5, causal=True)
    assert np.array_equal(o, ref_o.reshape(B * S, Hq, Dv))
    assert np.array_equal(lse, ref_lse.transpose(1, 0, 2).reshape(Hq, B * S))


def test_varlen_rows_and_unowned_rows():
    seq = [4, 0, 6]
    x = workloads.varlen_pack(seq, seq, 2, 1, 8, 8, dtype="bf16", seed=3, pad_q=2, pad_k=1)
    o, lse = oracle.sdpa_fwd_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], scale=0.3, causal=True)
    assert np.isnan(o[10:]).all() and np.isnan(lse[:, 10:]).all()  # padding rows belong to no sequence
    assert not np.isnan(o[:10]).any()
    # causal: the first row of each sequence is its first V row
    v = oracle.as_f64(x["v"])
    assert np.array_equal(o[0, 1], v[0, 0]) and np.array_equal(o[4, 0], v[4, 0])
    rows = np.array([[9, 1], [0, 0], [5, 1], [3, 0]])
    os_, ls = oracle.sdpa_fwd_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], scale=0.3, causal=True,
                                     rows=rows)
    for n, (i, h) in enumerate(rows):
        assert np.array_equal(os_[n], o[i, h]) and ls[n] == lse[h, i]
    with pytest.raises(AssertionError):
        oracle.sdpa_fwd_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], scale=0.3, rows=[[10, 0]])


def _torch_dequant_blocks(codes, scales, block):
    """Independent dequantisation with torch ops: each row's scale repeated over its block."""
    S = codes.shape[1]
    per_row = scales.double().repeat_interleave(block, dim=2)[:, :, :S]  # [B, H, S]
    return codes.double() * per_row.permute(0, 2, 1).unsqueeze(-1)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("v_int8", [False, True])
def test_int8_oracle_matches_torch_on_dequantized_operands(causal, v_int8):
    g = torch.Generator().manual_seed(51)
    B, Sq, Sk, Hq, Hkv, D = 2, 300, 260, 4, 2, 16
    q = torch.randint(-127, 128, (B, Sq, Hq, D), generator=g, dtype=torch.int8)
    k = torch.randint(-127, 128, (B, Sk, Hkv, D), generator=g, dtype=torch.int8)
    qs = torch.rand((B, Hq, 3), generator=g) * 0.02 + 0.001
    ks = torch.rand((B, Hkv, 3), generator=g) * 0.02 + 0.001
    if v_int8:
        v = torch.randint(-127, 128, (B, Sk, Hkv, D), generator=g, dtype=torch.int8)
        vs = torch.rand((B, Hkv, D), generator=g) * 0.01 + 0.001
        vt = v.double() * vs.double().unsqueeze(1)
    else:
        v, vs = _rand((B, Sk, Hkv, D), 52).to(torch.float16), None
        vt = v.double()
    o, lse = oracle.sdpa_fwd_int8(q, k, v, qs, ks, vs, scale=0.25, causal=causal)
    qt, kt = _torch_dequant_blocks(q, qs, 128), _torch_dequant_blocks(k, ks, 128)
    ref = _torch_sdpa(qt, kt, vt, None, 0.25, causal).numpy()
    ref_lse = _torch_lse(qt, kt, None, 0.25, causal).numpy()
    assert np.abs(o - ref).max() <= 1e-12
    assert np.abs(lse - ref_lse).max() <= 1e-12


def test_int8_block_scale_acts_on_its_rows_only():
    # doubling the scale of Q block 1 (rows 128..255) of one head changes exactly those rows
    x = workloads.int8_prefill(1, 2, 1, 300, 200, 32, seed=53)
    o1, l1 = oracle.sdpa_fwd_int8(x["q"], x["k"], x["v"], x["q_scale"], x["k_scale"], scale=0.2)
    qs = x["q_scale"].clone()
    qs[0, 1, 1] *= 2.0
    o2, l2 = oracle.sdpa_fwd_int8(x["q"], x["k"], x["v"], qs, x["k_scale"], scale=0.2)
    changed = np.abs(l2 - l1)[0] > 0  # [Hq, Sq]
    assert not changed[0].any()
    assert changed[1, 128:256].all() and not changed[1, :128].any() and not changed[1, 256:].any()
    assert np.array_equal(o1[0, :128], o2[0, :128]) and np.array_equal(o1[0, 256:], o2[0, 256:])


def test_int8_quantization_recipe():
    x = torch.randn(2, 300, 3, 16, generator=torch.Generator().manual_seed(54))
    x[1, 128:256, 2] = 0.0  # an all-zero block gets scale 1 and zero codes
    codes, scales = workloads.quantize_int8_blocks(x)
    assert scales.shape == (2, 3, 3) and codes.dtype == torch.int8
    deq = _torch_dequant_blocks(codes, scales, 128)
    per_row = scales.repeat_interleave(128, dim=2)[:, :, :300].permute(0, 2, 1).unsqueeze(-1)
    assert bool(((deq - x.double()).abs() <= per_row.double() / 2 + 1e-12).all())
    assert scales[1, 2, 1] == 1.0 and int(codes[1, 128:256, 2].abs().max()) == 0
    assert int(codes.abs().max()) == 127
    vc, vs = workloads.quantize_int8_channels(x)
    assert vs.shape == (2, 3, 16)
    assert bool(((vc.double() * vs.double().unsqueeze(1) - x.double()).abs() <= vs.double().unsqueeze(1) / 2 + 1e-12).all())


def test_key_split_recombines_exactly():
    # attention over all keys = the log-sum-exp merge of attention over two disjoint key ranges
    # (the algebra both split paths of the library rely on), to fp64 rounding
    B, Sq, Sk, Hq, Hkv, D = 1, 7, 40, 2, 1, 16
    q, k, v = _rand((B, Sq, Hq, D), 61), _rand((B, Sk, Hkv, D), 62), _rand((B, Sk, Hkv, D), 63)
    o, lse = oracle.sdpa_fwd(q, k, v, scale=0.6)
    o1, l1 = oracle.sdpa_fwd(q, k[:, :13], v[:, :13], scale=0.6)
    o2, l2 = oracle.sdpa_fwd(q, k[:, 13:], v[:, 13:], scale=0.6)
    m = np.maximum(l1, l2)
    lse_merged = m + np.log(np.exp(l1 - m) + np.exp(l2 - m))
    assert np.abs(lse_merged - lse).max() <= 1e-12
    w1 = np.exp(l1 - lse).transpose(0, 2, 1)[..., None]  # [B, Sq, Hq, 1]
    w2 = np.exp(l2 - lse).transpose(0, 2, 1)[..., None]
    assert np.abs(w1 * o1 + w2 * o2 - o).max() <= 1e-12


def test_scale_moves_between_q_and_the_softmax_scale():
    B, Sq, Sk, Hq, Hkv, D = 1, 9, 11, 2, 2, 8
    q, k, v = _rand((B, Sq, Hq, D), 64), _rand((B, Sk, Hkv, D), 65), _rand((B, Sk, Hkv, D), 66)
    o1, l1 = oracle.sdpa_fwd(q, k, v, scale=0.5, causal=True)
    o2, l2 = oracle.sdpa_fwd(q * 4.0, k, v, scale=0.125, causal=True)
    assert np.abs(o1 - o2).max() <= 1e-12 and np.abs(l1 - l2).max() <= 1e-12


def test_causal_rows_past_the_keys_see_every_key():
    # top-left alignment with Sq > Sk: rows i >= Sk - 1 see all keys, exactly as without causal masking
    B, Sq, Sk, Hq, Hkv, D = 1, 30, 12, 2, 1, 8
    q, k, v = _rand((B, Sq, Hq, D), 67), _rand((B, Sk, Hkv, D), 68), _rand((B, Sk, Hkv, D), 69)
    oc, lc = oracle.sdpa_fwd(q, k, v, scale=0.3, causal=True)
    on, ln = oracle.sdpa_fwd(q, k, v, scale=0.3, causal=False)
    assert np.array_equal(oc[:, Sk - 1:], on[:, Sk - 1:]) and np.array_equal(lc[:, :, Sk - 1:], ln[:, :, Sk - 1:])
    assert not np.allclose(oc[:, : Sk - 1], on[:, : Sk - 1])
