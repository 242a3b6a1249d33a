"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  The CUDA path (through the Python binding) and the fp64
oracle both consume the tensors made here, so both sides see bit-identical
inputs.

Seeds: every buffer set of workload ``index`` c and rotation r is drawn from
``torch.Generator('cpu').manual_seed(1000 * c + r)``.  Draw order is q, k, v,
then the mask (prefill); for decode it is q, kv_len, then per sequence the
valid K rows followed by the valid V rows (padding rows are never drawn).
Uniform[-1, 1] is ``2 * rand - 1`` in fp32; N(0, 1) is ``randn`` in fp32; the
cast to the stored type rounds to nearest even.  FP8 e4m3 codes are the
saturating RNE cast of ``x / s`` with the per-tensor scale ``s = amax / 448``.

The workload shapes follow the page "Xe2 ESIMD Flash Attention - SDP Prefill &
Decode", sections "GQA layout" (Q [q_len, headQ, HD], K/V [kv_len, headKv, HD])
and "Workflow" (small correctness size q=512, kv=1024), extended with a batch
dimension.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

E4M3_MAX = 448.0


@dataclass(frozen=True)
class Workload:
    name: str
    index: int            # 1-based workload number, feeds the seed
    kind: str             # "prefill" | "decode"
    B: int
    Hq: int
    Hkv: int
    Sq: int               # decode: 1
    Sk: int               # decode: padded cache length (max_kv)
    D: int
    Dv: int
    dtype: str            # "f16" | "bf16" | "e4m3"
    dist: str             # "uniform" | "normal"
    causal: bool = False
    mask: bool = False
    out_dtype: str = "bf16"
    kv_len_range: tuple = ()      # decode only: inclusive [lo, hi]
    masked_frac: float = 0.0      # additive mask: fraction of -inf entries
    full_row_frac: float = 0.0    # additive mask: fraction of fully -inf query rows
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def with_shape(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_prefill_f16_d64", 1, "prefill", B=1, Hq=1, Hkv=1, Sq=512, Sk=1024, D=64, Dv=64,
                 dtype="f16", dist="uniform", out_dtype="f16"),
        Workload("gqa_causal_prefill_bf16_d128", 2, "prefill", B=2, Hq=32, Hkv=8, Sq=4096, Sk=4096, D=128,
                 Dv=128, dtype="bf16", dist="normal", causal=True, out_dtype="bf16"),
        Workload("unaligned_mask_prefill_bf16_d128", 3, "prefill", B=3, Hq=28, Hkv=4, Sq=1000, Sk=3001, D=128,
                 Dv=128, dtype="bf16", dist="normal", mask=True, out_dtype="bf16", masked_frac=0.10,
                 full_row_frac=0.05),
        Workload("splitkv_decode_bf16_d128", 4, "decode", B=64, Hq=32, Hkv=8, Sq=1, Sk=16384, D=128, Dv=128,
                 dtype="bf16", dist="normal", out_dtype="bf16", kv_len_range=(1024, 16384)),
        Workload("mla_fp8_causal_prefill_d192", 5, "prefill", B=1, Hq=128, Hkv=128, Sq=8192, Sk=8192, D=192,
                 Dv=128, dtype="e4m3", dist="normal", causal=True, out_dtype="bf16"),
        # int8 Q/K codes with per-128-row-block scales, fp16 V (the SageV1 instance's head dim 128)
        Workload("int8_qk_causal_prefill_d128", 7, "prefill", B=2, Hq=32, Hkv=8, Sq=4096, Sk=4096, D=128,
                 Dv=128, dtype="i8", dist="normal", causal=True, out_dtype="f16", extra={"v": "f16"}),
        # MLA-shaped decode (QK over 192 dims, 128 value dims, as in the "MlaMmaOp" prefill) with 16
        # query heads per KV head, the widest group one decode tile holds
        Workload("mla_decode_bf16_d192_g16", 8, "decode", B=64, Hq=64, Hkv=4, Sq=1, Sk=16384, D=192, Dv=128,
                 dtype="bf16", dist="normal", out_dtype="bf16", kv_len_range=(1024, 16384)),
        # packed sequences: B sequence lengths drawn uniformly from len_range, keys = queries
        Workload("varlen_causal_prefill_bf16_d128", 6, "varlen", B=16, Hq=32, Hkv=8, Sq=8192, Sk=8192, D=128,
                 Dv=128, dtype="bf16", dist="normal", causal=True, out_dtype="bf16",
                 extra={"len_range": (64, 8192)}),
    ]
}

BY_INDEX = {w.index: w for w in WORKLOADS.values()}

_TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn, "i8": torch.int8}
INT8_MAX = 127.0
INT8_BLOCK = 128  # rows per Q / K scale block


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPE[name]


def generator(index: int, rotation: int = 0) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(1000 * index + rotation)
    return g


def _draw(g: torch.Generator, shape, dist: str) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    if dist == "normal":
        return torch.randn(shape, generator=g, dtype=torch.float32)
    raise ValueError(dist)


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor e4m3 quantisation of an fp32 tensor: (codes, scale) with x ~= codes * scale."""
    amax = float(x.abs().max())
    s = amax / E4M3_MAX if amax > 0 else 1.0
    codes = (x / s).to(torch.float8_e4m3fn)
    return codes, s


def quantize_int8_blocks(x: torch.Tensor, block: int = INT8_BLOCK):
    """Symmetric int8 codes of an fp32 [B, S, H, D] tensor with one scale per (b, h, block of
    ``block`` rows): scale = amax / 127 over the block's rows and channels (1 for an all-zero
    block), code = round-half-even(x / scale), which stays within [-127, 127].  Returns (codes
    [B, S, H, D] int8, scales [B, H, ceil(S / block)] fp32)."""
    B, S, H, D = x.shape
    nb = (S + block - 1) // block
    pad = torch.zeros((B, nb * block, H, D), dtype=torch.float32)
    pad[:, :S] = x
    amax = pad.view(B, nb, block, H, D).abs().amax(dim=(2, 4)).transpose(1, 2)  # [B, H, nb]
    scales = torch.where(amax > 0, amax / INT8_MAX, torch.ones_like(amax)).to(torch.float32).contiguous()
    per_row = scales.transpose(1, 2).repeat_interleave(block, dim=1)[:, :S]  # [B, S, H]
    codes = torch.round(x / per_row.unsqueeze(-1)).clamp(-INT8_MAX, INT8_MAX).to(torch.int8)
    return codes, scales


def quantize_int8_channels(x: torch.Tensor):
    """Symmetric int8 codes of an fp32 [B, S, H, D] tensor with one scale per (b, h, channel):
    amax over the rows / 127.  Returns (codes int8, scales [B, H, D] fp32)."""
    amax = x.abs().amax(dim=1)  # [B, H, D]
    scales = torch.where(amax > 0, amax / INT8_MAX, torch.ones_like(amax)).to(torch.float32).contiguous()
    codes = torch.round(x / scales.unsqueeze(1)).clamp(-INT8_MAX, INT8_MAX).to(torch.int8)
    return codes, scales


def int8_prefill(B, Hq, Hkv, Sq, Sk, D, v="f16", dist="normal", seed=0):
    """int8 Q/K codes with per-block scales; V as fp16 / bf16 values, or (v="i8") int8 codes with
    per-channel scales.  Draw order q, k, v in fp32, then quantisation."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    qf = _draw(g, (B, Sq, Hq, D), dist)
    kf = _draw(g, (B, Sk, Hkv, D), dist)
    vf = _draw(g, (B, Sk, Hkv, D), dist)
    q, q_scale = quantize_int8_blocks(qf)
    k, k_scale = quantize_int8_blocks(kf)
    if v == "i8":
        vv, v_scale = quantize_int8_channels(vf)
    else:
        vv, v_scale = vf.to(_TORCH_DTYPE[v]), None
    return {"q": q, "k": k, "v": vv, "q_scale": q_scale, "k_scale": k_scale, "v_scale": v_scale}


def int8_inputs(w: Workload, rotation: int = 0):
    return int8_prefill(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, v=w.extra.get("v", "f16"), dist=w.dist,
                        seed=1000 * w.index + rotation)


def _store(x: torch.Tensor, dtype: str):
    if dtype == "e4m3":
        return quantize_e4m3(x)
    return x.to(_TORCH_DTYPE[dtype]), 1.0


def make_mask(g: torch.Generator, B: int, Sq: int, Sk: int, masked_frac: float, full_row_frac: float):
    """Additive fp16 mask [B, Sq, Sk] of 0 / -inf: each entry -inf with probability ``masked_frac``,
    then round(full_row_frac * Sq) query rows per batch (a seeded permutation) set entirely -inf."""
    m = torch.zeros((B, Sq, Sk), dtype=torch.float16)
    hit = torch.rand((B, Sq, Sk), generator=g, dtype=torch.float32) < masked_frac
    m[hit] = float("-inf")
    n_full = int(round(full_row_frac * Sq))
    for b in range(B):
        rows = torch.randperm(Sq, generator=g)[:n_full]
        m[b, rows, :] = float("-inf")
    return m


def prefill_inputs(w: Workload, rotation: int = 0):
    """Q [B,Sq,Hq,D], K [B,Sk,Hkv,D], V [B,Sk,Hkv,Dv] (stored dtype) plus optional mask [B,Sq,Sk] fp16.

    For e4m3 the per-tensor scales are returned in ``descale`` = (s_q, s_k, s_v)."""
    assert w.kind == "prefill"
    g = generator(w.index, rotation)
    q, sq = _store(_draw(g, (w.B, w.Sq, w.Hq, w.D), w.dist), w.dtype)
    k, sk = _store(_draw(g, (w.B, w.Sk, w.Hkv, w.D), w.dist), w.dtype)
    v, sv = _store(_draw(g, (w.B, w.Sk, w.Hkv, w.Dv), w.dist), w.dtype)
    mask = make_mask(g, w.B, w.Sq, w.Sk, w.masked_frac, w.full_row_frac) if w.mask else None
    return {"q": q, "k": k, "v": v, "mask": mask, "descale": (sq, sk, sv)}


def decode_inputs(w: Workload, rotation: int = 0, pad_value: float = float("nan"), kv_len=None):
    """q [B,Hq,D], padded caches [B,max_kv,Hkv,D|Dv], kv_len int32 [B].

    Rows at or beyond kv_len[b] hold ``pad_value`` (NaN by default, so a kernel that reads them
    poisons its output)."""
    assert w.kind == "decode"
    g = generator(w.index, rotation)
    dt = _TORCH_DTYPE[w.dtype]
    q = _draw(g, (w.B, w.Hq, w.D), w.dist).to(dt)
    if kv_len is None:
        lo, hi = w.kv_len_range
        kv_len = torch.randint(lo, hi + 1, (w.B,), generator=g, dtype=torch.int64).to(torch.int32)
    else:
        kv_len = torch.as_tensor(kv_len, dtype=torch.int32)
    k = torch.full((w.B, w.Sk, w.Hkv, w.D), pad_value, dtype=dt)
    v = torch.full((w.B, w.Sk, w.Hkv, w.Dv), pad_value, dtype=dt)
    for b in range(w.B):
        n = int(kv_len[b])
        k[b, :n] = _draw(g, (n, w.Hkv, w.D), w.dist).to(dt)
        v[b, :n] = _draw(g, (n, w.Hkv, w.Dv), w.dist).to(dt)
    return {"q": q, "k": k, "v": v, "kv_len": kv_len}


def page_caches(k, v, page_size: int, seed: int, spare_pages: int = 0):
    """Scatter contiguous caches [B, max_kv, Hkv, .] into page pools [n_pages, page_size, Hkv, .].

    Logical page i of sequence b goes to physical page perm[b * max_pages + i] of a seeded random
    permutation over n_pages = B * max_pages + spare_pages; spare pages hold NaN.  The table is
    int32 [B, max_pages].  Works on any device (torch indexing only); max_kv must be a multiple of
    page_size."""
    B, max_kv = k.shape[0], k.shape[1]
    assert max_kv % page_size == 0
    max_pages = max_kv // page_size
    n_pages = B * max_pages + spare_pages
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    perm = torch.randperm(n_pages, generator=g)[: B * max_pages].to(k.device)
    pools = []
    for c in (k, v):
        pool = torch.full((n_pages, page_size, *c.shape[2:]), float("nan"), dtype=c.dtype, device=c.device)
        pool[perm] = c.reshape(B * max_pages, page_size, *c.shape[2:])
        pools.append(pool)
    table = perm.view(B, max_pages).to(torch.int32)
    return pools[0], pools[1], table


def custom_prefill(B, Hq, Hkv, Sq, Sk, D, Dv, dtype="bf16", dist="normal", seed=0, mask=False,
                   masked_frac=0.1, full_row_frac=0.05):
    """Small prefill cases for tests: same recipe, explicit seed."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    q, sq = _store(_draw(g, (B, Sq, Hq, D), dist), dtype)
    k, sk = _store(_draw(g, (B, Sk, Hkv, D), dist), dtype)
    v, sv = _store(_draw(g, (B, Sk, Hkv, Dv), dist), dtype)
    m = make_mask(g, B, Sq, Sk, masked_frac, full_row_frac) if mask else None
    return {"q": q, "k": k, "v": v, "mask": m, "descale": (sq, sk, sv)}


def varlen_pack(seq_q, seq_k, Hq, Hkv, D, Dv, dtype="bf16", dist="normal", seed=0, pad_q=0, pad_k=0):
    """Packed sequences: q [total_q, Hq, D], k [total_k, Hkv, D], v [total_k, Hkv, Dv] with sequence b
    on rows cu_q[b] .. cu_q[b+1] (keys likewise), cu_q / cu_k int32 [B + 1].  ``pad_q`` / ``pad_k``
    extra rows at the end belong to no sequence.  Draw order: q, k, v over all rows (e4m3: one
    per-tensor scale each)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    cu_q = torch.zeros(len(seq_q) + 1, dtype=torch.int32)
    cu_k = torch.zeros(len(seq_k) + 1, dtype=torch.int32)
    cu_q[1:] = torch.cumsum(torch.as_tensor(seq_q, dtype=torch.int64), 0).to(torch.int32)
    cu_k[1:] = torch.cumsum(torch.as_tensor(seq_k, dtype=torch.int64), 0).to(torch.int32)
    tq, tk = int(cu_q[-1]) + pad_q, int(cu_k[-1]) + pad_k
    q, sq = _store(_draw(g, (tq, Hq, D), dist), dtype)
    k, sk = _store(_draw(g, (tk, Hkv, D), dist), dtype)
    v, sv = _store(_draw(g, (tk, Hkv, Dv), dist), dtype)
    return {"q": q, "k": k, "v": v, "cu_q": cu_q, "cu_k": cu_k, "descale": (sq, sk, sv)}


def varlen_lengths(w: Workload, rotation: int = 0):
    """Sequence lengths of a packed workload: B draws, uniform over the inclusive len_range."""
    lo, hi = w.extra["len_range"]
    g = generator(w.index, rotation)
    return [int(x) for x in torch.randint(lo, hi + 1, (w.B,), generator=g, dtype=torch.int64)]


def varlen_inputs(w: Workload, rotation: int = 0):
    """Packed inputs of a varlen workload (query and key lengths equal)."""
    assert w.kind == "varlen"
    lens = varlen_lengths(w, rotation)
    x = varlen_pack(lens, lens, w.Hq, w.Hkv, w.D, w.Dv, w.dtype, w.dist, seed=1000 * w.index + rotation + 500)
    x["lengths"] = lens
    return x
