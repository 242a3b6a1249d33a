"""Shared helpers of the GPU parity tests: NaN/Inf count first, then max abs error."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances on O (absolute, vs the fp64 oracle on the same stored inputs).
TOL_16BIT = 1e-2
TOL_FP8 = 3e-2
# LSE = m + ln(l).  The decode sums l from the probabilities already rounded to the 16-bit
# type that feeds the P.V product (so that O is normalised by exactly the weights it used).
# Each rounded p has relative error <= u (unit roundoff of that type), so l, a sum of positive
# terms, has relative error <= u and |delta LSE| <= -ln(1 - u) ~ u.  Bound: u plus 1e-4 for
# fp32 score rounding and the approximate exp2/log2 units.  The prefill sums the fp32
# probabilities, so it meets these bounds with room; TOL_LSE_FP32_SUM is its own: fp32 sums of
# at most 16384 terms (partial sums per 128-key block) and the approximate exp2/log2 units.
U_BF16 = 2.0 ** -8
U_F16 = 2.0 ** -11
TOL_LSE_BF16 = U_BF16 + 1e-4   # bf16 P (bf16 inputs)
TOL_LSE_F16 = U_F16 + 1e-4     # f16 P (f16 and e4m3 inputs)
TOL_LSE_FP32_SUM = 1e-4        # the prefill's fp32 row sums
TOL_LSE = TOL_LSE_BF16


def nonfinite(a: np.ndarray) -> int:
    return int(np.count_nonzero(~np.isfinite(a)))


def assert_close(got, ref, tol, what="O"):
    got = np.asarray(got, dtype=np.float64)
    n_bad = nonfinite(got)
    assert n_bad == 0, f"{what}: {n_bad} NaN/Inf values"
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    assert err <= tol, f"{what}: max abs error {err:.3e} > {tol:.1e}"
    return err


def assert_lse_close(got, ref, tol=TOL_LSE):
    got = np.asarray(got, dtype=np.float64)
    assert not np.isnan(got).any(), "LSE: NaN"
    ninf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), ninf_ref), "LSE: -inf rows differ"
    fin = ~ninf_ref
    if fin.any():
        err = float(np.abs(got[fin] - ref[fin]).max())
        assert err <= tol, f"LSE: max abs error {err:.3e}"


def sample_rows(B, Hq, Sq, n, seed, extra=()):
    """(b, h, i) triples: tile edges, the first and last rows, plus seeded random ones."""
    g = np.random.default_rng(seed)
    rows = set()
    edges = [0, 1, 127, 128, 129, 255, 256, 257, Sq // 2, Sq - 2, Sq - 1]
    for i in edges:
        if 0 <= i < Sq:
            rows.add((int(g.integers(B)), int(g.integers(Hq)), i))
    for r in extra:
        rows.add(tuple(int(x) for x in r))
    while len(rows) < n:
        rows.add((int(g.integers(B)), int(g.integers(Hq)), int(g.integers(Sq))))
    return np.array(sorted(rows), dtype=np.int64)


def oracle_rows(q, k, v, mask, rows, *, scale, causal, descale=(1.0, 1.0, 1.0)):
    """Oracle O/LSE for selected rows, one (b, head) slice at a time so big tensors never go fp64 whole."""
    Hq, Hkv = q.shape[2], k.shape[2]
    group = Hq // Hkv
    Dv = v.shape[-1]
    o = np.empty((len(rows), Dv))
    lse = np.empty((len(rows),))
    by_head = {}
    for n, (b, h, i) in enumerate(rows):
        by_head.setdefault((b, h), []).append((n, i))
    for (b, h), items in by_head.items():
        kvh = h // group
        qs = q[b:b + 1, :, h:h + 1]
        ks = k[b:b + 1, :, kvh:kvh + 1]
        vs = v[b:b + 1, :, kvh:kvh + 1]
        ms = None if mask is None else mask[b:b + 1]
        sub = np.array([[0, 0, i] for _, i in items], dtype=np.int64)
        oo, ll = oracle.sdpa_fwd(qs, ks, vs, ms, scale=scale, causal=causal, rows=sub, descale=descale)
        for j, (n, _) in enumerate(items):
            o[n], lse[n] = oo[j], ll[j]
    return o, lse


def gather_rows(o_gpu: torch.Tensor, lse_gpu: torch.Tensor, rows):
    r = torch.as_tensor(rows, dtype=torch.long, device=o_gpu.device)
    o = o_gpu[r[:, 0], r[:, 2], r[:, 1]].float().cpu().numpy()
    lse = None if lse_gpu is None else lse_gpu[r[:, 0], r[:, 1], r[:, 2]].cpu().numpy()
    return o, lse
