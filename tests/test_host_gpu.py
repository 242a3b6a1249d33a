"""sdpa_fwd_host (host buffers, copies overlapped with compute over chunks of query rows) against
the device entry point and the fp64 oracle."""
import numpy as np
import pytest
import torch

import flash_attention_forward_gb300 as fa
import oracle
import workloads
from parity import TOL_16BIT, TOL_LSE_BF16, TOL_LSE_F16, assert_close, assert_lse_close

pytestmark = pytest.mark.gpu

DEV = "cuda"

# (B, Hq, Hkv, Sq, Sk, D, Dv): one chunk, several chunks with a ragged last one, fewer or more
# keys than queries (causal key prefixes clipped at Sk), the MLA head dims
SHAPES = [
    (1, 2, 1, 100, 77, 64, 64),
    (2, 4, 2, 1000, 1000, 128, 128),
    (1, 4, 4, 3000, 1200, 128, 128),
    (2, 2, 1, 700, 2000, 128, 128),
    (1, 2, 2, 2100, 2100, 192, 128),
]


def _pinned(x):
    return [x[n].pin_memory() for n in ("q", "k", "v")]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_host_call_matches_device_call_and_oracle(shape, causal):
    B, Hq, Hkv, Sq, Sk, D, Dv = shape
    dtype = "bf16" if D != 64 else "f16"
    x = workloads.custom_prefill(B, Hq, Hkv, Sq, Sk, D, Dv, dtype=dtype, seed=sum(shape) + causal)
    q, k, v = _pinned(x)
    o, lse = fa.sdpa_fwd_host(q, k, v, causal=causal)
    torch.cuda.synchronize()
    assert fa.sdpa_check_device_status() == fa.SDPA_OK
    od, ld = fa.sdpa_fwd(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), causal=causal)
    torch.cuda.synchronize()
    if causal:
        # the same key blocks in the same order for every row: bit for bit
        assert torch.equal(o, od.cpu()) and torch.equal(lse, ld.cpu())
    scale = 1.0 / np.sqrt(D)
    if Sq * Sk <= 2_000_000:
        ref_o, ref_lse = oracle.sdpa_fwd(x["q"], x["k"], x["v"], scale=scale, causal=causal)
        assert_close(o.float().numpy(), ref_o, TOL_16BIT)
        assert_lse_close(lse.numpy(), ref_lse, TOL_LSE_F16 if dtype == "f16" else TOL_LSE_BF16)
    else:
        assert_close(o.float().numpy(), od.float().cpu().numpy(), 2e-3)


def test_host_call_without_lse_and_repeated():
    x = workloads.custom_prefill(1, 2, 1, 600, 600, 128, 128, dtype="bf16", seed=5)
    q, k, v = _pinned(x)
    ws = torch.empty(fa.sdpa_fwd_host_workspace_size(1, 2, 1, 600, 600, 128, 128, True), dtype=torch.uint8,
                     device=DEV)
    o1, l1 = fa.sdpa_fwd_host(q, k, v, causal=True, return_lse=False, workspace=ws)
    o2, _ = fa.sdpa_fwd_host(q, k, v, causal=True, workspace=ws)
    torch.cuda.synchronize()
    assert l1 is None and torch.equal(o1, o2)


def test_host_call_validation():
    x = workloads.custom_prefill(1, 2, 1, 64, 64, 128, 128, dtype="bf16", seed=6)
    q, k, v = _pinned(x)
    with pytest.raises(fa.SdpaError) as e:
        fa.sdpa_fwd_host(q, k, v, workspace=torch.empty(16, dtype=torch.uint8, device=DEV))
    assert e.value.status == fa.SDPA_ERR_INVALID
    with pytest.raises(ValueError):
        fa.sdpa_fwd_host(q.to(DEV), k, v)
    assert fa.sdpa_check_device_status() == fa.SDPA_OK
