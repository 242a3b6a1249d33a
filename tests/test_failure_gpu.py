"""Failure detection without a GPU fault: a test hook withholds the first K/V stage of one
launch; every bounded wait must give up, the kernel must report SDPA_ERR_TIMEOUT through the
device status word, and the next call on the same context must be correct."""
import numpy as np
import pytest
import torch

import flash_attention_forward_gb300 as fa
import oracle
import workloads
from parity import TOL_16BIT, assert_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_stalled_stage_times_out_and_context_survives(dtype):
    D = 192 if dtype == "e4m3" else 128
    x = workloads.custom_prefill(1, 2, 2, 300, 500, D, 128, dtype=dtype, seed=51)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    scale = 1.0 / np.sqrt(D)

    def run():
        if dtype == "e4m3":
            return fa.sdpa_fwd_fp8(q, k, v, *x["descale"], scale=scale, causal=True)
        return fa.sdpa_fwd(q, k, v, scale=scale, causal=True)

    assert fa.sdpa_check_device_status() == fa.SDPA_OK
    assert fa.library().sdpa_debug_stall_next_call() == fa.SDPA_OK
    run()
    assert fa.sdpa_check_device_status() == fa.SDPA_ERR_TIMEOUT
    assert fa.sdpa_check_device_status() == fa.SDPA_OK  # reported once, then cleared
    o, _ = run()
    torch.cuda.synchronize()
    assert fa.sdpa_check_device_status() == fa.SDPA_OK
    ref, _ = oracle.sdpa_fwd(x["q"], x["k"], x["v"], scale=scale, causal=True, descale=x["descale"])
    assert_close(o.float().cpu().numpy(), ref, 3e-2 if dtype == "e4m3" else TOL_16BIT)
