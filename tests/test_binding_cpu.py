"""The Python binding on a machine without a GPU: it refuses host tensors (there is no CPU path)
and fails loudly when the compiled library is missing."""
import os
import subprocess
import sys

import pytest
import torch

import flash_attention_forward_gb300 as fa
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_host_tensors_are_refused():
    x = workloads.custom_prefill(1, 2, 1, 16, 16, 64, 64, dtype="bf16", seed=1)
    with pytest.raises(ValueError):
        fa.sdpa_fwd(x["q"], x["k"], x["v"])
    with pytest.raises(ValueError):
        fa.sdpa_fwd_fp8(x["q"].to(torch.float8_e4m3fn), x["k"].to(torch.float8_e4m3fn),
                        x["v"].to(torch.float8_e4m3fn), 1.0, 1.0, 1.0)
    p = workloads.varlen_pack([5, 7], [5, 7], 2, 1, 64, 64, dtype="bf16", seed=2)
    with pytest.raises(ValueError):
        fa.sdpa_fwd_varlen(p["q"], p["k"], p["v"], p["cu_q"], p["cu_k"], 7)
    i = workloads.int8_prefill(1, 2, 1, 16, 16, 64, seed=3)
    with pytest.raises(ValueError):
        fa.sdpa_fwd_int8(i["q"], i["k"], i["v"], i["q_scale"], i["k_scale"])
    d = workloads.decode_inputs(workloads.WORKLOADS["splitkv_decode_bf16_d128"].with_shape(B=2, Sk=64),
                                kv_len=[3, 64])
    with pytest.raises(ValueError):
        fa.sdpa_decode(d["q"], d["k"], d["v"], d["kv_len"])
    with pytest.raises(ValueError):
        fa.sdpa_decode_noalloc(d["q"], d["k"], d["v"], d["kv_len"])
    kp, vp, table = workloads.page_caches(d["k"], d["v"], 16, seed=3)
    with pytest.raises(ValueError):
        fa.sdpa_decode_paged(d["q"], kp, vp, table, d["kv_len"])


def test_missing_library_fails_loudly():
    code = ("import flash_attention_forward_gb300 as fa\n"
            "fa.LIB_PATH = '/nonexistent/libsdpa_gb300.so'\n"
            "try:\n    fa.library()\nexcept RuntimeError as e:\n    print('refused:', 'missing' in str(e))\n")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert out.stdout.strip() == "refused: True", out.stdout + out.stderr
