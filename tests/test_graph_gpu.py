"""The prefill and decode entry points inside a CUDA graph: captured once on static buffers,
replayed on new inputs, each replay equal to the eager call on the same inputs."""
import pytest
import torch

import flash_attention_forward_gb300 as fa
import workloads

pytestmark = pytest.mark.gpu

DEV = "cuda"


def test_prefill_graph_replays_match_eager():
    shape = (2, 8, 2, 700, 900, 128, 128)
    xs = [workloads.custom_prefill(*shape, dtype="bf16", seed=s) for s in (1, 2, 3)]
    q, k, v = (xs[0][n].to(DEV) for n in ("q", "k", "v"))
    B, Hq, Hkv, Sq, Sk, D, Dv = shape
    o = torch.empty((B, Sq, Hq, Dv), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=DEV)
    ws = torch.empty(max(16, fa.sdpa_fwd_workspace_size(B, Hq, Sq, Sk, Dv, False, False)), dtype=torch.uint8,
                     device=DEV)
    fa.sdpa_fwd(q, k, v, out=o, lse=lse, workspace=ws)  # first call outside capture (device lookups)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa.sdpa_fwd(q, k, v, out=o, lse=lse, workspace=ws)
    for x in xs:
        q.copy_(x["q"]), k.copy_(x["k"]), v.copy_(x["v"])
        g.replay()
        torch.cuda.synchronize()
        ro, rl = fa.sdpa_fwd(q, k, v)
        torch.cuda.synchronize()
        assert torch.equal(o, ro) and torch.equal(lse, rl)
    assert fa.sdpa_check_device_status() == fa.SDPA_OK


def test_decode_graph_replays_match_eager():
    w = workloads.WORKLOADS["splitkv_decode_bf16_d128"].with_shape(B=4, Sk=3000)
    xs = [workloads.decode_inputs(w, rotation=r, kv_len=lens, pad_value=0.0)
          for r, lens in enumerate(([3000, 1, 1500, 2049], [17, 3000, 0, 1024]))]
    q, k, v, kvl = (xs[0][n].to(DEV) for n in ("q", "k", "v", "kv_len"))
    o = torch.empty((w.B, w.Hq, w.Dv), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=DEV)
    ws = torch.empty(fa.sdpa_decode_workspace_size(w.B, w.Hq, w.Sk, w.Dv), dtype=torch.uint8, device=DEV)
    fa.sdpa_decode(q, k, v, kvl, scale=w.scale, out=o, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa.sdpa_decode(q, k, v, kvl, scale=w.scale, out=o, lse=lse, workspace=ws)
    for x in xs:
        q.copy_(x["q"]), k.copy_(x["k"]), v.copy_(x["v"]), kvl.copy_(x["kv_len"])
        g.replay()
        torch.cuda.synchronize()
        ro, rl = fa.sdpa_decode(q, k, v, kvl, scale=w.scale)
        torch.cuda.synchronize()
        assert torch.equal(o, ro) and torch.equal(lse, rl)
    assert fa.sdpa_check_device_status() == fa.SDPA_OK


def test_varlen_and_int8_graph_replays_match_eager():
    seq = [300, 5, 640]
    vx = workloads.varlen_pack(seq, seq, 4, 2, 128, 128, dtype="bf16", seed=8)
    q, k, v, cu_q, cu_k = (vx[n].to(DEV) for n in ("q", "k", "v", "cu_q", "cu_k"))
    ix = {n: (None if t is None else t.to(DEV))
          for n, t in workloads.int8_prefill(1, 4, 2, 500, 700, 128, v="i8", seed=9).items()}
    vo = torch.empty((q.shape[0], 4, 128), dtype=torch.bfloat16, device=DEV)
    vws = torch.empty(fa.sdpa_fwd_varlen_workspace_size(len(seq)), dtype=torch.uint8, device=DEV)
    io = torch.empty((1, 500, 4, 128), dtype=torch.float16, device=DEV)
    iws = torch.empty(fa.sdpa_fwd_int8_workspace_size(1, 4, 2, 500, 700, 128, True, True), dtype=torch.uint8,
                      device=DEV)
    iargs = (ix["q"], ix["k"], ix["v"], ix["q_scale"], ix["k_scale"], ix["v_scale"])

    def calls():
        fa.sdpa_fwd_varlen(q, k, v, cu_q, cu_k, max(seq), causal=True, out=vo, return_lse=False, workspace=vws)
        fa.sdpa_fwd_int8(*iargs, causal=True, out=io, return_lse=False, workspace=iws)

    calls()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        calls()
    for r in range(2):
        q.mul_(-1.0), ix["q"].neg_()  # new inputs in the static buffers
        g.replay()
        torch.cuda.synchronize()
        rv, _ = fa.sdpa_fwd_varlen(q, k, v, cu_q, cu_k, max(seq), causal=True)
        ri, _ = fa.sdpa_fwd_int8(*iargs, causal=True)
        torch.cuda.synchronize()
        assert torch.equal(vo[: int(cu_q[-1])], rv[: int(cu_q[-1])]) and torch.equal(io, ri)
    assert fa.sdpa_check_device_status() == fa.SDPA_OK
