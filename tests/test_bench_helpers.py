"""The benchmark's work counts, checked against brute force (CPU only)."""
import itertools

import bench
import workloads


def test_visible_pairs_match_brute_force():
    for Sq, Sk in itertools.product([1, 2, 5, 17, 130], [1, 3, 17, 129]):
        for causal in (False, True):
            brute = sum(1 for i in range(Sq) for j in range(Sk) if not causal or j <= i)
            assert bench.visible_pairs(Sq, Sk, causal) == brute, (Sq, Sk, causal)


def test_prefill_and_varlen_flops():
    w = workloads.WORKLOADS["gqa_causal_prefill_bf16_d128"]
    assert bench.prefill_flops(w) == 2.0 * 256 * 2 * 32 * (4096 * 4097 // 2)
    v = workloads.WORKLOADS["varlen_causal_prefill_bf16_d128"]
    lens = [3, 5, 1]
    assert bench.varlen_flops(v, lens) == sum(2.0 * 256 * 32 * L * (L + 1) // 2 for L in lens)
    # packing sequences of equal length gives the dense batch's count
    dense = w.with_shape(B=3, Sq=300, Sk=300)
    assert bench.varlen_flops(v.with_shape(Hq=32, D=128, Dv=128), [300] * 3) == bench.prefill_flops(dense)


def test_decode_bytes():
    w = workloads.WORKLOADS["splitkv_decode_bf16_d128"].with_shape(B=2)
    kv_len = [10, 1000]
    want = (10 + 1000) * 8 * 256 * 2 + 2 * 32 * 256 * 2
    assert bench.decode_bytes(w, kv_len) == want
