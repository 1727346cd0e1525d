"""The byte-counting convention used for every roofline figure.

Pinned to the fused-versus-unfused example of "Compilers and Kernels",
section "Roofline is a bound, not a stopwatch" (tests/golden/fusion_traffic_example.txt),
and to hand counts of the attention workloads.
"""
import os

import pytest

from attention_online_softmax_gb300 import roofline

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fusion_traffic_example.txt")


def load_golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, v = line.split()
        vals[k] = float(v)
    return vals


def test_fusion_example_traffic():
    g = load_golden()
    n, bpe = int(g["elements"]), int(g["bytes_per_element"])
    ops = n * 3
    # unfused: three kernels (mul, add, max), each reads one vector and writes one
    unfused = sum(roofline.materialized_traffic(n, bpe, reads=1, writes=1) for _ in range(3))
    fused = roofline.materialized_traffic(n, bpe, reads=1, writes=1)
    assert ops == g["operations"]
    assert unfused == g["unfused_bytes"] and fused == g["fused_bytes"]
    assert ops / unfused == pytest.approx(g["unfused_intensity"])
    assert ops / fused == pytest.approx(g["fused_intensity"])
    assert unfused / fused == pytest.approx(g["traffic_reduction"])


def test_attention_counts_by_hand():
    # tiny MHA B1 H2 N128 d64: Q,K,V,O bf16 = 4 * 2*128*64*2 B, LSE 2*128*4 B
    assert roofline.prefill_bytes(1, 2, 2, 128, 128, 64) == 4 * 32768 + 1024
    assert roofline.prefill_flops(1, 2, 128, 128, 64, False) == 4 * 2 * 128 * 128 * 64
    assert roofline.prefill_flops(4, 16, 512, 512, 64, True) == 2 * 4 * 16 * 512 * 512 * 64
    # GQA: K and V are counted once per key/value head
    assert roofline.prefill_bytes(1, 16, 2, 16384, 16384, 256) == (
        2 * 16 * 16384 * 256 * 2 + 2 * 2 * 16384 * 256 * 2 + 16 * 16384 * 4)
    # decode: 2 sequences of 17 and 32 tokens, 8 q heads over 2 kv heads, d 16
    b = roofline.decode_bytes([17, 32], 8, 2, 16, 16)
    assert b == 49 * 2 * 16 * 2 * 2 + 2 * 8 * 16 * 2 * 2 + 2 * 8 * 4 + (2 + 2) * 4 + 2 * 4


def test_roofline_bound_and_floor():
    p = roofline.Peaks(hbm_gbs=1000.0, bf16_tflops=100.0, bf16_tflops_sustained=90.0,
                       source="test")
    assert roofline.ridge(p) == pytest.approx(100.0)
    assert roofline.bound_rate(1e12, 1e9, p) == pytest.approx(1e14)  # I=1000 > ridge
    assert roofline.bound_rate(1e11, 1e10, p) == pytest.approx(1e13)  # I=10 < ridge
    assert roofline.time_floor_s(1e12, 1e9, p) == pytest.approx(0.01)


@pytest.mark.parametrize("Nq,Nk,causal,window", [(7, 7, True, 0), (5, 9, True, 3), (9, 5, True, 2),
                                                  (6, 11, False, 4), (8, 8, False, 0), (4, 4, True, 1)])
def test_allowed_pairs_brute_force(Nq, Nk, causal, window):
    # Count the pairs one by one from the mask's definition.
    diag = Nk - Nq
    n = 0
    for i in range(Nq):
        for j in range(Nk):
            if causal and j > i + diag:
                continue
            if window > 0 and j <= i + diag - window:
                continue
            n += 1
    assert roofline.allowed_pairs(Nq, Nk, causal, window) == n


def test_backward_and_paged_prefill_counts_by_hand():
    # Backward, B1 Hq4 Hkv2 N32 d16: Q, O, dO read and dQ written per query
    # head (4 bf16 tensors of 4*32*16), K, V read and dK, dV written per kv
    # head (4 of 2*32*16), LSE read (4*32 f32).
    assert roofline.bwd_bytes(1, 4, 2, 32, 32, 16) == 4 * (4 * 32 * 16 * 2) + 4 * (2 * 32 * 16 * 2) + 4 * 32 * 4
    # Chunked prefill: 2 sequences with 3 and 5 new tokens over contexts of
    # 20 and 5 tokens, Hq 4, Hkv 2, d 16, 16-token pages.  Q and O bf16 and
    # LSE f32 for the 8 new tokens; context K and V once per kv head; the
    # block-table entries used (2 + 1 pages); cu_seqlens (3) and seqlens (2).
    got = roofline.paged_prefill_bytes([3, 5], [20, 5], 4, 2, 16, 16)
    want = (8 * 4 * 16 * 2) * 2 + 8 * 4 * 4 + 25 * 2 * 16 * 2 * 2 + 3 * 4 + 5 * 4
    assert got == want
