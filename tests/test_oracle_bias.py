"""Pins for the oracle's additive bias C (left window, ALiBi slopes, dense bias).

"Compilers and Kernels", section "FlashAttention changes the algorithm around
IO": S = Q K^T / sqrt(d) + C with C in R U {-inf}.  The oracle's masked entry
point is pinned to a 50-digit decimal brute force that builds C itself, to
torch's float64 scaled_dot_product_attention with the same float mask, and to
equivalences: no options = the plain oracle; a window expressed as a -inf bias
= the window option; zero slopes / zero bias change nothing.
"""
from __future__ import annotations

import math
from decimal import Decimal, localcontext

import numpy as np
import pytest
import torch

import oracle
import oracle_mutants
from attention_online_softmax_gb300 import inputs
from test_oracle_pins import bf16_np, close

oracle_mutants.register_all()


def c_matrix(B, Hq, Nq, Nk, causal, window, slopes, bias):
    """C[b,h,i,j] in float64 (-inf for disallowed keys), built independently."""
    C = np.zeros((B, Hq, Nq, Nk))
    diag = Nk - Nq
    i = np.arange(Nq)[:, None]
    j = np.arange(Nk)[None, :]
    allowed = np.ones((Nq, Nk), dtype=bool)
    if causal:
        allowed &= j - i <= diag
    if window > 0:
        allowed &= j - i > diag - window
    for h in range(Hq):
        if slopes is not None:
            C[:, h] += float(slopes[h]) * (j - i - diag)
    if bias is not None:
        C += bias
    C[:, :, ~allowed] = -math.inf
    return C


def decimal_with_bias(q, k, v, scale, C):
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    rep = Hq // Hkv
    O = np.zeros((B, Hq, Nq, d))
    L = np.zeros((B, Hq, Nq))
    with localcontext() as ctx:
        ctx.prec = 50
        for b in range(B):
            for h in range(Hq):
                g = h // rep
                for i in range(Nq):
                    terms = []
                    for jj in range(Nk):
                        if C[b, h, i, jj] == -math.inf:
                            continue
                        s = sum(Decimal(float(q[b, h, i, c])) * Decimal(float(k[b, g, jj, c]))
                                for c in range(d)) * Decimal(float(scale)) + Decimal(float(C[b, h, i, jj]))
                        terms.append((s.exp(), jj))
                    if not terms:
                        L[b, h, i] = -math.inf
                        continue
                    z = sum(e for e, _ in terms)
                    for c in range(d):
                        O[b, h, i, c] = float(sum(e * Decimal(float(v[b, g, jj, c])) for e, jj in terms) / z)
                    L[b, h, i] = float(z.ln())
    return O, L


CASES = [
    # B, Hq, Hkv, Nq, Nk, d, causal, window, alibi, bias
    (1, 2, 2, 12, 12, 4, True, 5, False, False),
    (1, 2, 1, 7, 15, 4, True, 3, True, False),
    (1, 2, 2, 9, 9, 4, False, 0, True, True),
    (2, 2, 2, 6, 10, 4, False, 4, False, True),
    (1, 1, 1, 9, 5, 4, True, 2, True, True),   # rows without any key
]


@pytest.mark.parametrize("case", CASES)
def test_masked_oracle_matches_decimal_brute_force(case):
    B, Hq, Hkv, Nq, Nk, d, causal, window, use_alibi, use_bias = case
    x = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=700 + Nq + Nk, causal=causal)
    g = torch.Generator().manual_seed(5)
    slopes = (torch.rand(Hq, generator=g) * 0.5).numpy().astype(np.float32) if use_alibi else None
    bias_t = None
    bias_np = None
    if use_bias:
        bias_t = (torch.randn(B, Hq, Nq, Nk, generator=g) * 2).to(torch.bfloat16)
        bias_t[..., 0] = float("-inf")  # a disallowed key expressed through the bias
        bias_np = bf16_np(bias_t)
    O, L, _ = oracle.attention_masked(x.q, x.k, x.v, causal, x.scale, window_left=window,
                                      alibi=slopes, bias=bias_t,
                                      bias_strides=(Hq * Nq * Nk, Nq * Nk))
    C = c_matrix(B, Hq, Nq, Nk, causal, window, slopes, bias_np)
    Ob, Lb = decimal_with_bias(bf16_np(x.q), bf16_np(x.k), bf16_np(x.v), x.scale, C)
    assert close(O, Ob, 1e-12)
    assert close(L, Lb, 1e-12)


def test_masked_oracle_without_options_is_the_plain_oracle():
    x = inputs.prefill_inputs(2, 4, 2, 33, 47, 16, seed=711, causal=True)
    O1, L1, _ = oracle.attention(x.q, x.k, x.v, True, x.scale)
    O2, L2, _ = oracle.attention_masked(x.q, x.k, x.v, True, x.scale)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)
    O3, L3, _ = oracle.attention_masked(x.q, x.k, x.v, True, x.scale, window_left=1000,
                                        alibi=np.zeros(4, np.float32),
                                        bias=torch.zeros(1, 1, 33, 47, dtype=torch.bfloat16))
    np.testing.assert_allclose(O1, O3, atol=1e-14)
    np.testing.assert_allclose(L1, L3, atol=1e-14)


def test_window_equals_minus_inf_bias():
    B, H, N, d, W = 1, 2, 40, 16, 7
    x = inputs.prefill_inputs(B, H, H, N, N, d, seed=712, causal=True)
    O1, L1, _ = oracle.attention_masked(x.q, x.k, x.v, True, x.scale, window_left=W)
    i = torch.arange(N)[:, None]
    j = torch.arange(N)[None, :]
    bias = torch.where(j - i > -W, 0.0, float("-inf")).to(torch.bfloat16).expand(B, H, N, N).contiguous()
    O2, L2, _ = oracle.attention_masked(x.q, x.k, x.v, True, x.scale, bias=bias,
                                        bias_strides=(H * N * N, N * N))
    np.testing.assert_allclose(O1, O2, atol=1e-13)
    np.testing.assert_allclose(L1, L2, atol=1e-13)


def test_masked_oracle_against_torch_sdpa_float64():
    B, Hq, Hkv, Nq, Nk, d = 2, 4, 2, 21, 29, 16
    x = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=713, causal=True)
    g = torch.Generator().manual_seed(9)
    slopes = (torch.rand(Hq, generator=g) * 0.3).numpy().astype(np.float32)
    bias = (torch.randn(1, Hq, Nq, Nk, generator=g)).to(torch.bfloat16)  # broadcast over batch
    O, L, _ = oracle.attention_masked(x.q, x.k, x.v, True, x.scale, window_left=9, alibi=slopes,
                                      bias=bias, bias_strides=(0, Nq * Nk))
    C = torch.from_numpy(c_matrix(B, Hq, Nq, Nk, True, 9, slopes,
                                  np.broadcast_to(bf16_np(bias), (B, Hq, Nq, Nk))))
    q = x.q.double()
    k = x.k.double().repeat_interleave(2, dim=1)
    v = x.v.double().repeat_interleave(2, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=C, scale=x.scale)
    s = (q @ k.transpose(-1, -2)) * x.scale + C
    lse = torch.logsumexp(s, dim=-1)
    fin = torch.isfinite(lse).numpy()
    np.testing.assert_allclose(O[fin], ref.numpy()[fin], atol=1e-12)
    np.testing.assert_allclose(L[fin], lse.numpy()[fin], atol=1e-12)


def test_planted_alibi_sign_mistake_is_caught():
    # An ALiBi distance of the wrong sign (mutant 9) must fail the decimal pin.
    B, Hq, Hkv, Nq, Nk, d, causal, window = 1, 2, 1, 7, 15, 4, True, 3
    x = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=720, causal=causal)
    slopes = np.array([0.5, 0.25], dtype=np.float32)
    O, L, _ = oracle.attention_masked(x.q, x.k, x.v, causal, x.scale, window_left=window, alibi=slopes, mutant=9)
    C = c_matrix(B, Hq, Nq, Nk, causal, window, slopes, None)
    Ob, Lb = decimal_with_bias(bf16_np(x.q), bf16_np(x.k), bf16_np(x.v), x.scale, C)
    assert not (close(O, Ob, 1e-6) and close(L, Lb, 1e-6))


def test_planted_window_bound_mistake_is_caught():
    # A left window one key too wide (mutant 12) must fail the decimal pin.
    B, Hq, Hkv, Nq, Nk, d, causal, window = 1, 2, 1, 9, 13, 4, True, 4
    x = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=721, causal=causal)
    O, L, _ = oracle.attention_masked(x.q, x.k, x.v, causal, x.scale, window_left=window, mutant=12)
    C = c_matrix(B, Hq, Nq, Nk, causal, window, None, None)
    Ob, Lb = decimal_with_bias(bf16_np(x.q), bf16_np(x.k), bf16_np(x.v), x.scale, C)
    assert not (close(O, Ob, 1e-6) and close(L, Lb, 1e-6))
