"""Pins for the oracle's backward through the additive bias C (left window,
ALiBi, dense bias; "Compilers and Kernels", section "FlashAttention changes
the algorithm around IO": S = Q K^T / sqrt(d) + C).

The gradients of O with respect to Q, K, V keep the unbiased form with P the
biased weights.  The oracle's masked backward is pinned to torch autograd
through float64 scaled_dot_product_attention with the same additive mask, to
central finite differences of the oracle's own (separately pinned) masked
forward, and to the unbiased backward when C is zero.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from attention_online_softmax_gb300 import inputs
from test_oracle_pins import bf16_np


def dout_for(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


def mask_inputs(B, Hq, Nq, Nk, seed, alibi=True, bias=True):
    g = torch.Generator().manual_seed(seed)
    slopes = (torch.rand(Hq, generator=g) * 0.5).float() if alibi else None
    b = (torch.randn(B, Hq, Nq, Nk, generator=g) * 0.7).to(torch.bfloat16) if bias else None
    return slopes, b


def additive_mask(B, Hq, Nq, Nk, causal, window, slopes, bias):
    """C as a float64 [B, Hq, Nq, Nk] tensor, -inf where a key is disallowed."""
    i = torch.arange(Nq, dtype=torch.float64)[:, None]
    j = torch.arange(Nk, dtype=torch.float64)[None, :]
    diag = Nk - Nq
    c = torch.zeros(B, Hq, Nq, Nk, dtype=torch.float64)
    if slopes is not None:
        c = c + slopes.double()[None, :, None, None] * (j - i - diag)[None, None]
    if bias is not None:
        c = c + bias.double()
    allowed = torch.ones(Nq, Nk, dtype=torch.bool)
    if causal:
        allowed &= j <= i + diag
    if window > 0:
        allowed &= j > i + diag - window
    return c.masked_fill(~allowed[None, None], float("-inf"))


@pytest.mark.parametrize("causal,window,use_alibi,use_bias", [
    (True, 0, True, False), (False, 0, False, True), (True, 5, True, True), (False, 4, False, False)])
def test_masked_bwd_matches_torch_autograd_float64(causal, window, use_alibi, use_bias):
    B, Hq, Hkv, Nq, Nk, d = 2, 4, 2, 11, 14, 8   # Nq <= Nk: every row keeps its diagonal key
    x = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=80 + window, causal=causal)
    dout = dout_for((B, Hq, Nq, d), 81)
    slopes, bias = mask_inputs(B, Hq, Nq, Nk, 82, use_alibi, use_bias)
    dq, dk, dv, _ = oracle.attention_masked_bwd(x.q, x.k, x.v, dout, causal, x.scale, window_left=window,
                                                alibi=slopes, bias=bias,
                                                bias_strides=(Hq * Nq * Nk, Nq * Nk))
    q = x.q.double().requires_grad_()
    k = x.k.double().requires_grad_()
    v = x.v.double().requires_grad_()
    c = additive_mask(B, Hq, Nq, Nk, causal, window, slopes, bias)
    out = torch.nn.functional.scaled_dot_product_attention(
        q, k.repeat_interleave(Hq // Hkv, 1), v.repeat_interleave(Hq // Hkv, 1), attn_mask=c, scale=x.scale)
    out.backward(dout.double())
    np.testing.assert_allclose(dq, q.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, k.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, v.grad.numpy(), atol=1e-11)


def test_masked_bwd_matches_finite_differences_of_the_masked_forward():
    # Broadcast bias (one [Nq, Nk] plane for every batch and head), ALiBi,
    # window and causal together; Nq > Nk leaves the first rows without keys.
    B, Hq, Hkv, Nq, Nk, d = 1, 2, 1, 7, 5, 4
    causal, window = True, 3
    x = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=83, causal=causal)
    dout = dout_for((B, Hq, Nq, d), 84)
    _, bias = mask_inputs(1, 1, Nq, Nk, 85, alibi=False)
    slopes = torch.tensor([0.25, 0.125], dtype=torch.float32)
    kw = dict(window_left=window, alibi=slopes, bias=bias, bias_strides=(0, 0))
    dq, dk, dv, _ = oracle.attention_masked_bwd(x.q, x.k, x.v, dout, causal, x.scale, **kw)
    go = bf16_np(dout)
    base = {"q": bf16_np(x.q), "k": bf16_np(x.k), "v": bf16_np(x.v)}

    def loss(arrs):
        # sum(dO * O) from the plain definition on float64 inputs (the
        # oracle's masked forward takes bf16 inputs, which a step of 1e-6
        # cannot perturb).
        total = 0.0
        q, k, v = arrs["q"], arrs["k"], arrs["v"]
        diag = Nk - Nq
        for h in range(Hq):
            for i in range(Nq):
                js = [j for j in range(Nk) if j <= i + diag and j > i + diag - window]
                if not js:
                    continue
                s = np.array([q[0, h, i] @ k[0, 0, j] * x.scale + float(slopes[h]) * (j - i - diag)
                              + float(bias[0, 0, i, j].float()) for j in js])
                w = np.exp(s - s.max())
                w /= w.sum()
                total += float(go[0, h, i] @ (w @ v[0, 0, js]))
        return total

    # The plain definition above must agree with the oracle's masked forward
    # (pinned to printed decimals elsewhere) before its differences are used.
    o_ref = oracle.attention_masked(x.q, x.k, x.v, causal, x.scale, **kw)[0]
    assert abs(loss(base) - float(np.nansum(go * o_ref))) < 1e-12
    h = 1e-6
    rng = np.random.default_rng(9)
    for name, grad in (("q", dq), ("k", dk), ("v", dv)):
        for _ in range(8):
            idx = tuple(int(rng.integers(0, n)) for n in base[name].shape)
            plus = {**base, name: base[name].copy()}
            minus = {**base, name: base[name].copy()}
            plus[name][idx] += h
            minus[name][idx] -= h
            fd = (loss(plus) - loss(minus)) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])
    # rows without an allowed key take no gradient
    assert np.all(dq[0, :, :2] == 0.0)


def test_masked_bwd_without_bias_is_the_plain_backward():
    B, Hq, Hkv, Nq, Nk, d = 1, 4, 2, 13, 9, 8
    x = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=86, causal=True)
    dout = dout_for((B, Hq, Nq, d), 87)
    a = oracle.attention_masked_bwd(x.q, x.k, x.v, dout, True, x.scale)
    b = oracle.attention_bwd(x.q, x.k, x.v, dout, True, x.scale)
    for u, w in zip(a[:3], b[:3]):
        np.testing.assert_allclose(u, w, rtol=0, atol=1e-13)
