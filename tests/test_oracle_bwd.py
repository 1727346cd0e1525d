"""Pins for the oracle's backward pass (dQ, dK, dV).

The pages fix the forward ("Compilers and Kernels", section "FlashAttention
changes the algorithm around IO"); the backward is its derivative ("Tang: a
compiler that derives GPU kernels ...", abstract: gradients of comprehensions
are comprehensions).  The oracle is pinned to central finite differences of
an independent float64 forward, to torch autograd through float64
scaled_dot_product_attention, to the closed-form sums the softmax Jacobian
fixes, and to the reduction of grouped-query attention to repeated MHA.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import oracle_mutants
from attention_online_softmax_gb300 import inputs
from test_oracle_pins import bf16_np

oracle_mutants.register_all()


def dout_for(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


def forward_loss(q, k, v, dout, causal, scale):
    """sum(dO * O) for float64 numpy inputs, O from the plain definition."""
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    rep = Hq // Hkv
    total = 0.0
    for b in range(B):
        for h in range(Hq):
            g = h // rep
            s = q[b, h] @ k[b, g].T * scale
            if causal:
                i = np.arange(Nq)[:, None]
                j = np.arange(Nk)[None, :]
                s = np.where(j <= i + Nk - Nq, s, -np.inf)
            for i in range(Nq):
                if np.all(np.isneginf(s[i])):
                    continue
                w = np.exp(s[i] - s[i].max())
                w /= w.sum()
                total += float(dout[b, h, i] @ (w @ v[b, g]))
    return total


@pytest.mark.parametrize("causal,shape", [(False, (1, 2, 1, 5, 6, 4)), (True, (1, 2, 2, 6, 6, 4)),
                                          (True, (1, 1, 1, 7, 4, 3))])
def test_bwd_matches_finite_differences(causal, shape):
    B, Hq, Hkv, Nq, Nk, d = shape
    x = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=50 + Nq, causal=causal)
    dout = dout_for((B, Hq, Nq, d), 51)
    dq, dk, dv, _ = oracle.attention_bwd(x.q, x.k, x.v, dout, causal, x.scale)
    q, k, v, go = bf16_np(x.q), bf16_np(x.k), bf16_np(x.v), bf16_np(dout)
    h = 1e-6
    rng = np.random.default_rng(3)
    for name, arr, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, n)) for n in arr.shape)
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += h
            minus[idx] -= h
            args = {"q": q, "k": k, "v": v}
            fd = (forward_loss(**{**args, name: plus}, dout=go, causal=causal, scale=x.scale)
                  - forward_loss(**{**args, name: minus}, dout=go, causal=causal, scale=x.scale)) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_matches_torch_autograd_float64(causal):
    B, Hq, Hkv, Nq, Nk, d = 2, 4, 2, 9, 13, 8
    x = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=52, causal=causal)
    dout = dout_for((B, Hq, Nq, d), 53)
    dq, dk, dv, _ = oracle.attention_bwd(x.q, x.k, x.v, dout, causal, x.scale)
    q = x.q.double().requires_grad_()
    k = x.k.double().requires_grad_()
    v = x.v.double().requires_grad_()
    mask = None
    if causal:
        i = torch.arange(Nq)[:, None]
        j = torch.arange(Nk)[None, :]
        mask = j <= i + Nk - Nq
    out = torch.nn.functional.scaled_dot_product_attention(
        q, k.repeat_interleave(Hq // Hkv, 1), v.repeat_interleave(Hq // Hkv, 1), attn_mask=mask, scale=x.scale)
    out.backward(dout.double())
    np.testing.assert_allclose(dq, q.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, k.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, v.grad.numpy(), atol=1e-11)


def test_bwd_closed_form_sums():
    # Rows of P sum to 1: sum_j dV_j = sum_i dO_i.  Rows of dS sum to 0:
    # sum_j dK_j = 0.  (Non-causal: every row has keys.)
    B, H, Nq, Nk, d = 1, 3, 17, 23, 16
    x = inputs.prefill_inputs(B, H, H, Nq, Nk, d, seed=54, causal=False)
    dout = dout_for((B, H, Nq, d), 55)
    dq, dk, dv, _ = oracle.attention_bwd(x.q, x.k, x.v, dout, False, x.scale)
    np.testing.assert_allclose(dv.sum(axis=2), bf16_np(dout).sum(axis=2), atol=1e-12)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)


def test_bwd_gqa_is_repeated_mha_summed_over_the_group():
    B, Hq, Hkv, Nq, Nk, d = 1, 6, 2, 10, 12, 8
    x = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=56, causal=True)
    dout = dout_for((B, Hq, Nq, d), 57)
    dq, dk, dv, _ = oracle.attention_bwd(x.q, x.k, x.v, dout, True, x.scale)
    rep = Hq // Hkv
    dq2, dk2, dv2, _ = oracle.attention_bwd(x.q, x.k.repeat_interleave(rep, 1), x.v.repeat_interleave(rep, 1),
                                            dout, True, x.scale)
    np.testing.assert_allclose(dq, dq2, atol=1e-13)
    np.testing.assert_allclose(dk, dk2.reshape(B, Hkv, rep, Nk, d).sum(axis=2), atol=1e-13)
    np.testing.assert_allclose(dv, dv2.reshape(B, Hkv, rep, Nk, d).sum(axis=2), atol=1e-13)


def test_bwd_rows_without_keys_take_no_gradient():
    # Causal with Nq > Nk: the first Nq - Nk rows see no key.
    x = inputs.prefill_inputs(1, 1, 1, 8, 3, 4, seed=58, causal=True)
    dout = dout_for((1, 1, 8, 4), 59)
    dq, dk, dv, _ = oracle.attention_bwd(x.q, x.k, x.v, dout, True, x.scale)
    assert np.all(dq[0, 0, :5] == 0.0)
    assert np.any(dq[0, 0, 5:] != 0.0)


@pytest.mark.parametrize("mutant", [6, 7])
def test_planted_backward_mistakes_are_caught(mutant):
    # A dropped D term (6) or a dropped dK scale (7) must fail the autograd pin.
    B, Hq, Hkv, Nq, Nk, d = 1, 2, 1, 9, 13, 8
    x = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=60, causal=True)
    dout = dout_for((B, Hq, Nq, d), 61)
    dq, dk, dv, _ = oracle.attention_bwd(x.q, x.k, x.v, dout, True, x.scale, mutant=mutant)
    q = x.q.double().requires_grad_()
    k = x.k.double().requires_grad_()
    v = x.v.double().requires_grad_()
    i = torch.arange(Nq)[:, None]
    j = torch.arange(Nk)[None, :]
    out = torch.nn.functional.scaled_dot_product_attention(
        q, k.repeat_interleave(Hq // Hkv, 1), v.repeat_interleave(Hq // Hkv, 1), attn_mask=j <= i + Nk - Nq,
        scale=x.scale)
    out.backward(dout.double())
    agree = (np.allclose(dq, q.grad.numpy(), atol=1e-9) and np.allclose(dk, k.grad.numpy(), atol=1e-9)
             and np.allclose(dv, v.grad.numpy(), atol=1e-9))
    assert not agree


@pytest.mark.parametrize("causal,shape", [(False, (1, 2, 1, 5, 6, 4)), (True, (1, 2, 2, 6, 6, 4)),
                                          (True, (1, 1, 1, 7, 4, 3))])
def test_bwd_dq_rows_match_finite_differences(causal, shape):
    # The per-row dQ function against central differences of the plain
    # forward, on every row (rows without keys included).
    B, Hq, Hkv, Nq, Nk, d = shape
    x = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=60 + Nq, causal=causal)
    dout = dout_for((B, Hq, Nq, d), 61)
    rows = np.arange(B * Hq * Nq)
    got = oracle.attention_bwd_dq_rows(x.q, x.k, x.v, dout, causal, x.scale, rows)
    q, k, v, go = bf16_np(x.q), bf16_np(x.k), bf16_np(x.v), bf16_np(dout)
    h = 1e-6
    rng = np.random.default_rng(5)
    for r in rows:
        c = int(rng.integers(0, d))
        idx = np.unravel_index(int(r), (B, Hq, Nq)) + (c,)
        plus, minus = q.copy(), q.copy()
        plus[idx] += h
        minus[idx] -= h
        fd = (forward_loss(plus, k, v, go, causal, x.scale) - forward_loss(minus, k, v, go, causal, x.scale)) / (2 * h)
        assert abs(fd - got[r, c]) <= 1e-6 * max(1.0, abs(fd)), (r, c, fd, got[r, c])


def test_bwd_dq_rows_equal_the_full_backward():
    # Sampled rows of a GQA causal case with Nq != Nk, in shuffled order.
    B, Hq, Hkv, Nq, Nk, d = 2, 4, 2, 37, 53, 16
    x = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=62, causal=True)
    dout = dout_for((B, Hq, Nq, d), 63)
    dq = oracle.attention_bwd(x.q, x.k, x.v, dout, True, x.scale)[0].reshape(-1, d)
    rows = np.random.default_rng(7).permutation(B * Hq * Nq)[:40]
    got = oracle.attention_bwd_dq_rows(x.q, x.k, x.v, dout, True, x.scale, rows)
    np.testing.assert_allclose(got, dq[rows], rtol=0, atol=1e-13)
    with pytest.raises(ValueError):
        oracle.attention_bwd_dq_rows(x.q, x.k, x.v, dout, True, x.scale, [B * Hq * Nq])
