"""GPU parity of the backward through the additive bias C (left window,
ALiBi slopes, dense bias) against the oracle's masked backward.

The forward is attn_fwd_masked with the same bias (its bf16 O and f32 LSE
feed the backward, as in training); gradients are checked elementwise with
the bound of test_gpu_bwd.grad_bound, in both output dtypes, with NaN-filled
outputs so that a missed write fails.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from attention_online_softmax_gb300 import configs, inputs
from test_gpu_bwd import dout_for, grad_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def abi():
    from attention_online_softmax_gb300 import build
    build.build()
    from attention_online_softmax_gb300 import abi as mod
    return mod


def bias_strides(bias, B, Hq):
    if bias is None:
        return (0, 0)
    return (bias.stride(0) if bias.shape[0] == B else 0, bias.stride(1) if bias.shape[1] == Hq else 0)


def run_masked_bwd(abi, x, dout, window, slopes, bias, g_dtype):
    dev = torch.device("cuda")
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    B, Hq, Nq, d = q.shape
    sl = None if slopes is None else slopes.to(dev)
    bb = None if bias is None else bias.to(dev)
    o = torch.empty((B, Hq, Nq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    abi.attn_fwd_masked(q, k, v, o, lse, x.causal, x.scale, window_left=window, alibi=sl, bias=bb)
    dq = torch.full(q.shape, float("nan"), dtype=g_dtype, device=dev)
    dk = torch.full(k.shape, float("nan"), dtype=g_dtype, device=dev)
    dv = torch.full(v.shape, float("nan"), dtype=g_dtype, device=dev)
    abi.attn_bwd(q, k, v, o, dout.to(dev), lse, dq, dk, dv, x.causal, x.scale, window_left=window, alibi=sl,
                 bias=bb)
    torch.cuda.synchronize()
    assert abi.attn_get_device_status() == 0
    return dq.double().cpu().numpy(), dk.double().cpu().numpy(), dv.double().cpu().numpy()


def check_masked_bwd(abi, x, seed, window=0, slopes=None, bias=None, dtypes=(torch.bfloat16, torch.float32)):
    B, Hq = x.q.shape[:2]
    dout = dout_for(x.q.shape, seed)
    ref = oracle.attention_masked_bwd(x.q, x.k, x.v, dout, x.causal, x.scale, window_left=window,
                                      alibi=None if slopes is None else slopes.numpy(), bias=bias,
                                      bias_strides=bias_strides(bias, B, Hq))[:3]
    for g_dtype in dtypes:
        got = run_masked_bwd(abi, x, dout, window, slopes, bias, g_dtype)
        for name, a, r in zip(("dq", "dk", "dv"), got, ref):
            assert np.all(np.isfinite(a)), f"{name}: non-finite values"
            err = np.abs(a - r)
            assert np.all(err <= grad_bound(r, g_dtype == torch.bfloat16)), (
                f"{name} ({g_dtype}): max|err| {err.max():.3e}, max|ref| {np.abs(r).max():.3e}")


CASES = [
    # B, Hq, Hkv, Nq, Nk, d, causal, window, alibi, bias shape kind, -inf fraction
    (1, 2, 2, 256, 256, 128, True, 100, False, None, 0.0),     # window inside one key tile's reach
    (1, 4, 2, 300, 300, 64, True, 200, True, None, 0.0),       # window + ALiBi, GQA, ragged
    (2, 2, 2, 200, 301, 128, False, 0, False, "full", 0.05),   # dense bias, odd Nk
    (1, 2, 1, 129, 260, 64, True, 0, True, "batch", 0.1),      # ALiBi + bias broadcast over the batch
    (1, 4, 2, 384, 384, 128, True, 130, True, "head", 0.0),    # everything, several key tiles
    (1, 2, 2, 200, 200, 256, True, 96, True, None, 0.0),       # d = 256: window + ALiBi
    (1, 4, 2, 192, 250, 256, False, 0, False, "full", 0.05),   # d = 256: dense bias
]


def bias_shape(kind, B, Hq, Nq, Nk):
    return {"full": (B, Hq, Nq, Nk), "batch": (1, Hq, Nq, Nk), "head": (B, 1, Nq, Nk)}[kind]


@pytest.mark.parametrize("case", CASES)
def test_masked_bwd(abi, case):
    B, Hq, Hkv, Nq, Nk, d, causal, window, use_alibi, kind, frac = case
    x = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=8000 + Nq + d, causal=causal)
    slopes = inputs.alibi_slopes(Hq) if use_alibi else None
    bias = None
    if kind is not None:
        bias = inputs.bias_inputs(bias_shape(kind, B, Hq, Nq, Nk), seed=8100 + Nq, neg_inf_frac=frac)
    check_masked_bwd(abi, x, seed=8200 + Nq, window=window, slopes=slopes, bias=bias)


def test_masked_bwd_rows_all_minus_inf(abi):
    # Query rows whose bias is -inf for every key take no gradient (LSE = -inf).
    B, Hq, Nq, Nk, d = 1, 2, 150, 300, 128
    x = inputs.prefill_inputs(B, Hq, Hq, Nq, Nk, d, seed=8300, causal=False)
    bias = inputs.bias_inputs((B, Hq, Nq, Nk), seed=8301, neg_inf_rows=5)
    check_masked_bwd(abi, x, seed=8302, bias=bias, dtypes=(torch.float32,))


def test_masked_bwd_no_bias_is_the_plain_backward(abi):
    # A zero window and no slopes or bias take the unbiased kernel: bitwise
    # equal dK, dV to attn_bwd.
    x = inputs.prefill_inputs(1, 2, 2, 256, 256, 128, seed=8400, causal=True)
    dout = dout_for(x.q.shape, 8401)
    a = run_masked_bwd(abi, x, dout, 0, None, None, torch.float32)
    from test_gpu_bwd import run_bwd
    b = run_bwd(abi, x, dout, torch.float32)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])


@pytest.mark.parametrize("cfg", [configs.WINDOW, configs.ALIBI_BIAS], ids=lambda c: c.name)
def test_masked_bwd_full_config_sampled_heads(abi, cfg):
    # The masked workloads' backward at full size, checked on (batch, head)
    # slices: with Hq = Hkv a head's gradients depend on that head's inputs
    # (and its plane of the bias) only, so the oracle runs on the slices alone.
    c = cfg
    x = inputs.prefill_inputs(c.B, c.Hq, c.Hkv, c.Nq, c.Nk, c.d, c.seed, c.causal)
    slopes = inputs.alibi_slopes(c.Hq) if c.alibi else None
    bias = None
    if c.bias is not None:
        shape = (c.B if c.bias == "full" else 1, c.Hq, c.Nq, c.Nk)
        bias = inputs.bias_inputs(shape, seed=c.seed + 100)
    g = torch.Generator().manual_seed(c.seed + 50)
    dout = torch.randn(x.q.shape, generator=g).to(torch.bfloat16)
    got = run_masked_bwd(abi, x, dout, c.window, slopes, bias, torch.float32)
    for b, h in ((0, 0), (c.B - 1, c.Hq - 1)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        bsl = None
        if bias is not None:
            bsl = bias[(slice(0, 1) if bias.shape[0] == 1 else slice(b, b + 1), slice(h, h + 1))].contiguous()
        ref = oracle.attention_masked_bwd(
            x.q[sl].contiguous(), x.k[sl].contiguous(), x.v[sl].contiguous(), dout[sl].contiguous(), c.causal,
            x.scale, window_left=c.window, alibi=None if slopes is None else slopes[h:h + 1].numpy(),
            bias=bsl, bias_strides=(0, 0))[:3]
        for name, a, r in zip(("dq", "dk", "dv"), got, ref):
            err = np.abs(a[sl] - r)
            assert np.all(err <= grad_bound(r, False)), (name, b, h, err.max())
