"""GPU parity of the attention backward (dQ, dK, dV) against the f64 oracle.

The kernel takes the forward's bf16 O and f32 LSE from ``attn_fwd`` (as a
training step would) and rounds P and dS to bf16 before their tensor-core
products; the oracle differentiates the exact softmax in float64.  Each
gradient is checked elementwise against a bound derived from that arithmetic
(see ``grad_bound``), in both output modes, with every output buffer
NaN-prefilled so that a missed write fails.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from attention_online_softmax_gb300 import configs, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def abi():
    from attention_online_softmax_gb300 import build
    build.build()
    from attention_online_softmax_gb300 import abi as mod
    return mod


def dout_for(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


def run_bwd(abi, x, dout, g_dtype):
    dev = torch.device("cuda")
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    B, Hq, Nq, d = q.shape
    o = torch.empty((B, Hq, Nq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    abi.attn_fwd(q, k, v, o, lse, x.causal, x.scale)
    dq = torch.full(q.shape, float("nan"), dtype=g_dtype, device=dev)
    dk = torch.full(k.shape, float("nan"), dtype=g_dtype, device=dev)
    dv = torch.full(v.shape, float("nan"), dtype=g_dtype, device=dev)
    abi.attn_bwd(q, k, v, o, dout.to(dev), lse, dq, dk, dv, x.causal, x.scale)
    torch.cuda.synchronize()
    assert abi.attn_get_device_status() == 0
    return dq.double().cpu().numpy(), dk.double().cpu().numpy(), dv.double().cpu().numpy()


def grad_bound(ref, bf16_out):
    """Allowed |error| per element.

    The kernel's weights P and dS enter the tensor cores as bf16 (relative
    rounding 2^-9 each), D = rowsum(dO * O) uses the bf16-rounded O, and the
    sums run in f32.  Each gradient element is a sum of such rounded terms,
    so its error is a few 2^-9 of the size of the terms, which the largest
    |value| of the gradient tensor bounds; measured worst cases sit near
    2.5 * 2^-9 of max|ref|.  We allow 4 * 2^-9 = 2^-7 of max|ref|, plus half a
    bf16 ulp of each element when the output is bf16.
    """
    tol = 2.0 ** -7 * np.abs(ref).max(initial=0.0)
    if bf16_out:
        tol = tol + 2.0 ** -9 * np.abs(ref)
    return tol


def check_bwd(abi, x, seed):
    dout = dout_for(x.q.shape, seed)
    ref = oracle.attention_bwd(x.q, x.k, x.v, dout, x.causal, x.scale)[:3]
    worst = {}
    for g_dtype in (torch.bfloat16, torch.float32):
        got = run_bwd(abi, x, dout, g_dtype)
        for name, a, r in zip(("dq", "dk", "dv"), got, ref):
            assert np.all(np.isfinite(a)), f"{name}: non-finite values"
            err = np.abs(a - r)
            bound = grad_bound(r, g_dtype == torch.bfloat16)
            assert np.all(err <= bound), (f"{name} ({g_dtype}): max|err| {err.max():.3e}, "
                                          f"max|ref| {np.abs(r).max():.3e}")
            scale = np.abs(r).max(initial=0.0)
            worst[(name, str(g_dtype))] = err.max(initial=0.0) / (scale if scale > 0 else 1.0)
    return worst


SHAPES = [
    # B, Hq, Hkv, Nq, Nk, d, causal
    (1, 2, 2, 128, 128, 64, False),
    (1, 2, 2, 128, 128, 128, True),
    (1, 2, 2, 200, 200, 64, True),      # ragged
    (2, 4, 2, 77, 300, 128, True),      # Nq < Nk, GQA
    (1, 2, 1, 300, 77, 128, True),      # Nq > Nk: rows without keys
    (1, 8, 2, 256, 384, 64, False),     # GQA 4:1, several key tiles
    (2, 4, 4, 640, 640, 128, True),
    # d = 256: two CTAs per key tile (head-dim halves), 64-query items.
    (1, 2, 2, 128, 128, 256, False),
    (1, 2, 2, 200, 200, 256, True),     # ragged
    (2, 4, 2, 77, 300, 256, True),      # Nq < Nk (Nq not a multiple of 4), GQA
    (1, 2, 1, 300, 77, 256, True),      # Nq > Nk: rows without keys
    (1, 8, 2, 256, 384, 256, False),    # GQA 4:1, several key tiles
    (1, 4, 1, 640, 640, 256, True),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_bwd_shapes(abi, shape):
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    x = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=7000 + Nq + Nk + d, causal=causal)
    check_bwd(abi, x, seed=7100 + Nq)


def test_bwd_larger(abi):
    x = inputs.prefill_inputs(1, 8, 8, 1024, 1024, 128, seed=7200, causal=True)
    check_bwd(abi, x, seed=7201)


def test_bwd_zero_queries_or_keys(abi):
    dev = torch.device("cuda")
    # Nk = 0: dQ = 0.
    x = inputs.prefill_inputs(1, 2, 2, 64, 0, 64, seed=7300, causal=False)
    dout = dout_for(x.q.shape, 7301).to(dev)
    q = x.q.to(dev)
    o = torch.zeros_like(q)
    lse = torch.full((1, 2, 64), float("-inf"), dtype=torch.float32, device=dev)
    dq = torch.full(q.shape, float("nan"), dtype=torch.float32, device=dev)
    k = torch.empty((1, 2, 0, 64), dtype=torch.bfloat16, device=dev)
    abi.attn_bwd(q, k, k, o, dout, lse, dq, k.float(), k.float(), False, x.scale)
    torch.cuda.synchronize()
    assert torch.all(dq == 0)


def test_bwd_dk_dv_deterministic(abi):
    x = inputs.prefill_inputs(1, 4, 2, 512, 512, 128, seed=7400, causal=True)
    dout = dout_for(x.q.shape, 7401)
    a = run_bwd(abi, x, dout, torch.float32)
    b = run_bwd(abi, x, dout, torch.float32)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    np.testing.assert_allclose(a[0], b[0], atol=1e-5)  # dQ: atomic summation order


def test_bwd_large_score_range(abi):
    # K scaled by 8: peaky weights, many rows dominated by one key.
    x = inputs.prefill_inputs(1, 2, 2, 384, 384, 128, seed=7500, causal=True, k_scale=8.0)
    check_bwd(abi, x, seed=7501)


def test_bwd_full_config_sampled_heads(abi):
    # The benchmark's backward launch (causal MHA B2 H32 N4096 d128) checked on
    # two (batch, head) slices: with Hq = Hkv a head's gradients depend on that
    # head's inputs only, so the oracle runs on the slices alone.
    c = configs.LONG
    x = inputs.prefill_inputs(c.B, c.Hq, c.Hkv, c.Nq, c.Nk, c.d, c.seed, c.causal)
    g = torch.Generator().manual_seed(c.seed + 50)
    dout = torch.randn(x.q.shape, generator=g).to(torch.bfloat16)
    got = run_bwd(abi, x, dout, torch.float32)
    for b, h in ((0, 0), (1, 31)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle.attention_bwd(x.q[sl].contiguous(), x.k[sl].contiguous(), x.v[sl].contiguous(),
                                   dout[sl].contiguous(), True, x.scale)[:3]
        for name, a, r in zip(("dq", "dk", "dv"), got, ref):
            err = np.abs(a[sl] - r)
            assert np.all(err <= grad_bound(r, False)), (name, b, h, err.max())


def test_bwd_d256_gqa_shape_shorter(abi):
    # The long d = 256 workload's head layout (B1, 16 query heads on 2 kv
    # heads, causal) at N = 2048, every gradient element against the oracle.
    c = configs.GQA256
    x = inputs.prefill_inputs(c.B, c.Hq, c.Hkv, 2048, 2048, c.d, seed=c.seed + 60, causal=c.causal)
    check_bwd(abi, x, seed=c.seed + 61)


def test_bwd_d256_full_config_sampled(abi):
    # The benchmark's d = 256 backward launch (causal GQA B1 Hq16 Hkv2 N16384)
    # checked on seeded query rows of dQ, which the oracle computes one by
    # one, and on the closed-form sums over keys that hold at any size:
    # rows of P sum to 1 (sum_j dV_j = sum of dO over the rows that see a
    # key) and rows of dS sum to 0 (sum_j dK_j = 0).
    c = configs.GQA256
    x = inputs.prefill_inputs(c.B, c.Hq, c.Hkv, c.Nq, c.Nk, c.d, c.seed, c.causal)
    g = torch.Generator().manual_seed(c.seed + 50)
    dout = torch.randn(x.q.shape, generator=g).to(torch.bfloat16)
    dq, dk, dv = run_bwd(abi, x, dout, torch.float32)
    rows = np.random.default_rng(c.seed + 51).choice(c.B * c.Hq * c.Nq, size=96, replace=False)
    ref = oracle.attention_bwd_dq_rows(x.q, x.k, x.v, dout, True, x.scale, rows)
    got = dq.reshape(-1, c.d)[rows]
    assert np.all(np.abs(got - ref) <= grad_bound(ref, False)), np.abs(got - ref).max()
    # Sums over keys, per (batch, kv head, column).  The kernel rounds P and
    # dS to bf16 (2^-9 relative): the sums carry about 2^-9 of the summed
    # magnitudes, which the bounds below allow four times over.
    go = dout.double().numpy().reshape(c.B, c.Hkv, c.Hq // c.Hkv, c.Nq, c.d)
    want_dv = go.sum(axis=(2, 3))   # causal with Nq == Nk: every row sees a key
    tol_dv = 2.0 ** -7 * np.abs(dv).sum(axis=2) + 1e-3
    assert np.all(np.abs(dv.sum(axis=2) - want_dv) <= tol_dv), np.abs(dv.sum(axis=2) - want_dv).max()
    tol_dk = 2.0 ** -7 * np.abs(dk).sum(axis=2) + 1e-3
    assert np.all(np.abs(dk.sum(axis=2)) <= tol_dk), np.abs(dk.sum(axis=2)).max()
