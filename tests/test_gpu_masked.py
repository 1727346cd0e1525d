"""GPU parity of the additive bias C (left window, ALiBi slopes, dense bias).

"Compilers and Kernels", section "FlashAttention changes the algorithm around
IO": S = Q K^T / sqrt(d) + C, C in R U {-inf}.  ``attn_fwd_masked`` (through
the C ABI) against the oracle's ``attention_masked`` on the same seeded
inputs, with the tolerances of the plain parity tests: max|dO| <= 1e-2,
max|dLSE| <= 1e-3, the -inf LSE pattern exact (rows whose every key is
disallowed give O = 0 and LSE = -inf).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from attention_online_softmax_gb300 import inputs
from test_gpu_parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def abi():
    from attention_online_softmax_gb300 import build
    build.build()
    from attention_online_softmax_gb300 import abi as mod
    return mod


def bias_shape(kind, B, Hq, Nq, Nk):
    return {"full": (B, Hq, Nq, Nk), "head": (B, 1, Nq, Nk), "batch": (1, Hq, Nq, Nk),
            "both": (1, 1, Nq, Nk)}[kind]


def run_masked(abi, x, window, slopes, bias, o_dtype):
    dev = torch.device("cuda")
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    B, Hq, Nq, d = q.shape
    o = torch.full((B, Hq, Nq, d), float("nan"), dtype=o_dtype, device=dev)
    lse = torch.full((B, Hq, Nq), float("nan"), dtype=torch.float32, device=dev)
    abi.attn_fwd_masked(q, k, v, o, lse, x.causal, x.scale, window_left=window,
                        alibi=None if slopes is None else slopes.to(dev),
                        bias=None if bias is None else bias.to(dev))
    torch.cuda.synchronize()
    assert abi.attn_get_device_status() == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


def check_masked(abi, x, window=0, slopes=None, bias=None):
    B, Hq, Nq, _ = x.q.shape
    Nk = x.k.shape[2]
    strides = (0, 0)
    if bias is not None:
        strides = (bias.stride(0) if bias.shape[0] == B else 0,
                   bias.stride(1) if bias.shape[1] == Hq else 0)
    o_ref, lse_ref, _ = oracle.attention_masked(
        x.q, x.k, x.v, x.causal, x.scale, window_left=window,
        alibi=None if slopes is None else slopes.numpy(), bias=bias, bias_strides=strides)
    out = []
    for dt in (torch.bfloat16, torch.float32):
        o, lse = run_masked(abi, x, window, slopes, bias, dt)
        out.append(compare(o, lse, o_ref, lse_ref, dt == torch.bfloat16))
    return out, lse_ref


MASKED = [
    # B, Hq, Hkv, Nq, Nk, d, causal, window, alibi, bias kind, -inf fraction
    (1, 4, 2, 600, 600, 128, True, 100, False, None, 0.0),     # sliding window: early tiles skipped
    (1, 2, 2, 300, 900, 64, False, 257, False, None, 0.0),     # window without causal, Nk > Nq
    (1, 2, 2, 777, 777, 128, True, 1, False, None, 0.0),       # window of one key: the diagonal
    (2, 4, 4, 333, 333, 128, True, 0, True, None, 0.0),        # ALiBi, causal
    (1, 8, 2, 256, 512, 64, True, 0, True, None, 0.0),         # ALiBi with GQA
    (1, 2, 2, 200, 301, 128, False, 0, False, "full", 0.05),   # dense bias, odd Nk: odd row starts
    (2, 3, 3, 130, 77, 64, False, 0, False, "head", 0.0),      # bias broadcast over heads
    (2, 2, 1, 129, 260, 128, True, 0, False, "batch", 0.1),    # bias broadcast over the batch
    (1, 2, 2, 150, 150, 256, True, 64, True, "batch", 0.0),    # all terms, d = 256
    (1, 2, 2, 300, 77, 128, True, 20, True, "full", 0.0),      # Nq > Nk: rows without keys
    (1, 4, 4, 513, 1025, 64, False, 300, True, "both", 0.02),  # all terms, d = 64, ragged
]


@pytest.mark.parametrize("case", MASKED)
def test_masked_prefill(abi, case):
    B, Hq, Hkv, Nq, Nk, d, causal, window, use_alibi, kind, frac = case
    x = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=4000 + Nq + Nk + d, causal=causal)
    slopes = inputs.alibi_slopes(Hq) if use_alibi else None
    bias = None
    if kind is not None:
        bias = inputs.bias_inputs(bias_shape(kind, B, Hq, Nq, Nk), seed=4100 + Nq, neg_inf_frac=frac)
    check_masked(abi, x, window, slopes, bias)


def test_bias_rows_all_minus_inf(abi):
    # Query rows whose bias is -inf for every key: O = 0, LSE = -inf.
    B, Hq, Nq, Nk, d = 1, 2, 260, 300, 128
    x = inputs.prefill_inputs(B, Hq, Hq, Nq, Nk, d, seed=4200, causal=False)
    bias = inputs.bias_inputs((B, Hq, Nq, Nk), seed=4201, neg_inf_rows=5)
    _, lse_ref = check_masked(abi, x, bias=bias)
    assert np.isneginf(lse_ref).sum() == 5


def test_two_tile_units_with_window(abi):
    # Enough (batch, head) units that the plain path pairs two query tiles per
    # CTA; the window moves each unit's first key tile.
    x = inputs.prefill_inputs(1, 320, 64, 500, 500, 64, seed=4300, causal=True)
    check_masked(abi, x, window=130)


def test_wide_window_is_the_plain_kernel(abi):
    # A window longer than every row's key range disallows nothing: the result
    # is bitwise that of attn_fwd.
    x = inputs.prefill_inputs(1, 4, 2, 700, 900, 128, seed=4400, causal=True)
    dev = torch.device("cuda")
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    o1 = torch.empty((1, 4, 700, 128), dtype=torch.bfloat16, device=dev)
    l1 = torch.empty((1, 4, 700), dtype=torch.float32, device=dev)
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    abi.attn_fwd(q, k, v, o1, l1, True, x.scale)
    abi.attn_fwd_masked(q, k, v, o2, l2, True, x.scale, window_left=2000)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_masked_arguments_rejected(abi):
    x = inputs.prefill_inputs(1, 2, 2, 64, 64, 64, seed=4500, causal=False)
    dev = torch.device("cuda")
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    o = torch.empty((1, 2, 64, 64), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((1, 2, 64), dtype=torch.float32, device=dev)
    with pytest.raises(abi.AttnError):
        abi.attn_fwd_masked(q, k, v, o, lse, False, x.scale, window_left=-1)
    raw = torch.zeros(1 + 2 * 64 * 64, dtype=torch.bfloat16, device=dev)
    misaligned = raw[1:].view(1, 2, 64, 64)  # 2-byte aligned only
    with pytest.raises(abi.AttnError):
        abi.attn_fwd_masked(q, k, v, o, lse, False, x.scale, bias=misaligned)
