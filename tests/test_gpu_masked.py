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
from attention_online_softmax_gb300 import configs, inputs
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
    # Nk a multiple of 8: the bias is staged into shared memory by TMA
    (1, 2, 2, 200, 304, 128, False, 0, False, "full", 0.05),
    (2, 3, 3, 130, 64, 64, False, 0, False, "head", 0.0),      # one partial key tile
    (2, 2, 1, 129, 256, 128, True, 0, False, "batch", 0.1),
    (1, 2, 2, 152, 152, 256, True, 64, True, "batch", 0.0),
    (1, 4, 4, 513, 1024, 64, False, 300, True, "both", 0.02),
    (1, 2, 2, 300, 80, 128, True, 20, True, "full", 0.0),
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


@pytest.mark.parametrize("kind", [None, "batch", "full"])  # ALiBi alone, staged bias, direct bias
def test_alibi_slopes_of_either_sign(abi, kind):
    # With ALiBi slopes the key tiles are taken from the last to the first.
    # Positive slopes put each row's maximum on the first tile taken;
    # negative ones (and a steep mix) make it grow on every tile, so O is
    # rescaled after every key tile: the result must not depend on which.
    B, Hq, Nq, Nk, d = 1, 4, 300, 1100 if kind != "full" else 1101, 128
    x = inputs.prefill_inputs(B, Hq, Hq, Nq, Nk, d, seed=4150, causal=False)
    slopes = inputs.alibi_slopes(Hq) * torch.tensor([-1.0, 1.0, -8.0, 0.5])
    bias = None
    if kind is not None:
        bias = inputs.bias_inputs(bias_shape(kind, B, Hq, Nq, Nk), seed=4151, neg_inf_frac=0.02)
    check_masked(abi, x, slopes=slopes, bias=bias)


@pytest.mark.parametrize("Nk", [300, 296])  # direct and staged bias reads
def test_bias_rows_all_minus_inf(abi, Nk):
    # Query rows whose bias is -inf for every key: O = 0, LSE = -inf.
    B, Hq, Nq, d = 1, 2, 260, 128
    x = inputs.prefill_inputs(B, Hq, Hq, Nq, Nk, d, seed=4200, causal=False)
    bias = inputs.bias_inputs((B, Hq, Nq, Nk), seed=4201, neg_inf_rows=5)
    _, lse_ref = check_masked(abi, x, bias=bias)
    assert np.isneginf(lse_ref).sum() == 5


@pytest.mark.parametrize("d", [64, 128, 256])
def test_staged_and_direct_bias_reads_agree(abi, d):
    # The same bias through the shared-memory staging path (16-byte aligned
    # copy) and through direct loads (a copy 4 bytes off the 16-byte grid)
    # gives bitwise the same result: both add the same terms in the same order.
    B, Hq, Nq, Nk = 1, 2, 300, 512
    x = inputs.prefill_inputs(B, Hq, Hq, Nq, Nk, d, seed=4250 + d, causal=True)
    bias = inputs.bias_inputs((B, Hq, Nq, Nk), seed=4251, neg_inf_frac=0.05)
    dev = torch.device("cuda")
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    aligned = bias.to(dev)
    raw = torch.empty(bias.numel() + 8, dtype=torch.bfloat16, device=dev)
    off = raw[2:2 + bias.numel()].view(bias.shape)  # 4-byte aligned, not 16
    off.copy_(aligned)
    assert off.data_ptr() % 16 != 0 and aligned.data_ptr() % 16 == 0
    slopes = inputs.alibi_slopes(Hq).to(dev)
    outs = []
    for b in (aligned, off):
        o = torch.empty((B, Hq, Nq, d), dtype=torch.float32, device=dev)
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
        abi.attn_fwd_masked(q, k, v, o, lse, True, x.scale, window_left=400, alibi=slopes, bias=b)
        outs.append((o, lse))
    torch.cuda.synchronize()
    assert abi.attn_get_device_status() == 0
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


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


@pytest.mark.parametrize("cfg", configs.MASKED_CONFIGS, ids=lambda c: c.name)
def test_masked_configs(abi, cfg):
    # The additive-bias workloads the benchmark times, on a seeded row subset.
    x = inputs.prefill_inputs(cfg.B, cfg.Hq, cfg.Hkv, cfg.Nq, cfg.Nk, cfg.d, cfg.seed, cfg.causal)
    rows = inputs.check_rows(x.generator, cfg.B, cfg.Hq, cfg.Nq, cfg.check_rows_per_head)
    slopes = inputs.alibi_slopes(cfg.Hq) if cfg.alibi else None
    bias = None
    if cfg.bias is not None:
        shape = (cfg.B if cfg.bias == "full" else 1, cfg.Hq, cfg.Nq, cfg.Nk)
        bias = inputs.bias_inputs(shape, seed=cfg.seed + 100)
    strides = (0, 0)
    if bias is not None:
        strides = (bias.stride(0) if bias.shape[0] == cfg.B else 0, bias.stride(1))
    o_ref, lse_ref, _ = oracle.attention_masked(
        x.q, x.k, x.v, cfg.causal, x.scale, window_left=cfg.window,
        alibi=None if slopes is None else slopes.numpy(), bias=bias, bias_strides=strides, rows=rows)
    for dt in (torch.bfloat16, torch.float32):
        o, lse = run_masked(abi, x, cfg.window, slopes, bias, dt)
        d = o.shape[-1]
        compare(o.reshape(-1, d)[rows.numpy()], lse.reshape(-1)[rows.numpy()], o_ref, lse_ref,
                dt == torch.bfloat16)
