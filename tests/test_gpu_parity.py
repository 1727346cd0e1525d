"""GPU parity: the CUDA kernels, called through the C ABI, against the f64 oracle.

Tolerance (bf16 inputs, f32 accumulation): max|dO| <= 1e-2 and
max|dLSE| <= 1e-3.  bf16 output rounding alone exceeds 1e-2 once |O| >= 4
(half an ulp is 2^-6 there), so bf16-output elements with |O_ref| >= 4 are
gated through the float32-output mode of the same kernel instead, which must
meet 1e-2 everywhere.  Every output buffer is prefilled with NaN so a missed
write fails.  Large configurations are compared on a seeded subset of query
rows (>= 256 per head plus the first and last row).
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from attention_online_softmax_gb300 import configs, inputs

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module")
def abi():
    from attention_online_softmax_gb300 import build
    build.build()
    from attention_online_softmax_gb300 import abi as mod
    return mod


def run_fwd(abi, x, o_dtype=torch.bfloat16):
    dev = torch.device("cuda")
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    B, Hq, Nq, d = q.shape
    o = torch.full((B, Hq, Nq, d), float("nan"), dtype=o_dtype, device=dev)
    lse = torch.full((B, Hq, Nq), float("nan"), dtype=torch.float32, device=dev)
    abi.attn_fwd(q, k, v, o, lse, x.causal, x.scale)
    torch.cuda.synchronize()
    assert abi.attn_get_device_status() == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


def compare(o, lse, o_ref, lse_ref, bf16_out: bool):
    o = o.reshape(o_ref.shape).astype(np.float64)
    lse = lse.reshape(lse_ref.shape).astype(np.float64)
    assert np.all(np.isfinite(o)), "non-finite O (missed write or NaN read)"
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isneginf(lse), ~fin), "LSE -inf pattern differs"
    dl = np.abs(lse[fin] - lse_ref[fin]).max(initial=0.0)
    do = np.abs(o - o_ref)
    big = np.abs(o_ref) >= 4.0
    gated = do[~big] if bf16_out else do
    worst = gated.max(initial=0.0)
    assert worst <= O_TOL, f"max|dO| = {worst}"
    assert dl <= LSE_TOL, f"max|dLSE| = {dl}"
    return worst, dl, int(big.sum())


def check_prefill(abi, x, rows=None):
    o_ref, lse_ref, _ = oracle.attention(x.q, x.k, x.v, x.causal, x.scale, rows=rows)
    results = []
    for dt in (torch.bfloat16, torch.float32):
        o, lse = run_fwd(abi, x, dt)
        d = o.shape[-1]
        if rows is not None:
            o = o.reshape(-1, d)[rows.numpy()]
            lse = lse.reshape(-1)[rows.numpy()]
        results.append(compare(o, lse, o_ref, lse_ref, dt == torch.bfloat16))
    return results


SMALL_PREFILL = [
    # B, Hq, Hkv, Nq, Nk, d, causal
    (1, 2, 2, 128, 128, 64, False),
    (1, 2, 2, 200, 200, 64, False),     # ragged in both dims
    (2, 3, 3, 77, 300, 128, True),      # Nq < Nk, bottom-right causal
    (1, 2, 2, 300, 77, 128, True),      # Nq > Nk: rows without keys
    (1, 4, 2, 257, 257, 128, True),     # GQA, ragged
    (1, 8, 1, 129, 520, 256, False),    # MQA, d = 256
    (1, 2, 2, 384, 384, 256, True),
    (2, 2, 2, 1, 1, 64, False),         # one key
    (1, 2, 2, 1, 700, 128, True),       # single query row (decode-like)
]


@pytest.mark.parametrize("shape", SMALL_PREFILL)
def test_prefill_small_shapes(abi, shape):
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    x = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=1000 + Nq + Nk + d, causal=causal)
    check_prefill(abi, x)


# Enough (batch, head) x 256-row units that the library pairs two query tiles
# per CTA; ragged tails leave the second tile of the last unit partly or
# entirely past Nq.
TWO_TILE = [
    (1, 200, 200, 500, 500, 64, True),
    (2, 100, 20, 300, 420, 128, True),
    (1, 320, 320, 300, 300, 128, False),
]


@pytest.mark.parametrize("shape", TWO_TILE)
def test_prefill_two_tile_units(abi, shape):
    B, Hq, Hkv, Nq, Nk, d, causal = shape
    x = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=3000 + Nq + Hq, causal=causal)
    check_prefill(abi, x)


def test_prefill_zero_keys(abi):
    x = inputs.prefill_inputs(1, 2, 2, 64, 0, 128, seed=5, causal=False)
    o, lse = run_fwd(abi, x)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_prefill_large_score_range_rescaling(abi):
    # K scaled by 8: scores spread widely, the running max moves often.
    x = inputs.prefill_inputs(1, 2, 2, 640, 640, 128, seed=6, causal=True, k_scale=8.0)
    check_prefill(abi, x)


@pytest.mark.parametrize("cfg", [configs.TINY, configs.BLOCK, configs.LONG, configs.LONG_K4,
                                 configs.GQA256], ids=lambda c: c.name)
def test_prefill_configs(abi, cfg):
    x = inputs.prefill_inputs(cfg.B, cfg.Hq, cfg.Hkv, cfg.Nq, cfg.Nk, cfg.d, cfg.seed, cfg.causal,
                              k_scale=cfg.k_scale)
    rows = None
    if cfg.check_rows_per_head is not None:
        rows = inputs.check_rows(x.generator, cfg.B, cfg.Hq, cfg.Nq, cfg.check_rows_per_head)
    check_prefill(abi, x, rows)


def test_prefill_is_deterministic(abi):
    x = inputs.prefill_inputs(1, 4, 4, 1000, 1000, 128, seed=7, causal=True)
    o1, l1 = run_fwd(abi, x)
    o2, l2 = run_fwd(abi, x)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("d,two", [(64, False), (128, True), (256, False)])
def test_prefill_output_only_16_byte_aligned(abi, d, two):
    # O at an address that is 16-byte but not 32-byte aligned (the contract's
    # minimum) takes the epilogue's 16-byte stores: bitwise the result written
    # to an aligned O.
    heads = 160 if two else 2
    x = inputs.prefill_inputs(1, heads, heads, 300, 300, d, seed=7100 + d, causal=True)
    dev = torch.device("cuda")
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    shape = (1, heads, 300, d)
    n = math.prod(shape)
    o_al = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    raw = torch.empty(n + 16, dtype=torch.bfloat16, device=dev)
    o_off = raw[8:8 + n].view(shape)  # 16 bytes past a 256-byte aligned base
    assert o_off.data_ptr() % 32 == 16 and o_al.data_ptr() % 32 == 0
    outs = []
    for o in (o_al, o_off):
        lse = torch.empty((1, heads, 300), dtype=torch.float32, device=dev)
        abi.attn_fwd(q, k, v, o, lse, True, x.scale)
        outs.append((o.clone(), lse))
    torch.cuda.synchronize()
    assert abi.attn_get_device_status() == 0
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_prefill_output_depends_on_every_input(abi):
    # Perturb one element of Q, K and V in turn: the affected rows must change.
    x = inputs.prefill_inputs(1, 2, 2, 256, 256, 64, seed=8, causal=False)
    o0, l0 = run_fwd(abi, x)
    for name in ("q", "k", "v"):
        y = inputs.prefill_inputs(1, 2, 2, 256, 256, 64, seed=8, causal=False)
        t = getattr(y, name)
        t[0, 1, 200, 5] = t[0, 1, 200, 5] + 3.0
        o1, l1 = run_fwd(abi, y)
        assert not np.array_equal(o0, o1), name


# ------------------------------------------------------------------ decode
def run_decode(abi, d_in, o_dtype=torch.bfloat16):
    dev = torch.device("cuda")
    q = d_in.q.to(dev)
    kc, vc = d_in.kcache.to(dev), d_in.vcache.to(dev)
    bt, sl = d_in.block_table.to(dev), d_in.seqlens.to(dev)
    S, Hq, d = q.shape
    Hkv = kc.shape[2]
    o = torch.full((S, Hq, d), float("nan"), dtype=o_dtype, device=dev)
    lse = torch.full((S, Hq), float("nan"), dtype=torch.float32, device=dev)
    max_len = int(d_in.seqlens.max().item()) if S else 0
    nbytes = abi.attn_decode_workspace_size(S, Hq, Hkv, d, max_len)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    ws.fill_(0xFF)  # NaN pattern: partials must all be written before use
    abi.attn_decode_paged(q, kc, vc, bt, sl, o, lse, max_len, d_in.scale, ws)
    torch.cuda.synchronize()
    assert abi.attn_get_device_status() == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


def check_decode(abi, d_in):
    o_ref, lse_ref, _ = oracle.decode_paged(d_in.q, d_in.kcache, d_in.vcache, d_in.block_table,
                                            d_in.seqlens, d_in.scale)
    for dt in (torch.bfloat16, torch.float32):
        o, lse = run_decode(abi, d_in, dt)
        compare(o, lse, o_ref, lse_ref, dt == torch.bfloat16)


SMALL_DECODE = [
    # num_seqs, Hq, Hkv, d, lengths
    (5, 32, 8, 128, [1, 15, 16, 17, 300]),
    (3, 8, 8, 64, [0, 33, 700]),            # empty sequence, G = 1
    (4, 16, 2, 128, [1000, 1, 257, 64]),    # G = 8
    (2, 8, 4, 256, [513, 2048]),            # d = 256, G = 2
    (3, 16, 4, 64, [4096, 100, 4095]),
    (1, 4, 4, 128, [8192]),                 # one long sequence: many small chunks
]


@pytest.mark.parametrize("case", SMALL_DECODE)
def test_decode_small_cases(abi, case):
    S, Hq, Hkv, d, lens = case
    pages = sum((L + 15) // 16 for L in lens) + 7
    d_in = inputs.decode_inputs(S, Hq, Hkv, d, 0, max(lens), num_pages=pages, page_size=16,
                                seed=2000 + sum(lens), lengths=lens,
                                max_pages_per_seq=(max(lens) + 15) // 16 + 1)
    check_decode(abi, d_in)


PAGED_DECODE = [
    # num_seqs, Hq, Hkv, d, page_size, lengths
    (4, 32, 8, 128, 32, [1, 31, 33, 700]),       # contexts ending mid-page
    (3, 16, 4, 64, 64, [64, 65, 1500]),
    (3, 8, 2, 256, 128, [127, 128, 2049]),
    (5, 32, 2, 128, 16, [17, 300, 1, 4000, 256]),  # a group of 16 query heads
    (3, 64, 4, 64, 128, [900, 1, 5000]),           # group of 16, 128-token pages
    (2, 16, 1, 256, 32, [70, 3000]),               # MQA-style group of 16 at d = 256
]


@pytest.mark.parametrize("case", PAGED_DECODE)
def test_decode_page_sizes_and_groups(abi, case):
    S, Hq, Hkv, d, page, lens = case
    pages = sum((L + page - 1) // page for L in lens) + 5
    d_in = inputs.decode_inputs(S, Hq, Hkv, d, 0, max(lens), num_pages=pages, page_size=page,
                                seed=3000 + sum(lens) + page, lengths=lens,
                                max_pages_per_seq=(max(lens) + page - 1) // page + 1)
    check_decode(abi, d_in)


def test_decode_workspace_reuse_determinism_and_graph_replay(abi):
    # One workspace for several calls: its merge counters must come back
    # reset, so a second call (other inputs), a repeat of the first (bitwise
    # equal) and two replays of a captured call (same epoch) all merge right.
    dev = torch.device("cuda")
    cases = [inputs.decode_inputs(6, 32, 8, 128, 300, 3000, num_pages=1200, page_size=16, seed=41),
             inputs.decode_inputs(6, 32, 8, 128, 300, 3000, num_pages=1200, page_size=16, seed=42)]
    need = max(abi.attn_decode_workspace_size(6, 32, 8, 128, c.max_seqlen) for c in cases)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=dev)

    def call(c, o, lse):
        abi.attn_decode_paged(c.q.to(dev), c.kcache.to(dev), c.vcache.to(dev), c.block_table.to(dev),
                              c.seqlens.to(dev), o, lse, c.max_seqlen, c.scale, ws)

    outs = []
    for c in cases + cases[:1]:
        o = torch.full((6, 32, 128), float("nan"), dtype=torch.bfloat16, device=dev)
        lse = torch.full((6, 32), float("nan"), dtype=torch.float32, device=dev)
        call(c, o, lse)
        torch.cuda.synchronize()
        assert abi.attn_get_device_status() == 0
        outs.append((o.float().cpu().numpy(), lse.cpu().numpy()))
    for c, (o, lse) in zip(cases, outs):
        o_ref, lse_ref, _ = oracle.decode_paged(c.q, c.kcache, c.vcache, c.block_table, c.seqlens, c.scale)
        compare(o, lse, o_ref, lse_ref, True)
    assert np.array_equal(outs[0][0], outs[2][0]) and np.array_equal(outs[0][1], outs[2][1])

    c = cases[1]
    q, kc, vc = c.q.to(dev), c.kcache.to(dev), c.vcache.to(dev)
    bt, sl = c.block_table.to(dev), c.seqlens.to(dev)
    o = torch.full((6, 32, 128), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((6, 32), float("nan"), dtype=torch.float32, device=dev)
    abi.attn_decode_paged(q, kc, vc, bt, sl, o, lse, c.max_seqlen, c.scale, ws)  # warm-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            abi.attn_decode_paged(q, kc, vc, bt, sl, o, lse, c.max_seqlen, c.scale, ws)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert abi.attn_get_device_status() == 0
        assert np.array_equal(o.float().cpu().numpy(), outs[1][0])
        assert np.array_equal(lse.cpu().numpy(), outs[1][1])


def test_prefill_graph_replay(abi):
    # A captured prefill keeps its work-counter slot; consecutive replays
    # must each compute every unit (the slot is freed by each replay's last
    # fetch).
    dev = torch.device("cuda")
    x = inputs.prefill_inputs(1, 8, 8, 1000, 1000, 128, seed=43, causal=True)
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    abi.attn_fwd(q, k, v, o, lse, True, x.scale)
    torch.cuda.synchronize()
    ref_o, ref_l = o.float().cpu().numpy(), lse.cpu().numpy()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            abi.attn_fwd(q, k, v, o, lse, True, x.scale)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert abi.attn_get_device_status() == 0
        assert np.array_equal(o.float().cpu().numpy(), ref_o)
        assert np.array_equal(lse.cpu().numpy(), ref_l)


def test_decode_config(abi):
    c = configs.DECODE
    d_in = inputs.decode_inputs(c.num_seqs, c.Hq, c.Hkv, c.d, c.len_lo, c.len_hi, c.num_pages,
                                c.page_size, c.seed)
    check_decode(abi, d_in)


def test_decode_bad_block_table_is_reported_not_read(abi):
    d_in = inputs.decode_inputs(2, 8, 2, 128, 0, 40, num_pages=8, page_size=16, seed=9,
                                lengths=[40, 20], max_pages_per_seq=4)
    d_in.block_table[1, 0] = 1 << 20  # outside the pool: TMA fills zeros, status flags it
    dev = torch.device("cuda")
    o = torch.empty((2, 8, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((2, 8), dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, abi.attn_decode_workspace_size(2, 8, 2, 128, 40)), dtype=torch.uint8,
                     device=dev)
    abi.attn_decode_paged(d_in.q.to(dev), d_in.kcache.to(dev), d_in.vcache.to(dev),
                          d_in.block_table.to(dev), d_in.seqlens.to(dev), o, lse, 40, d_in.scale, ws)
    assert abi.attn_get_device_status() == 7
    assert abi.attn_get_device_status() == 0  # reading clears it


def test_prefill_uneven_scheduling_groups(abi):
    # 67 heads of 16 two-tile units: no divisor of 67 near the two-wave group
    # size, so the heads are scheduled in groups of 23, 23 and 21; every unit
    # of the short last group must still be computed once.
    x = inputs.prefill_inputs(1, 67, 67, 4096, 4096, 64, seed=9, causal=True)
    rows = inputs.check_rows(x.generator, 1, 67, 4096, 24)
    check_prefill(abi, x, rows)
