"""GPU parity of chunked prefill against a paged KV cache (ragged sequences).

``attn_prefill_paged`` through the C ABI against the oracle's
``prefill_paged`` on the same seeded inputs, with the tolerances of the plain
parity tests (max|dO| <= 1e-2, max|dLSE| <= 1e-3, exact -inf LSE pattern).
Every cache slot past a context and every unused page holds bf16 NaN, so a
value row read past a context's end, or a stray page, shows up as NaN.
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


def run_paged(abi, x, causal, window, o_dtype):
    dev = torch.device("cuda")
    q = x.q.to(dev)
    total_q, Hq, d = q.shape
    o = torch.full((total_q, Hq, d), float("nan"), dtype=o_dtype, device=dev)
    lse = torch.full((total_q, Hq), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.full((max(16, abi.attn_prefill_paged_workspace_size(x.seqlens_k.numel())),), 0xFF,
                    dtype=torch.uint8, device=dev)
    abi.attn_prefill_paged(q, x.kcache.to(dev), x.vcache.to(dev), x.block_table.to(dev),
                           x.cu_seqlens_q.to(dev), x.seqlens_k.to(dev), o, lse, causal, x.scale,
                           window_left=window, workspace=ws)
    torch.cuda.synchronize()
    assert abi.attn_get_device_status() == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


def check_paged(abi, x, causal, window=0, rows=None):
    o_ref, lse_ref, _ = oracle.prefill_paged(x.q, x.kcache, x.vcache, x.block_table, x.cu_seqlens_q,
                                             x.seqlens_k, causal, x.scale, window_left=window, rows=rows)
    for dt in (torch.bfloat16, torch.float32):
        o, lse = run_paged(abi, x, causal, window, dt)
        if rows is not None:
            d = o.shape[-1]
            o = o.reshape(-1, d)[rows]
            lse = lse.reshape(-1)[rows]
        compare(o, lse, o_ref, lse_ref, dt == torch.bfloat16)
    return lse_ref


PAGED = [
    # q_lens, k_lens, Hq, Hkv, d, page_size, causal, window
    ([512], [512], 8, 2, 128, 16, True, 0),                          # a whole prompt through pages
    ([200, 1, 77, 300], [1000, 33, 77, 301], 8, 2, 128, 16, True, 0),  # ragged; contexts end mid-page
    ([129, 64], [500, 64], 4, 4, 64, 32, True, 0),
    ([100, 260], [300, 1030], 8, 1, 256, 16, True, 0),               # d = 256, MQA
    ([50, 300], [700, 300], 4, 2, 128, 64, False, 0),                # non-causal, 64-slot pages
    ([400], [2000], 4, 4, 128, 128, True, 300),                      # left window, 128-slot pages
    ([300], [200], 2, 2, 128, 16, True, 0),                          # k_len < q_len: rows without keys
    ([0, 130, 0, 7], [50, 130, 0, 9], 4, 2, 64, 16, True, 0),        # empty chunks and contexts
    ([5, 3], [0, 3], 2, 1, 128, 16, True, 0),                        # a chunk with no context at all
    # One page per key tile: with d = 64 it is one box, and the second
    # producer warp has none (it still arrives on every item's barrier);
    # with d = 256 each producer warp has one box of it.
    ([129, 64], [500, 70], 4, 4, 64, 128, True, 0),
    ([100, 260], [300, 1030], 8, 1, 256, 128, True, 0),
]


@pytest.mark.parametrize("case", PAGED)
def test_paged_prefill(abi, case):
    q_lens, k_lens, Hq, Hkv, d, ps, causal, window = case
    pages = sum((k + ps - 1) // ps for k in k_lens) + 9
    x = inputs.paged_prefill_inputs(q_lens, k_lens, Hq, Hkv, d, num_pages=pages, page_size=ps,
                                    seed=6000 + sum(q_lens) + d,
                                    max_pages_per_seq=max((k + ps - 1) // ps for k in k_lens) + 2)
    check_paged(abi, x, causal, window)


# Enough heads that the library pairs two query tiles per unit; ragged chunks
# leave a unit's second tile partly or wholly past its sequence.
TWO_TILE = [
    ([300, 1, 200, 77], [1000, 33, 300, 77], 160, 32, 64, 16, True, 0),
    ([260, 520], [900, 520], 128, 16, 128, 16, True, 0),
    ([384, 129], [384, 700], 128, 32, 128, 32, False, 0),
]


@pytest.mark.parametrize("case", TWO_TILE)
def test_paged_prefill_two_tile_units(abi, case):
    q_lens, k_lens, Hq, Hkv, d, ps, causal, window = case
    pages = sum((k + ps - 1) // ps for k in k_lens) + 9
    x = inputs.paged_prefill_inputs(q_lens, k_lens, Hq, Hkv, d, num_pages=pages, page_size=ps,
                                    seed=6500 + sum(q_lens) + d)
    g = torch.Generator().manual_seed(6501)
    total = x.q.shape[0] * Hq
    rows = np.concatenate([torch.randperm(total, generator=g)[:20000].numpy(), [0, total - 1]])
    check_paged(abi, x, causal, window, rows=rows)


def test_one_token_chunks_match_the_oracle_decode(abi):
    # One new token per sequence is paged decode; the prefill kernel handles it too.
    k_lens = [1, 17, 64, 200, 5, 4097]
    x = inputs.paged_prefill_inputs([1] * 6, k_lens, 8, 2, 128, num_pages=400, page_size=16, seed=6100)
    lse_ref = check_paged(abi, x, True)
    _, lse_dec, _ = oracle.decode_paged(x.q, x.kcache, x.vcache, x.block_table, x.seqlens_k, x.scale)
    np.testing.assert_allclose(lse_ref, lse_dec, atol=1e-12)


def test_bad_block_table_is_reported_not_read(abi):
    x = inputs.paged_prefill_inputs([40, 20], [40, 20], 4, 2, 128, num_pages=8, page_size=16, seed=6200,
                                    max_pages_per_seq=4)
    x.block_table[1, 0] = 1 << 20
    dev = torch.device("cuda")
    o = torch.empty((60, 4, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((60, 4), dtype=torch.float32, device=dev)
    abi.attn_prefill_paged(x.q.to(dev), x.kcache.to(dev), x.vcache.to(dev), x.block_table.to(dev),
                           x.cu_seqlens_q.to(dev), x.seqlens_k.to(dev), o, lse, True, x.scale)
    assert abi.attn_get_device_status() == 7
    assert abi.attn_get_device_status() == 0


def test_paged_prefill_is_deterministic(abi):
    x = inputs.paged_prefill_inputs([300, 200], [900, 250], 8, 2, 128, num_pages=100, page_size=16, seed=6300)
    o1, l1 = run_paged(abi, x, True, 0, torch.bfloat16)
    o2, l2 = run_paged(abi, x, True, 0, torch.bfloat16)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_chunked_prefill_config(abi):
    # The benchmark's chunked-prefill workload on a seeded row subset.
    c = configs.CHUNKED
    x = inputs.paged_prefill_inputs(*configs.chunked_lengths(c), c.Hq, c.Hkv, c.d, num_pages=c.num_pages,
                                    page_size=c.page_size, seed=c.seed)
    g = torch.Generator().manual_seed(c.seed + 1)
    total = x.q.shape[0] * c.Hq
    rows = torch.randperm(total, generator=g)[:4096].numpy()
    rows = np.concatenate([rows, [0, total - 1]])
    check_paged(abi, x, True, 0, rows=rows)


def test_more_sequences_than_the_plan_ranks(abi):
    # Past 1024 sequences the plan kernel keeps the given dispatch order
    # instead of ranking by context length; every row must still be right.
    n = 1100
    g = torch.Generator().manual_seed(6600)
    q_lens = torch.randint(0, 3, (n,), generator=g).tolist()
    k_lens = [q + int(e) for q, e in zip(q_lens, torch.randint(0, 40, (n,), generator=g).tolist())]
    pages = sum((k + 15) // 16 for k in k_lens) + 9
    x = inputs.paged_prefill_inputs(q_lens, k_lens, 4, 2, 64, num_pages=pages, page_size=16, seed=6601)
    check_paged(abi, x, True)


def test_equal_context_lengths_tie_in_index_order(abi):
    # Ranked dispatch with ties (equal contexts) and a spread of lengths.
    q_lens = [100, 37, 100, 1, 256, 100]
    k_lens = [600, 600, 100, 600, 900, 600]
    pages = sum((k + 15) // 16 for k in k_lens) + 9
    x = inputs.paged_prefill_inputs(q_lens, k_lens, 8, 2, 128, num_pages=pages, page_size=16, seed=6602)
    check_paged(abi, x, True)
