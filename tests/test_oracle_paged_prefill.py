"""Pins for the oracle's chunked prefill against a paged KV cache.

"Don't Write Kernels, Derive Them", section "What happened" (paged KV-cache
access among the operations the method covers) and "Compilers and Kernels",
section "FlashAttention changes the algorithm around IO" (the attention each
query row computes).  The paged oracle is pinned to a 50-digit decimal brute
force over K/V rows the test gathers itself, to the plain oracle on the same
gathered rows, to paged decode (one new token per sequence), and to the
invariance of the result under a relabelling of the page pool.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import oracle_mutants
from attention_online_softmax_gb300 import inputs
from test_oracle_bias import decimal_with_bias
from test_oracle_pins import bf16_np, close

oracle_mutants.register_all()


def gather(x, s):
    """K and V rows [k_len, Hkv, d] of sequence s, read through the block table."""
    L = int(x.seqlens_k[s])
    ps = x.page_size
    ks, vs = [], []
    for t in range(L):
        page = int(x.block_table[s, t // ps])
        ks.append(x.kcache[page, t % ps])
        vs.append(x.vcache[page, t % ps])
    if not ks:
        shape = (0,) + tuple(x.kcache.shape[2:])
        return torch.empty(shape, dtype=torch.bfloat16), torch.empty(shape, dtype=torch.bfloat16)
    return torch.stack(ks), torch.stack(vs)


def seq_slice(x, s):
    a, b = int(x.cu_seqlens_q[s]), int(x.cu_seqlens_q[s + 1])
    return a, b


CASES = [
    # q_lens, k_lens, Hq, Hkv, d, page_size, causal, window
    ([3, 1, 4], [7, 5, 4], 2, 1, 4, 4, True, 0),
    ([2, 3], [9, 3], 2, 2, 4, 2, True, 3),
    ([4, 2], [6, 11], 2, 1, 4, 4, False, 0),
    ([5, 0, 2], [3, 4, 0], 1, 1, 4, 2, True, 0),   # rows without keys, empty chunk, empty context
]


@pytest.mark.parametrize("case", CASES)
def test_paged_prefill_matches_decimal_brute_force(case):
    q_lens, k_lens, Hq, Hkv, d, ps, causal, window = case
    x = inputs.paged_prefill_inputs(q_lens, k_lens, Hq, Hkv, d, num_pages=sum(k_lens) // ps + 6,
                                    page_size=ps, seed=900 + sum(q_lens))
    O, L, _ = oracle.prefill_paged(x.q, x.kcache, x.vcache, x.block_table, x.cu_seqlens_q, x.seqlens_k,
                                   causal, x.scale, window_left=window)
    for s in range(len(q_lens)):
        a, b = seq_slice(x, s)
        nq, nk = b - a, k_lens[s]
        if nq == 0:
            continue
        k, v = gather(x, s)
        qs = bf16_np(x.q[a:b].permute(1, 0, 2).unsqueeze(0))            # [1, Hq, nq, d]
        ks = bf16_np(k.permute(1, 0, 2).unsqueeze(0))                   # [1, Hkv, nk, d]
        vs = bf16_np(v.permute(1, 0, 2).unsqueeze(0))
        C = np.zeros((1, Hq, nq, nk))
        i = np.arange(nq)[:, None]
        j = np.arange(nk)[None, :]
        allowed = np.ones((nq, nk), dtype=bool)
        if causal:
            allowed &= j <= i + nk - nq
        if window > 0:
            allowed &= j > i + nk - nq - window
        C[:, :, ~allowed] = -math.inf
        Ob, Lb = decimal_with_bias(qs, ks, vs, x.scale, C)
        assert close(O[a:b].transpose(1, 0, 2), Ob[0], 1e-12)
        assert close(L[a:b].T, Lb[0], 1e-12)


def test_paged_prefill_is_the_plain_oracle_on_gathered_rows():
    q_lens, k_lens = [37, 1, 64, 20], [100, 33, 64, 150]
    x = inputs.paged_prefill_inputs(q_lens, k_lens, 4, 2, 16, num_pages=50, page_size=8, seed=901)
    O, L, _ = oracle.prefill_paged(x.q, x.kcache, x.vcache, x.block_table, x.cu_seqlens_q, x.seqlens_k,
                                   True, x.scale)
    for s in range(len(q_lens)):
        a, b = seq_slice(x, s)
        k, v = gather(x, s)
        Op, Lp, _ = oracle.attention(x.q[a:b].permute(1, 0, 2).unsqueeze(0).contiguous(),
                                     k.permute(1, 0, 2).unsqueeze(0).contiguous(),
                                     v.permute(1, 0, 2).unsqueeze(0).contiguous(), True, x.scale)
        np.testing.assert_allclose(O[a:b], Op[0].transpose(1, 0, 2), atol=1e-13)
        np.testing.assert_allclose(L[a:b], Lp[0].T, atol=1e-13)


def test_one_new_token_is_paged_decode():
    # A chunk of one token per sequence attends its whole context: paged decode.
    k_lens = [1, 17, 64, 200, 5]
    x = inputs.paged_prefill_inputs([1] * 5, k_lens, 8, 2, 32, num_pages=60, page_size=16, seed=902)
    O, L, _ = oracle.prefill_paged(x.q, x.kcache, x.vcache, x.block_table, x.cu_seqlens_q, x.seqlens_k,
                                   True, x.scale)
    Od, Ld, _ = oracle.decode_paged(x.q, x.kcache, x.vcache, x.block_table, x.seqlens_k, x.scale)
    np.testing.assert_allclose(O, Od, atol=1e-13)
    np.testing.assert_allclose(L, Ld, atol=1e-13)


def test_relabelling_the_page_pool_changes_nothing():
    q_lens, k_lens = [9, 30], [40, 30]
    x = inputs.paged_prefill_inputs(q_lens, k_lens, 2, 1, 8, num_pages=20, page_size=4, seed=903)
    O1, L1, _ = oracle.prefill_paged(x.q, x.kcache, x.vcache, x.block_table, x.cu_seqlens_q, x.seqlens_k,
                                     True, x.scale)
    g = torch.Generator().manual_seed(7)
    perm = torch.randperm(20, generator=g)           # new page p holds old page perm[p]
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(20)
    bt2 = inv[x.block_table.long()].to(torch.int32)
    O2, L2, _ = oracle.prefill_paged(x.q, x.kcache[perm], x.vcache[perm], bt2, x.cu_seqlens_q,
                                     x.seqlens_k, True, x.scale)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)


def test_rows_subset_matches_full():
    x = inputs.paged_prefill_inputs([50, 70], [120, 70], 4, 4, 16, num_pages=30, page_size=8, seed=904)
    O, L, _ = oracle.prefill_paged(x.q, x.kcache, x.vcache, x.block_table, x.cu_seqlens_q, x.seqlens_k,
                                   True, x.scale, window_left=33)
    rows = np.array([0, 3, 199, 200, 479])
    Or, Lr, _ = oracle.prefill_paged(x.q, x.kcache, x.vcache, x.block_table, x.cu_seqlens_q, x.seqlens_k,
                                     True, x.scale, window_left=33, rows=rows)
    np.testing.assert_array_equal(Or, O.reshape(-1, 16)[rows])
    np.testing.assert_array_equal(Lr, L.reshape(-1)[rows])


def test_bad_block_table_entry_is_rejected():
    x = inputs.paged_prefill_inputs([2], [10], 1, 1, 4, num_pages=4, page_size=4, seed=905)
    x.block_table[0, 1] = 99
    with pytest.raises(ValueError):
        oracle.prefill_paged(x.q, x.kcache, x.vcache, x.block_table, x.cu_seqlens_q, x.seqlens_k,
                             True, x.scale)


@pytest.mark.parametrize("mutant", [8, 10])
def test_planted_paged_mistakes_are_caught(mutant):
    # A causal bound off by one (8) or a wrong kv head (10) must fail the pin
    # against the plain oracle on gathered rows.
    q_lens, k_lens = [37, 20], [100, 150]
    x = inputs.paged_prefill_inputs(q_lens, k_lens, 4, 2, 16, num_pages=40, page_size=8, seed=906)
    O, L, _ = oracle.prefill_paged(x.q, x.kcache, x.vcache, x.block_table, x.cu_seqlens_q, x.seqlens_k,
                                   True, x.scale, mutant=mutant)
    agree = True
    for s in range(len(q_lens)):
        a, b = seq_slice(x, s)
        k, v = gather(x, s)
        Op, Lp, _ = oracle.attention(x.q[a:b].permute(1, 0, 2).unsqueeze(0).contiguous(),
                                     k.permute(1, 0, 2).unsqueeze(0).contiguous(),
                                     v.permute(1, 0, 2).unsqueeze(0).contiguous(), True, x.scale)
        agree = agree and np.allclose(O[a:b], Op[0].transpose(1, 0, 2), atol=1e-9)
    assert not agree
