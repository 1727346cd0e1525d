"""Pins for the CPU oracle: it is checked against things other than itself.

Every check here runs on the CPU.  The oracle is pinned to
  * an independent brute force in 50-digit decimal arithmetic of the
    definition "softmax(QK^T/sqrt(d) + C) V" ("Compilers and Kernels",
    section "FlashAttention changes the algorithm around IO"), written without
    the max shift, so a wrong shift, scale, mask, head map or normaliser shows;
  * closed forms (Q = 0, causal row 0, uniform V, a dominant one-hot score);
  * invariants (permutation of keys, convex hull of V, GQA = repeated MHA,
    paged = contiguous);
  * the textbook routine torch.nn.functional.scaled_dot_product_attention in
    float64, with torch.logsumexp for the row LSE;
  * planted mistakes: each mutant build of the oracle must fail a pin.
"""
from __future__ import annotations

import math
import random
from decimal import Decimal, localcontext

import numpy as np
import pytest
import torch

import oracle
import oracle_mutants
from attention_online_softmax_gb300 import inputs

oracle_mutants.register_all()


def bf16_np(t: torch.Tensor) -> np.ndarray:
    return t.float().double().numpy()


# ---------------------------------------------------------------- brute force
def decimal_attention(q, k, v, causal, scale):
    """Plain definition in 50-digit decimals, no max shift.

    q: [B,Hq,Nq,d], k/v: [B,Hkv,Nk,d] (float64 arrays holding bf16 values,
    converted to Decimal exactly).  Key j is allowed for query i iff not causal
    or j - i <= Nk - Nq.  Returns O [B,Hq,Nq,d] and LSE [B,Hq,Nq] as floats.
    """
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    rep = Hq // Hkv
    O = np.zeros((B, Hq, Nq, d))
    L = np.zeros((B, Hq, Nq))
    with localcontext() as ctx:
        ctx.prec = 50
        sc = Decimal(float(scale))
        for b in range(B):
            for h in range(Hq):
                g = h // rep
                K = [[Decimal(float(x)) for x in row] for row in k[b, g]]
                V = [[Decimal(float(x)) for x in row] for row in v[b, g]]
                for i in range(Nq):
                    qi = [Decimal(float(x)) for x in q[b, h, i]]
                    allowed = [j for j in range(Nk) if (not causal) or (j - i <= Nk - Nq)]
                    if not allowed:
                        L[b, h, i] = -math.inf
                        continue
                    e = {}
                    for j in allowed:
                        s = sum(qi[c] * K[j][c] for c in range(d)) * sc
                        e[j] = s.exp()
                    z = sum(e.values())
                    for c in range(d):
                        O[b, h, i, c] = float(sum(e[j] * V[j][c] for j in allowed) / z)
                    L[b, h, i] = float(z.ln())
    return O, L


BRUTE_CASES = [
    # B, Hq, Hkv, Nq, Nk, d, causal
    (1, 2, 2, 16, 16, 8, False),
    (1, 2, 2, 12, 12, 8, True),
    (1, 1, 1, 5, 9, 4, True),     # Nq < Nk: bottom-right causal
    (1, 1, 1, 9, 5, 4, True),     # Nq > Nk: first rows have no allowed key
    (2, 4, 2, 7, 11, 6, False),   # GQA, ragged sizes
    (1, 4, 1, 6, 6, 8, True),     # MQA
]


def close(a, b, tol):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    both_inf = np.isneginf(a) & np.isneginf(b)
    with np.errstate(invalid="ignore"):
        diff = np.where(both_inf, 0.0, np.abs(a - b))
    return bool(np.all(np.isfinite(diff)) and diff.max(initial=0.0) <= tol)


@pytest.mark.parametrize("case", BRUTE_CASES)
def test_oracle_matches_decimal_brute_force(case):
    B, Hq, Hkv, Nq, Nk, d, causal = case
    x = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=100 + sum(case[:-1]), causal=causal)
    O, L, _ = oracle.attention(x.q, x.k, x.v, causal, x.scale)
    Ob, Lb = decimal_attention(bf16_np(x.q), bf16_np(x.k), bf16_np(x.v), causal, x.scale)
    assert close(O, Ob, 1e-12)
    assert close(L, Lb, 1e-12)


# ----------------------------------------------------------- closed forms
def test_zero_query_gives_mean_of_allowed_values():
    B, H, N, d = 1, 2, 37, 16
    x = inputs.prefill_inputs(B, H, H, N, N, d, seed=7, causal=True)
    q0 = torch.zeros_like(x.q)
    O, L, _ = oracle.attention(q0, x.k, x.v, True, x.scale)
    V = bf16_np(x.v)
    for h in range(H):
        for i in range(N):
            np.testing.assert_allclose(O[0, h, i], V[0, h, : i + 1].mean(axis=0), atol=1e-13)
            assert abs(L[0, h, i] - math.log(i + 1)) < 1e-13
    O, L, _ = oracle.attention(q0, x.k, x.v, False, x.scale)
    np.testing.assert_allclose(O[0, 1, 5], V[0, 1].mean(axis=0), atol=1e-13)
    assert abs(L[0, 0, 3] - math.log(N)) < 1e-13


def test_causal_row_zero_returns_first_value_row():
    x = inputs.prefill_inputs(2, 3, 3, 20, 20, 32, seed=8, causal=True)
    O, L, _ = oracle.attention(x.q, x.k, x.v, True, x.scale)
    Q, K, V = bf16_np(x.q), bf16_np(x.k), bf16_np(x.v)
    for b in range(2):
        for h in range(3):
            np.testing.assert_array_equal(O[b, h, 0], V[b, h, 0])
            assert abs(L[b, h, 0] - x.scale * float(Q[b, h, 0] @ K[b, h, 0])) < 1e-12


def test_uniform_values_return_the_constant():
    x = inputs.prefill_inputs(1, 2, 2, 24, 40, 16, seed=9, causal=False)
    v = torch.full_like(x.v, 1.75)
    O, _, _ = oracle.attention(x.q, x.k, v, False, x.scale)
    np.testing.assert_allclose(O, 1.75, atol=1e-14)


def test_one_hot_dominant_score_selects_its_value_row():
    # q = c e_1, K[j*] = c e_1, every other key orthogonal to e_1: the score
    # gap is Delta = scale c^2 and O -> V[j*] within (n-1) e^-Delta 2 max|V|.
    n, d, c, jstar = 33, 16, 8.0, 11
    x = inputs.prefill_inputs(1, 1, 1, 1, n, d, seed=10, causal=False)
    q = torch.zeros(1, 1, 1, d)
    q[..., 0] = c
    k = x.k.float().clone()
    k[..., 0] = 0.0
    k[0, 0, jstar] = 0.0
    k[0, 0, jstar, 0] = c
    q, k = q.to(torch.bfloat16), k.to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    O, L, _ = oracle.attention(q, k, x.v, False, scale)
    V = bf16_np(x.v)
    delta = scale * c * c
    bound = (n - 1) * math.exp(-delta) * 2 * np.abs(V).max()
    assert np.abs(O[0, 0, 0] - V[0, 0, jstar]).max() <= bound
    assert abs(L[0, 0, 0] - delta) <= 2 * (n - 1) * math.exp(-delta)


# --------------------------------------------------------------- invariants
def test_key_permutation_invariance_and_convex_hull():
    x = inputs.prefill_inputs(1, 2, 2, 10, 50, 8, seed=11, causal=False)
    perm = torch.randperm(50, generator=torch.Generator().manual_seed(0))
    O1, L1, _ = oracle.attention(x.q, x.k, x.v, False, x.scale)
    O2, L2, _ = oracle.attention(x.q, x.k[:, :, perm], x.v[:, :, perm], False, x.scale)
    np.testing.assert_allclose(O1, O2, atol=1e-13)
    np.testing.assert_allclose(L1, L2, atol=1e-13)
    V = bf16_np(x.v)
    lo = V.min(axis=2)[:, :, None, :]
    hi = V.max(axis=2)[:, :, None, :]
    assert np.all(O1 >= lo - 1e-13) and np.all(O1 <= hi + 1e-13)


def test_gqa_equals_mha_with_repeated_kv_heads():
    x = inputs.prefill_inputs(2, 8, 2, 13, 21, 16, seed=12, causal=True)
    O1, L1, _ = oracle.attention(x.q, x.k, x.v, True, x.scale)
    k = x.k.repeat_interleave(4, dim=1)
    v = x.v.repeat_interleave(4, dim=1)
    O2, L2, _ = oracle.attention(x.q, k, v, True, x.scale)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)


def test_row_subset_matches_full_evaluation():
    x = inputs.prefill_inputs(2, 4, 2, 33, 33, 16, seed=13, causal=True)
    O, L, _ = oracle.attention(x.q, x.k, x.v, True, x.scale)
    rows = inputs.check_rows(x.generator, 2, 4, 33, 5)
    Os, Ls, _ = oracle.attention(x.q, x.k, x.v, True, x.scale, rows=rows)
    np.testing.assert_array_equal(Os, O.reshape(-1, 16)[rows.numpy()])
    np.testing.assert_array_equal(Ls, L.reshape(-1)[rows.numpy()])


def test_fully_masked_rows_are_zero_with_minus_inf_lse():
    x = inputs.prefill_inputs(1, 1, 1, 9, 4, 8, seed=14, causal=True)
    O, L, _ = oracle.attention(x.q, x.k, x.v, True, x.scale)
    # Nk - Nq = -5: rows 0..4 have no allowed key.
    assert np.all(O[0, 0, :5] == 0.0) and np.all(np.isneginf(L[0, 0, :5]))
    assert np.all(np.isfinite(L[0, 0, 5:]))


def test_textbook_sdpa_float64_cross_check():
    for causal, (Nq, Nk) in [(False, (19, 23)), (True, (17, 17)), (True, (6, 14))]:
        x = inputs.prefill_inputs(2, 4, 2, Nq, Nk, 16, seed=15 + Nq, causal=causal)
        O, L, _ = oracle.attention(x.q, x.k, x.v, causal, x.scale)
        q = x.q.double()
        k = x.k.double().repeat_interleave(2, dim=1)
        v = x.v.double().repeat_interleave(2, dim=1)
        mask = None
        if causal:
            i = torch.arange(Nq)[:, None]
            j = torch.arange(Nk)[None, :]
            mask = (j - i) <= (Nk - Nq)
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask,
                                                               scale=x.scale)
        s = (q @ k.transpose(-1, -2)) * x.scale
        if mask is not None:
            s = s.masked_fill(~mask, -math.inf)
        lse = torch.logsumexp(s, dim=-1)
        np.testing.assert_allclose(O, ref.numpy(), atol=1e-12)
        np.testing.assert_allclose(L, lse.numpy(), atol=1e-12)


# ------------------------------------------------------------------ decode
def test_paged_decode_equals_contiguous_attention():
    d = inputs.decode_inputs(5, 8, 2, 16, 1, 70, num_pages=40, page_size=16, seed=16,
                             max_pages_per_seq=5)
    O, L, _ = oracle.decode_paged(d.q, d.kcache, d.vcache, d.block_table, d.seqlens, d.scale)
    for s in range(5):
        n = int(d.seqlens[s])
        pages = d.block_table[s, : (n + 15) // 16].long()
        k = d.kcache[pages].reshape(-1, 2, 16)[:n].permute(1, 0, 2).unsqueeze(0)
        v = d.vcache[pages].reshape(-1, 2, 16)[:n].permute(1, 0, 2).unsqueeze(0)
        q = d.q[s].reshape(1, 8, 1, 16)
        Oc, Lc, _ = oracle.attention(q, k.contiguous(), v.contiguous(), False, d.scale)
        np.testing.assert_array_equal(O[s], Oc[0, :, 0])
        np.testing.assert_array_equal(L[s], Lc[0, :, 0])
        assert np.all(np.isfinite(O[s]))  # no NaN slot was read


def test_paged_decode_zero_length_sequence():
    d = inputs.decode_inputs(3, 4, 4, 8, 0, 0, num_pages=4, page_size=16, seed=17,
                             max_pages_per_seq=2, lengths=[0, 17, 1])
    O, L, _ = oracle.decode_paged(d.q, d.kcache, d.vcache, d.block_table, d.seqlens, d.scale)
    assert np.all(O[0] == 0) and np.all(np.isneginf(L[0]))
    V = bf16_np(d.vcache)
    page = int(d.block_table[2, 0])
    np.testing.assert_array_equal(O[2], V[page, 0])


def test_planted_decode_layout_mistake_is_caught():
    # A page read with its slot and head axes swapped (mutant 11) must fail the
    # gathered-rows pin (or read a NaN slot).
    d = inputs.decode_inputs(5, 8, 2, 16, 1, 70, num_pages=40, page_size=16, seed=16,
                             max_pages_per_seq=5)
    O, L, _ = oracle.decode_paged(d.q, d.kcache, d.vcache, d.block_table, d.seqlens, d.scale, mutant=11)
    agree = True
    for s in range(5):
        n = int(d.seqlens[s])
        pages = d.block_table[s, : (n + 15) // 16].long()
        k = d.kcache[pages].reshape(-1, 2, 16)[:n].permute(1, 0, 2).unsqueeze(0)
        v = d.vcache[pages].reshape(-1, 2, 16)[:n].permute(1, 0, 2).unsqueeze(0)
        q = d.q[s].reshape(1, 8, 1, 16)
        Oc, Lc, _ = oracle.attention(q, k.contiguous(), v.contiguous(), False, d.scale)
        agree = agree and np.allclose(O[s], Oc[0, :, 0], atol=1e-9) and np.allclose(L[s], Lc[0, :, 0], atol=1e-9)
    assert not agree


# ------------------------------------------------------------------ mutants
def _mutant_fails(mutant: int) -> bool:
    for case in BRUTE_CASES:
        B, Hq, Hkv, Nq, Nk, d, causal = case
        x = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, d, seed=200 + sum(case[:-1]), causal=causal)
        O, L, _ = oracle.attention(x.q, x.k, x.v, causal, x.scale, mutant=mutant)
        Ob, Lb = decimal_attention(bf16_np(x.q), bf16_np(x.k), bf16_np(x.v), causal, x.scale)
        if not (close(O, Ob, 1e-6) and close(L, Lb, 1e-6)):
            return True
    return False


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5])
def test_planted_oracle_mistakes_are_caught(mutant):
    assert _mutant_fails(mutant)


def test_thread_count_does_not_change_results():
    x = inputs.prefill_inputs(1, 4, 4, 64, 64, 32, seed=18, causal=True)
    O1, L1, t1 = oracle.attention(x.q, x.k, x.v, True, x.scale, threads=1)
    O2, L2, t2 = oracle.attention(x.q, x.k, x.v, True, x.scale, threads=0)
    assert t1 == 1 and t2 >= 1
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)
