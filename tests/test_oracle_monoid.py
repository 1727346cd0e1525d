"""Pins for the online-softmax recurrence and the merge of partial states.

"Compilers and Kernels", section "FlashAttention changes the algorithm around
IO": the block recurrence keeps the numerator and denominator of the full
softmax in exact arithmetic, so over ANY partition of the allowed keys it must
reproduce the two-pass oracle to rounding (1e-12 in float64).  The merge of
partial states (the reading of "online softmax as a monoid" in the Tang
abstract) must be associative and commutative with identity (-inf, 0, 0); a
block with no allowed key is that identity.
"""
from __future__ import annotations

import math
import random

import numpy as np
import pytest
import torch

import oracle
from oracle import monoid
from attention_online_softmax_gb300 import inputs


def scores_and_values(seed, n=97, d=16, causal_row=None, k_scale=1.0):
    x = inputs.prefill_inputs(1, 1, 1, 1 if causal_row is None else n, n, d, seed=seed,
                              causal=causal_row is not None, k_scale=k_scale)
    q = x.q.double()[0, 0]
    k = x.k.double()[0, 0]
    v = x.v.double()[0, 0].numpy()
    row = 0 if causal_row is None else causal_row
    s = (k @ q[row]).numpy() * x.scale
    if causal_row is not None:
        s[np.arange(n) > causal_row] = -math.inf
    return x, s, v, row


def random_partition(n, rng):
    cuts = sorted(rng.sample(range(1, n), rng.randint(0, min(12, n - 1))))
    bounds = [0] + cuts + [n]
    return [np.arange(a, b) for a, b in zip(bounds[:-1], bounds[1:])]


@pytest.mark.parametrize("seed", range(6))
def test_recurrence_over_random_partitions_equals_definition(seed):
    rng = random.Random(seed)
    k_scale = 4.0 if seed % 2 else 1.0
    causal_row = None if seed < 3 else 50
    x, s, v, row = scores_and_values(300 + seed, causal_row=causal_row, k_scale=k_scale)
    causal = causal_row is not None
    rows = None if not causal else [row]
    O, L, _ = oracle.attention(x.q, x.k, x.v, causal, x.scale, rows=rows)
    O = O.reshape(-1, O.shape[-1])[0]
    L = float(np.asarray(L).reshape(-1)[0])
    for _ in range(20):
        part = random_partition(len(s), rng)
        st = monoid.recurrence(s, v, part)
        Oo, Lo = monoid.finalize(st)
        assert np.abs(Oo - O).max() <= 1e-12
        assert abs(Lo - L) <= 1e-12


def tree_merge(states, rng):
    states = list(states)
    while len(states) > 1:
        i = rng.randrange(len(states) - 1)
        states[i:i + 2] = [monoid.merge(states[i], states[i + 1])]
    return states[0]


@pytest.mark.parametrize("seed", range(6))
def test_merge_is_associative_and_commutative(seed):
    rng = random.Random(1000 + seed)
    _, s, v, _ = scores_and_values(400 + seed, k_scale=4.0 if seed % 2 else 1.0)
    ref = monoid.finalize(monoid.block_state(s, v))
    for _ in range(20):
        part = random_partition(len(s), rng)
        blocks = [monoid.block_state(s[idx], v[idx]) for idx in part]
        t1 = monoid.finalize(tree_merge(blocks, rng))           # random bracketing
        rng.shuffle(blocks)
        t2 = monoid.finalize(tree_merge(blocks, rng))           # random order too
        for O, L in (t1, t2):
            assert np.abs(O - ref[0]).max() <= 1e-12
            assert abs(L - ref[1]) <= 1e-12


def test_identity_and_masked_blocks():
    _, s, v, _ = scores_and_values(500)
    a = monoid.block_state(s[:40], v[:40])
    e = monoid.identity(v.shape[1])
    for m in (monoid.merge(a, e), monoid.merge(e, a)):
        assert m.m == a.m and m.l == a.l and np.array_equal(m.o, a.o)
    masked = monoid.block_state(np.full(7, -math.inf), v[:7])
    assert masked.m == -math.inf and masked.l == 0.0 and not masked.o.any()
    ee = monoid.merge(e, e)
    assert monoid.finalize(ee)[1] == -math.inf


def test_stored_output_form_merges_like_states():
    # Partials stored as (O_s, lse_s) merge to the same result: LSE =
    # logsumexp_s(lse_s), O = sum_s exp(lse_s - LSE) O_s.
    rng = random.Random(7)
    _, s, v, _ = scores_and_values(600, k_scale=4.0)
    ref = monoid.finalize(monoid.block_state(s, v))
    part = random_partition(len(s), rng)
    stored = [monoid.finalize(monoid.block_state(s[i], v[i])) for i in part]
    states = [monoid.from_output(o, l) for o, l in stored]
    O, L = monoid.finalize(tree_merge(states, rng))
    lses = np.array([l for _, l in stored])
    Lx = lses.max() + math.log(np.exp(lses - lses.max()).sum())
    Ox = sum(math.exp(l - Lx) * o for o, l in stored)
    for a, b in ((O, ref[0]), (Ox, ref[0])):
        assert np.abs(a - b).max() <= 1e-12
    assert abs(L - ref[1]) <= 1e-12 and abs(Lx - ref[1]) <= 1e-12


def test_split_decode_partials_reproduce_decode_oracle():
    # Decode splits a sequence's keys into chunks and merges the chunk states;
    # the merged result must equal the decode oracle for every head.
    d = inputs.decode_inputs(3, 8, 2, 16, 1, 300, num_pages=64, page_size=16, seed=19,
                             max_pages_per_seq=19)
    O, L, _ = oracle.decode_paged(d.q, d.kcache, d.vcache, d.block_table, d.seqlens, d.scale)
    rng = random.Random(3)
    for s in range(3):
        n = int(d.seqlens[s])
        pages = d.block_table[s, : (n + 15) // 16].long()
        K = d.kcache[pages].double().reshape(-1, 2, 16)[:n]
        V = d.vcache[pages].double().reshape(-1, 2, 16)[:n]
        for h in range(8):
            g = h // 4
            sc = (K[:, g] @ d.q[s, h].double()).numpy() * d.scale
            chunk = rng.choice([16, 32, 64, 256])
            parts = [np.arange(a, min(n, a + chunk)) for a in range(0, n, chunk)]
            st = tree_merge([monoid.block_state(sc[i], V[i, g].numpy()) for i in parts], rng)
            Om, Lm = monoid.finalize(st)
            assert np.abs(Om - O[s, h]).max() <= 1e-12
            assert abs(Lm - L[s, h]) <= 1e-12


def test_planted_missing_rescale_is_caught(monkeypatch):
    # Drop the correction alpha_t = exp(m_{t-1} - m_t) (every nonempty part
    # weighted 1): the recurrence over a partition with a rising max must
    # then miss the definition, which is what the partition pin checks.
    x, s, v, row = scores_and_values(305, k_scale=4.0)
    O, L, _ = oracle.attention(x.q, x.k, x.v, False, x.scale)
    O = O.reshape(-1, O.shape[-1])[0]
    L = float(np.asarray(L).reshape(-1)[0])
    order = np.argsort(s)  # ascending scores: the running max rises at every block
    part = [order[i:i + 8] for i in range(0, len(s), 8)]
    Oo, Lo = monoid.finalize(monoid.recurrence(s, v, part))
    assert np.abs(Oo - O).max() <= 1e-12 and abs(Lo - L) <= 1e-12  # the unplanted recurrence agrees
    monkeypatch.setattr(monoid, "_weight", lambda m_part, m: 0.0 if m_part == -math.inf else 1.0)
    Oo, Lo = monoid.finalize(monoid.recurrence(s, v, part))
    assert np.abs(Oo - O).max() > 1e-6 or abs(Lo - L) > 1e-6
