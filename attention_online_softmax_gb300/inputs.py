"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds none of the attention arithmetic: it only draws random
numbers and lays them out.  Both the tests (which feed the oracle and the
kernels) and the benchmark import it; it imports neither side.

Recipe (the pages name no generator; this is the reading used throughout):

* ``g = torch.Generator('cpu').manual_seed(seed)``; every draw comes from it
  in the order documented below, as float32 ``torch.randn`` rounded to
  bfloat16 (round-to-nearest-even by ``Tensor.to``).
* Prefill draws Q [B,Hq,Nq,d], then K [B,Hkv,Nk,d], then V [B,Hkv,Nk,d].
  ``k_scale`` multiplies the bf16 K afterwards (4 is exact: a power of two).
* Paged decode draws the lengths ``randint(lo, hi + 1, (S,))``, one pool
  permutation ``randperm(num_pages)``, q [S,Hq,d], then for each sequence in
  order its K and V rows [L_s, Hkv, d].  Sequence s owns the next
  ceil(L_s / page_size) pages of the permutation (no page is shared).  Every
  slot the cache does not use -- tail slots of a sequence's last page and whole
  unused pages -- holds bf16 NaN, so a stray read shows up in parity.  Unused
  block-table entries point at a NaN page when one exists.
* Row subsets for large configurations continue on the same generator after
  the data: per (b, h), ``randperm(Nq)[:per_head]`` plus rows 0 and Nq-1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

BF16_NAN = float("nan")


def _randn_bf16(g: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(tuple(shape), generator=g, dtype=torch.float32).to(torch.bfloat16)


@dataclass
class PrefillInputs:
    q: torch.Tensor  # [B, Hq, Nq, d] bf16
    k: torch.Tensor  # [B, Hkv, Nk, d] bf16
    v: torch.Tensor  # [B, Hkv, Nk, d] bf16
    causal: bool
    scale: float
    generator: torch.Generator

    @property
    def shape(self):
        B, Hq, Nq, d = self.q.shape
        return B, Hq, self.k.shape[1], Nq, self.k.shape[2], d


def prefill_inputs(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int,
                   seed: int, causal: bool, k_scale: float = 1.0,
                   scale: float | None = None) -> PrefillInputs:
    g = torch.Generator("cpu").manual_seed(int(seed))
    q = _randn_bf16(g, (B, Hq, Nq, d))
    k = _randn_bf16(g, (B, Hkv, Nk, d))
    v = _randn_bf16(g, (B, Hkv, Nk, d))
    if k_scale != 1.0:
        k = (k.float() * k_scale).to(torch.bfloat16)
    if scale is None:
        scale = float(torch.tensor(1.0 / math.sqrt(d), dtype=torch.float32))
    return PrefillInputs(q, k, v, bool(causal), float(scale), g)


def check_rows(g: torch.Generator, B: int, Hq: int, Nq: int, per_head: int) -> torch.Tensor:
    """Flat row ids ((b*Hq + h)*Nq + i) of a seeded subset, sorted per head."""
    out = []
    for bh in range(B * Hq):
        pick = torch.randperm(Nq, generator=g)[:per_head]
        rows = torch.unique(torch.cat([pick, torch.tensor([0, Nq - 1])]))
        out.append(rows + bh * Nq)
    return torch.cat(out).to(torch.int64)


@dataclass
class DecodeInputs:
    q: torch.Tensor            # [S, Hq, d] bf16
    kcache: torch.Tensor       # [P, page_size, Hkv, d] bf16
    vcache: torch.Tensor       # [P, page_size, Hkv, d] bf16
    block_table: torch.Tensor  # [S, max_pages] int32
    seqlens: torch.Tensor      # [S] int32
    scale: float
    page_size: int
    max_seqlen: int
    generator: torch.Generator


def decode_inputs(num_seqs: int, Hq: int, Hkv: int, d: int, len_lo: int, len_hi: int,
                  num_pages: int, page_size: int, seed: int,
                  max_pages_per_seq: int | None = None,
                  lengths: list[int] | None = None,
                  scale: float | None = None) -> DecodeInputs:
    """Paged KV cache with seeded lengths (or explicit ``lengths``)."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    if lengths is None:
        lens = torch.randint(len_lo, len_hi + 1, (num_seqs,), generator=g, dtype=torch.int64)
    else:
        lens = torch.tensor(list(lengths), dtype=torch.int64)
        if lens.numel() != num_seqs:
            raise ValueError("lengths must have num_seqs entries")
    perm = torch.randperm(num_pages, generator=g)
    q = _randn_bf16(g, (num_seqs, Hq, d))
    pages_needed = [(int(L) + page_size - 1) // page_size for L in lens.tolist()]
    if max_pages_per_seq is None:
        max_pages_per_seq = max(1, (int(len_hi) + page_size - 1) // page_size)
    if sum(pages_needed) > num_pages:
        raise ValueError("page pool too small for the drawn lengths")
    if max(pages_needed + [0]) > max_pages_per_seq:
        raise ValueError("max_pages_per_seq too small for the drawn lengths")
    kc = torch.full((num_pages, page_size, Hkv, d), BF16_NAN, dtype=torch.bfloat16)
    vc = torch.full((num_pages, page_size, Hkv, d), BF16_NAN, dtype=torch.bfloat16)
    used = sum(pages_needed)
    spare = int(perm[used]) if used < num_pages else 0
    bt = torch.full((num_seqs, max_pages_per_seq), spare, dtype=torch.int32)
    cursor = 0
    for s, L in enumerate(lens.tolist()):
        npg = pages_needed[s]
        pages = perm[cursor:cursor + npg]
        cursor += npg
        bt[s, :npg] = pages.to(torch.int32)
        ks = _randn_bf16(g, (L, Hkv, d))
        vs = _randn_bf16(g, (L, Hkv, d))
        if L == 0:
            continue
        full = L // page_size
        if full:
            kc[pages[:full]] = ks[:full * page_size].reshape(full, page_size, Hkv, d)
            vc[pages[:full]] = vs[:full * page_size].reshape(full, page_size, Hkv, d)
        rem = L - full * page_size
        if rem:
            kc[pages[full], :rem] = ks[full * page_size:]
            vc[pages[full], :rem] = vs[full * page_size:]
    if scale is None:
        scale = float(torch.tensor(1.0 / math.sqrt(d), dtype=torch.float32))
    return DecodeInputs(q, kc, vc, bt, lens.to(torch.int32), float(scale), page_size,
                        int(lens.max().item()) if num_seqs else 0, g)


def alibi_slopes(Hq: int) -> torch.Tensor:
    """Per-head ALiBi slopes as float32 [Hq]: the geometric sequence
    2^(-8 (h + 1) / Hq) of the ALiBi recipe (an input of the biased kernel,
    not part of the attention arithmetic)."""
    h = torch.arange(1, Hq + 1, dtype=torch.float64)
    return torch.pow(2.0, -8.0 * h / Hq).to(torch.float32)


def bias_inputs(shape, seed: int, std: float = 2.0, neg_inf_frac: float = 0.0,
                neg_inf_rows: int = 0) -> torch.Tensor:
    """A dense additive bias [Bb, Hb, Nq, Nk] as bf16 (Bb, Hb may be 1 for
    broadcasting): ``std * randn`` from its own generator, then a random
    ``neg_inf_frac`` of the entries set to -inf, then ``neg_inf_rows`` random
    query rows of the first (batch, head) slice set to -inf entirely."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    b = torch.randn(tuple(shape), generator=g, dtype=torch.float32) * std
    if neg_inf_frac > 0:
        b[torch.rand(tuple(shape), generator=g) < neg_inf_frac] = float("-inf")
    if neg_inf_rows > 0:
        rows = torch.randperm(shape[2], generator=g)[:neg_inf_rows]
        b[0, 0, rows, :] = float("-inf")
    return b.to(torch.bfloat16)


@dataclass
class PagedPrefillInputs:
    q: torch.Tensor             # [total_q, Hq, d] bf16, sequences packed in order
    kcache: torch.Tensor        # [P, page_size, Hkv, d] bf16
    vcache: torch.Tensor        # [P, page_size, Hkv, d] bf16
    block_table: torch.Tensor   # [S, max_pages] int32
    cu_seqlens_q: torch.Tensor  # [S + 1] int32
    seqlens_k: torch.Tensor     # [S] int32 (context length, new tokens included)
    scale: float
    page_size: int
    max_seqlen_q: int
    generator: torch.Generator


def paged_prefill_inputs(q_lens: list[int], k_lens: list[int], Hq: int, Hkv: int, d: int,
                         num_pages: int, page_size: int, seed: int,
                         max_pages_per_seq: int | None = None,
                         scale: float | None = None) -> PagedPrefillInputs:
    """Chunked prefill: sequence s appends q_lens[s] new tokens to a context
    that then holds k_lens[s] tokens in the paged cache.

    Draw order: ``perm = randperm(num_pages)``, q [total_q, Hq, d], then for
    each sequence its K and V rows [k_lens[s], Hkv, d].  Pages are handed out
    from the permutation in sequence order; unused slots and pages hold bf16
    NaN and unused block-table entries point at a NaN page when one exists,
    as for paged decode.
    """
    if len(q_lens) != len(k_lens):
        raise ValueError("q_lens and k_lens differ in length")
    S = len(q_lens)
    g = torch.Generator("cpu").manual_seed(int(seed))
    perm = torch.randperm(num_pages, generator=g)
    total_q = int(sum(q_lens))
    q = _randn_bf16(g, (total_q, Hq, d))
    pages_needed = [(int(L) + page_size - 1) // page_size for L in k_lens]
    if max_pages_per_seq is None:
        max_pages_per_seq = max([1] + pages_needed)
    if sum(pages_needed) > num_pages:
        raise ValueError("page pool too small for the context lengths")
    if max(pages_needed + [0]) > max_pages_per_seq:
        raise ValueError("max_pages_per_seq too small for the context lengths")
    kc = torch.full((num_pages, page_size, Hkv, d), BF16_NAN, dtype=torch.bfloat16)
    vc = torch.full((num_pages, page_size, Hkv, d), BF16_NAN, dtype=torch.bfloat16)
    used = sum(pages_needed)
    spare = int(perm[used]) if used < num_pages else 0
    bt = torch.full((S, max_pages_per_seq), spare, dtype=torch.int32)
    cursor = 0
    for s, L in enumerate(int(x) for x in k_lens):
        npg = pages_needed[s]
        pages = perm[cursor:cursor + npg]
        cursor += npg
        bt[s, :npg] = pages.to(torch.int32)
        ks = _randn_bf16(g, (L, Hkv, d))
        vs = _randn_bf16(g, (L, Hkv, d))
        full = L // page_size
        if full:
            kc[pages[:full]] = ks[:full * page_size].reshape(full, page_size, Hkv, d)
            vc[pages[:full]] = vs[:full * page_size].reshape(full, page_size, Hkv, d)
        rem = L - full * page_size
        if rem:
            kc[pages[full], :rem] = ks[full * page_size:]
            vc[pages[full], :rem] = vs[full * page_size:]
    cu = torch.zeros(S + 1, dtype=torch.int32)
    if S:
        cu[1:] = torch.cumsum(torch.tensor([int(x) for x in q_lens], dtype=torch.int64), 0).to(torch.int32)
    if scale is None:
        scale = float(torch.tensor(1.0 / math.sqrt(d), dtype=torch.float32))
    return PagedPrefillInputs(q, kc, vc, bt, cu, torch.tensor([int(x) for x in k_lens], dtype=torch.int32),
                              float(scale), page_size, max([0] + [int(x) for x in q_lens]), g)
