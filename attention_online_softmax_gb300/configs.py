"""The synthetic workloads this library is measured and checked on.

Each entry names what the workload is, with its sizes.  Inputs come from
``inputs.py`` with the listed seed.  ``check_rows_per_head`` is the size of the
seeded query-row subset used when the CPU oracle cannot afford every row.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class PrefillConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    seed: int
    k_scale: float = 1.0
    check_rows_per_head: int | None = None  # None: every row
    window: int = 0            # left window (0: none)
    alibi: bool = False        # per-head ALiBi slopes
    bias: str | None = None    # dense bias: None, "full" [B,Hq,Nq,Nk] or "batch" [1,Hq,Nq,Nk]


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    num_seqs: int
    Hq: int
    Hkv: int
    d: int
    len_lo: int
    len_hi: int
    num_pages: int
    page_size: int
    seed: int


TINY = PrefillConfig("tiny_mha_b1_h2_n128_d64", 1, 2, 2, 128, 128, 64, False, 0)
BLOCK = PrefillConfig("causal_mha_b4_h16_n512_d64", 4, 16, 16, 512, 512, 64, True, 1)
LONG = PrefillConfig("causal_mha_b2_h32_n4096_d128", 2, 32, 32, 4096, 4096, 128, True, 2,
                     check_rows_per_head=256)
LONG_K4 = PrefillConfig("causal_mha_b2_h32_n4096_d128_kx4", 2, 32, 32, 4096, 4096, 128, True, 2,
                        k_scale=4.0, check_rows_per_head=256)
GQA256 = PrefillConfig("causal_gqa16to2_b1_n16384_d256", 1, 16, 2, 16384, 16384, 256, True, 3,
                       check_rows_per_head=256)
DECODE = DecodeConfig("paged_gqa32to8_decode_64seq_d128_len512to8192", 64, 32, 8, 128,
                      512, 8192, 40000, 16, 4)

PREFILL_CONFIGS = (TINY, BLOCK, LONG, LONG_K4, GQA256)
# Workloads whose backward is timed (the forward's O and LSE as inputs).
BWD_CONFIGS = (LONG, GQA256)

# Additive-bias workloads ("Compilers and Kernels": S = Q K^T / sqrt(d) + C).
WINDOW = PrefillConfig("causal_window1024_b2_h32_n4096_d128", 2, 32, 32, 4096, 4096, 128, True, 5,
                       check_rows_per_head=64, window=1024)
ALIBI_BIAS = PrefillConfig("alibi_densebias_b1_h16_n2048_d128", 1, 16, 16, 2048, 2048, 128, False, 6,
                           check_rows_per_head=64, alibi=True, bias="batch")
MASKED_CONFIGS = (WINDOW, ALIBI_BIAS)


@dataclass(frozen=True)
class ChunkedConfig:
    """Chunked prefill against a paged KV cache: each sequence appends
    ``chunk`` new tokens to a cached context of U[ctx_lo, ctx_hi] tokens."""
    name: str
    num_seqs: int
    chunk: int
    ctx_lo: int
    ctx_hi: int
    Hq: int
    Hkv: int
    d: int
    num_pages: int
    page_size: int
    seed: int


CHUNKED = ChunkedConfig("chunked_prefill_16seq_512new_ctx0to8192_gqa32to8_d128", 16, 512, 0, 8192, 32, 8, 128,
                        12000, 16, 7)


def chunked_lengths(c: ChunkedConfig):
    """(q_lens, k_lens) of a chunked-prefill workload: contexts drawn as
    ``randint(ctx_lo, ctx_hi + 1)`` from a generator seeded with ``seed``."""
    import torch
    g = torch.Generator("cpu").manual_seed(int(c.seed))
    ctx = torch.randint(c.ctx_lo, c.ctx_hi + 1, (c.num_seqs,), generator=g).tolist()
    return [c.chunk] * c.num_seqs, [int(x) + c.chunk for x in ctx]


ALL = {c.name: c for c in PREFILL_CONFIGS + MASKED_CONFIGS + (DECODE, CHUNKED)}
