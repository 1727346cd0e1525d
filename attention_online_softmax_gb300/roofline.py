"""Algorithmic work and traffic of the attention path, and the roofline bound.

Conventions ("Compilers and Kernels", section "Roofline is a bound, not a
stopwatch"): intensity I = F / Q, attainable rate P_bound = min(P_max,
B_max * I), time floor T >= max(F / P_max, Q / B_max), with measured ceilings.
Traffic is counted the way that section's fused-versus-unfused example counts
it: every materialised tensor costs one full pass over HBM for each read and
each write, with no credit for cache retention across kernels.

Prefill FLOPs are 4*B*Hq*Nq*Nk*d (two matrix products), halved for causal
masking.  Prefill bytes are one pass over Q, K, V (bf16; K and V once per
key/value head), O (bf16) and LSE (f32).  Decode bytes are the K and V rows of
every cached token (once per key/value head: a query group shares each read),
plus q, O, LSE, the block-table entries used and the sequence lengths.  Split
partials written by the decode path are overhead, not algorithmic traffic.
"""
from __future__ import annotations

import json
import math
import os
from dataclasses import dataclass

BF16 = 2
F32 = 4
I32 = 4


def materialized_traffic(elements: int, bytes_per_element: int, reads: int, writes: int) -> int:
    """Bytes moved when ``reads`` + ``writes`` full tensors cross HBM."""
    return int(elements) * int(bytes_per_element) * (int(reads) + int(writes))


def prefill_flops(B: int, Hq: int, Nq: int, Nk: int, d: int, causal: bool) -> float:
    f = 4.0 * B * Hq * Nq * Nk * d
    return f / 2.0 if causal else f


def allowed_pairs(Nq: int, Nk: int, causal: bool, window: int = 0) -> int:
    """Number of (query, key) pairs the mask allows in one (batch, head):
    row i sees keys [max(0, i + Nk - Nq - window + 1), min(Nk - 1, i + Nk - Nq)]
    (the lower end only with a window, the upper only when causal)."""
    import numpy as np
    i = np.arange(Nq, dtype=np.int64)
    diag = Nk - Nq
    hi = np.minimum(Nk - 1, i + diag) if causal else np.full(Nq, Nk - 1, dtype=np.int64)
    lo = np.maximum(0, i + diag - window + 1) if window > 0 else np.zeros(Nq, dtype=np.int64)
    return int(np.clip(hi - lo + 1, 0, None).sum())


def masked_flops(B: int, Hq: int, Nq: int, Nk: int, d: int, causal: bool, window: int = 0) -> float:
    """4 d flops (two d-long dot products, multiply + add) per allowed pair."""
    return 4.0 * B * Hq * d * allowed_pairs(Nq, Nk, causal, window)


def prefill_bytes(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int) -> int:
    q = B * Hq * Nq * d * BF16
    kv = 2 * B * Hkv * Nk * d * BF16
    o = B * Hq * Nq * d * BF16
    lse = B * Hq * Nq * F32
    return q + kv + o + lse


def bwd_bytes(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int) -> int:
    """Backward: Q, O, dO read and dQ written (bf16) per query head; K, V read
    and dK, dV written per kv head; LSE read (f32)."""
    qside = B * Hq * Nq * d * BF16 * 4
    kside = B * Hkv * Nk * d * BF16 * 4
    return qside + kside + B * Hq * Nq * F32


def paged_prefill_bytes(q_lens, k_lens, Hq: int, Hkv: int, d: int, page_size: int) -> int:
    """Chunked prefill: new-token Q, O (bf16) and LSE (f32), each sequence's
    context K and V once per KV head, and the block-table entries used."""
    tq = sum(int(x) for x in q_lens)
    kv = sum(int(x) for x in k_lens) * Hkv * d * BF16 * 2
    bt = sum((int(L) + page_size - 1) // page_size for L in k_lens) * I32
    return tq * Hq * d * BF16 * 2 + tq * Hq * F32 + kv + bt + (len(q_lens) * 2 + 1) * I32


def decode_bytes(seqlens, Hq: int, Hkv: int, d: int, page_size: int) -> int:
    lens = [int(x) for x in seqlens]
    kv = sum(lens) * Hkv * d * BF16 * 2
    q = len(lens) * Hq * d * BF16
    o = len(lens) * Hq * d * BF16
    lse = len(lens) * Hq * F32
    bt = sum((L + page_size - 1) // page_size for L in lens) * I32
    sl = len(lens) * I32
    return kv + q + o + lse + bt + sl


def decode_flops(seqlens, Hq: int, d: int) -> float:
    return 4.0 * sum(int(x) for x in seqlens) * Hq * d


@dataclass(frozen=True)
class Peaks:
    hbm_gbs: float
    bf16_tflops: float
    bf16_tflops_sustained: float
    source: str  # "measured" or "fallback"


FALLBACK = Peaks(6800.0, 1900.0, 1700.0, "fallback")


def load_peaks(path: str | None = None) -> Peaks:
    """Ceilings from MEASURED_PEAKS.json at the repository root, else fallback."""
    if path is None:
        path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
    except (OSError, ValueError):
        return FALLBACK

    def pick(*names):
        for n in names:
            cur = j
            ok = True
            for part in n.split("."):
                if isinstance(cur, dict) and part in cur:
                    cur = cur[part]
                else:
                    ok = False
                    break
            if ok and isinstance(cur, (int, float)):
                return float(cur)
        return None

    hbm = pick("hbm_gbs", "hbm.gbs", "hbm_copy_gbs")
    tf = pick("bf16_tflops", "bf16.tflops", "bf16_dense_tflops")
    tfs = pick("bf16_tflops_sustained", "bf16.tflops_sustained")
    if hbm is None or tf is None:
        return FALLBACK
    return Peaks(hbm, tf, tfs if tfs is not None else tf, "measured")


def time_floor_s(flops: float, nbytes: float, peaks: Peaks, sustained: bool = False) -> float:
    p = (peaks.bf16_tflops_sustained if sustained else peaks.bf16_tflops) * 1e12
    b = peaks.hbm_gbs * 1e9
    return max(flops / p, nbytes / b)


def bound_rate(flops: float, nbytes: float, peaks: Peaks) -> float:
    """P_bound = min(P_max, B_max * I) in FLOP/s."""
    if nbytes <= 0:
        return peaks.bf16_tflops * 1e12
    return min(peaks.bf16_tflops * 1e12, peaks.hbm_gbs * 1e9 * flops / nbytes)


def ridge(peaks: Peaks) -> float:
    return peaks.bf16_tflops * 1e12 / (peaks.hbm_gbs * 1e9)


def fmt_frac(x: float) -> float:
    return float(f"{x:.4f}") if math.isfinite(x) else x
