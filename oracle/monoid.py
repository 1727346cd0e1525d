"""Online softmax as a recurrence over key blocks and as a monoid -- TEST ONLY.

Float64 numpy restatements, used by the tests to pin the semantics that the
CUDA kernels implement (the per-tile recurrence in prefill, the split partials
and their merge in paged decode).  Nothing here is imported by the CUDA path.

Sources
-------
"Compilers and Kernels", section "FlashAttention changes the algorithm around
IO", the block recurrence: for one query row, start from m = -inf, l = 0,
o = 0; for each key block B_t take b_t = max S over the block, m_t =
max(m_{t-1}, b_t), alpha_t = exp(m_{t-1} - m_t), l_t = alpha_t l_{t-1} +
sum_j exp(S_j - m_t), o_t = alpha_t o_{t-1} + sum_j exp(S_j - m_t) v_j, and
finish with O = o_T / l_T.  The same section states that this keeps the same
numerator and denominator as the full softmax in exact arithmetic.

"Tang: a compiler that derives GPU kernels ..." (abstract): the flash schedule
comes from recognising online softmax as a monoid.  The pages print only the
sequential step above, so the binary merge is this reading of it:

    (m_a, l_a, o_a) (+) (m_b, l_b, o_b) = (m, e^{m_a-m} l_a + e^{m_b-m} l_b,
                                              e^{m_a-m} o_a + e^{m_b-m} o_b),
    m = max(m_a, m_b), identity (-inf, 0, 0).

The sequential step is the merge with a single block's state on the right.
Where a running max is -inf (nothing allowed yet) its weight is taken as 0
instead of exp(-inf - -inf); merging with the identity returns the other
operand unchanged.
"""
from __future__ import annotations

import math

import numpy as np


class State:
    """Partial softmax state of one query row: running max, sum, numerator."""

    __slots__ = ("m", "l", "o")

    def __init__(self, m: float, l: float, o: np.ndarray):
        self.m = float(m)
        self.l = float(l)
        self.o = np.asarray(o, dtype=np.float64)

    def __repr__(self) -> str:  # pragma: no cover - debugging aid
        return f"State(m={self.m}, l={self.l}, o={self.o})"


def identity(dv: int) -> State:
    return State(-math.inf, 0.0, np.zeros(dv))


def _weight(m_part: float, m: float) -> float:
    # exp(m_part - m), with an empty part (m_part = -inf) weighing 0.
    if m_part == -math.inf:
        return 0.0
    return math.exp(m_part - m)


def merge(a: State, b: State) -> State:
    """Associative, commutative merge of two partial states (identity (-inf,0,0))."""
    m = max(a.m, b.m)
    if m == -math.inf:
        return identity(a.o.shape[0])
    wa, wb = _weight(a.m, m), _weight(b.m, m)
    return State(m, wa * a.l + wb * b.l, wa * a.o + wb * b.o)


def block_state(scores: np.ndarray, values: np.ndarray) -> State:
    """State of one key block: scores [n] (-inf = disallowed), values [n, dv]."""
    scores = np.asarray(scores, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    dv = values.shape[1]
    allowed = scores > -math.inf
    if not allowed.any():
        return identity(dv)
    b = float(scores[allowed].max())
    p = np.where(allowed, np.exp(np.where(allowed, scores, 0.0) - b), 0.0)
    return State(b, float(p.sum()), p @ values)


def recurrence(scores: np.ndarray, values: np.ndarray, partition) -> State:
    """The page's sequential recurrence over the blocks listed in ``partition``.

    ``partition`` is a list of index arrays covering the keys in order.  Each
    step takes b_t, updates m_t, rescales by alpha_t and adds the block's
    exp(S - m_t) terms, exactly in the order the recurrence is printed.
    """
    scores = np.asarray(scores, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    m = -math.inf
    l = 0.0
    o = np.zeros(values.shape[1])
    for idx in partition:
        s = scores[idx]
        allowed = s > -math.inf
        b_t = float(s[allowed].max()) if allowed.any() else -math.inf
        m_t = max(m, b_t)
        if m_t == -math.inf:
            continue  # nothing allowed so far: state stays (-inf, 0, 0)
        alpha = _weight(m, m_t)
        p = np.where(allowed, np.exp(np.where(allowed, s, 0.0) - m_t), 0.0)
        l = alpha * l + float(p.sum())
        o = alpha * o + p @ values[idx]
        m = m_t
    return State(m, l, o)


def finalize(st: State):
    """(O, LSE) of a state: O = o / l, LSE = m + ln l; empty -> (0, -inf)."""
    if st.l == 0.0:
        return np.zeros_like(st.o), -math.inf
    return st.o / st.l, st.m + math.log(st.l)


def from_output(o_row: np.ndarray, lse: float) -> State:
    """The equivalent stored form (O_s, lse_s) of a partial, as a state.

    A partial stored as normalised output O_s = o_s / l_s and lse_s =
    m_s + ln l_s is the state (lse_s, 1, O_s): scaling (m, l, o) by a common
    factor leaves every merge result unchanged.
    """
    if lse == -math.inf:
        return identity(np.asarray(o_row).shape[0])
    return State(lse, 1.0, np.asarray(o_row, dtype=np.float64))
