"""Oracle for fused attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never imports, links or calls it, and it imports nothing from the CUDA
library.  Inputs reach both sides from the seeded generators in
``attention_online_softmax_gb300.inputs``, which hold none of the method's
arithmetic.

Contents
--------
``attn_oracle.c``   plain two-pass attention and paged decode in double
                    precision (C, OpenMP over query rows); see its header for
                    the passages it follows and the readings it takes.
``monoid.py``       the online-softmax recurrence and the associative merge of
                    partial states (m, l, o), in float64 numpy, written from the
                    same pages; used by the tests to pin the merge semantics.

Every function here is pinned by ``tests/test_oracle_*.py`` against brute
force, closed forms and invariants; none of its expected values comes from the
CUDA path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
#: the C source of the oracle
SOURCE = _SRC
_LOCK = threading.Lock()
_LIBS: dict[int, ctypes.CDLL] = {}
# Patched copies of the source with one planted mistake each, registered by
# the test-suite under a number (``mutant=`` of the functions below).
_MUTANT_SOURCES: dict[int, str] = {}


def register_source(mutant: int, path: str) -> None:
    """Use the C file at ``path`` for ``mutant=mutant`` (mutant > 0)."""
    if mutant <= 0:
        raise ValueError("mutant numbers are positive; 0 is the oracle itself")
    with _LOCK:
        _MUTANT_SOURCES[mutant] = path
        _LIBS.pop(mutant, None)


def lib_path(mutant: int = 0) -> str:
    name = "liboracle.so" if mutant == 0 else f"liboracle_mutant{mutant}.so"
    return os.path.join(_HERE, "_build", name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the C oracle (or a registered mutant copy) with gcc (-O2,
    OpenMP).  Returns the .so path."""
    src = _SRC
    if mutant != 0:
        src = _MUTANT_SOURCES.get(mutant)
        if src is None:
            raise ValueError(f"no source registered for mutant {mutant}")
    out = lib_path(mutant)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load(mutant: int = 0) -> ctypes.CDLL:
    with _LOCK:
        lib = _LIBS.get(mutant)
        if lib is None:
            lib = ctypes.CDLL(build(mutant))
            p = ctypes.c_void_p
            i = ctypes.c_int
            lib.oracle_attention.argtypes = [p, p, p, i, i, i, i, i, i, i,
                                             ctypes.c_float, p, ctypes.c_int64,
                                             p, p, i]
            lib.oracle_attention.restype = i
            lib.oracle_decode_paged.argtypes = [p, p, p, p, p, i, i, i, i, i,
                                                i, i, ctypes.c_float, p, i,
                                                p, p, i]
            lib.oracle_decode_paged.restype = i
            i64 = ctypes.c_int64
            lib.oracle_attention_masked.argtypes = [p, p, p, i, i, i, i, i, i, i,
                                                    ctypes.c_float, i, p, p, i64, i64,
                                                    p, i64, p, p, i]
            lib.oracle_attention_masked.restype = i
            lib.oracle_prefill_paged.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, i, i, i,
                                                 ctypes.c_float, p, i64, p, p, i]
            lib.oracle_prefill_paged.restype = i
            lib.oracle_attention_bwd.argtypes = [p, p, p, p, i, i, i, i, i, i, i, ctypes.c_float,
                                                 p, p, p, i]
            lib.oracle_attention_bwd.restype = i
            lib.oracle_attention_bwd_dq_rows.argtypes = [p, p, p, p, i, i, i, i, i, i, i, ctypes.c_float,
                                                         p, i64, p, i]
            lib.oracle_attention_bwd_dq_rows.restype = i
            lib.oracle_attention_masked_bwd.argtypes = [p, p, p, p, i, i, i, i, i, i, i, ctypes.c_float,
                                                        i, p, p, i64, i64, p, p, p, i]
            lib.oracle_attention_masked_bwd.restype = i
            _LIBS[mutant] = lib
        return lib


def _bits(x) -> np.ndarray:
    """bf16 data as a contiguous uint16 numpy array of its bit patterns.

    Accepts a torch bfloat16 tensor (any device: it is copied to host) or a
    numpy uint16 array.
    """
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("numpy input must hold bf16 bit patterns as uint16")
        return np.ascontiguousarray(x)
    import torch
    if x.dtype != torch.bfloat16:
        raise TypeError(f"expected bfloat16, got {x.dtype}")
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def attention(q, k, v, causal: bool, scale: float, rows=None, threads: int = 0,
              mutant: int = 0):
    """softmax(scale * Q K^T + mask) V and the row logsumexp, in float64.

    q: [B, Hq, Nq, d], k, v: [B, Hkv, Nk, d] (bf16).  ``rows`` selects flat
    query rows ((b*Hq + h)*Nq + i); None means all rows.  Returns
    (O [nrows, d] float64, LSE [nrows] float64, threads_used); with rows=None
    O is reshaped to [B, Hq, Nq, d] and LSE to [B, Hq, Nq].
    """
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    if qb.ndim != 4 or kb.ndim != 4 or vb.shape != kb.shape:
        raise ValueError("q must be [B,Hq,Nq,d]; k, v [B,Hkv,Nk,d]")
    B, Hq, Nq, d = qb.shape
    Bk, Hkv, Nk, dk = kb.shape
    if Bk != B or dk != d:
        raise ValueError("q/k shape mismatch")
    if rows is None:
        nrows = B * Hq * Nq
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.size
    o = np.empty((nrows, d), dtype=np.float64)
    lse = np.empty((nrows,), dtype=np.float64)
    rc = _load(mutant).oracle_attention(
        _ptr(qb), _ptr(kb), _ptr(vb), B, Hq, Hkv, Nq, Nk, d, int(bool(causal)),
        float(scale), None if rows_arr is None else _ptr(rows_arr), nrows,
        _ptr(o), _ptr(lse), int(threads))
    if rc < 0:
        raise ValueError(f"oracle_attention rejected its arguments ({rc})")
    if rows is None:
        o = o.reshape(B, Hq, Nq, d)
        lse = lse.reshape(B, Hq, Nq)
    return o, lse, rc


def attention_masked(q, k, v, causal: bool, scale: float, window_left: int = 0, alibi=None,
                     bias=None, bias_strides=(0, 0), rows=None, threads: int = 0, mutant: int = 0):
    """Attention with the additive bias C = causal mask + left window + ALiBi
    + dense bias (see oracle_attention_masked in attn_oracle.c), float64.

    alibi: [Hq] float32 slopes or None; bias: bf16 tensor addressed as
    bias[b*sb + h*sh + i*Nk + j] with bias_strides = (sb, sh) in elements, or
    None.  Returns (O, LSE, threads) shaped like ``attention``.
    """
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    B, Hq, Nq, d = qb.shape
    _, Hkv, Nk, _ = kb.shape
    al = None if alibi is None else np.ascontiguousarray(np.asarray(_host(alibi), dtype=np.float32))
    bb = None if bias is None else _bits(bias).reshape(-1)
    if rows is None:
        nrows = B * Hq * Nq
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.size
    o = np.empty((nrows, d), dtype=np.float64)
    lse = np.empty((nrows,), dtype=np.float64)
    rc = _load(mutant).oracle_attention_masked(
        _ptr(qb), _ptr(kb), _ptr(vb), B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), float(scale),
        int(window_left), None if al is None else _ptr(al), None if bb is None else _ptr(bb),
        int(bias_strides[0]), int(bias_strides[1]),
        None if rows_arr is None else _ptr(rows_arr), nrows, _ptr(o), _ptr(lse), int(threads))
    if rc < 0:
        raise ValueError(f"oracle_attention_masked rejected its arguments ({rc})")
    if rows is None:
        o = o.reshape(B, Hq, Nq, d)
        lse = lse.reshape(B, Hq, Nq)
    return o, lse, rc


def decode_paged(q, kcache, vcache, block_table, seqlens, scale: float,
                 seqs=None, threads: int = 0, mutant: int = 0):
    """One-row attention per (sequence, query head) over a paged KV cache.

    q: [S, Hq, d]; kcache, vcache: [P, page_size, Hkv, d] (bf16);
    block_table: [S, max_pages] int32; seqlens: [S] int32.  Returns
    (O [n, Hq, d] float64, LSE [n, Hq] float64, threads_used) for the selected
    sequences (all when ``seqs`` is None).
    """
    qb, kb, vb = _bits(q), _bits(kcache), _bits(vcache)
    bt = np.ascontiguousarray(np.asarray(_host(block_table), dtype=np.int32))
    sl = np.ascontiguousarray(np.asarray(_host(seqlens), dtype=np.int32))
    S, Hq, d = qb.shape
    P, page, Hkv, dk = kb.shape
    if dk != d or vb.shape != kb.shape or bt.shape[0] != S or sl.shape != (S,):
        raise ValueError("decode shape mismatch")
    if seqs is None:
        n = S
        seqs_arr = None
    else:
        seqs_arr = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
        n = seqs_arr.size
    o = np.empty((n, Hq, d), dtype=np.float64)
    lse = np.empty((n, Hq), dtype=np.float64)
    rc = _load(mutant).oracle_decode_paged(
        _ptr(qb), _ptr(kb), _ptr(vb), _ptr(bt), _ptr(sl), S, Hq, Hkv, d, page,
        P, bt.shape[1], float(scale), None if seqs_arr is None else _ptr(seqs_arr),
        n, _ptr(o), _ptr(lse), int(threads))
    if rc < 0:
        raise ValueError(f"oracle_decode_paged rejected its arguments ({rc})")
    return o, lse, rc


def attention_bwd(q, k, v, dout, causal: bool, scale: float, threads: int = 0, mutant: int = 0):
    """Gradients (dQ, dK, dV) of the attention output for the upstream
    gradient dout (see oracle_attention_bwd in attn_oracle.c), float64.

    q, dout: [B, Hq, Nq, d]; k, v: [B, Hkv, Nk, d] (bf16).  Returns
    (dQ [B,Hq,Nq,d], dK [B,Hkv,Nk,d], dV [B,Hkv,Nk,d], threads_used).
    """
    qb, kb, vb, gb = _bits(q), _bits(k), _bits(v), _bits(dout)
    B, Hq, Nq, d = qb.shape
    _, Hkv, Nk, _ = kb.shape
    if gb.shape != qb.shape or vb.shape != kb.shape:
        raise ValueError("q/dout or k/v shape mismatch")
    dq = np.empty((B, Hq, Nq, d), dtype=np.float64)
    dk = np.empty((B, Hkv, Nk, d), dtype=np.float64)
    dv = np.empty((B, Hkv, Nk, d), dtype=np.float64)
    rc = _load(mutant).oracle_attention_bwd(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(gb), B, Hq, Hkv, Nq, Nk, d,
                                      int(bool(causal)), float(scale), _ptr(dq), _ptr(dk), _ptr(dv),
                                      int(threads))
    if rc < 0:
        raise ValueError(f"oracle_attention_bwd rejected its arguments ({rc})")
    return dq, dk, dv, rc


def attention_masked_bwd(q, k, v, dout, causal: bool, scale: float, window_left: int = 0, alibi=None,
                         bias=None, bias_strides=(0, 0), threads: int = 0):
    """Gradients (dQ, dK, dV) of attention_masked's output for the upstream
    gradient dout (see oracle_attention_masked_bwd in attn_oracle.c), float64.

    alibi, bias and bias_strides as in attention_masked.  Returns
    (dQ [B,Hq,Nq,d], dK [B,Hkv,Nk,d], dV [B,Hkv,Nk,d], threads_used).
    """
    qb, kb, vb, gb = _bits(q), _bits(k), _bits(v), _bits(dout)
    B, Hq, Nq, d = qb.shape
    _, Hkv, Nk, _ = kb.shape
    if gb.shape != qb.shape or vb.shape != kb.shape:
        raise ValueError("q/dout or k/v shape mismatch")
    al = None if alibi is None else np.ascontiguousarray(np.asarray(_host(alibi), dtype=np.float32))
    if al is not None and al.shape != (Hq,):
        raise ValueError("alibi must have one slope per query head")
    bb = None if bias is None else _bits(bias).reshape(-1)
    dq = np.empty((B, Hq, Nq, d), dtype=np.float64)
    dk = np.empty((B, Hkv, Nk, d), dtype=np.float64)
    dv = np.empty((B, Hkv, Nk, d), dtype=np.float64)
    rc = _load().oracle_attention_masked_bwd(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(gb), B, Hq, Hkv, Nq, Nk, d,
                                             int(bool(causal)), float(scale), int(window_left),
                                             None if al is None else _ptr(al), None if bb is None else _ptr(bb),
                                             int(bias_strides[0]), int(bias_strides[1]), _ptr(dq), _ptr(dk),
                                             _ptr(dv), int(threads))
    if rc < 0:
        raise ValueError(f"oracle_attention_masked_bwd rejected its arguments ({rc})")
    return dq, dk, dv, rc


def attention_bwd_dq_rows(q, k, v, dout, causal: bool, scale: float, rows, threads: int = 0):
    """dQ of the listed flat query rows ((b * Hq + h) * Nq + i) only, by the
    same per-row steps as attention_bwd (see oracle_attention_bwd_dq_rows in
    attn_oracle.c), float64: [len(rows), d].  Costs one row's keys per row.
    """
    qb, kb, vb, gb = _bits(q), _bits(k), _bits(v), _bits(dout)
    B, Hq, Nq, d = qb.shape
    _, Hkv, Nk, _ = kb.shape
    if gb.shape != qb.shape or vb.shape != kb.shape:
        raise ValueError("q/dout or k/v shape mismatch")
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.empty((r.shape[0], d), dtype=np.float64)
    rc = _load().oracle_attention_bwd_dq_rows(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(gb), B, Hq, Hkv, Nq, Nk, d,
                                              int(bool(causal)), float(scale), _ptr(r), int(r.shape[0]),
                                              _ptr(out), int(threads))
    if rc < 0:
        raise ValueError(f"oracle_attention_bwd_dq_rows rejected its arguments ({rc})")
    return out


def prefill_paged(q, kcache, vcache, block_table, cu_seqlens_q, seqlens_k, causal: bool,
                  scale: float, window_left: int = 0, rows=None, threads: int = 0, mutant: int = 0):
    """Chunked prefill of ragged sequences against a paged KV cache (see
    oracle_prefill_paged in attn_oracle.c), float64.

    q: [total_q, Hq, d]; kcache, vcache: [P, page_size, Hkv, d] (bf16);
    block_table: [S, max_pages] int32; cu_seqlens_q: [S + 1] int32;
    seqlens_k: [S] int32.  ``rows`` selects flat (token * Hq + h) rows.
    Returns (O [total_q, Hq, d] or [nrows, d], LSE [total_q, Hq] or [nrows],
    threads_used).
    """
    qb, kb, vb = _bits(q), _bits(kcache), _bits(vcache)
    bt = np.ascontiguousarray(np.asarray(_host(block_table), dtype=np.int32))
    cu = np.ascontiguousarray(np.asarray(_host(cu_seqlens_q), dtype=np.int32))
    sk = np.ascontiguousarray(np.asarray(_host(seqlens_k), dtype=np.int32))
    total_q, Hq, d = qb.shape
    P, page, Hkv, dk = kb.shape
    S = sk.shape[0]
    if dk != d or vb.shape != kb.shape or cu.shape != (S + 1,) or bt.shape[0] != S:
        raise ValueError("paged prefill shape mismatch")
    if S and int(cu[-1]) != total_q:
        raise ValueError("cu_seqlens_q[-1] must equal total_q")
    if rows is None:
        nrows = total_q * Hq
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.size
    o = np.empty((nrows, d), dtype=np.float64)
    lse = np.empty((nrows,), dtype=np.float64)
    rc = _load(mutant).oracle_prefill_paged(
        _ptr(qb), _ptr(kb), _ptr(vb), _ptr(bt), _ptr(cu), _ptr(sk), S, Hq, Hkv, d, page, P,
        bt.shape[1] if bt.ndim == 2 else 0, int(bool(causal)), int(window_left), float(scale),
        None if rows_arr is None else _ptr(rows_arr), nrows, _ptr(o), _ptr(lse), int(threads))
    if rc < 0:
        raise ValueError(f"oracle_prefill_paged rejected its arguments ({rc})")
    if rows is None:
        o = o.reshape(total_q, Hq, d)
        lse = lse.reshape(total_q, Hq)
    return o, lse, rc


def _host(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return x
