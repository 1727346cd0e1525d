"""Thin ctypes binding of the C ABI in include/attn.h (argument marshalling only).

Each function has the name of the C entry point it calls.  Tensors are
PyTorch CUDA tensors (torch is used for device memory and streams only); the
binding checks dtype / contiguity / device, passes raw pointers and sizes, and
raises ``AttnError`` on a non-OK status.  Every step of the computation runs in
the CUDA kernels of libattn_gb300.so: there is no other code path.  Importing
this module when the library has not been built raises ``ImportError``.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

_LIB_PATH = _build.LIB

if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"libattn_gb300.so is not built ({_LIB_PATH}); run "
        "`python -m attention_online_softmax_gb300.build` (needs nvcc)")

_lib = ctypes.CDLL(_LIB_PATH)

_vp = ctypes.c_void_p
_i = ctypes.c_int
_lib.attn_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, ctypes.c_float, _i, _vp]
_lib.attn_fwd.restype = _i
class AttnMask(ctypes.Structure):
    """Mirror of attn_mask in include/attn.h."""
    _fields_ = [("window_left", ctypes.c_int), ("alibi_slopes", ctypes.c_void_p),
                ("bias", ctypes.c_void_p), ("bias_stride_b", ctypes.c_longlong),
                ("bias_stride_h", ctypes.c_longlong)]


_lib.attn_fwd_masked.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, ctypes.c_float,
                                 ctypes.POINTER(AttnMask), _i, _vp]
_lib.attn_fwd_masked.restype = _i
_lib.attn_prefill_paged_workspace_size.argtypes = [_i]
_lib.attn_prefill_paged_workspace_size.restype = ctypes.c_size_t
_lib.attn_prefill_paged.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i,
                                    _i, _i, ctypes.c_float, _vp, ctypes.c_size_t, _i, _vp]
_lib.attn_prefill_paged.restype = _i
_lib.attn_bwd_workspace_size.argtypes = [_i, _i, _i, _i]
_lib.attn_bwd_workspace_size.restype = ctypes.c_size_t
_lib.attn_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, ctypes.c_float,
                          _i, _vp, ctypes.c_size_t, _vp]
_lib.attn_bwd.restype = _i
_lib.attn_bwd_masked.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i,
                                 ctypes.c_float, ctypes.POINTER(AttnMask), _i, _vp, ctypes.c_size_t, _vp]
_lib.attn_bwd_masked.restype = _i
_lib.attn_probe_dram_latency.argtypes = [_vp, ctypes.c_size_t, _i, _vp, _vp]
_lib.attn_probe_dram_latency.restype = _i
_lib.attn_decode_workspace_size.argtypes = [_i, _i, _i, _i, _i]
_lib.attn_decode_workspace_size.restype = ctypes.c_size_t
_lib.attn_decode_paged.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i,
                                   ctypes.c_float, _vp, ctypes.c_size_t, _i, _vp]
_lib.attn_decode_paged.restype = _i
_lib.attn_decode_paged_static.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i,
                                          _i, ctypes.c_float, _i, _vp]
_lib.attn_decode_paged_static.restype = _i
_lib.attn_selftest_wait_timeout.argtypes = [ctypes.c_uint32, _vp]
_lib.attn_selftest_wait_timeout.restype = _i
_lib.attn_get_device_status.argtypes = [_vp]
_lib.attn_get_device_status.restype = _i
_lib.attn_status_string.argtypes = [_i]
_lib.attn_status_string.restype = ctypes.c_char_p
_lib.attn_launch_count.argtypes = []
_lib.attn_launch_count.restype = ctypes.c_uint64
_lib.attn_abi_version.argtypes = []
_lib.attn_abi_version.restype = _i
_lib.attn_fwd_kernel_name.argtypes = [_i, _i, _i, _i]
_lib.attn_fwd_kernel_name.restype = ctypes.c_char_p
_lib.attn_decode_kernel_name.argtypes = [_i, _i, _i, _i, _i]
_lib.attn_decode_kernel_name.restype = ctypes.c_char_p

ATTN_OK = 0
ATTN_BF16 = 0
ATTN_F32 = 1

#: every symbol include/attn.h declares
EXPORTS = ("attn_fwd", "attn_fwd_masked", "attn_prefill_paged_workspace_size", "attn_prefill_paged",
           "attn_bwd_workspace_size", "attn_bwd", "attn_bwd_masked", "attn_probe_dram_latency",
           "attn_decode_workspace_size", "attn_decode_paged", "attn_decode_paged_static",
           "attn_get_device_status", "attn_selftest_wait_timeout", "attn_status_string",
           "attn_launch_count", "attn_abi_version", "attn_fwd_kernel_name", "attn_decode_kernel_name")

#: size of the scratch array built into the library for attn_decode_paged_static
STATIC_SCRATCH_BYTES = 64 << 20


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {attn_status_string(status)} (status {status})")


def lib() -> ctypes.CDLL:
    return _lib


def attn_status_string(status: int) -> str:
    return _lib.attn_status_string(int(status)).decode()


def attn_launch_count() -> int:
    return int(_lib.attn_launch_count())


def attn_abi_version() -> int:
    return int(_lib.attn_abi_version())


def attn_fwd_kernel_name(B: int, Hq: int, Nq: int, d: int) -> str:
    """The kernel instantiation attn_fwd launches for these sizes ("" if rejected)."""
    return _lib.attn_fwd_kernel_name(int(B), int(Hq), int(Nq), int(d)).decode()


def attn_decode_kernel_name(num_seqs: int, Hq: int, Hkv: int, d: int, max_seqlen: int) -> str:
    """The kernel instantiation attn_decode_paged launches for these sizes ("" if rejected)."""
    return _lib.attn_decode_kernel_name(int(num_seqs), int(Hq), int(Hkv), int(d), int(max_seqlen)).decode()


def _stream_ptr(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _check(status: int, where: str) -> None:
    if status != ATTN_OK:
        raise AttnError(status, where)


def _need(t, dtype, name):
    import torch
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return torch


def attn_fwd(q, k, v, o, lse, causal: bool, scale: float, stream=None) -> None:
    """q [B,Hq,Nq,d], k/v [B,Hkv,Nk,d] bf16 -> o [B,Hq,Nq,d] (bf16|f32), lse [B,Hq,Nq] f32."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    _need(lse, torch.float32, "lse")
    if o.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("o must be bfloat16 or float32")
    _need(o, o.dtype, "o")
    B, Hq, Nq, d = q.shape
    _, Hkv, Nk, _ = k.shape
    if tuple(o.shape) != (B, Hq, Nq, d) or tuple(lse.shape) != (B, Hq, Nq) or v.shape != k.shape:
        raise ValueError("shape mismatch between q, k, v, o, lse")
    st = _lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nk, d,
                       int(bool(causal)), float(scale),
                       ATTN_F32 if o.dtype == torch.float32 else ATTN_BF16, _stream_ptr(stream))
    _check(st, "attn_fwd")


def attn_fwd_masked(q, k, v, o, lse, causal: bool, scale: float, window_left: int = 0, alibi=None,
                    bias=None, stream=None) -> None:
    """attn_fwd with an additive bias: a left window, per-head ALiBi slopes
    (CUDA float32 [Hq]) and/or a dense bf16 bias broadcastable to
    [B, Hq, Nq, Nk] (its last two dimensions contiguous)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    _need(lse, torch.float32, "lse")
    if o.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("o must be bfloat16 or float32")
    _need(o, o.dtype, "o")
    B, Hq, Nq, d = q.shape
    _, Hkv, Nk, _ = k.shape
    if tuple(o.shape) != (B, Hq, Nq, d) or tuple(lse.shape) != (B, Hq, Nq) or v.shape != k.shape:
        raise ValueError("shape mismatch between q, k, v, o, lse")
    m = _mask_struct(Hq, B, Nq, Nk, window_left, alibi, bias)
    st = _lib.attn_fwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nk, d,
                              int(bool(causal)), float(scale), ctypes.byref(m),
                              ATTN_F32 if o.dtype == torch.float32 else ATTN_BF16, _stream_ptr(stream))
    _check(st, "attn_fwd_masked")


def attn_prefill_paged_workspace_size(num_seqs: int) -> int:
    return int(_lib.attn_prefill_paged_workspace_size(int(num_seqs)))


def attn_prefill_paged(q, kcache, vcache, block_table, cu_seqlens_q, seqlens_k, o, lse, causal: bool,
                       scale: float, window_left: int = 0, workspace=None, stream=None) -> None:
    """Chunked prefill against a paged KV cache; shapes as in include/attn.h.
    ``workspace``: CUDA uint8 tensor of attn_prefill_paged_workspace_size(S)
    bytes (allocated here when None)."""
    import torch
    _need(q, torch.bfloat16, "q")
    _need(kcache, torch.bfloat16, "kcache")
    _need(vcache, torch.bfloat16, "vcache")
    _need(block_table, torch.int32, "block_table")
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q")
    _need(seqlens_k, torch.int32, "seqlens_k")
    _need(lse, torch.float32, "lse")
    if o.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("o must be bfloat16 or float32")
    _need(o, o.dtype, "o")
    total_q, Hq, d = q.shape
    P, page_size, Hkv, dk = kcache.shape
    S = seqlens_k.numel()
    if dk != d or vcache.shape != kcache.shape or cu_seqlens_q.numel() != S + 1 or block_table.dim() != 2 \
            or block_table.shape[0] != S or tuple(o.shape) != (total_q, Hq, d) or tuple(lse.shape) != (total_q, Hq):
        raise ValueError("paged prefill shape mismatch")
    need = attn_prefill_paged_workspace_size(S)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    st = _lib.attn_prefill_paged(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(block_table), _ptr(cu_seqlens_q),
                                 _ptr(seqlens_k), _ptr(o), _ptr(lse), S, total_q, Hq, Hkv, d, page_size, P,
                                 block_table.shape[1], int(bool(causal)), int(window_left), float(scale),
                                 _ptr(workspace), workspace.numel(),
                                 ATTN_F32 if o.dtype == torch.float32 else ATTN_BF16, _stream_ptr(stream))
    _check(st, "attn_prefill_paged")


def attn_bwd_workspace_size(B: int, Hq: int, Nq: int, d: int) -> int:
    return int(_lib.attn_bwd_workspace_size(int(B), int(Hq), int(Nq), int(d)))


def _mask_struct(Hq: int, B: int, Nq: int, Nk: int, window_left: int, alibi, bias):
    import torch
    m = AttnMask(int(window_left), None, None, 0, 0)
    if alibi is not None:
        _need(alibi, torch.float32, "alibi")
        if alibi.numel() != Hq:
            raise ValueError("alibi must hold Hq slopes")
        m.alibi_slopes = alibi.data_ptr()
    if bias is not None:
        if bias.dtype != torch.bfloat16 or not bias.is_cuda or bias.dim() != 4:
            raise TypeError("bias must be a 4-D CUDA bfloat16 tensor")
        if tuple(bias.shape[2:]) != (Nq, Nk) or (Nk > 1 and bias.stride(3) != 1) or \
                (Nq > 1 and bias.stride(2) != Nk):
            raise ValueError("bias must end in contiguous [Nq, Nk]")
        m.bias = bias.data_ptr()
        m.bias_stride_b = bias.stride(0) if bias.shape[0] == B else 0
        m.bias_stride_h = bias.stride(1) if bias.shape[1] == Hq else 0
    return m


def attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, causal: bool, scale: float, workspace=None, stream=None,
             window_left: int = 0, alibi=None, bias=None) -> None:
    """Backward of attn_fwd (or, with window_left / alibi / bias, of
    attn_fwd_masked with the same bias): dq [B,Hq,Nq,d], dk, dv [B,Hkv,Nk,d]
    (all bf16 or all f32) from q, k, v, the forward's o and lse, and the
    upstream dout."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _need(t, torch.bfloat16, n)
    _need(lse, torch.float32, "lse")
    gd = dq.dtype
    if gd not in (torch.bfloat16, torch.float32) or dk.dtype != gd or dv.dtype != gd:
        raise TypeError("dq, dk, dv must all be bfloat16 or all float32")
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _need(t, gd, n)
    B, Hq, Nq, d = q.shape
    _, Hkv, Nk, _ = k.shape
    if (v.shape != k.shape or o.shape != q.shape or dout.shape != q.shape or tuple(lse.shape) != (B, Hq, Nq)
            or dq.shape != q.shape or dk.shape != k.shape or dv.shape != k.shape):
        raise ValueError("backward shape mismatch")
    need = attn_bwd_workspace_size(B, Hq, Nq, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    gdt = ATTN_F32 if gd == torch.float32 else ATTN_BF16
    if window_left or alibi is not None or bias is not None:
        m = _mask_struct(Hq, B, Nq, Nk, window_left, alibi, bias)
        st = _lib.attn_bwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                                  _ptr(dv), B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), float(scale),
                                  ctypes.byref(m), gdt, _ptr(workspace), workspace.numel(), _stream_ptr(stream))
        _check(st, "attn_bwd_masked")
        return
    st = _lib.attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                       B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), float(scale), gdt, _ptr(workspace),
                       workspace.numel(), _stream_ptr(stream))
    _check(st, "attn_bwd")


def attn_probe_dram_latency(chain, hops: int, out_ns, stream=None) -> None:
    """chain: CUDA int32 tensor (a cycle of indices, see include/attn.h);
    out_ns: CUDA int64 tensor of 2 elements."""
    import torch
    _need(chain, torch.int32, "chain")
    _need(out_ns, torch.int64, "out_ns")
    _check(_lib.attn_probe_dram_latency(_ptr(chain), chain.numel(), int(hops), _ptr(out_ns), _stream_ptr(stream)),
           "attn_probe_dram_latency")


def attn_decode_workspace_size(num_seqs: int, Hq: int, Hkv: int, d: int, max_seqlen: int) -> int:
    return int(_lib.attn_decode_workspace_size(num_seqs, Hq, Hkv, d, max_seqlen))


def attn_decode_paged(q, kcache, vcache, block_table, seqlens, o, lse, max_seqlen: int,
                      scale: float, workspace, stream=None) -> None:
    """Paged decode; shapes as in include/attn.h.  ``workspace`` is a CUDA uint8
    tensor of at least attn_decode_workspace_size(...) bytes (or None when that
    size is 0)."""
    import torch
    _need(q, torch.bfloat16, "q")
    _need(kcache, torch.bfloat16, "kcache")
    _need(vcache, torch.bfloat16, "vcache")
    _need(block_table, torch.int32, "block_table")
    _need(seqlens, torch.int32, "seqlens")
    _need(lse, torch.float32, "lse")
    _need(o, o.dtype, "o")
    S, Hq, d = q.shape
    P, page, Hkv, _ = kcache.shape
    ws_bytes = 0
    if workspace is not None:
        ws_bytes = workspace.numel() * workspace.element_size()
    st = _lib.attn_decode_paged(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(block_table), _ptr(seqlens),
                                _ptr(o), _ptr(lse), S, Hq, Hkv, d, page, P, block_table.shape[1],
                                int(max_seqlen), float(scale), _ptr(workspace), ws_bytes,
                                ATTN_F32 if o.dtype == torch.float32 else ATTN_BF16,
                                _stream_ptr(stream))
    _check(st, "attn_decode_paged")


def attn_decode_paged_static(q, kcache, vcache, block_table, seqlens, o, lse, max_seqlen: int,
                             scale: float, stream=None) -> None:
    """attn_decode_paged without a workspace: the library's built-in scratch
    array holds the split partials, so nothing is allocated for the call.

    For callers that cannot allocate device memory themselves (all of it owned
    by a framework's fixed pool, or a loop where an allocation's implicit device
    synchronisation is not acceptable).  Calls that can overlap on the GPU
    share the one array and must be ordered on one stream; the first call on a
    device looks up the array's address and should come before any stream
    capture.  Workloads whose split partials exceed STATIC_SCRATCH_BYTES raise
    AttnError (status ATTN_ERR_WORKSPACE).
    """
    import torch
    _need(q, torch.bfloat16, "q")
    _need(kcache, torch.bfloat16, "kcache")
    _need(vcache, torch.bfloat16, "vcache")
    _need(block_table, torch.int32, "block_table")
    _need(seqlens, torch.int32, "seqlens")
    _need(lse, torch.float32, "lse")
    _need(o, o.dtype, "o")
    S, Hq, d = q.shape
    P, page, Hkv, _ = kcache.shape
    st = _lib.attn_decode_paged_static(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(block_table),
                                       _ptr(seqlens), _ptr(o), _ptr(lse), S, Hq, Hkv, d, page, P,
                                       block_table.shape[1], int(max_seqlen), float(scale),
                                       ATTN_F32 if o.dtype == torch.float32 else ATTN_BF16,
                                       _stream_ptr(stream))
    _check(st, "attn_decode_paged_static")


def attn_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Launch the failure-detection self-test (a wait that must time out)."""
    _check(_lib.attn_selftest_wait_timeout(int(limit_us), _stream_ptr(stream)),
           "attn_selftest_wait_timeout")


def attn_get_device_status(stream=None) -> int:
    return int(_lib.attn_get_device_status(_stream_ptr(stream)))
