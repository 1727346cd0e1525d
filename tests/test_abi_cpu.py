"""C ABI checks that need no GPU: the library loads, exports every declared
symbol, and rejects bad arguments before touching the device.

Only argument combinations that are rejected before any CUDA call are passed
with fake (never dereferenced) pointers.
"""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from attention_online_softmax_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")

OK, INVALID, UNSUPPORTED, MISALIGNED, WORKSPACE, LAUNCH, TIMEOUT, BOUNDS, NO_DEVICE = range(9)
FAKE = 0x10000      # 16-byte aligned, never dereferenced
ODD = 0x10008       # 8-byte aligned only


@pytest.fixture(scope="module")
def abi():
    build.build()
    from attention_online_softmax_gb300 import abi as mod
    return mod


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)))


def test_header_declares_the_documented_entry_points():
    syms = declared_symbols()
    for name in ("attn_fwd", "attn_decode_paged", "attn_decode_workspace_size",
                 "attn_get_device_status", "attn_status_string"):
        assert name in syms


PAGE_TITLES = ("Compilers and Kernels", "Tang: a compiler that derives GPU kernels and bounds how fast they can run",
               "Don't Write Kernels, Derive Them")


def declaration_comments():
    """(name, the comment block that documents it) for every ATTN_API declaration."""
    text = open(HEADER).read()
    out = []
    for m in re.finditer(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text):
        start = text.rfind("/*", 0, m.start())
        end = text.find("*/", start)
        assert 0 <= start < end < m.start(), m.group(1)
        out.append((m.group(1), " ".join(text[start:end].replace("*", " ").split())))
    return out


def test_every_declaration_cites_its_passage_or_says_it_has_none():
    decls = declaration_comments()
    assert len(decls) == len(declared_symbols())
    for name, comment in decls:
        cited = re.search(r'Source: "([^"]+)"', comment)
        if cited:
            assert cited.group(1) in PAGE_TITLES, (name, cited.group(1))
        else:
            assert "no counterpart" in comment, name
    cites = dict(decls)
    for name in ("attn_fwd", "attn_decode_paged", "attn_decode_workspace_size", "attn_fwd_masked",
                 "attn_prefill_paged", "attn_bwd"):
        assert "Source:" in cites[name], name


def test_fwd_kernel_name_follows_the_dispatch(abi):
    # Names only; no launch.  d = 256 never takes two query tiles per unit.
    assert abi.attn_fwd_kernel_name(1, 16, 16384, 256) == "prefill_fwd_kernel<256,1,5,0,0>"
    assert abi.attn_fwd_kernel_name(1, 2, 128, 64).startswith("prefill_fwd_kernel<64,1,")
    assert abi.attn_fwd_kernel_name(2, 32, 4096, 128).startswith("prefill_fwd_kernel<128,2,")
    assert abi.attn_fwd_kernel_name(1, 2, 128, 96) == ""


def test_library_exports_every_declared_symbol(abi):
    lib = ctypes.CDLL(build.LIB)
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert set(declared_symbols()) == set(abi.EXPORTS)
    assert abi.attn_abi_version() == 1


def test_status_strings(abi):
    assert abi.attn_status_string(OK) == "ok"
    names = {abi.attn_status_string(s) for s in range(9)}
    assert len(names) == 9
    assert abi.attn_status_string(99) == "unknown status"


def fwd(abi, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, Hq=2, Hkv=2, Nq=128, Nk=128, d=64,
        causal=0, scale=0.125, dt=0):
    return abi.lib().attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, scale, dt, None)


def test_fwd_rejects_bad_arguments_before_any_launch(abi):
    before = abi.attn_launch_count()
    assert fwd(abi, d=96) == UNSUPPORTED
    assert fwd(abi, d=32) == UNSUPPORTED
    assert fwd(abi, Hq=3, Hkv=2) == INVALID
    assert fwd(abi, Hkv=0) == INVALID
    assert fwd(abi, B=-1) == INVALID
    assert fwd(abi, Nq=-4) == INVALID
    assert fwd(abi, scale=float("nan")) == INVALID
    assert fwd(abi, scale=float("inf")) == INVALID
    assert fwd(abi, scale=0.0) == INVALID
    assert fwd(abi, scale=-0.125) == INVALID
    assert fwd(abi, dt=7) == INVALID
    assert fwd(abi, q=ODD) == MISALIGNED
    assert fwd(abi, o=0) == MISALIGNED
    assert fwd(abi, lse=ODD) == MISALIGNED
    assert fwd(abi, k=0) == MISALIGNED
    # empty outputs are a no-op, with any pointers
    assert fwd(abi, Nq=0, q=0, o=0, lse=0) == OK
    assert fwd(abi, B=0, q=0) == OK
    assert abi.attn_launch_count() == before


def test_fwd_without_device_reports_no_device(abi):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; valid arguments would launch")
    assert fwd(abi) in (NO_DEVICE, UNSUPPORTED)


def dec(abi, num_seqs=4, Hq=32, Hkv=8, d=128, page=16, pages=100, max_pages=32, max_len=512,
        ws=FAKE, ws_bytes=1 << 40, scale=0.088, dt=0, q=FAKE, bt=FAKE, sl=FAKE):
    return abi.lib().attn_decode_paged(q, FAKE, FAKE, bt, sl, FAKE, FAKE, num_seqs, Hq, Hkv, d, page,
                                       pages, max_pages, max_len, scale, ws, ws_bytes, dt, None)


def test_decode_rejects_bad_arguments(abi):
    before = abi.attn_launch_count()
    assert dec(abi, page=8) == UNSUPPORTED
    assert dec(abi, page=48) == UNSUPPORTED
    assert dec(abi, page=256) == UNSUPPORTED
    assert dec(abi, d=80) == UNSUPPORTED
    assert dec(abi, Hq=128, Hkv=4) == UNSUPPORTED     # group of 32
    assert dec(abi, Hq=24, Hkv=8) == UNSUPPORTED      # group of 3
    assert dec(abi, Hq=30, Hkv=8) == INVALID
    assert dec(abi, max_len=513, max_pages=32) == INVALID  # beyond the block table
    assert dec(abi, pages=0) == INVALID
    assert dec(abi, num_seqs=-1) == INVALID
    assert dec(abi, scale=float("nan")) == INVALID
    assert dec(abi, scale=-1.0) == INVALID
    assert dec(abi, bt=ODD) == MISALIGNED
    assert dec(abi, sl=0) == MISALIGNED
    need = abi.attn_decode_workspace_size(4, 32, 8, 128, 512)
    assert need > 0
    assert dec(abi, ws_bytes=need - 1) == WORKSPACE
    assert dec(abi, ws=0) == WORKSPACE
    assert dec(abi, num_seqs=0, q=0) == OK
    assert abi.attn_launch_count() == before


def test_decode_workspace_size_is_a_pure_plan(abi):
    ws = abi.attn_decode_workspace_size
    up = lambda n: (n + 255) // 256 * 256

    def expect(S, Hq, splits, d):
        # split partials: d + 1 floats per sequence, split and query head
        return up(S * splits * Hq * (d + 1) * 4)
    # 64 sequences x 8 kv heads: one 8-head group per CTA, 256-token chunks,
    # ceil(8192 / 256) = 32 splits.
    assert ws(64, 32, 8, 128, 8192) == expect(64, 32, 32, 128)
    # a sequence that fits one chunk needs no partials
    assert ws(4096, 32, 8, 128, 256) == 0
    assert ws(1, 32, 8, 128, 0) == 0
    # few sequences: smaller chunks to fill the GPU, more splits
    assert ws(1, 8, 8, 128, 4096) == expect(1, 8, 64, 128)
    # a group of 16 query heads: two warps per kv head, 4 kv heads per CTA
    assert ws(64, 64, 4, 128, 8192) == expect(64, 64, 32, 128)
    assert ws(4, 30, 8, 128, 512) == 0          # invalid -> 0
    assert ws(4, 32, 8, 96, 512) == 0
    assert ws(4, 128, 4, 128, 512) == 0         # group of 32
    assert ws(64, 32, 8, 128, 8192) == ws(64, 32, 8, 128, 8192)


def test_decode_kernel_name_follows_the_plan(abi):
    combine = " + decode_combine_kernel"
    assert abi.attn_decode_kernel_name(64, 32, 8, 128, 8192) == "decode_split_kernel<128,4,1>" + combine
    assert abi.attn_decode_kernel_name(8, 64, 4, 64, 1000) == "decode_split_kernel<64,8,2>" + combine
    assert abi.attn_decode_kernel_name(8, 8, 8, 256, 1000) == "decode_split_kernel<256,1,1>" + combine
    assert abi.attn_decode_kernel_name(4096, 32, 8, 128, 256) == "decode_split_kernel<128,4,1>"
    assert abi.attn_decode_kernel_name(8, 24, 8, 128, 1000) == ""


def test_bwd_workspace_size(abi):
    # D per query row (f32) and the f32 dQ accumulator [B, Hq, Nq, d], each
    # rounded up to 256 bytes.
    ws = abi.attn_bwd_workspace_size
    up = lambda n: (n + 255) // 256 * 256
    for B, Hq, Nq in ((2, 32, 4096), (1, 3, 77), (1, 1, 1)):
        rows = B * Hq * Nq
        for d in (64, 128, 256):
            assert ws(B, Hq, Nq, d) == up(rows * 4) + up(rows * d * 4)
    for bad in ((1, 2, 64, 32), (1, 2, 64, 96), (1, 0, 64, 128), (-1, 2, 64, 128)):
        assert ws(*bad) == 0


def test_paged_prefill_workspace_size(abi):
    # Unit prefix sums (num_seqs + 1 int32) and the dispatch order (num_seqs
    # int32), each rounded up to 256 bytes.
    ws = abi.attn_prefill_paged_workspace_size
    up = lambda n: (n + 255) // 256 * 256
    for n in (0, 1, 16, 63, 64, 1000, 5000):
        assert ws(n) == up((n + 1) * 4) + up(n * 4)
    assert ws(-1) == 0
