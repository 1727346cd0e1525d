"""The allocation-free paged decode entry point (attn_decode_paged_static).

Some callers cannot allocate device memory for a workspace: their device
memory is all owned by a host framework's fixed pool, or they run in a loop
where an allocation (which may synchronise the device) is not acceptable.
attn_decode_paged_static serves them from a scratch array built into the
library.  These tests call it through the C ABI and check that it returns what
attn_decode_paged (caller-provided workspace) returns -- bit for bit, since
both run the same deterministic kernels on the same inputs, so a partial
overwrite of the shared array cannot hide behind a tolerance -- on two calls
in a row with different inputs (the shared array keeps the previous call's
contents), and that a workload too large for the array is refused without a
launch.

This file is named so that pytest collects it last.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from attention_online_softmax_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def abi():
    from attention_online_softmax_gb300 import build
    build.build()
    from attention_online_softmax_gb300 import abi as mod
    return mod


def device_inputs(d_in, dev):
    return (d_in.q.to(dev), d_in.kcache.to(dev), d_in.vcache.to(dev), d_in.block_table.to(dev),
            d_in.seqlens.to(dev))


def both_paths(abi, d_in):
    dev = torch.device("cuda")
    q, kc, vc, bt, sl = device_inputs(d_in, dev)
    S, Hq, d = q.shape
    Hkv = kc.shape[2]
    need = abi.attn_decode_workspace_size(S, Hq, Hkv, d, d_in.max_seqlen)
    assert 0 < need <= abi.STATIC_SCRATCH_BYTES  # the static path really uses its scratch
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    o_ref = torch.full((S, Hq, d), float("nan"), dtype=torch.bfloat16, device=dev)
    l_ref = torch.full((S, Hq), float("nan"), dtype=torch.float32, device=dev)
    abi.attn_decode_paged(q, kc, vc, bt, sl, o_ref, l_ref, d_in.max_seqlen, d_in.scale, ws)
    o = torch.full_like(o_ref, float("nan"))
    l = torch.full_like(l_ref, float("nan"))
    abi.attn_decode_paged_static(q, kc, vc, bt, sl, o, l, d_in.max_seqlen, d_in.scale)
    torch.cuda.synchronize()
    assert abi.attn_get_device_status() == 0
    return (o.float().cpu().numpy(), l.cpu().numpy(), o_ref.float().cpu().numpy(),
            l_ref.cpu().numpy())


def test_static_scratch_matches_workspace_path_on_consecutive_calls(abi):
    cases = [
        inputs.decode_inputs(24, 32, 8, 128, 1, 3000, num_pages=4800, page_size=16, seed=31,
                             max_pages_per_seq=188),
        inputs.decode_inputs(9, 16, 2, 128, 700, 5000, num_pages=3000, page_size=16, seed=32,
                             max_pages_per_seq=313),
    ]
    for d_in in cases:  # two calls in a row; the second sees the first's leftovers
        o, l, o_ref, l_ref = both_paths(abi, d_in)
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
        assert np.array_equal(o, o_ref)
        assert np.array_equal(l, l_ref)


def test_static_scratch_refuses_workloads_larger_than_the_array(abi):
    # 4096 sequences of up to 8192 tokens: far more split partials than the array holds.
    need = abi.attn_decode_workspace_size(4096, 32, 8, 128, 8192)
    assert need > abi.STATIC_SCRATCH_BYTES
    before = abi.attn_launch_count()
    # Null pointers: were the size check ever to stop refusing this, the call
    # would still return ATTN_ERR_MISALIGNED before any launch.
    st = abi.lib().attn_decode_paged_static(None, None, None, None, None, None, None, 4096, 32, 8, 128, 16,
                                            40000, 512, 8192, 0.088, 0, None)
    assert st == 4  # ATTN_ERR_WORKSPACE, before any launch
    assert abi.attn_launch_count() == before
