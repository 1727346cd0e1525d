"""Failure detection without a GPU fault.

Every pipeline wait in the kernels is bounded: when it runs out it records
ATTN_ERR_TIMEOUT in the device status word and the kernel unwinds and returns.
The self-test kernel makes one such wait run out on purpose (a barrier phase
that can never complete, with a short limit) -- nothing traps, faults or hangs
-- and the context must stay usable afterwards.  Host-side failures (bad
arguments) are covered in test_abi_cpu.py.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from attention_online_softmax_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def abi():
    from attention_online_softmax_gb300 import build
    build.build()
    from attention_online_softmax_gb300 import abi as mod
    return mod


def test_expired_wait_reports_timeout_and_context_survives(abi):
    assert abi.attn_get_device_status() == 0
    t0 = time.perf_counter()
    abi.attn_selftest_wait_timeout(20000)  # 20 ms limit
    assert abi.attn_get_device_status() == 6  # ATTN_ERR_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert 0.015 <= elapsed < 5.0
    assert abi.attn_get_device_status() == 0  # reading cleared it
    # the context still runs real work correctly
    x = inputs.prefill_inputs(1, 2, 2, 200, 200, 64, seed=42, causal=True)
    dev = torch.device("cuda")
    o = torch.empty((1, 2, 200, 64), dtype=torch.float32, device=dev)
    lse = torch.empty((1, 2, 200), dtype=torch.float32, device=dev)
    abi.attn_fwd(x.q.to(dev), x.k.to(dev), x.v.to(dev), o, lse, True, x.scale)
    torch.cuda.synchronize()
    assert abi.attn_get_device_status() == 0
    o_ref, l_ref, _ = oracle.attention(x.q, x.k, x.v, True, x.scale)
    assert np.abs(o.cpu().numpy() - o_ref).max() <= 1e-2
    assert np.abs(lse.cpu().numpy() - l_ref).max() <= 1e-3


def test_selftest_rejects_bad_limits(abi):
    for bad in (0, 2_000_000):
        with pytest.raises(abi.AttnError):
            abi.attn_selftest_wait_timeout(bad)
