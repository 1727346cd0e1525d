"""The DRAM-latency probe behind the decode time floor (attn_probe_dram_latency).

The probe follows idx = chain[idx] from index 0.  On a chain whose cycle is
known, the last index after `hops` hops is fixed, so the test checks the walk
itself (not only that a time came back); an entry pointing outside the chain
must be reported by the kernel's own bounds check (ATTN_ERR_BOUNDS) without
being used as an index.
"""
from __future__ import annotations

import pytest
import torch

pytestmark = pytest.mark.gpu

BOUNDS = 7


@pytest.fixture(scope="module")
def abi():
    from attention_online_softmax_gb300 import build
    build.build()
    from attention_online_softmax_gb300 import abi as mod
    return mod


def cycle_chain(n: int, seed: int):
    """chain[perm[i]] = perm[i + 1]: one cycle through all n entries."""
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(n, generator=g)
    chain = torch.empty(n, dtype=torch.int32)
    chain[perm] = torch.roll(perm, -1).to(torch.int32)
    return chain, perm.tolist()


@pytest.mark.parametrize("n,hops", [(1, 5), (37, 100), (4096, 3000)])
def test_probe_walks_a_known_chain(abi, n, hops):
    chain, perm = cycle_chain(n, seed=n)
    expect = perm[(perm.index(0) + hops) % n]
    dev = torch.device("cuda")
    out = torch.full((2,), -1, dtype=torch.int64, device=dev)
    abi.attn_probe_dram_latency(chain.to(dev), hops, out)
    torch.cuda.synchronize()
    assert abi.attn_get_device_status() == 0
    ns, last = out.cpu().tolist()
    assert last == expect
    assert ns > 0


def test_probe_reports_an_entry_outside_the_chain(abi):
    # 0 -> 3 -> 2 -> 1000 (outside a 4-entry chain): the walk stops at the bad
    # entry, which is never dereferenced.
    chain = torch.tensor([3, 0, 1000, 2], dtype=torch.int32)
    dev = torch.device("cuda")
    out = torch.full((2,), -1, dtype=torch.int64, device=dev)
    abi.attn_probe_dram_latency(chain.to(dev), 10, out)
    torch.cuda.synchronize()
    assert abi.attn_get_device_status() == BOUNDS
    assert out.cpu().tolist() == [0, 1000]
    assert abi.attn_get_device_status() == 0  # reading the status cleared it
