"""Multi-process (gloo, world_size 2, CPU) checks of the N>1 paths.

* bench.py's whole-job aggregation: max over ranks of the timed region and
  value = world * steps * floor / max time.
* The one real exchange step of the attention path when a sequence's keys are
  sharded over ranks: each rank computes its shard's partial (O_r, LSE_r); the
  partials are all-gathered and merged with the online-softmax monoid (the
  merge reading of "online softmax as a monoid", Tang abstract).  The merged
  result must equal the unsharded oracle.  The merge is not a sum, so an
  all-reduce of O would be wrong; the test shows that too.
"""
from __future__ import annotations

import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, fn, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            init_method=f"tcp://127.0.0.1:{port}")
    try:
        q.put((rank, fn(rank, world)))
    except Exception as e:  # pragma: no cover - surfaced in the parent
        q.put((rank, e))
    finally:
        dist.destroy_process_group()


def run_ranks(fn, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, fn, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = {}
    for _ in range(world):
        r, v = q.get(timeout=120)
        out[r] = v
    for p in procs:
        p.join(timeout=60)
    for r, v in out.items():
        if isinstance(v, Exception):
            raise v
    return out


def _bench_aggregation(rank, world):
    import bench
    t = bench.max_over_ranks(1.0 + rank, world)
    return t, bench.aggregate_value(0.5, 10, t, world)


def test_bench_aggregation_takes_the_slowest_rank():
    out = run_ranks(_bench_aggregation)
    for r in range(2):
        t, v = out[r]
        assert t == 2.0
        assert v == pytest.approx(2 * 10 * 0.5 / 2.0)


def _sharded_decode(rank, world):
    import oracle
    from oracle import monoid
    from attention_online_softmax_gb300 import inputs
    x = inputs.prefill_inputs(1, 8, 2, 1, 1000, 64, seed=77, causal=False)
    # rank r owns keys [r*N/world, (r+1)*N/world)
    n = x.k.shape[2]
    lo, hi = rank * n // world, (rank + 1) * n // world
    o, l, _ = oracle.attention(x.q, x.k[:, :, lo:hi].contiguous(), x.v[:, :, lo:hi].contiguous(),
                               False, x.scale)
    part = torch.cat([torch.from_numpy(o.reshape(8, 64)),
                      torch.from_numpy(l.reshape(8, 1))], dim=1)
    gathered = [torch.empty_like(part) for _ in range(world)]
    dist.all_gather(gathered, part)
    merged_o, merged_l = [], []
    for h in range(8):
        st = monoid.identity(64)
        for g in gathered:
            st = monoid.merge(st, monoid.from_output(g[h, :64].numpy(), float(g[h, 64])))
        oo, ll = monoid.finalize(st)
        merged_o.append(oo)
        merged_l.append(ll)
    summed = part.clone()
    dist.all_reduce(summed)  # the wrong exchange: a plain sum of outputs
    full_o, full_l, _ = oracle.attention(x.q, x.k, x.v, False, x.scale)
    return (np.abs(np.array(merged_o) - full_o.reshape(8, 64)).max(),
            np.abs(np.array(merged_l) - full_l.reshape(8)).max(),
            np.abs(summed[:, :64].numpy() - full_o.reshape(8, 64)).max())


def test_kv_sharded_partials_merge_to_the_unsharded_result():
    out = run_ranks(_sharded_decode)
    for r in range(2):
        do, dl, dsum = out[r]
        assert do <= 1e-12 and dl <= 1e-12
        assert dsum > 1e-3
