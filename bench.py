#!/usr/bin/env python3
"""Benchmark of the fused-attention hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  * prefill: attn_fwd on the long causal MHA workload (B=2, H=32, Nq=Nk=4096,
    d=128, bf16, seed 2), and
  * paged decode: attn_decode_paged on 64 sequences, Hq=32 over Hkv=8, d=128,
    lengths uniform in [512, 8192] (seed 4), 16-token pages in a 40000-page pool.

Metric: the step's roofline floor (prefill FLOPs at the measured dense-bf16
peak, decode bytes at the measured HBM bandwidth; T >= max(F/P, Q/B) for each
kernel) divided by the measured step time, summed over GPUs.  At N=1 this is
the fraction of roofline the step reaches.  Inputs are resident in HBM; L2 is
flushed (256 MiB write) before every timed step.  The same metric is also
measured end to end through the C ABI from pinned host buffers ("e2e").

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from attention_online_softmax_gb300 import configs, inputs, roofline  # noqa: E402

METRIC = "attention prefill TFLOP/s & decode HBM GB/s, each as fraction of roofline"
UNIT = "fraction of roofline (step floor time / step time, summed over GPUs)"
WORKLOAD = ("prefill causal MHA B2 H32 N4096 d128 bf16 + paged GQA decode 64 seqs Hq32 Hkv8 d128 "
            "len U[512,8192] 16-token pages in a 40000-page pool")
PROFILE_DIR = os.path.join(ROOT, "profiles")
_CSRC = os.path.join(ROOT, "attention_online_softmax_gb300", "csrc")
# The sources that define each profiled kernel: its own header, the shared PTX
# helpers and the launch code that sets its stages and scheduling.
KERNEL_SOURCES = {
    "prefill_fwd_c3": [os.path.join(_CSRC, f) for f in ("ptx.cuh", "prefill_fwd.cuh", "attn_api.cu")],
    "decode_c5": [os.path.join(_CSRC, f) for f in ("ptx.cuh", "decode.cuh", "attn_api.cu")],
}


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES[kernel]:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_from_profiles(kernel: str) -> float | None:
    """Per-launch DRAM bytes recorded in profiles/traffic.txt for this kernel's
    source hash (lines: `<kernel> <source-hash> <bytes>`); None when the kernel
    changed since the capture."""
    path = os.path.join(PROFILE_DIR, "traffic.txt")
    want = kernel_source_hash(kernel)
    try:
        for line in open(path):
            parts = line.split()
            if len(parts) == 3 and parts[0] == kernel and parts[1] == want:
                return float(parts[2])
    except OSError:
        pass
    return None


# ---------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(floor_s: float, steps: int, total_max_s: float, world: int) -> float:
    """Whole-job value: every rank runs `steps` steps of the same workload
    (weak scaling, no collective on the data path); the job's time is the
    slowest rank's, so value = world * steps * floor / max-over-ranks time."""
    return world * steps * floor_s / total_max_s


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", self.gpu], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.file.name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def gpu_index_for(local_rank: int) -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


# ---------------------------------------------------------------- workloads
def make_decode_inputs():
    c = configs.DECODE
    return inputs.decode_inputs(c.num_seqs, c.Hq, c.Hkv, c.d, c.len_lo, c.len_hi, c.num_pages,
                                c.page_size, c.seed)


def make_prefill_inputs(c=configs.LONG):
    return inputs.prefill_inputs(c.B, c.Hq, c.Hkv, c.Nq, c.Nk, c.d, c.seed, c.causal,
                                 k_scale=c.k_scale)


def make_mask_inputs(c):
    """ALiBi slopes and dense bias of an additive-bias workload (None when unused)."""
    slopes = inputs.alibi_slopes(c.Hq) if c.alibi else None
    bias = None
    if c.bias is not None:
        shape = (c.B if c.bias == "full" else 1, c.Hq, c.Nq, c.Nk)
        bias = inputs.bias_inputs(shape, seed=c.seed + 100)
    return slopes, bias


def floors(peaks, pre_flops, pre_bytes, dec_flops, dec_bytes):
    f_pre = roofline.time_floor_s(pre_flops, pre_bytes, peaks)
    f_dec = roofline.time_floor_s(dec_flops, dec_bytes, peaks)
    return f_pre, f_dec


# ---------------------------------------------------------------- CPU oracle sample
def oracle_sample(peaks, xp, xd, target_s: float, threads: int = 0):
    """Time the oracle on a bounded, seeded sample of the step's workload.

    Sample: the same fraction f of prefill query rows (seeded, spread over all
    heads) and of decode sequences; f is calibrated so the run takes about
    target_s.  Returns (floor_time_of_sample, seconds, threads, description).
    """
    import numpy as np
    import oracle

    P, Dc = configs.LONG, configs.DECODE
    total_rows = P.B * P.Hq * P.Nq
    g = torch.Generator().manual_seed(1234)
    order = torch.randperm(total_rows, generator=g)
    seq_order = torch.randperm(Dc.num_seqs, generator=g)

    def work_of(n_rows, n_seqs):
        rows = order[:n_rows]
        i = (rows % P.Nq).double()
        allowed = torch.clamp(i + 1 + (P.Nk - P.Nq), 0, P.Nk) if P.causal else torch.full_like(i, P.Nk)
        flops = float(4.0 * allowed.sum().item() * P.d)
        seqs = seq_order[:n_seqs]
        lens = [int(xd.seqlens[s]) for s in seqs.tolist()]
        dbytes = roofline.decode_bytes(lens, Dc.Hq, Dc.Hkv, Dc.d, Dc.page_size) if lens else 0
        dflops = roofline.decode_flops(lens, Dc.Hq, Dc.d)
        return (flops / (peaks.bf16_tflops * 1e12)
                + roofline.time_floor_s(dflops, dbytes, peaks)), rows, seqs

    def run(n_rows, n_seqs):
        _, rows, seqs = work_of(n_rows, n_seqs)
        t0 = time.perf_counter()
        _, _, th1 = oracle.attention(xp.q, xp.k, xp.v, P.causal, xp.scale, rows=rows.numpy(),
                                     threads=threads)
        th2 = th1
        if n_seqs:
            _, _, th2 = oracle.decode_paged(xd.q, xd.kcache, xd.vcache, xd.block_table, xd.seqlens,
                                            xd.scale, seqs=seqs.numpy(), threads=threads)
        return time.perf_counter() - t0, max(th1, th2)

    frac = 1.0 / 512
    t, th = run(max(1, int(total_rows * frac)), max(1, int(round(Dc.num_seqs * frac))))
    frac = min(1.0, frac * target_s / max(t, 1e-3))
    n_rows = max(1, int(total_rows * frac))
    n_seqs = max(1, int(round(Dc.num_seqs * frac)))
    floor, _, _ = work_of(n_rows, n_seqs)
    t, th = run(n_rows, n_seqs)
    desc = (f"{n_rows} of {total_rows} prefill query rows (seeded) and {n_seqs} of {Dc.num_seqs} "
            f"decode sequences (all heads): fraction {frac:.4f} of one step")
    return floor, t, th, desc, (n_rows, n_seqs)


# ---------------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    if rank != 0:
        return 0
    peaks = roofline.load_peaks()
    xp = make_prefill_inputs()
    xd = make_decode_inputs()
    floor, t, th, desc, sizes = oracle_sample(peaks, xp, xd, target_s=2.0)
    import oracle
    P = configs.LONG
    g = torch.Generator().manual_seed(1234)
    rows = torch.randperm(P.B * P.Hq * P.Nq, generator=g)[: sizes[0]].numpy()
    seqs = torch.randperm(configs.DECODE.num_seqs, generator=g)[: sizes[1]].numpy()

    def one():
        t0 = time.perf_counter()
        oracle.attention(xp.q, xp.k, xp.v, P.causal, xp.scale, rows=rows)
        oracle.decode_paged(xd.q, xd.kcache, xd.vcache, xd.block_table, xd.seqlens, xd.scale, seqs=seqs)
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        one()
    times = [one() for _ in range(args.steps)]
    total = sum(times)
    value = floor * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 inputs)",
        "config": {"workload": WORKLOAD, "sample": desc, "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": th, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm
def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the per-config table")
    ap.add_argument("--profile", choices=["prefill", "prefill_d256", "tiny", "block", "decode", "bwd", "bwd_d256", "chunked",
                                          "alibi"],
                    default=None,
                    help="run one kernel of the step a few times (for an ncu capture) and exit")
    args = ap.parse_args(argv)
    rank, world, local = dist_env()
    if args.profile:
        return profile_one(args.profile)

    if args.impl == "reference":
        dist_init(world, "gloo")
        return run_reference(args, rank, world)

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    if local == 0:
        from attention_online_softmax_gb300 import build
        build.build()
    barrier(world)
    from attention_online_softmax_gb300 import abi

    peaks = roofline.load_peaks()
    P, Dc = configs.LONG, configs.DECODE
    xp = make_prefill_inputs()
    xd = make_decode_inputs()
    pre_flops = roofline.prefill_flops(P.B, P.Hq, P.Nq, P.Nk, P.d, P.causal)
    pre_bytes = roofline.prefill_bytes(P.B, P.Hq, P.Hkv, P.Nq, P.Nk, P.d)
    lens = xd.seqlens.tolist()
    dec_bytes = roofline.decode_bytes(lens, Dc.Hq, Dc.Hkv, Dc.d, Dc.page_size)
    dec_flops = roofline.decode_flops(lens, Dc.Hq, Dc.d)
    f_pre, f_dec = floors(peaks, pre_flops, pre_bytes, dec_flops, dec_bytes)

    # device buffers
    q, k, v = xp.q.to(dev), xp.k.to(dev), xp.v.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    dq = xd.q.to(dev)
    kc, vc = xd.kcache.to(dev), xd.vcache.to(dev)
    bt, sl = xd.block_table.to(dev), xd.seqlens.to(dev)
    do = torch.empty_like(dq)
    dlse = torch.empty(dq.shape[:2], dtype=torch.float32, device=dev)
    ws_bytes = abi.attn_decode_workspace_size(Dc.num_seqs, Dc.Hq, Dc.Hkv, Dc.d, xd.max_seqlen)
    ws = torch.empty(max(16, ws_bytes), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def prefill():
        abi.attn_fwd(q, k, v, o, lse, P.causal, xp.scale, stream)

    def decode():
        abi.attn_decode_paged(dq, kc, vc, bt, sl, do, dlse, xd.max_seqlen, xd.scale, ws, stream)

    for _ in range(max(3, args.warmup)):
        prefill()
        decode()
    torch.cuda.synchronize()
    if abi.attn_get_device_status() != 0:
        raise SystemExit("device status error after warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(gpu_index_for(local))
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    launches0 = abi.attn_launch_count()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        prefill()
        ev[i][1].record(stream)
        decode()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    launches = abi.attn_launch_count() - launches0
    clocks = sampler.stop()
    t_pre = [ev[i][0].elapsed_time(ev[i][1]) * 1e-3 for i in range(args.steps)]
    t_dec = [ev[i][1].elapsed_time(ev[i][2]) * 1e-3 for i in range(args.steps)]
    total = sum(a + b for a, b in zip(t_pre, t_dec))
    total_max = max_over_ranks(total, world, dev)
    value = aggregate_value(f_pre + f_dec, args.steps, total_max, world)
    if abi.attn_get_device_status() != 0:
        raise SystemExit("device status error in the timed region")

    mean_pre = statistics.fmean(t_pre)
    mean_dec = statistics.fmean(t_dec)
    pre_tflops = pre_flops / mean_pre / 1e12
    dec_gbs = dec_bytes / mean_dec / 1e9

    # ---- end to end through the C ABI from pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(abi, xp, xd, dev, stream, min(args.steps, 5), f_pre + f_dec, world)

    extra = None
    if not args.no_extra and rank == 0:
        extra = per_config_table(abi, dev, stream, peaks, with_cpu=not args.no_cpu_baseline)

    # Decode time floor: traffic at the measured bandwidth plus the launches
    # and one DRAM round trip the split/combine stage cannot avoid.
    launch_s, dram_s = launch_and_latency_floor(dev, stream, abi)
    dec_kernels = 2 if ws_bytes > 0 else 1  # split kernel (+ combine when sequences span chunks)
    dec_floor = dec_bytes / (peaks.hbm_gbs * 1e9) + dec_kernels * launch_s + dram_s

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        floor, t, th, desc, _ = oracle_sample(peaks, xp, xd, target_s=12.0)
        cpu = {"value": floor / t, "unit": UNIT, "cores": th, "kind": "oracle", "sample": desc,
               "seconds": t}

    if rank == 0:
        peak_src = "of measured" if peaks.source == "measured" else "of fallback"
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": 1e3 * total_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 inputs, NaN-filled unused cache pages)",
            "config": {"workload": WORKLOAD, "l2": "flushed before every timed step (256 MiB write)",
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "peaks": peak_src},
            "prefill": {"tflops": pre_tflops, "frac": pre_tflops * 1e12 / (peaks.bf16_tflops * 1e12),
                        "ms": mean_pre * 1e3, "floor_ms": f_pre * 1e3},
            "decode": {"gbs": dec_gbs, "frac": dec_gbs / peaks.hbm_gbs, "ms": mean_dec * 1e3,
                       "floor_ms": f_dec * 1e3, "bytes": dec_bytes,
                       "time_floor": {"ms": dec_floor * 1e3, "traffic_ms": f_dec * 1e3,
                                      "launch_us": launch_s * 1e6, "kernels": dec_kernels,
                                      "dram_latency_us": dram_s * 1e6,
                                      "measured_over_floor": mean_dec / dec_floor}},
            "roofline": {"bound": "tensor", "kernel": abi.attn_fwd_kernel_name(P.B, P.Hq, P.Nq, P.d),
                         "achieved": pre_tflops, "peak": peaks.bf16_tflops, "unit": "TFLOP/s",
                         "frac": pre_tflops / peaks.bf16_tflops, "peak_source": peak_src,
                         "traffic": traffic_from_profiles("prefill_fwd_c3"),
                         "algorithmic": {"flops": pre_flops, "bytes": pre_bytes}},
            "roofline_decode": {"bound": "hbm",
                                "kernel": abi.attn_decode_kernel_name(Dc.num_seqs, Dc.Hq, Dc.Hkv, Dc.d, xd.max_seqlen),
                                "achieved": dec_gbs, "peak": peaks.hbm_gbs, "unit": "GB/s",
                                "frac": dec_gbs / peaks.hbm_gbs, "peak_source": peak_src,
                                "traffic": traffic_from_profiles("decode_c5")},
            "gpu_launches": launches,
            "clocks": clocks,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "per_config": extra,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def profile_one(which: str, launches: int = 3) -> int:
    """A few launches of one kernel on its bench workload, nothing else timed."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from attention_online_softmax_gb300 import build
    build.build()
    from attention_online_softmax_gb300 import abi
    if which.startswith("prefill") or which in ("bwd", "bwd_d256", "tiny", "block"):
        c = {"prefill_d256": configs.GQA256, "bwd_d256": configs.GQA256, "tiny": configs.TINY,
             "block": configs.BLOCK}.get(which, configs.LONG)
        x = make_prefill_inputs(c)
        q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        if which.startswith("bwd"):
            # The backward of a long causal workload (its forward once first).
            abi.attn_fwd(q, k, v, o, lse, c.causal, x.scale)
            g = torch.Generator().manual_seed(c.seed + 50)
            dout = torch.randn(q.shape, generator=g).to(torch.bfloat16).to(dev)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            ws = torch.empty(abi.attn_bwd_workspace_size(c.B, c.Hq, c.Nq, c.d), dtype=torch.uint8, device=dev)
            for _ in range(launches):
                abi.attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, c.causal, x.scale, workspace=ws)
        else:
            for _ in range(launches):
                abi.attn_fwd(q, k, v, o, lse, c.causal, x.scale)
    elif which == "alibi":
        # The ALiBi + dense-bias workload: its forward, then its backward.
        c = configs.ALIBI_BIAS
        x = make_prefill_inputs(c)
        q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        slopes, bias = make_mask_inputs(c)
        kw = dict(window_left=c.window, alibi=slopes.to(dev), bias=bias.to(dev))
        for _ in range(launches):
            abi.attn_fwd_masked(q, k, v, o, lse, c.causal, x.scale, **kw)
        g = torch.Generator().manual_seed(c.seed + 50)
        dout = torch.randn(q.shape, generator=g).to(torch.bfloat16).to(dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(abi.attn_bwd_workspace_size(c.B, c.Hq, c.Nq, c.d), dtype=torch.uint8, device=dev)
        for _ in range(launches):
            abi.attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, c.causal, x.scale, workspace=ws, **kw)
    elif which == "chunked":
        c = configs.CHUNKED
        q_lens, k_lens = configs.chunked_lengths(c)
        x = inputs.paged_prefill_inputs(q_lens, k_lens, c.Hq, c.Hkv, c.d, num_pages=c.num_pages,
                                        page_size=c.page_size, seed=c.seed)
        q = x.q.to(dev)
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
        args = (q, x.kcache.to(dev), x.vcache.to(dev), x.block_table.to(dev), x.cu_seqlens_q.to(dev),
                x.seqlens_k.to(dev), o, lse, True, x.scale)
        ws = torch.empty(max(16, abi.attn_prefill_paged_workspace_size(c.num_seqs)), dtype=torch.uint8, device=dev)
        for _ in range(launches):
            abi.attn_prefill_paged(*args, workspace=ws)
    else:
        Dc = configs.DECODE
        xd = make_decode_inputs()
        dq, kc, vc = xd.q.to(dev), xd.kcache.to(dev), xd.vcache.to(dev)
        bt, sl = xd.block_table.to(dev), xd.seqlens.to(dev)
        do = torch.empty_like(dq)
        dlse = torch.empty(dq.shape[:2], dtype=torch.float32, device=dev)
        ws = torch.empty(max(16, abi.attn_decode_workspace_size(Dc.num_seqs, Dc.Hq, Dc.Hkv, Dc.d,
                                                                xd.max_seqlen)),
                         dtype=torch.uint8, device=dev)
        for _ in range(launches):
            abi.attn_decode_paged(dq, kc, vc, bt, sl, do, dlse, xd.max_seqlen, xd.scale, ws)
    torch.cuda.synchronize()
    st = abi.attn_get_device_status()
    print(json.dumps({"profile": which, "launches": abi.attn_launch_count(), "status": st}))
    return 0 if st == 0 else 1


def launch_and_latency_floor(dev, stream, abi=None, reps: int = 200):
    """Measured costs a GEMV-class stage cannot avoid beyond its traffic.

    launch_s: the GPU-side interval between dependent one-element kernels
    replayed from a CUDA graph (the cost each additional kernel in a chain
    adds, without host launch overhead); dram_s: one DRAM round
    trip, from a single thread chasing dependent loads through a cycle of
    128-byte lines in a buffer larger than L2 (flushed first), the elapsed
    time divided by the hops (`attn_probe_dram_latency`).  Used for the decode
    time floor: traffic at the measured HBM bandwidth + launches * launch_s +
    dram_s ("Tang: a compiler that derives GPU kernels ...": the time floor of
    a GEMV-class stage).
    """
    # GPU-side cost of one more kernel in a chain: `reps` one-element kernels
    # captured in a CUDA graph (no host launch overhead), replayed and timed.
    x = torch.zeros(1, device=dev)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for _ in range(20):
            x.add_(1)
    torch.cuda.current_stream(dev).wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(reps):
            x.add_(1)
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    graph.replay()
    e1.record()
    torch.cuda.synchronize()
    launch_s = e0.elapsed_time(e1) * 1e-3 / reps
    del graph
    if abi is None:
        return launch_s, 0.0
    # A random cycle through 2M lines of 128 bytes (256 MiB): entry 32*a holds 32*next(a).
    lines = 1 << 21
    g = torch.Generator().manual_seed(1234)
    perm = torch.randperm(lines, generator=g).to(dev)
    chain = torch.zeros(lines * 32, dtype=torch.int32, device=dev)
    chain[perm * 32] = (torch.roll(perm, -1) * 32).to(torch.int32)
    # Line 0 lies on the cycle, so the chase may start at index 0.
    out = torch.zeros(2, dtype=torch.int64, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    hops = 2000
    ns = []
    for _ in range(5):
        flush.zero_()
        abi.attn_probe_dram_latency(chain, hops, out, stream)
        torch.cuda.synchronize()
        ns.append(int(out[0].item()) / hops)
    del chain, flush, perm
    return launch_s, statistics.median(ns) * 1e-9


def measure_e2e(abi, xp, xd, dev, stream, steps, floor_s, world):
    """Same step from pinned host memory: H2D of every input, both calls, D2H of O and LSE."""
    P, Dc = configs.LONG, configs.DECODE
    host_in = [t.pin_memory() for t in (xp.q, xp.k, xp.v, xd.q, xd.kcache, xd.vcache,
                                        xd.block_table, xd.seqlens)]
    dev_in = [torch.empty_like(t, device=dev) for t in host_in]
    o = torch.empty_like(dev_in[0])
    lse = torch.empty(xp.q.shape[:3], dtype=torch.float32, device=dev)
    do = torch.empty_like(dev_in[3])
    dlse = torch.empty(xd.q.shape[:2], dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, abi.attn_decode_workspace_size(Dc.num_seqs, Dc.Hq, Dc.Hkv, Dc.d,
                                                            xd.max_seqlen)),
                     dtype=torch.uint8, device=dev)
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse, do, dlse)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)

    def step():
        for d_, h_ in zip(dev_in, host_in):
            d_.copy_(h_, non_blocking=True)
        q, k, v, dq, kc, vc, bt, sl = dev_in
        abi.attn_fwd(q, k, v, o, lse, P.causal, xp.scale, stream)
        abi.attn_decode_paged(dq, kc, vc, bt, sl, do, dlse, xd.max_seqlen, xd.scale, ws, stream)
        for h_, d_ in zip(host_out, (o, lse, do, dlse)):
            h_.copy_(d_, non_blocking=True)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    t = max_over_ranks(e0.elapsed_time(e1) * 1e-3, world, dev)
    return {"value": world * steps * floor_s / t, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": 1e3 * t / steps, "steps": steps}


def back_to_back_us(make_call, set_bytes: int, calls: int = 20, reps: int = 10) -> float:
    """Per-call time of a small workload issued back to back: CUDA graphs of
    `calls` calls, each call on its own copy of the inputs, the copies cycled
    so that a copy is used again only after more than 256 MiB of other inputs
    (more than L2) have been touched: every call starts from a cold L2 without
    a flush kernel between calls.  The events bracket a whole graph, so the
    launch latency of one graph is spread over `calls` calls.

    make_call(i) -> a zero-argument callable on input copy i (it allocates the
    copy)."""
    nsets = max(2, -(-(256 << 20) // max(1, set_bytes)) + 1)
    ngraphs = -(-nsets // calls)
    fns = [make_call(i) for i in range(nsets)]
    for f in fns[: min(nsets, 3)]:
        f()
    torch.cuda.synchronize()
    graphs = []
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for g in range(ngraphs):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=side):
                for i in range(calls):
                    fns[(g * calls + i) % nsets]()
            graphs.append(gr)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for gr in graphs:
        gr.replay()
    torch.cuda.synchronize()
    ts = []
    for r in range(reps):
        for gr in graphs:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            gr.replay()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e-3 / calls)
    return statistics.median(ts) * 1e6


def gpu_median(call, stream, flush, reps: int, graph: bool = True):
    """Median, p10, p90 seconds of `call` on the device (L2 flushed before each rep).

    With `graph`, the call is captured once into a CUDA graph and each rep
    replays it, so the events bracket the kernels alone: an eager call from
    Python can leave the GPU idle while the host prepares the launch, which
    for a kernel of a few microseconds would be most of what the events see.
    """
    # `call` launches on torch's current stream (it must not name a stream:
    # under capture the current stream is the capturing one).
    for _ in range(3):
        call()
    run = call
    if graph:
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                call()
        stream.wait_stream(side)
        g.replay()
        torch.cuda.synchronize()
        run = g.replay
    ts = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e-3)
    ts.sort()
    return statistics.median(ts), ts[len(ts) // 10], ts[(9 * len(ts)) // 10]


# ---------------------------------------------------------------- CPU oracle per workload
# The oracle (f64, C with OpenMP over rows) timed on the host cores beside each
# workload's GPU time: a baseline, not the target.  Small workloads run whole;
# large ones on a seeded sample of query rows calibrated to about `target_s`,
# extrapolated to the whole workload by allowed (query, key) pairs (the
# oracle's work per row is proportional to the keys the row sees).
CPU_TARGET_S = 1.5


def _row_keys(rows, Nq: int, Nk: int, causal: bool, window: int = 0):
    import numpy as np
    i = np.asarray(rows, dtype=np.int64) % Nq
    diag = Nk - Nq
    hi = np.minimum(Nk - 1, i + diag) if causal else np.full(i.shape, Nk - 1)
    lo = np.maximum(0, i + diag - window + 1) if window > 0 else np.zeros(i.shape, dtype=np.int64)
    return np.clip(hi - lo + 1, 0, None)


def _calibrated(run, total_rows: int, seed: int, first: int = 64, target_s: float = CPU_TARGET_S):
    """run(rows) -> (seconds, threads) on a seeded sample sized to ~target_s."""
    g = torch.Generator().manual_seed(seed)
    order = torch.randperm(total_rows, generator=g).numpy()
    n = min(total_rows, first)
    t, th = run(order[:n])
    if n < total_rows and t < target_s:
        n = min(total_rows, max(n + 1, int(n * target_s / max(t, 1e-4))))
        t, th = run(order[:n])
    return order[:n], t, th


def cpu_prefill(c, x):
    import numpy as np
    import oracle
    total = c.B * c.Hq * c.Nq
    masked = bool(c.window or c.alibi or c.bias is not None)
    slopes, bias, strides = None, None, (0, 0)
    if masked:
        slopes, bias = make_mask_inputs(c)
        if bias is not None:
            strides = (bias.stride(0) if bias.shape[0] == c.B else 0, bias.stride(1))

    def run(rows):
        t0 = time.perf_counter()
        if masked:
            _, _, th = oracle.attention_masked(x.q, x.k, x.v, c.causal, x.scale, window_left=c.window,
                                               alibi=slopes, bias=bias, bias_strides=strides, rows=rows)
        else:
            _, _, th = oracle.attention(x.q, x.k, x.v, c.causal, x.scale, rows=rows)
        return time.perf_counter() - t0, th

    rows, t, th = _calibrated(run, total, seed=c.seed + 900)
    full_pairs = c.B * c.Hq * roofline.allowed_pairs(c.Nq, c.Nk, c.causal, c.window)
    sample_pairs = int(_row_keys(rows, c.Nq, c.Nk, c.causal, c.window).sum())
    out = {"kind": "oracle", "cores": th, "sample_rows": int(len(rows)), "total_rows": total,
           "seconds": t, "rows_per_s": len(rows) / t}
    if len(rows) == total:
        out["full_s"] = t
    else:
        out["extrapolated_full_s"] = t * full_pairs / max(sample_pairs, 1)
        out["extrapolation"] = "sample time x (all allowed pairs / sampled rows' allowed pairs)"
    if c is configs.TINY:
        t0 = time.perf_counter()
        _, _, th1 = oracle.attention(x.q, x.k, x.v, c.causal, x.scale, threads=1)
        out["full_s_1_thread"] = time.perf_counter() - t0
        out["threads_1"] = th1
    return out


def cpu_decode(xd):
    import oracle
    t0 = time.perf_counter()
    _, _, th = oracle.decode_paged(xd.q, xd.kcache, xd.vcache, xd.block_table, xd.seqlens, xd.scale)
    t = time.perf_counter() - t0
    return {"kind": "oracle", "cores": th, "full_s": t, "seconds": t,
            "sample": "every sequence and head"}


def cpu_chunked(c, x, q_lens, k_lens):
    import numpy as np
    import oracle
    total = sum(q_lens) * c.Hq
    # allowed keys of each packed (token, head) row: token i of a chunk sees
    # keys 0 .. i + k_len - q_len (causal).
    keys = np.concatenate([np.arange(q) + (k - q) + 1 for q, k in zip(q_lens, k_lens)])

    def run(rows):
        t0 = time.perf_counter()
        _, _, th = oracle.prefill_paged(x.q, x.kcache, x.vcache, x.block_table, x.cu_seqlens_q, x.seqlens_k,
                                        True, x.scale, rows=rows)
        return time.perf_counter() - t0, th

    rows, t, th = _calibrated(run, total, seed=c.seed + 900)
    full_pairs = int(keys.sum()) * c.Hq
    sample_pairs = int(keys[np.asarray(rows) // c.Hq].sum())
    return {"kind": "oracle", "cores": th, "sample_rows": int(len(rows)), "total_rows": total, "seconds": t,
            "rows_per_s": len(rows) / t, "extrapolated_full_s": t * full_pairs / max(sample_pairs, 1),
            "extrapolation": "sample time x (all allowed pairs / sampled rows' allowed pairs)"}


def cpu_bwd(c, x, dout):
    import oracle
    # One query head with its kv head.  For causal Nq == Nk only the first
    # n0 rows are run: that prefix is the same computation for its rows (a
    # row sees only keys up to itself).  Extrapolated to the workload by
    # allowed (query, key) pairs.
    n0 = min(c.Nq, 4096 if c.d <= 128 else 2048) if (c.causal and c.Nq == c.Nk) else c.Nq
    nk0 = n0 if (c.causal and c.Nq == c.Nk) else c.Nk
    sl = (slice(0, 1), slice(0, 1), slice(0, n0))
    slk = (slice(0, 1), slice(0, 1), slice(0, nk0))
    t0 = time.perf_counter()
    _, _, _, th = oracle.attention_bwd(x.q[sl].contiguous(), x.k[slk].contiguous(), x.v[slk].contiguous(),
                                       dout[sl].contiguous(), c.causal, x.scale)
    t = time.perf_counter() - t0

    def pairs(nq, nk):
        return nq * (nq + 1) / 2 if (c.causal and nq == nk) else nq * nk
    full = t * c.B * c.Hq * pairs(c.Nq, c.Nk) / pairs(n0, nk0)
    sample = "one (batch, query head) slice" + (f", its first {n0} rows" if n0 < c.Nq else "")
    return {"kind": "oracle", "cores": th, "seconds": t, "sample": sample,
            "extrapolated_full_s": full, "extrapolation": "sample time x (all allowed pairs / sampled pairs)"}


def cpu_bwd_masked(c, x, dout, slopes, bias):
    import oracle
    # One (batch, head) slice (MHA: every head costs the same allowed pairs).
    sl = (slice(0, 1), slice(0, 1))
    bsl = None if bias is None else bias[sl].contiguous()
    t0 = time.perf_counter()
    _, _, _, th = oracle.attention_masked_bwd(
        x.q[sl].contiguous(), x.k[sl].contiguous(), x.v[sl].contiguous(), dout[sl].contiguous(), c.causal,
        x.scale, window_left=c.window, alibi=None if slopes is None else slopes[:1].numpy(), bias=bsl,
        bias_strides=(0, 0))
    t = time.perf_counter() - t0
    return {"kind": "oracle", "cores": th, "seconds": t, "sample": "one (batch, head) slice of the workload",
            "extrapolated_full_s": t * c.B * c.Hq, "extrapolation": "slice time x B*Hq (equal heads)"}


def _row(t, p10, p90, fl, by, peaks, cpu, **extra):
    bound = roofline.bound_rate(fl, by, peaks)
    out = {"us": t * 1e6, "tflops": fl / t / 1e12, "frac_of_peak": fl / t / (peaks.bf16_tflops * 1e12),
           "frac_of_bound": fl / t / bound, "p10_us": p10 * 1e6, "p90_us": p90 * 1e6}
    out.update(extra)
    if cpu is not None:
        full = cpu.get("full_s", cpu.get("extrapolated_full_s"))
        out["cpu"] = cpu
        out["gpu_speedup_over_cpu"] = full / t
    return out


def per_config_table(abi, dev, stream, peaks, reps: int = 30, with_cpu: bool = True):
    """Each workload timed alone (median of reps, L2 flushed before each), with
    the oracle timed beside it on the host cores."""
    out = {}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for c in configs.PREFILL_CONFIGS:
        x = make_prefill_inputs(c)
        q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        fwd = lambda: abi.attn_fwd(q, k, v, o, lse, c.causal, x.scale)  # noqa: E731
        t, p10, p90 = gpu_median(fwd, stream, flush, reps)
        fl = roofline.prefill_flops(c.B, c.Hq, c.Nq, c.Nk, c.d, c.causal)
        by = roofline.prefill_bytes(c.B, c.Hq, c.Hkv, c.Nq, c.Nk, c.d)
        extra = {"kernel": abi.attn_fwd_kernel_name(c.B, c.Hq, c.Nq, c.d), "timing": "CUDA-graph replay"}
        if t < 50e-6:
            # the same call issued eagerly from Python: includes the host's launch latency
            extra["us_eager"] = gpu_median(fwd, stream, flush, reps, graph=False)[0] * 1e6
            # A one-element add timed the same way: the harness's own floor
            # (event, graph launch and kernel start) that a single call pays.
            one = torch.zeros(1, device=dev)
            extra["us_single_call_floor"] = gpu_median(lambda: one.add_(1.0), stream, flush, reps)[0] * 1e6
            # Back to back, every call cold in L2 (inputs cycled through more
            # than L2): the per-call time of a stream of such calls.
            def make_call(i, c=c, x=x):
                qi, ki, vi = (x.q.to(dev), x.k.to(dev), x.v.to(dev)) if i > 0 else (q, k, v)
                oi, li = torch.empty_like(qi), torch.empty(qi.shape[:3], dtype=torch.float32, device=dev)
                return lambda: abi.attn_fwd(qi, ki, vi, oi, li, c.causal, x.scale)
            set_bytes = 4 * q.numel() * 2 + lse.numel() * 4
            extra["us_back_to_back"] = back_to_back_us(make_call, set_bytes)
            extra["back_to_back"] = "20 calls per CUDA graph, inputs cycled through > 256 MiB (cold L2, no flush)"
        out[c.name] = _row(t, p10, p90, fl, by, peaks, cpu_prefill(c, x) if with_cpu else None, **extra)
        del q, k, v, o, lse
    for c in configs.MASKED_CONFIGS:
        x = make_prefill_inputs(c)
        q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        slopes, bias = make_mask_inputs(c)
        slopes = None if slopes is None else slopes.to(dev)
        bias = None if bias is None else bias.to(dev)

        def call():
            abi.attn_fwd_masked(q, k, v, o, lse, c.causal, x.scale, window_left=c.window, alibi=slopes,
                                bias=bias)
        t, p10, p90 = gpu_median(call, stream, flush, reps)
        fl = roofline.masked_flops(c.B, c.Hq, c.Nq, c.Nk, c.d, c.causal, c.window)
        by = roofline.prefill_bytes(c.B, c.Hq, c.Hkv, c.Nq, c.Nk, c.d)
        if bias is not None:
            by += bias.numel() * 2
        out[c.name] = _row(t, p10, p90, fl, by, peaks, cpu_prefill(c, x) if with_cpu else None,
                           flops="4 d per allowed (query, key) pair")
        del q, k, v, o, lse, slopes, bias
    # Backward of the long causal workloads (forward output and LSE as inputs).
    for c in configs.BWD_CONFIGS:
        x = make_prefill_inputs(c)
        q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        abi.attn_fwd(q, k, v, o, lse, c.causal, x.scale, stream)
        g = torch.Generator().manual_seed(c.seed + 50)
        dout_h = torch.randn(x.q.shape, generator=g).to(torch.bfloat16)
        dout = dout_h.to(dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(abi.attn_bwd_workspace_size(c.B, c.Hq, c.Nq, c.d), dtype=torch.uint8, device=dev)
        t, p10, p90 = gpu_median(
            lambda: abi.attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, c.causal, x.scale, workspace=ws),
            stream, flush, reps)
        fl = 2.5 * roofline.prefill_flops(c.B, c.Hq, c.Nq, c.Nk, c.d, c.causal)
        by = roofline.bwd_bytes(c.B, c.Hq, c.Hkv, c.Nq, c.Nk, c.d)
        cpu = cpu_bwd(c, x, dout_h) if with_cpu else None
        out["bwd_" + c.name] = _row(t, p10, p90, fl, by, peaks, cpu,
                                    flops="5 products of 2 N^2 d per head = 2.5x the forward's")
        del q, k, v, o, lse, dout, dq, dk, dv, ws
    # Backward through the additive bias (the masked forward's O and LSE as inputs).
    for c in configs.MASKED_CONFIGS:
        x = make_prefill_inputs(c)
        q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        slopes, bias = make_mask_inputs(c)
        slopes_d = None if slopes is None else slopes.to(dev)
        bias_d = None if bias is None else bias.to(dev)
        kw = dict(window_left=c.window, alibi=slopes_d, bias=bias_d)
        abi.attn_fwd_masked(q, k, v, o, lse, c.causal, x.scale, **kw)
        g = torch.Generator().manual_seed(c.seed + 50)
        dout_h = torch.randn(x.q.shape, generator=g).to(torch.bfloat16)
        dout = dout_h.to(dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(abi.attn_bwd_workspace_size(c.B, c.Hq, c.Nq, c.d), dtype=torch.uint8, device=dev)
        t, p10, p90 = gpu_median(
            lambda: abi.attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, c.causal, x.scale, workspace=ws, **kw),
            stream, flush, reps)
        fl = 2.5 * roofline.masked_flops(c.B, c.Hq, c.Nq, c.Nk, c.d, c.causal, c.window)
        by = roofline.bwd_bytes(c.B, c.Hq, c.Hkv, c.Nq, c.Nk, c.d)
        if bias is not None:
            by += bias.numel() * 2
        cpu = cpu_bwd_masked(c, x, dout_h, slopes, bias) if with_cpu else None
        out["bwd_" + c.name] = _row(t, p10, p90, fl, by, peaks, cpu,
                                    flops="2.5 x (4 d per allowed (query, key) pair)")
        del q, k, v, o, lse, dout, dq, dk, dv, ws, slopes_d, bias_d
    # Chunked prefill against the paged cache.
    c = configs.CHUNKED
    q_lens, k_lens = configs.chunked_lengths(c)
    x = inputs.paged_prefill_inputs(q_lens, k_lens, c.Hq, c.Hkv, c.d, num_pages=c.num_pages,
                                    page_size=c.page_size, seed=c.seed)
    q = x.q.to(dev)
    kc, vc = x.kcache.to(dev), x.vcache.to(dev)
    bt, cu, sk = x.block_table.to(dev), x.cu_seqlens_q.to(dev), x.seqlens_k.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, abi.attn_prefill_paged_workspace_size(c.num_seqs)), dtype=torch.uint8, device=dev)
    t, p10, p90 = gpu_median(
        lambda: abi.attn_prefill_paged(q, kc, vc, bt, cu, sk, o, lse, True, x.scale, workspace=ws),
        stream, flush, reps)
    fl = sum(4.0 * c.Hq * c.d * roofline.allowed_pairs(a, b, True) for a, b in zip(q_lens, k_lens))
    by = roofline.paged_prefill_bytes(q_lens, k_lens, c.Hq, c.Hkv, c.d, c.page_size)
    out[c.name] = _row(t, p10, p90, fl, by, peaks, cpu_chunked(c, x, q_lens, k_lens) if with_cpu else None,
                       flops="4 d per allowed (query, key) pair")
    del q, kc, vc, o, lse, ws
    # Paged decode alone (HBM-bound: reported as GB/s against the copy ceiling).
    Dc = configs.DECODE
    xd = make_decode_inputs()
    dq_, kc, vc = xd.q.to(dev), xd.kcache.to(dev), xd.vcache.to(dev)
    bt, sl = xd.block_table.to(dev), xd.seqlens.to(dev)
    do = torch.empty_like(dq_)
    dlse = torch.empty(dq_.shape[:2], dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, abi.attn_decode_workspace_size(Dc.num_seqs, Dc.Hq, Dc.Hkv, Dc.d, xd.max_seqlen)),
                     dtype=torch.uint8, device=dev)
    t, p10, p90 = gpu_median(
        lambda: abi.attn_decode_paged(dq_, kc, vc, bt, sl, do, dlse, xd.max_seqlen, xd.scale, ws),
        stream, flush, reps)
    by = roofline.decode_bytes(xd.seqlens.tolist(), Dc.Hq, Dc.Hkv, Dc.d, Dc.page_size)
    row = {"us": t * 1e6, "gbs": by / t / 1e9, "frac_of_hbm": by / t / (peaks.hbm_gbs * 1e9),
           "p10_us": p10 * 1e6, "p90_us": p90 * 1e6, "bytes": by}
    if with_cpu:
        row["cpu"] = cpu_decode(xd)
        row["gpu_speedup_over_cpu"] = row["cpu"]["full_s"] / t
    out[Dc.name] = row
    del dq_, kc, vc, bt, sl, do, dlse, ws
    torch.cuda.empty_cache()
    return out


if __name__ == "__main__":
    sys.exit(main())
