#!/usr/bin/env python
"""Benchmark of the per-rank LAGA compute on GB300.

One step = the whole hot path on one batch: laga_fwd (latent LayerNorm,
RoPE, head-shard up-projection, causal attention forward) followed by
laga_bwd (attention backward, up-projection backward, LayerNorm/RoPE
backward) of a 16-head DeepSeek-V3-dim shard at S=16384 (bf16 operands,
fp32 accumulation).  Inputs are seeded synthetic tensors of the workload's
shapes and distributions.

value = attention fwd+bwd algorithmic FLOPs (H*S^2*1152, causal S^2/2
pairs) / the full step time, in TFLOP/s; the step time includes the
up-projection and the norm kernels, so value under-states the attention
kernels' own rate (reported separately as attn_kernels_tflops).

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank computes its own head shard of an N*16-head layer
(no collective on the data path: weak scaling); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LAGA attn fwd+bwd TFLOP/s (V3 dims, 16-head shard, S=16K); % of BF16 peak"
UNIT = "TFLOP/s"
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=2, help="workload configuration (default 2)")
    ap.add_argument("--form", default="laga", choices=["laga", "explicit", "laga_fused"])
    ap.add_argument("--no-block-variant", action="store_true",
                    help="skip the timing of the full attention block beside the main line")
    ap.add_argument("--block-d-model", type=int, default=7168,
                    help="hidden size of the attention block variant (DeepSeek-V3: 7168)")
    ap.add_argument("--no-fused-variant", action="store_true",
                    help="skip the timing of the fused up-projection form beside the main line")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--seq", type=int, default=0,
                    help="override the sequence length (smaller cases for profiling)")
    ap.add_argument("--sweep", action="store_true",
                    help="sequence/head sweep of LAGA and the absorbed form: throughput and "
                         "measured activation memory against the closed form (one JSON line "
                         "per point)")
    ap.add_argument("--sweep-S", default="2048,4096,8192,16384,32768")
    ap.add_argument("--sweep-H", default="8,16,32")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mma-rates", action="store_true",
                    help="tensor-core issue rate per MMA shape and accumulator interleaving "
                         "(laga_diag_mma_rate), one JSON line per case")
    ap.add_argument("--single-stream", action="store_true",
                    help="laga_bwd on the compute stream alone instead of laga_bwd_overlap "
                         "(dQ kernel on a second stream of the caller's)")
    return ap.parse_args()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), float(pk["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="laga_clocks_", suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(rows[0][2]), "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows), "reasons": reasons}


# ----------------------------------------------------------------- ncu traffic
def ncu_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes of one kernel from its committed ncu summary, if
    the summary was taken on the current kernel source (same sha256)."""
    import hashlib
    import re
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    src = re.search(r"source_sha256:\s*([0-9a-f]+)\s+(\S+)", txt)
    if not m or not src:
        return None
    f = os.path.join(ROOT, src.group(2))
    if not os.path.exists(f) or hashlib.sha256(open(f, "rb").read()).hexdigest() != src.group(1):
        return None
    return float(m.group(1))


# ----------------------------------------------------------------- kernels' work
def kernel_work(name: str, S: int, H: int, B: int = 1):
    """(bound, algorithmic units per launch) of each library kernel: FLOPs
    for tensor-core work, DRAM bytes for the HBM-bound kernels."""
    pairs = B * H * S * S / 2.0
    T, R = B * S, B * S * H
    table = {
        "attn_fwd": ("tensor", pairs * (2 * 192 + 2 * 128)),
        # the backward's algorithmic FLOPs, split between its two kernels:
        # S^T, dP^T, dV and dK in the key-stationary one, dQ in the other
        # (whose recomputed S and dP are not counted)
        "attn_bwd_dkdv": ("tensor", pairs * (2 * 192 + 2 * 128 + 2 * 128 + 2 * 192)),
        "attn_bwd_dq": ("tensor", pairs * 2 * 192),
        # the fused form's dK/dV kernel also rebuilds K/V = L W (1x the up-projection)
        "attn_bwd_dkdv_fused": ("tensor", pairs * (2 * 192 + 2 * 128 + 2 * 128 + 2 * 192)
                                + 2.0 * T * 512 * H * 256),
        "upproj": ("tensor", 2.0 * T * 512 * H * 256),
        "upproj_dw": ("tensor", 2.0 * T * 512 * H * 256),
        "upproj_dl": ("tensor", 2.0 * T * 512 * H * 256),
        # HBM-bound: bytes read + written once
        "prep_fwd": ("hbm", T * 576 * 2 + R * 64 * 2 + T * (512 * 2 + 8 + 64 * 2) + R * 64 * 2),
        "bwd_pre": ("hbm", 2 * R * 128 * 2 + R * 4),
        "dq_final": ("hbm", R * 192 * 4 + R * 192 * 2),
        "norm_bwd": ("hbm", T * 512 * 4 + T * 576 * 2 + T * 8 + R * 64 * 4 + T * 576 * 4),
    }
    return table.get(name, ("hbm", None))


def attention_flops(S, H, B=1):
    pairs = B * H * S * S / 2.0
    return pairs * (2 * 192 + 2 * 128), pairs * (6 * 192 + 4 * 128)


# ----------------------------------------------------------------- CPU oracle
def oracle_sample(wl, S_sample: int, heads: int = 1):
    """Time the fp64 oracle's fwd+bwd of `heads` heads of the workload on the
    first S_sample tokens; returns (seconds, attention FLOPs of the sample)."""
    import dataclasses
    import oracle
    from laga_inputs import as_f64, make_inputs
    sub = dataclasses.replace(wl, S=S_sample, H=heads, n_h_total=heads, head_offset=0)
    cpu = make_inputs(sub)
    a = {k: as_f64(v) for k, v in cpu.items()}
    d = oracle.Dims(S=sub.S, H=heads)
    t0 = time.perf_counter()
    _, _, st = oracle.forward(a["q"], a["c"], a["w"], a["gamma"], a["cos"], a["sin"], d)
    oracle.backward(st, a["dO"])
    dt = time.perf_counter() - t0
    f, b = attention_flops(S_sample, heads)
    return dt, f + b


def run_reference(args, rank):
    from laga_inputs import config
    if rank != 0:
        return
    wl = config(args.config)
    S_sample = min(wl.S, 8192)
    times, flops = [], 0.0
    for i in range(args.warmup + args.steps):
        dt, flops = oracle_sample(wl, S_sample)
        if i >= args.warmup:
            times.append(dt)
    sec = sum(times) / len(times)
    value = flops / sec / 1e12
    sample = (f"fp64 NumPy oracle fwd+bwd of 1 head on the first {S_sample} tokens of the "
              f"{wl.name} workload per step")
    cores = os.cpu_count()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "S": wl.S, "H": wl.H, "sample_S": S_sample,
                       "sample_heads": 1},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- ranks
def rank_workload(base, rank: int, world: int):
    """Rank r computes heads [r*H, (r+1)*H) of a world*H-head layer: the
    shards partition the heads, no data-path collective (weak scaling)."""
    import dataclasses
    return dataclasses.replace(base, n_h_total=base.H * world, head_offset=base.H * rank)


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The slowest rank's time (the job's time) on every rank."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- end to end
def end_to_end(args, cpu, dev, stream, step, outs, world, attn_flops):
    """The same metric through the public API with host buffers, as a
    training loop would run it: every step copies its inputs from pinned
    host memory to the device and every output back to pinned host memory,
    all inside the timed region.  Inputs and outputs are double-buffered on
    the device, so the copies of one step overlap the compute of its
    neighbours (host-to-device and device-to-host on their own streams)."""
    import torch
    host_in = {k: v.pin_memory() for k, v in cpu.items()}
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(x.numel() * x.element_size() for x in outs)
    dev_in = [{k: torch.empty_like(v, device=dev) for k, v in cpu.items()} for _ in range(2)]
    dev_out = [outs, [torch.empty_like(x) for x in outs]]
    host_out = [[torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in outs]
                for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(n):
        done = [None, None]                # compute of the step that last used slot
        freed = [None, None]               # device-to-host copy that last read slot
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        start.record(s_in)
        stream.wait_event(start)
        s_out.wait_event(start)
        for i in range(n):
            k = i % 2
            if done[k] is not None:
                s_in.wait_event(done[k])
            with torch.cuda.stream(s_in):
                for name in dev_in[k]:
                    dev_in[k][name].copy_(host_in[name], non_blocking=True)
            landed = torch.cuda.Event()
            landed.record(s_in)
            stream.wait_event(landed)
            if freed[k] is not None:
                stream.wait_event(freed[k])
            step(dev_in[k], dev_out[k])
            done[k] = torch.cuda.Event()
            done[k].record(stream)
            s_out.wait_event(done[k])
            with torch.cuda.stream(s_out):
                for x, hx in zip(dev_out[k], host_out[k]):
                    hx.copy_(x, non_blocking=True)
            freed[k] = torch.cuda.Event()
            freed[k].record(s_out)
        end.record(s_out)
        torch.cuda.synchronize(dev)
        return start.elapsed_time(end) / n

    run(2)                                 # warms the pinned copies and streams
    ms = run(args.e2e_steps)
    return {"value": round(world * attn_flops / (ms * 1e-3) / 1e12, 3), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3),
            "pipelined": "inputs and outputs double-buffered; copies overlap neighbouring steps"}


# ----------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import dataclasses
    import torch
    import torch.distributed as dist
    import sequence_latent_norm_gb300 as pkg
    from laga_inputs import config, make_inputs

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    base = config(args.config, **({"S": args.seq} if args.seq else {}))
    wl = rank_workload(base, rank, world)
    S, H, B = wl.S, wl.H, wl.B

    # CPU baseline first (rank 0, one GPU only): the oracle as it stands.
    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        nh = min(4, base.H)
        dt, fl = oracle_sample(base, base.S, nh)
        cpu_baseline = {"value": fl / dt / 1e12, "unit": UNIT, "cores": os.cpu_count(),
                        "kind": "oracle",
                        "sample": f"fp64 NumPy oracle fwd+bwd of {nh} of the {H} heads over all "
                                  f"{S} tokens ({dt:.1f} s)"}

    cpu = make_inputs(wl)
    t = {k: v.to(dev) for k, v in cpu.items()}
    shard = pkg.Shard(S=S, H=H, n_h_total=wl.n_h_total, head_offset=wl.head_offset, B=B,
                      io_dtype=wl.dtype, form=args.form)
    run = pkg.Laga(shard, device=dev)
    _ = run.ws_bwd
    f32 = torch.float32
    o = torch.empty(B, S, H, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, H, S, dtype=f32, device=dev)
    dq = torch.empty(B, S, H, 192, dtype=torch.bfloat16, device=dev)
    dc = torch.empty(B, S, 576, dtype=f32, device=dev)
    dw = torch.empty(512, H * 256, dtype=f32, device=dev)
    dg = torch.empty(512, dtype=f32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    aux = None if args.single_stream else torch.cuda.Stream(dev)

    launches = [0]

    def step(tt, oo=None):
        o_, lse_, dq_, dc_, dw_, dg_ = oo if oo is not None else (o, lse, dq, dc, dw, dg)
        run.forward(tt["q"], tt["c"], tt["w"], tt["gamma"], tt["cos"], tt["sin"], o_, lse_)
        n = pkg._lib.last_launch_count()
        run.backward(tt["q"], tt["c"], tt["w"], tt["gamma"], tt["cos"], tt["sin"], o_, lse_,
                     tt["dO"], dq_, dc_, dw_, dg_, aux_stream=aux)
        launches[0] = n + pkg._lib.last_launch_count()

    for _ in range(args.warmup):
        step(t)
    torch.cuda.synchronize(dev)
    pkg._lib.sync_check()

    def barrier():
        if world > 1:
            dist.barrier()

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = None
    clocks = ClockSampler(gpu_id)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()                      # L2 flush, outside the timed events
        ev[i][0].record(stream)
        step(t)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    pkg._lib.sync_check()
    # per-kernel times from a second pass of the same steps, with the
    # library's event pairs around every launch (kept out of the timed pass)
    pkg._lib.profile_reset()
    pkg._lib.profile_enable(True)
    for i in range(args.steps):
        flush.zero_()
        step(t)
    torch.cuda.synchronize(dev)
    pkg._lib.profile_enable(False)
    prof = pkg._lib.profile_read()
    pkg._lib.sync_check()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    ms_per_step = total_ms / args.steps
    fwd_f, bwd_f = attention_flops(S, H, B)
    attn_flops = fwd_f + bwd_f
    value = world * attn_flops / (ms_per_step * 1e-3) / 1e12

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(args, cpu, dev, stream, step, [o, lse, dq, dc, dw, dg], world,
                         attn_flops)

    # ---- per-kernel rates and the roofline of the dominant kernel
    peak_tf, peak_gbs, peak_src = measured_peaks()
    kernels = {}
    for name, (ms, n) in prof.items():
        bound, units = kernel_work(name, S, H, B)
        per = ms / n
        ent = {"launches_per_step": n / args.steps, "ms_per_launch": round(per, 4),
               "share": round(ms / sum(v[0] for v in prof.values()), 4)}
        if units is not None:
            rate = units / (per * 1e-3)
            ent["achieved"] = round(rate / 1e12 if bound == "tensor" else rate / 1e9, 2)
            ent["unit"] = "TFLOP/s" if bound == "tensor" else "GB/s"
        kernels[name] = ent
    top = max(prof.items(), key=lambda kv: kv[1][0])[0]
    bound, units = kernel_work(top, S, H, B)
    per_ms = prof[top][0] / prof[top][1]
    if bound == "tensor":
        ach = units / (per_ms * 1e-3) / 1e12
        roof = {"kernel": top, "bound": "tensor", "achieved": round(ach, 2), "peak": peak_tf,
                "unit": "TFLOP/s", "frac": round(ach / peak_tf, 4),
                "peak_source": f"{peak_src} bf16 dense (burst)"}
    else:
        ach = units / (per_ms * 1e-3) / 1e9
        roof = {"kernel": top, "bound": "hbm", "achieved": round(ach, 1), "peak": peak_gbs,
                "unit": "GB/s", "frac": round(ach / peak_gbs, 4),
                "peak_source": f"{peak_src} HBM copy"}
    roof["traffic"] = ncu_traffic(top, base.name)
    # the variants run on the same inputs with the main line's workspaces
    # and outputs released, so that each is timed in the memory state it
    # would have alone
    del run, o, lse, dq, dc, dw, dg
    torch.cuda.empty_cache()
    fused = None
    if args.form == "laga" and world == 1 and not args.no_fused_variant:
        fused = fused_variant(args, wl, t, dev, stream, flush, peak_tf, gpu_id)
    block = None
    if args.form == "laga" and world == 1 and not args.no_block_variant:
        block = block_variant(args, wl, dev, stream, flush, gpu_id)
    attn_ms = sum(prof[k][0] for k in prof if k.startswith("attn")) / args.steps
    up_f = 3 * 2.0 * B * S * 512 * H * 256
    line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": base.name, "B": B, "S": S, "H": H, "n_h_total": wl.n_h_total,
                       "d_nope": 128, "d_rope": 64, "d_v": 128, "d_kv": 512, "form": args.form,
                       "parallelism": f"{world} independent head shards (no data-path collective)",
                       "l2": "flushed between steps by a 512 MB write outside the timed events",
                       "value_definition": "H*S^2*1152 attention FLOPs / full hot-path step time",
                       "backward_call": ("laga_bwd (one stream)" if aux is None else
                                         "laga_bwd_overlap (dQ kernel on a second caller "
                                         "stream)")},
            "pct_of_bf16_peak": round(100 * value / world / peak_tf, 2),
            # the same work counted over the exact S(S+1)/2 causal pairs
            "value_exact_causal_pairs": round(value * (S + 1) / S, 3),
            "attn_kernels_tflops": round(attn_flops / (attn_ms * 1e-3) / 1e12, 2),
            "block_tflops": round((attn_flops + up_f) / (ms_per_step * 1e-3) / 1e12, 2),
            "wall_s_timed": round(t_wall, 3),
            "clocks": clk,
            "e2e": e2e,
            "gpu_launches": launches[0] * args.steps,
            "roofline": roof, "kernels": kernels, "cpu_baseline": cpu_baseline,
            "fused_upproj_variant": fused, "attention_block_variant": block}
    if rank == 0:
        print(json.dumps(line), flush=True)


def fused_variant(args, wl, t, dev, stream, flush, peak_tf, gpu_id=None):
    """The fused up-projection form on the same inputs: step time (fwd +
    bwd, one stream), its dK/dV kernel's rate and the saved-activation
    bytes of both forms."""
    import torch
    import sequence_latent_norm_gb300 as pkg
    S, H, B = wl.S, wl.H, wl.B
    shard = pkg.Shard(S=S, H=H, n_h_total=wl.n_h_total, head_offset=wl.head_offset, B=B,
                      io_dtype=wl.dtype, form="laga_fused")
    run = pkg.Laga(shard, device=dev)
    base_dims = pkg.Shard(S=S, H=H, n_h_total=wl.n_h_total, head_offset=wl.head_offset, B=B,
                          io_dtype=wl.dtype, form="laga").dims()

    def step():
        o, lse = run.forward(t["q"], t["c"], t["w"], t["gamma"], t["cos"], t["sin"])
        run.backward(t["q"], t["c"], t["w"], t["gamma"], t["cos"], t["sin"], o, lse, t["dO"])

    clocks = ClockSampler(gpu_id)
    clocks.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    pkg._lib.sync_check()
    ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    pkg._lib.profile_reset()
    pkg._lib.profile_enable(True)
    for _ in range(args.steps):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    pkg._lib.profile_enable(False)
    prof = pkg._lib.profile_read()
    pkg._lib.sync_check()
    clk = clocks.stop()
    k = "attn_bwd_dkdv_fused"
    per = prof[k][0] / prof[k][1]
    _, units = kernel_work(k, S, H, B)
    fwd_f, bwd_f = attention_flops(S, H, B)
    return {"form": "laga_fused", "ms_per_step": round(ms, 4),
            "value": round((fwd_f + bwd_f) / (ms * 1e-3) / 1e12, 3), "unit": UNIT,
            "dkdv_fused_ms_per_launch": round(per, 4),
            "dkdv_fused_tflops": round(units / (per * 1e-3) / 1e12, 2),
            "dkdv_fused_frac": round(units / (per * 1e-3) / 1e12 / peak_tf, 4),
            "saved_bytes": run.saved_bytes, "saved_bytes_laga": pkg._lib.workspace_bytes(base_dims, pkg._lib.WS_SAVED),
            "fwd_scratch_bytes": run.fwd_bytes, "clocks": clk}


def block_variant(args, wl, dev, stream, flush, gpu_id=None):
    """The full attention block (W_q, W_kv_a, the library's LAGA compute,
    W_o; forward + backward) around the same shard: one rank's block holds
    the shard's heads over the whole sequence, i.e. the per-rank work of a
    sequence-parallel layer with P * H heads at degree P for the three
    projections' head-wise GEMMs.  Returns its step time, tokens/s and the
    rate of all its FLOPs."""
    import torch
    import sequence_latent_norm_gb300 as pkg
    from laga_inputs import make_block_inputs
    from sequence_latent_norm_gb300.block import LagaAttentionBlock
    S, H, B, d = wl.S, wl.H, wl.B, args.block_d_model
    t = {k: v.to(dev) for k, v in make_block_inputs(wl, d).items()}
    blk = LagaAttentionBlock.single(H, S, B=B, device=dev)

    def step():
        blk.forward(t["h"], t["w_q"], t["w_kva"], t["gamma"], t["w_kvb"], t["w_o"], t["cos"],
                    t["sin"])
        blk.backward(t["dy"])

    clocks = ClockSampler(gpu_id)
    clocks.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    pkg._lib.sync_check()
    clk = clocks.stop()
    ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    fwd_f, bwd_f = attention_flops(S, H, B)
    # W_q, W_kv_a and W_o: one GEMM per weight forward, two backward
    proj = 3 * 2.0 * B * S * d * (H * 192 + 576 + H * 128)
    up = 3 * 2.0 * B * S * 512 * H * 256
    return {"workload": f"MLA attention block, {H} heads, S={S}, d_model={d}, B={B}",
            "ms_per_step": round(ms, 4), "tokens_per_s": round(B * S / (ms * 1e-3), 1),
            "tflops_all_gemms_and_attention": round((fwd_f + bwd_f + proj + up) / (ms * 1e-3) / 1e12,
                                                    2),
            "projections": "W_q, W_kv_a, W_o as torch matmuls (cuBLAS), bf16 in and out",
            "clocks": clk}


# ----------------------------------------------------------------- sweep
def run_sweep(args):
    """S x H grid for the LAGA and absorbed forms (DeepSeek-V3 dims, bf16):
    fwd+bwd time, attention TFLOP/s, and the measured peak device memory of a
    forward (saved activations + outputs) against the per-token closed form
    (absorbed: q_absorbed and the latent accumulator, n_h*d_kv each; LAGA:
    per-head K/V, n_h*(d_nope+d_v))."""
    import torch
    import sequence_latent_norm_gb300 as pkg
    from laga_inputs import config, make_inputs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    for S in [int(x) for x in args.sweep_S.split(",")]:
        for H in [int(x) for x in args.sweep_H.split(",")]:
            wl = config(4, S=S, H=H, n_h_total=H)
            cpu = make_inputs(wl)
            t = {k: v.to(dev) for k, v in cpu.items()}
            peak = {}
            for form in ("laga", "absorbed"):
                torch.cuda.synchronize(dev)
                torch.cuda.empty_cache()
                torch.cuda.reset_peak_memory_stats(dev)
                base = torch.cuda.memory_allocated(dev)
                run = pkg.Laga(pkg.Shard(S=S, H=H, form=form), device=dev)
                o, lse = run.forward(t["q"], t["c"], t["w"], t["gamma"], t["cos"], t["sin"])
                torch.cuda.synchronize(dev)
                peak[form] = torch.cuda.max_memory_allocated(dev) - base
                times = []
                for it in range(2):
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    o, lse = run.forward(t["q"], t["c"], t["w"], t["gamma"], t["cos"], t["sin"], o, lse)
                    run.backward(t["q"], t["c"], t["w"], t["gamma"], t["cos"], t["sin"], o, lse, t["dO"])
                    b.record()
                    torch.cuda.synchronize(dev)
                    times.append(a.elapsed_time(b))
                pkg._lib.sync_check()
                ms = times[-1]
                f, bw = attention_flops(S, H)
                line = {"sweep": "config4", "form": form, "S": S, "H": H, "ms_fwd_bwd": round(ms, 3),
                        "attn_tflops": round((f + bw) / (ms * 1e-3) / 1e12, 2),
                        "peak_fwd_bytes": peak[form],
                        "saved_workspace_bytes": run.saved_bytes}
                if form == "absorbed":
                    per_tok = (2 * H * 512 - H * 256) * 2
                    line["measured_gap_bytes"] = peak["absorbed"] - peak["laga"]
                    line["closed_form_gap_bytes"] = S * per_tok
                    line["gap_ratio"] = round(line["measured_gap_bytes"] / line["closed_form_gap_bytes"], 4)
                print(json.dumps(line), flush=True)
                del run, o, lse
                torch.cuda.empty_cache()


# ----------------------------------------------------------------- MMA rates
def run_mma_rates():
    """SM clocks per tcgen05.mma (M=128, K=16, bf16 -> fp32) on every SM, by
    N, operand form and accumulator interleaving; the peak per-SM rate the
    measured bf16 GEMM peak implies is printed beside them."""
    import torch
    import sequence_latent_norm_gb300 as pkg
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    cyc = torch.zeros(n_sm, dtype=torch.int64, device=dev)
    peak_tf, _, src = measured_peaks()
    forms = {0: "ss", 1: "ts", 2: "ss/ts alternating"}
    bgs = {0: "none", 1: "TMEM loads", 2: "shared-memory stores", 3: "TMA bulk copies",
           4: "TMEM stores", 5: "exp + FMA"}
    n_instr = 8160
    cases = []
    for n in (64, 128, 192, 256):
        for op in (0, 1):
            for bmn in (0, 1):
                for bg in (0, 1, 2):
                    cases.append((op | (bmn << 2) | (bg << 3), n, 1, 1))
    for op in (0, 1, 2):
        for n_acc, run in ((2, 1), (2, 4), (3, 1)):
            cases.append((op, 128, n_acc, run))
    for n in (64, 128, 256):
        for op in (0, 1):
            for bg in (0, 1, 3, 4, 5):
                cases.append((op | 4 | (bg << 3) | 64, n, 1, 1))
    # how long one 32-column TMEM load (with its wait) takes while the tensor
    # core streams MMAs into other columns
    for n in (64, 128, 256):
        form = 1 | 4 | (1 << 3) | 64 | 128
        for rep in range(2):
            pkg._lib.diag_mma_rate(form, n, 1, 1, n_instr, n_sm, cyc.data_ptr())
            torch.cuda.synchronize(dev)
        c = cyc.cpu().double()
        print(json.dumps({"tmem_load_latency": {"clk_per_32_column_load": float(c.median()),
                                                "alongside": f"ts N={n} MMAs, N(0,1)-like"}}),
              flush=True)
    # one dependent broadcast 16-byte shared-memory load, with the tensor
    # core idle (a single MMA) and while it streams MMAs of each form
    for op in (0, 1):
        for n, instr in ((128, 48), (128, n_instr), (256, n_instr)):
            form = op | 4 | (6 << 3) | 64 | 128
            for rep in range(2):
                pkg._lib.diag_mma_rate(form, n, 1, 1, instr, n_sm, cyc.data_ptr())
                torch.cuda.synchronize(dev)
            c = cyc.cpu().double()
            print(json.dumps({"smem_broadcast_load_latency": {
                "clk_per_load": float(c.median()),
                "alongside": f"{forms[op]} N={n} MMAs x {instr}"}}), flush=True)
    # one issuing thread against two (lane 0 of two warps, own accumulators)
    for n in (64, 128):
        for op in (0, 1):
            cases.append((op | 4 | 64 | 256, n, 1, 1))
    for form, n, n_acc, run in cases:
        for rep in range(2):           # the first launch warms clocks and caches
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            pkg._lib.diag_mma_rate(form, n, n_acc, run, n_instr, n_sm, cyc.data_ptr())
            b.record()
            torch.cuda.synchronize(dev)
        c = cyc.cpu().double()
        if (c == 0).any():
            raise RuntimeError("laga_diag_mma_rate: a bounded wait gave up")
        clk = float(c.median()) / n_instr
        flop = 2.0 * 128 * n * 16
        # cross-check of the clock count: the launch's FLOPs over its event time
        tflops = n_sm * n_instr * flop / (a.elapsed_time(b) * 1e-3) / 1e12
        print(json.dumps({"mma_rate": {"form": forms[form & 3],
                                       "b_major": "MN" if form & 4 else "K",
                                       "background": bgs[(form >> 3) & 7],
                                       "operands": "N(0,1)-like" if form & 64 else "small",
                                       "issuers": 2 if form & 256 else 1,
                                       "N": n,
                                       "accumulators": n_acc,
                                       "run": run, "clk_per_mma": round(clk, 1),
                                       "flop_per_clk_per_sm": round(flop / clk),
                                       "launch_tflops": round(tflops, 1),
                                       "sms": n_sm, "mmas_per_sm": n_instr}}), flush=True)
    print(json.dumps({"mma_rate_reference": {
        "measured_bf16_peak_tflops": peak_tf, "peak_source": src,
        "flop_per_clk_per_sm_at_2070_mhz": round(peak_tf * 1e12 / (n_sm * 2.07e9))}}), flush=True)


def main():
    args = parse_args()
    if args.mma_rates:
        run_mma_rates()
        return
    if args.sweep:
        run_sweep(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch.distributed as dist
        import torch
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
