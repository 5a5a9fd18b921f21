#!/usr/bin/env python
"""Throughput of the bounded-activation DiT block forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

A step is one pass of the whole hot path (every block of the workload, plus
the final layer when it has one) over one batch of seeded synthetic tokens
already resident in HBM.  The forward is in place on the residual stream, so
step i+1 runs on step i's output (the work per step does not depend on the
values).  W untimed warm-up steps, then exactly K steps between CUDA events
on the launching stream, bracketed by a barrier and a device synchronize;
the max over ranks is reported.  Inputs are larger than L2 (x alone is
4*T*D bytes, K/V another 4*T*D), so L2 is not flushed between steps.

One JSON line is printed by rank 0.  ``value`` is block-tokens per second
(tokens x blocks per step / step time) summed over ranks.  With N > 1 every
rank runs an independent replica (the path has no exchange step on one GPU;
"scaling": "weak").

``--impl reference`` times the float64 CPU oracle instead, on a bounded
sample of the same workload (see ``cpu_sample``).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "dit4_int8_final_T32768_D3072"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                  "bf16_tflops_sustained": 1700.0}

# kernel kind -> source file(s) whose hash keys the ncu traffic figure
KIND_SOURCE = {"attention": ("attention.cu", "attn_sched.h"), "modln": "modln.cu",
               "final": "final.cu", "gemm_kv": "gemm.cu", "gemm_q": "gemm.cu",
               "gemm_o": "gemm.cu", "gemm_swiglu": "gemm.cu",
               "gemm_down": "gemm.cu"}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--weight-scratch", choices=("on", "off"), default="off",
                    help="int8 blocks: expand each phase's weights to bf16 in a "
                         "scratch ahead of the GEMMs (exact; same result bits) "
                         "instead of converting them in the GEMM main loop")
    ap.add_argument("--no-alt", action="store_true",
                    help="skip the extra int8 weight-scratch measurement")
    ap.add_argument("--mlp-chunk", type=int, default=None,
                    help="override the workload's MLP token chunk (0: all tokens)")
    ap.add_argument("--attn-chunk", type=int, default=None,
                    help="override the workload's attention query slab (0: all tokens)")
    ap.add_argument("--kv-offload", type=int, default=0,
                    help="key block size: keep K/V of all tokens in pinned host memory "
                         "and stream them back in blocks of this many keys (0: resident)")
    ap.add_argument("--lora", type=int, default=0,
                    help="rank of activation-space LoRA adapters on all five "
                         "linears of every block (0: none)")
    ap.add_argument("--qk", choices=("none", "axial"), default="none",
                    help="add the per-head Q/K RMSNorm + rotary embedding "
                         "(axial video angles) to every block")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=256,
                    help="token rows in the oracle's timed sample")
    ap.add_argument("--oracle", choices=("sample", "full"), default="sample",
                    help="--impl reference: time the oracle on a row sample of "
                         "the workload, or on the whole block (every token)")
    ap.add_argument("--cpu-threads", type=int, default=0,
                    help="BLAS threads of the oracle (0: every core of the process)")
    return ap.parse_args(argv)


# ------------------------------------------------------------------ helpers

def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_sha(names):
    """First 16 hex digits of the sha256 of the kernel's source file(s)."""
    h = hashlib.sha256()
    for name in ((names,) if isinstance(names, str) else names):
        with open(os.path.join(ROOT, "memory_bounded_video_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(kind, workload):
    """DRAM bytes per launch from a committed ncu capture, if the kernel's
    source is unchanged since (else None)."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    e = t.get(workload, {}).get(kind)
    if not e or e.get("source_sha") != source_sha(KIND_SOURCE[kind]):
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id=None):
        self.proc = None
        self.path = None
        self.device_id = device_id

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}",
               "--format=csv,noheader,nounits", "-lms", "200"]
        if self.device_id:
            cmd += ["-i", self.device_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append(dict(sm=float(parts[1]), sm_max=float(parts[2]),
                                     power=float(parts[3]),
                                     hw_slowdown=parts[5] == "Active",
                                     hw_thermal=parts[6] == "Active",
                                     sw_thermal=parts[7] == "Active",
                                     sw_power_cap=parts[8] == "Active"))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        pmax = max(r["power"] for r in rows)
        loaded = [r for r in rows if r["power"] >= 0.5 * pmax] or rows
        reasons = sorted({k for r in loaded for k in
                          ("hw_slowdown", "hw_thermal", "sw_thermal",
                           "sw_power_cap") if r[k]})
        names = {"hw_thermal": "hw_thermal_slowdown",
                 "sw_thermal": "sw_thermal_slowdown"}
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
                "sm_max_mhz": max(r["sm_max"] for r in rows),
                "reasons": [names.get(k, k) for k in reasons],
                "samples": len(rows), "power_w_max": pmax}


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank time over all ranks (identity on one rank).  Runs
    on whatever process group is initialised (NCCL on GPUs, gloo in the CPU
    tests)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job throughput of `world` independent replicas: the units all
    ranks processed over the slowest rank's time."""
    return units_per_rank * world / (ms_max / 1e3)


def block_flops(T: int, D: int, F: int) -> int:
    """Algorithmic flops of one block: the Q, K, V projections (6 D^2 per
    token, Q counted once), the O projection (2 D^2), the SwiGLU MLP (6 D F)
    and the two attention contractions (4 T D per query token).  Norms,
    softmax and elementwise work are not counted."""
    return T * (8 * D * D + 6 * D * F) + 4 * T * T * D


def step_stats(ms_list):
    """Median, min and max of per-step milliseconds."""
    return {"median": round(statistics.median(ms_list), 4),
            "min": round(min(ms_list), 4), "max": round(max(ms_list), 4)}


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ oracle (CPU) leg

def cpu_sample(cfg, inp, rows_n, steps=1, warmup=0, qk=None, loras=None):
    """Time the float64 oracle on a bounded sample of the workload.

    Per block: K and V of all T tokens are computed first (untimed set-up, the
    oracle's own projection); the timed sample is the K/V projection of
    `rows_n` token rows plus every other stage of the block for those rows,
    attending to all T keys, plus the final layer on those rows when the
    workload has one.  Throughput = blocks x rows / time."""
    import numpy as np
    from oracle import block as ob

    T, D, H = cfg["T"], cfg["D"], cfg["heads"]
    rows = np.linspace(0, T - 1, rows_n).astype(np.int64)
    x = inp.x.double().numpy()
    blocks = []
    for bw, mod in zip(inp.blocks, inp.mods):
        if bw.int8:
            w = ob.DitWeights(**{k: ob.dequant_int8(v.numpy(), bw.scales[k].numpy())
                                 for k, v in bw.named().items()})
        else:
            w = ob.DitWeights(**{k: v.double().numpy() for k, v in bw.named().items()})
        blocks.append((w, mod.double().numpy()))
    l64 = [None] * len(blocks)
    if loras is not None:
        l64 = [{k: (A.double().numpy(), B.double().numpy(), al)
                for k, (A, B, al) in lo.items()} for lo in loras]
    # set-up: K/V of every token for the first block, by the oracle's own
    # projection; every block's sampled rows attend to that key/value set
    # (the oracle's cost does not depend on the values, and this keeps the
    # untimed set-up to one full projection)
    w0, mod0 = blocks[0]
    a = ob.ln_modulate(x, mod0[0], mod0[1])
    _, wk, wv = w0.q_k_v()
    qk64 = None
    if qk is not None:
        qk64 = {k: (v.double().numpy() if hasattr(v, "double") else v)
                for k, v in qk.items()}
    Dm = cfg["D"]
    kproj = a @ wk.T + ob.lora_delta(a, None if l64[0] is None else l64[0]["qkv"],
                                     slice(Dm, 2 * Dm))
    vproj = a @ wv.T + ob.lora_delta(a, None if l64[0] is None else l64[0]["qkv"],
                                     slice(2 * Dm, 3 * Dm))
    kv = (ob.qk_transform(kproj, H, None if qk64 is None else qk64["k_norm"],
                          None if qk64 is None else qk64["cos"],
                          None if qk64 is None else qk64["sin"]), vproj)
    del a
    kvs = [kv] * len(blocks)
    wf = None
    if inp.wf is not None:
        wf = (ob.dequant_int8(inp.wf.numpy(), inp.wf_scale.numpy())
              if inp.wf_scale is not None else inp.wf.double().numpy())
        mod_f = inp.mod_f.double().numpy()

    def one():
        t0 = time.perf_counter()
        for (w, mod), kv, lo in zip(blocks, kvs, l64):
            a = ob.ln_modulate(x[rows], mod[0], mod[1])
            _, wk, wv = w.q_k_v()
            ad = None if lo is None else lo["qkv"]
            _ = (a @ wk.T + ob.lora_delta(a, ad, slice(Dm, 2 * Dm)),
                 a @ wv.T + ob.lora_delta(a, ad, slice(2 * Dm, 3 * Dm)))
            ob.dit_block_rows(x, w, mod, H, rows, kv=kv, qk=qk64, lora=lo)
        if wf is not None:
            ob.final_layer(x[rows], wf, mod_f)
        return time.perf_counter() - t0

    for _ in range(warmup):
        one()
    times = [one() for _ in range(steps)]
    per_step = sum(times) / len(times)
    value = len(blocks) * rows_n / per_step
    sample = (f"{rows_n} of {T} token rows per block (their K/V projection, "
              f"LN-mod, Q, attention against all {T} keys, O-proj, SwiGLU MLP"
              + (", final layer" if wf is not None else "")
              + (", Q/K RMSNorm + rotary" if qk64 is not None else "")
              + (", LoRA adapters" if loras is not None else "")
              + f") x {len(blocks)} block(s), float64 numpy oracle; K/V of all "
              "tokens precomputed untimed (first block's, reused as every "
              "block's key/value set)")
    return value, per_step, sample, times


def cpu_full(cfg, inp, steps=1, warmup=0):
    """Time the float64 oracle on the whole workload: every block over all T
    tokens (unchunked), plus the final layer when the workload has one.
    Throughput = blocks x T / time."""
    from oracle import block as ob

    H = cfg["heads"]
    x0 = inp.x.double().numpy()
    blocks = []
    for bw, mod in zip(inp.blocks, inp.mods):
        if bw.int8:
            w = ob.DitWeights(**{k: ob.dequant_int8(v.numpy(), bw.scales[k].numpy())
                                 for k, v in bw.named().items()})
        else:
            w = ob.DitWeights(**{k: v.double().numpy() for k, v in bw.named().items()})
        blocks.append((w, mod.double().numpy()))
    wf = None
    if inp.wf is not None:
        wf = (ob.dequant_int8(inp.wf.numpy(), inp.wf_scale.numpy())
              if inp.wf_scale is not None else inp.wf.double().numpy())
        mod_f = inp.mod_f.double().numpy()

    def one():
        t0 = time.perf_counter()
        x = x0
        for w, mod in blocks:
            x = ob.dit_block(x, w, mod, H)
        if wf is not None:
            ob.final_layer(x, wf, mod_f)
        return time.perf_counter() - t0

    for _ in range(warmup):
        one()
    times = [one() for _ in range(steps)]
    per_step = sum(times) / len(times)
    value = len(blocks) * cfg["T"] / per_step
    sample = (f"whole workload: {len(blocks)} block(s) x {cfg['T']} tokens, unchunked"
              + (", final layer" if wf is not None else "")
              + ", float64 numpy oracle")
    return value, per_step, sample, times


# ------------------------------------------------------------------ GPU leg

def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from memory_bounded_video_gb300 import build as dbuild
    from memory_bounded_video_gb300 import ditstream, runner, synth

    cfg = dict(synth.WORKLOADS[args.workload])
    if args.mlp_chunk is not None:
        cfg["mlp_chunk"] = args.mlp_chunk
    if args.attn_chunk is not None:
        cfg["attn_chunk"] = args.attn_chunk
    T, D, H, F = cfg["T"], cfg["D"], cfg["heads"], cfg["F"]
    dev_name = f"cuda:{local_rank}"
    torch.cuda.set_device(local_rank)
    dbuild.build()
    ditstream.load()

    inp = synth.make_workload(args.workload, seed=rank)
    dev = runner.upload(inp, dev_name)
    scratch = cfg["int8"] and args.weight_scratch == "on"
    stack = runner.DitStack(T, D, H, F, cfg["mlp_chunk"], cfg["attn_chunk"],
                            cfg["ffn_slice"], device=dev_name, lora_rank=args.lora,
                            weight_scratch=scratch, kv_offload=args.kv_offload)
    loras = dls = None
    if args.lora:
        loras = [synth.make_lora(D, F, args.lora, seed=100 * rank + i)
                 for i in range(cfg["blocks"])]
        dls = [runner.upload_lora(lo, b) for lo, b in zip(loras, dev.blocks)]
    qk = dqk = None
    if args.qk != "none":
        qk = synth.make_qk(T, D // H, seed=rank, angles=args.qk)
        dqk = runner.upload_qk(qk, dev_name)
    x = dev.x.clone()
    stream = torch.cuda.current_stream()
    mem0 = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()

    def step():
        stack.forward(x, dev, stream, qk=dqk, lora=dls)

    for _ in range(args.warmup):
        step()
    stack.check(stream)
    peak_fwd = torch.cuda.max_memory_allocated() - mem0

    def barrier():
        if world > 1:
            dist.barrier()

    def timed_steps(k, fn):
        """Run fn() k times with a CUDA event on `stream` between steps;
        returns the per-step ms and the total ms (first event to last)."""
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(k + 1)]
        barrier()
        torch.cuda.synchronize()
        ev[0].record(stream)
        for i in range(k):
            fn()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        barrier()
        return ([ev[i].elapsed_time(ev[i + 1]) for i in range(k)],
                ev[0].elapsed_time(ev[k]))

    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local_rank).uuid)
    except Exception:
        uuid = None

    # headline: no per-kernel instrumentation, one event between steps
    clocks = ClockSampler(uuid)
    clocks.start()
    per_step, ms = timed_steps(args.steps, step)
    clk = clocks.stop()
    stack.check(stream)
    ms = max_over_ranks(ms, world, dev_name)

    # second pass of the same steps with every launch bracketed by events:
    # the per-kernel breakdown and the dominant kernel's roofline
    stack.plan.profile_enable(True)
    stack.plan.profile_read()
    per_step_prof, ms_prof = timed_steps(args.steps, step)
    prof = stack.plan.profile_read()
    stack.plan.profile_enable(False)
    stack.check(stream)

    blocks = cfg["blocks"]
    tokens_per_step = blocks * T
    value = replica_throughput(tokens_per_step * args.steps, world, ms)
    ms_per_step = ms / args.steps
    flops_step = blocks * block_flops(T, D, F)
    if args.lora:  # u = x A^T and the u B^T K-steps of the five adapted linears
        flops_step += blocks * T * 2 * args.lora * (9 * D + 3 * F)
    peaks, peak_src = load_peaks()
    tflops = flops_step / (ms_per_step / 1e3) / 1e12
    # the kernels run at the bench's clocks, not at the power-capped clock of
    # the sustained cuBLAS loop: the burst figure is the denominator
    tpeak = peaks["bf16_tflops"]

    # per-kernel breakdown and the dominant kernel's roofline
    kernels = {}
    total_k = sum(v["ms"] for v in prof.values()) or 1.0
    for k, v in prof.items():
        if v["launches"]:
            kernels[k] = dict(launches=v["launches"], ms=round(v["ms"], 4),
                              share=round(v["ms"] / total_k, 4))
            if v["unit"] == "flops":
                kernels[k]["tflops"] = round(v["work"] / (v["ms"] / 1e3) / 1e12, 1)
            else:
                kernels[k]["gbs"] = round(v["work"] / (v["ms"] / 1e3) / 1e9, 1)
    dom = max(prof, key=lambda k: prof[k]["ms"])
    d = prof[dom]
    if d["unit"] == "flops":
        achieved = d["work"] / (d["ms"] / 1e3) / 1e12
        roof = dict(bound="tensor", achieved=round(achieved, 2), peak=tpeak,
                    unit="TFLOP/s", frac=round(achieved / tpeak, 4))
        peak_note = f"bf16_tflops (burst) of {peak_src}"
    else:
        achieved = d["work"] / (d["ms"] / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = dict(bound="hbm", achieved=round(achieved, 1), peak=peak,
                    unit="GB/s", frac=round(achieved / peak, 4))
        peak_note = f"hbm_gbs of {peak_src}"
    roof["traffic"] = traffic_for(dom, args.workload)
    roof["kernel"] = dom
    roof["launch_ms"] = round(d["ms"] / d["launches"], 4)
    roof["work_per_launch"] = d["work"] / d["launches"]
    roof["peak_source"] = peak_note
    roof["timing"] = ("CUDA events around every launch on the launching stream, "
                      "in a second pass of the same steps (the headline pass "
                      "runs without them)")

    line = {
        "metric": "DiT-block tokens/s @32k tokens, % BF16 tensor peak, "
                  "peak activation GiB",
        "value": round(value, 1),
        "unit": "block-tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "step_ms": step_stats(per_step),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 (fp32 accumulate, fp32 residual)",
        "data": "synthetic (seeded N(0,1) tokens, N(0,0.02) weights)",
        "config": {"workload": args.workload, "T": T, "D": D, "heads": H,
                   "head_dim": D // H, "ffn": F, "blocks": blocks,
                   "final_layer": cfg["final"], "int8_weights": cfg["int8"],
                   "mlp_chunk_tokens": cfg["mlp_chunk"],
                   "attn_chunk_tokens": cfg["attn_chunk"],
                   "ffn_slice": cfg["ffn_slice"] or F,
                   "l2": "not flushed: inputs larger than L2 "
                         f"(x {4 * T * D / 2**20:.0f} MiB, K/V "
                         f"{4 * T * D / 2**20:.0f} MiB per block)",
                   "qk_transform": (None if qk is None else
                                    f"q/k rmsnorm + {args.qk} rotary"),
                   "lora_rank": args.lora or None,
                   "kv_offload_key_block": args.kv_offload or None,
                   "int8_weight_scratch_gib": (round(stack.plan.weight_scratch_bytes()
                                                     / 2**30, 4) if scratch else None),
                   "parallelism": f"replicas x{world}"},
        "tflops": round(tflops, 2),
        "tensor_peak_frac": round(tflops / tpeak, 4),
        "tensor_peak_frac_sustained": round(tflops / peaks["bf16_tflops_sustained"], 4),
        "peak_source": f"bf16_tflops (burst) of {peak_src}",
        "peak_activation_gib": round(stack.plan.workspace_bytes() / 2**30, 4),
        "activation_beyond_kv_gib": round(
            (stack.plan.workspace_bytes() - (0 if args.kv_offload else 4 * T * D)) / 2**30, 4),
        "measured_forward_alloc_gib": round(peak_fwd / 2**30, 4),
        "roofline": roof,
        "kernels": kernels,
        "instrumented_pass": {"ms_per_step": round(ms_prof / args.steps, 4),
                              "step_ms": step_stats(per_step_prof),
                              "kernel_ms_per_step": round(total_k / args.steps, 4)},
        "gpu_launches": int(sum(v["launches"] for v in prof.values())),
        "clocks": clk,
    }

    # e2e through the public API with host buffers: every step's tokens come
    # from pinned host memory and its result goes back to pinned host memory
    # (DitStack.forward_host: a copy stream moves step i + 1 in and step
    # i - 1 out while step i computes)
    if not args.no_e2e:
        x_host = inp.x.pin_memory()
        res_shape = (T, 64) if cfg["final"] else (T, D)
        out_host = torch.empty(res_shape, dtype=torch.float32).pin_memory()
        k_e2e = max(20, args.steps)

        def e2e_run(k):
            stack.forward_host([x_host] * k, dev, [out_host] * k, stream,
                               qk=dqk, lora=dls)

        e2e_run(2)
        torch.cuda.synchronize()
        stack.check()
        # the host -> device copy of one step's tokens alone, on a side stream
        cs = torch.cuda.Stream()
        xd = torch.empty_like(dev.x)
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        with torch.cuda.stream(cs):
            c0.record(cs)
            for _ in range(5):
                xd.copy_(x_host, non_blocking=True)
            c1.record(cs)
        torch.cuda.synchronize()
        h2d_ms = c0.elapsed_time(c1) / 5
        del xd
        clocks_e = ClockSampler(uuid)
        clocks_e.start()
        barrier()
        torch.cuda.synchronize()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        e2e_run(k_e2e)
        f1.record(stream)
        torch.cuda.synchronize()
        barrier()
        clk_e = clocks_e.stop()
        stack.check()
        ms_e2e = max_over_ranks(f0.elapsed_time(f1), world, dev_name)
        line["e2e"] = {"value": round(replica_throughput(tokens_per_step * k_e2e, world,
                                                         ms_e2e), 1),
                       "unit": "block-tokens/s",
                       "h2d_bytes_per_step": 4 * T * D,
                       "d2h_bytes_per_step": 4 * res_shape[0] * res_shape[1],
                       "steps": k_e2e,
                       "ms_per_step": round(ms_e2e / k_e2e, 4),
                       "h2d_ms_per_step_alone": round(h2d_ms, 4),
                       "clocks": clk_e,
                       "copies": "pinned host memory; step i+1's input copied in and step "
                                 "i-1's result copied out on a copy stream during step i's "
                                 "kernels (DitStack.forward_host); the first step's copy-in "
                                 "is not overlapped"}

    # int8 workloads: the same plan and inputs with the bf16 weight scratch
    # bound (weights expanded ahead of the GEMMs instead of converted in
    # their main loop; same output bits), timed the same way
    if cfg["int8"] and not scratch and not args.no_alt:
        buf = torch.empty(stack.plan.weight_scratch_bytes(), dtype=torch.uint8,
                          device=dev_name)
        stack.plan.bind_weight_scratch(buf)
        for _ in range(2):
            step()
        stack.check(stream)
        per_alt, ms_alt = timed_steps(args.steps, step)
        stack.check(stream)
        ms_alt = max_over_ranks(ms_alt, world, dev_name) / args.steps
        stack.plan.bind_weight_scratch(None)
        del buf
        tf_alt = flops_step / (ms_alt / 1e3) / 1e12
        line["int8_weight_scratch"] = {
            "note": "same workload, int8 weights expanded to bf16 (exact) into a "
                    "scratch ahead of the GEMMs instead of converted in the GEMM "
                    "main loop; same output bits",
            "ms_per_step": round(ms_alt, 4),
            "step_ms": step_stats(per_alt),
            "value": round(replica_throughput(tokens_per_step, world, ms_alt), 1),
            "unit": "block-tokens/s",
            "tflops": round(tf_alt, 2),
            "tensor_peak_frac": round(tf_alt / tpeak, 4),
            "scratch_gib": round(stack.plan.weight_scratch_bytes() / 2**30, 4)}

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, per, sample, _ = cpu_sample(cfg, inp, args.cpu_rows, qk=qk, loras=loras)
        line["cpu_baseline"] = {"value": round(v, 2), "unit": "block-tokens/s",
                                "cores": cpu_cores(), "kind": "oracle",
                                "sample": sample,
                                "seconds_per_sample": round(per, 3)}
    return line


def run_reference(args):
    from memory_bounded_video_gb300 import synth

    cfg = dict(synth.WORKLOADS[args.workload])
    inp = synth.make_workload(args.workload, seed=0)
    qk = None
    if args.qk != "none":
        qk = synth.make_qk(cfg["T"], cfg["D"] // cfg["heads"], seed=0, angles=args.qk)
    loras = None
    if args.lora:
        loras = [synth.make_lora(cfg["D"], cfg["F"], args.lora, seed=i)
                 for i in range(cfg["blocks"])]
    if args.oracle == "full":
        value, per_step, sample, times = cpu_full(cfg, inp, steps=args.steps,
                                                  warmup=args.warmup)
    else:
        value, per_step, sample, times = cpu_sample(cfg, inp, args.cpu_rows,
                                                    steps=args.steps,
                                                    warmup=args.warmup, qk=qk,
                                                    loras=loras)
    T = cfg["T"]
    return {
        "impl": "reference",
        "metric": "DiT-block tokens/s @32k tokens, % BF16 tensor peak, "
                  "peak activation GiB",
        "value": round(value, 3), "unit": "block-tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(per_step * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": args.workload, "T": T, "D": cfg["D"],
                   "heads": cfg["heads"], "ffn": cfg["F"],
                   "blocks": cfg["blocks"], "final_layer": cfg["final"],
                   "int8_weights": cfg["int8"],
                   "qk_transform": (None if qk is None else
                                    f"q/k rmsnorm + {args.qk} rotary"),
                   "lora_rank": args.lora or None},
        "cpu_baseline": {"value": round(value, 3), "unit": "block-tokens/s",
                         "cores": args.cpu_threads or cpu_cores(), "kind": "oracle",
                         "sample": sample,
                         "seconds_per_step": step_stats(times)},
        "e2e": {"value": round(value, 3), "unit": "block-tokens/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    if args.cpu_threads:  # before numpy's BLAS starts its thread pool
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = str(args.cpu_threads)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
