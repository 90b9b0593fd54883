#!/usr/bin/env python3
"""Benchmark of the GLA forward hot path on GB300 (one JSON line on stdout).

Default workload (N=1): the chunked forward at B=2, H=16, T=32768, dk=128,
dv=256 (the long-sequence prefill workload the prefill roofline target is
stated on), plus the decode step at B=256, H=32, dk=dv=128 reported under
"decode".  A step is one gla_chunk_fwd call over the whole batch, inputs
resident in HBM (2.15 GB of inputs, far larger than the 129 MB L2, so no L2
flush is needed between steps).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the only reference this method
has here) on a bounded sample of the same workload, on the host cores.
Multi-GPU (torchrun): every rank runs its own replica of the workload (heads
are independent; there is no exchange step), value = all ranks' tokens / the
slowest rank's time.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GLA chunk-fwd tokens/s (B·H·T) and % roofline; decode steps/s and HBM GB/s"
BWD_METRIC = "GLA chunk-bwd tokens/s (B·H·T): gradients of q, k, v, log_alpha and h0"
GDN_METRIC = "Gated DeltaNet forward tokens/s (B·H·T)"
# fp32 FMA peak of the SM array: 152 SMs x 128 fp32 lanes x 2 flops x 2070 MHz (max SM clock)
FP32_SIMT_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------------- workloads

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the chunked
# forward kernel's launch in one call (the FULL pass with the fused correction;
# the small hT combine that follows it is not counted), measured with ncu on the
# long workload (B2 H16 T32768 dk128 dv256) at full size, with the kernel
# sources whose hash is given.  Any change to those sources makes the figure
# stale: it is then reported as null.
MEASURED_TRAFFIC = {"workload": "B2-H16-T32768-dk128-dv256", "sources": "2061b6c4cb81ba29",
                    "bytes_per_call": 1642785280 + 515365120}
TRAFFIC_SOURCES = ["gla_chunk.cu", "gla_chunk_kernel.cuh", "gla_ptx.cuh"]


# ncu DRAM bytes (read + write) of one gla_chunk_bwd call on the long workload,
# all six launches, for the backward sources hashed in "sources": captured at
# B=1 H=4 (2,048 chunks) and scaled by the chunks of the long workload (16,384;
# every chunk's inputs, states and gradients move once per launch)
MEASURED_BWD_TRAFFIC = {"workload": "B2-H16-T32768-dk128-dv256", "sources": "78ecd605f9e52d28",
                        "bytes_per_call": 8 * (810_661_632 + 474_801_408 + 769_031_680
                                               + 994_191_360 + 134_400)}
BWD_TRAFFIC_SOURCES = ["gla_backward.cu", "gla_ptx.cuh"]


# ncu DRAM bytes (read + write) of one gla_gdn_chunk_fwd call (the WY pre-pass and
# the sequential kernel) at the long shape B=2 H=16 T=32768 dk=128 dv=256, for the
# sources hashed in "sources"; scaled by the heads a call covers (every head
# streams its own rows and scratch once)
MEASURED_GDN_CHUNK_TRAFFIC = {"T": 32768, "dk": 128, "dv": 256, "heads": 32,
                              "sources": "314d585fa2cf92a6",
                              "bytes_per_call": 277083136 + 347115008 + 1489071616 + 512064768}
GDN_CHUNK_TRAFFIC_SOURCES = ["gla_gdn_chunk.cu", "gla_ptx.cuh"]


# ncu DRAM bytes (read + write) of one gla_gdn_fwd launch, captured at B=1, H=8 of
# the long shape (T=32768, dk=128, dv=256) and scaled by the heads a launch
# covers (traffic per head is fixed: every head streams its own rows once)
MEASURED_GDN_TRAFFIC = {"T": 32768, "dk": 128, "dv": 256, "heads": 8, "sources": "ef91c872e7aeb93f",
                        "bytes_per_launch": 272358144 + 110092032}
GDN_TRAFFIC_SOURCES = ["gla_gdn.cu"]


# ncu DRAM bytes (read + write) of one decode step at B=256 H=32 dk=dv=128 (the 5th
# launch of a run: 6.715 TB/s x 152.93 us), for the decode source hashed in "sources".
# Part of the state is still in L2 from the previous step, so DRAM moves 0.95x the
# algorithmic bytes.
MEASURED_DECODE_TRAFFIC = {"sources": "96841f7d24f0df73", "bytes_per_step": 1026925000}
DECODE_TRAFFIC_SOURCES = ["gla_decode.cu"]


def kernel_sources_hash(files=None) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in (TRAFFIC_SOURCES if files is None else files):
        with open(os.path.join(ROOT, "chunkwise_linear_rnn_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(cfg):
    if cfg.name != MEASURED_TRAFFIC["workload"]:
        return None
    try:
        if kernel_sources_hash() != MEASURED_TRAFFIC["sources"]:
            return None
    except OSError:
        return None
    return MEASURED_TRAFFIC["bytes_per_call"]


def measured_bwd_traffic(cfg):
    if cfg.name != MEASURED_BWD_TRAFFIC["workload"]:
        return None
    try:
        if kernel_sources_hash(BWD_TRAFFIC_SOURCES) != MEASURED_BWD_TRAFFIC["sources"]:
            return None
    except OSError:
        return None
    return MEASURED_BWD_TRAFFIC["bytes_per_call"]


def measured_gdn_traffic(cfg):
    m = MEASURED_GDN_TRAFFIC
    if (cfg.T, cfg.dk, cfg.dv) != (m["T"], m["dk"], m["dv"]):
        return None
    try:
        if kernel_sources_hash(GDN_TRAFFIC_SOURCES) != m["sources"]:
            return None
    except OSError:
        return None
    return m["bytes_per_launch"] * cfg.B * cfg.H // m["heads"]


def measured_gdn_chunk_traffic(cfg):
    m = MEASURED_GDN_CHUNK_TRAFFIC
    if (cfg.T, cfg.dk, cfg.dv) != (m["T"], m["dk"], m["dv"]):
        return None
    try:
        if kernel_sources_hash(GDN_CHUNK_TRAFFIC_SOURCES) != m["sources"]:
            return None
    except OSError:
        return None
    return m["bytes_per_call"] * cfg.B * cfg.H // m["heads"]


def chunk_bytes(cfg, n_states: int | None = None, gate_per_head: bool = False) -> int:
    """Algorithmic bytes of one chunked forward: each input read once, each output written once.

    n_states: the (sequence, head) states read and written (default B * H);
    gate_per_head: one fp32 gate per token instead of one per key channel.
    """
    gate = 4 if gate_per_head else 4 * cfg.dk
    per_token = 2 * cfg.dk + 2 * cfg.dk + 2 * cfg.dv + gate + 2 * cfg.dv
    if n_states is None:
        n_states = cfg.B * cfg.H
    state = n_states * cfg.dk * cfg.dv * 4 * (2 if cfg.sigma_h0 is not None else 1)
    return cfg.tokens * per_token + state


def bwd_bytes(cfg, n_states: int | None = None) -> int:
    """Algorithmic bytes of one backward call: q, k, v, log alpha, d_o, h0 and dhT read
    once; dq, dk, dv, dlog alpha and dh0 written once (n_states = sequences x heads)."""
    per_token = 2 * cfg.dk * 2 + cfg.dv * 2 + cfg.dk * 4 + cfg.dv * 2 \
        + 2 * cfg.dk * 2 + cfg.dv * 2 + cfg.dk * 4
    n = cfg.B * cfg.H if n_states is None else n_states
    return cfg.tokens * per_token + 3 * n * cfg.dk * cfg.dv * 4


def packed_lengths(total: int, n: int, seed: int) -> list:
    """A seeded mix of n sequence lengths (log-normal weights, sigma 1) summing to total."""
    import numpy as np
    w = np.random.default_rng(seed).lognormal(0.0, 1.0, size=n)
    lens = np.maximum(1, np.floor(w / w.sum() * total)).astype(np.int64)
    lens[int(np.argmax(lens))] += total - int(lens.sum())
    return [int(x) for x in lens]


# tokens per chunk of the chunked forward kernel
KERNEL_CHUNK = 128


def chunk_flops(cfg, C: int = KERNEL_CHUNK) -> int:
    """Algorithmic flops (causal entries only) at chunk size C, as counted for the roofline."""
    return cfg.tokens * ((C + 1) * (cfg.dk + cfg.dv) + 4 * cfg.dk * cfg.dv)


def roofline(byts: int, flops: int, seconds: float, pk: dict, pk_kind: str,
             tensor_peak_key: str = "bf16_tflops") -> dict:
    """Roofline of one launch: the slower of its bytes at the HBM peak and its flops at
    the bf16 tensor peak binds; `frac` = roofline time / measured time, and `achieved`
    is the binding quantity's rate.  Both fractions are returned."""
    hbm_gbs = byts / seconds / 1e9
    tflops = flops / seconds / 1e12
    t_hbm = byts / (pk["hbm_gbs"] * 1e9)
    t_tc = flops / (pk[tensor_peak_key] * 1e12)
    out = {"peak_kind": pk_kind, "algorithmic_bytes_per_launch": int(byts),
           "flops_per_launch": int(flops), "hbm_frac": hbm_gbs / pk["hbm_gbs"],
           "tensor_frac": tflops / pk[tensor_peak_key], "tensor_peak_tflops": pk[tensor_peak_key],
           "tensor_peak_key": tensor_peak_key}
    if t_hbm >= t_tc:
        out.update({"bound": "hbm", "achieved": hbm_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": hbm_gbs / pk["hbm_gbs"]})
    else:
        out.update({"bound": "tensor", "achieved": tflops, "peak": pk[tensor_peak_key],
                    "unit": "TFLOP/s", "frac": tflops / pk[tensor_peak_key]})
    # the order the contract lists the keys in
    return {k: out[k] for k in ("bound", "achieved", "peak", "unit", "frac")} | out


def decode_bytes(cfg) -> int:
    return cfg.B * cfg.H * (8 * cfg.dk * cfg.dv + 2 * cfg.dk + 2 * cfg.dk + 4 * cfg.dk
                            + 2 * cfg.dv + 2 * cfg.dv)


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"gla_bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}",
                                          f"--query-gpu={self.QUERY}", "--format=csv,noheader",
                                          "-lms", "20"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return self
        # nvidia-smi takes a moment to start: wait (bounded) for its first line so that
        # the samples cover the timed region rather than only what follows it.
        deadline = time.time() + 5.0
        while time.time() < deadline and self.proc.poll() is None:
            try:
                if os.path.getsize(self.path) > 0:
                    break
            except OSError:
                pass
            time.sleep(0.01)
        self.first_line = self._count()
        return self

    def _count(self) -> int:
        try:
            with open(self.path) as f:
                return sum(1 for _ in f)
        except OSError:
            return 0

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            lines = open(self.path).read().splitlines()
            # drop the sample(s) written before the timed region started
            inside = lines[getattr(self, "first_line", 0):]
            # a region shorter than the sampling period keeps the sample nearest to it
            for line in (inside or lines[-1:]):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1].split()[0]))
                    smax = float(parts[2].split()[0])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------------------- our arm

class Ranks:
    """The replicas' rank helpers: a barrier and the maximum over ranks.

    With a process group (any backend; NCCL on the GPU machine, gloo in the CPU
    tests) they go through it; alone they are a device synchronisation and
    the identity.  `device` is where the reduction tensor lives.
    """

    def __init__(self, dist=None, device=None):
        import torch
        self.dist = dist
        self.device = device if device is not None else torch.device("cpu")

    def barrier(self):
        import torch
        if self.dist is not None:
            self.dist.barrier()
        if self.device.type == "cuda":
            torch.cuda.synchronize(self.device)

    def max_over_ranks(self, x: float) -> float:
        import torch
        if self.dist is None:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=self.device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())


def replica_inputs(cfg, rank: int, device):
    """Rank `rank`'s replica of a fixed-length workload: the seeded synthetic
    inputs drawn with seed = rank, so that each rank works on its own shard
    (a distinct draw of the same distribution) and no data crosses ranks."""
    from synth import make_config_inputs
    return make_config_inputs(cfg, seed=rank, device=device)


def job_tokens(cfg, world: int) -> int:
    """Tokens the whole job processes per step: every rank's replica."""
    return cfg.tokens * world


def run_ours(args, rank, world, local_rank):
    import torch
    import __graft_entry__ as ge
    ge.build()
    import chunkwise_linear_rnn_gb300 as gla

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    ranks = Ranks(dist, dev)
    barrier, max_over_ranks = ranks.barrier, ranks.max_over_ranks

    pk, pk_kind = peaks()
    cfg = chunk_config(args)
    line = None
    if args.only == "bwd":
        return bwd_leg(args, cfg, world, rank, dev, gla, barrier, max_over_ranks, pk, pk_kind)
    if args.only == "gdn":
        return gdn_leg(args, cfg, world, rank, dev, gla, barrier, max_over_ranks, pk, pk_kind)
    if args.only != "decode":
        line = chunk_leg(args, cfg, world, rank, dev, gla, barrier, max_over_ranks, pk, pk_kind)
    else:
        line = {"metric": METRIC, "value": None, "unit": "tokens/s", "n_gpus": world,
                "steps": 0, "warmup": args.warmup, "note": "chunked forward skipped (--only decode)"}
    if (args.only == "both" and args.workload == "long" and not args.varlen
            and args.gate == "channel" and not (args.batch or args.heads)):
        # the other prefill workloads of the same kernel, secondary numbers on the line
        import argparse as _ap
        for wl, steps in (("medium", 100), ("very_long", 20)):
            wargs = _ap.Namespace(**vars(args))
            wargs.workload, wargs.no_e2e = wl, True
            wargs.steps, wargs.warmup = min(args.steps, steps), max(args.warmup, 3)
            w = chunk_leg(wargs, chunk_config(wargs), world, rank, dev, gla, barrier,
                          max_over_ranks, pk, pk_kind)
            line[wl] = {"metric": w["metric"], "value": w["value"], "unit": w["unit"],
                        "ms_per_step": w["ms_per_step"], "steps": w["steps"],
                        "workload": w["config"]["workload"], "roofline": w["roofline"],
                        "gpu_launches": w["gpu_launches"], "clocks": w["clocks"]}
    if args.only != "chunk":
        line["decode"] = decode_leg(args, world, rank, dev, gla, barrier, max_over_ranks, pk)
    if args.only == "both" and not args.varlen and args.gate == "channel":
        # the backward on the same workload, a secondary number on the same line
        import argparse as _ap
        bargs = _ap.Namespace(**vars(args))
        bargs.steps, bargs.warmup, bargs.no_e2e = min(args.steps, 20), max(args.warmup, 3), True
        b = bwd_leg(bargs, cfg, world, rank, dev, gla, barrier, max_over_ranks, pk, pk_kind)
        line["backward"] = {"metric": b["metric"], "value": b["value"], "unit": b["unit"],
                            "ms_per_step": b["ms_per_step"], "steps": b["steps"],
                            "workload": b["config"]["workload"], "roofline": b["roofline"],
                            "gpu_launches": b["gpu_launches"], "clocks": b["clocks"]}
        # the gated delta rule forward on the same shape, likewise secondary; its failure
        # is reported in place and never costs the primary line
        gargs = _ap.Namespace(**vars(args))
        gargs.steps, gargs.warmup, gargs.no_e2e = min(args.steps, 10), max(args.warmup, 3), True
        try:
            gd = gdn_leg(gargs, cfg, world, rank, dev, gla, barrier, max_over_ranks, pk, pk_kind)
            line["gated_delta_rule"] = {
                "metric": gd["metric"], "value": gd["value"], "unit": gd["unit"],
                "ms_per_step": gd["ms_per_step"], "steps": gd["steps"],
                "workload": gd["config"]["workload"], "roofline": gd["roofline"],
                "gpu_launches": gd["gpu_launches"], "clocks": gd["clocks"]}
        except Exception as exc:  # noqa: BLE001
            log(f"gated delta rule leg failed: {exc!r}")
            line["gated_delta_rule"] = {"error": repr(exc)[:300]}
    return line


def chunk_config(args):
    """The workload's ChunkConfig, with --batch / --heads overrides (used for small profiles)."""
    import dataclasses
    from synth import CHUNK_CONFIGS
    cfg = CHUNK_CONFIGS[args.workload]
    if args.batch or args.heads:
        B = args.batch or cfg.B
        H = args.heads or cfg.H
        cfg = dataclasses.replace(cfg, B=B, H=H, name=f"B{B}-H{H}-T{cfg.T}-dk{cfg.dk}-dv{cfg.dv}")
    return cfg


def chunk_leg(args, cfg, world, rank, dev, gla, barrier, max_over_ranks, pk, pk_kind):
    import torch
    from synth import make_chunk_inputs
    stream = torch.cuda.current_stream(dev)
    n_states = None
    packed = None
    if args.varlen and args.gate == "head":
        raise SystemExit("--gate head takes fixed-length batches only")
    if args.varlen:
        # the same tokens per head, packed: --varlen sequences of mixed lengths
        # through gla_chunk_fwd_varlen (q, k, v, gates drawn as for the workload)
        per_head = cfg.B * cfg.T
        lens = packed_lengths(per_head, args.varlen, seed=1234 + rank)
        cu = [0]
        for n in lens:
            cu.append(cu[-1] + n)
        q, k, v, a, _ = make_chunk_inputs(1, cfg.H, per_head, cfg.dk, cfg.dv, sigma_z=cfg.sigma_z,
                                          tau=cfg.tau, seed=rank, device=dev)
        q, k, v, a = (t[0] for t in (q, k, v, a))
        h0 = None
        if cfg.sigma_h0 is not None:
            g = torch.Generator(device=dev)
            g.manual_seed(5678 + rank)
            h0 = torch.randn(len(lens), cfg.H, cfg.dk, cfg.dv, generator=g, device=dev,
                             dtype=torch.float32).mul_(cfg.sigma_h0)
        o = torch.empty(cfg.H, per_head, cfg.dv, dtype=torch.bfloat16, device=dev)
        hT = torch.empty(len(lens), cfg.H, cfg.dk, cfg.dv, dtype=torch.float32, device=dev)
        n_states = len(lens) * cfg.H
        srt = sorted(lens)
        packed = {"sequences": len(lens), "min_len": srt[0], "median_len": srt[len(srt) // 2],
                  "max_len": srt[-1], "lengths": "log-normal weights (sigma 1), seed 1234"}

        def step():
            gla.gla_chunk_fwd_varlen(q, k, v, a, cu, cfg.scale, h0, out=o, final_state=hT)

        launches_per_step = gla.gla_chunk_fwd_varlen_plan(cu, cfg.H, cfg.dk, cfg.dv)["launches"]
    else:
        q, k, v, a, h0 = replica_inputs(cfg, rank, dev)
        if args.gate == "head":
            a = a[..., 0].contiguous()   # one gate per token and head (its first channel's draw)
        o = torch.empty(cfg.B, cfg.H, cfg.T, cfg.dv, dtype=torch.bfloat16, device=dev)
        hT = torch.empty(cfg.B, cfg.H, cfg.dk, cfg.dv, dtype=torch.float32, device=dev)

        def step():
            gla.gla_chunk_fwd(q, k, v, a, cfg.scale, h0, out=o, final_state=hT)

        launches_per_step = gla.gla_chunk_fwd_plan(cfg.B, cfg.H, cfg.T, cfg.dk, cfg.dv)["launches"]
    for _ in range(args.warmup):
        step()
    barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with ClockSampler(dev.index) as clk:
        barrier()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for s, e in ev:
            s.record(stream)
            step()
            e.record(stream)
        t_end.record(stream)
        barrier()
    total_ms = max_over_ranks(t_start.elapsed_time(t_end))
    per_launch_ms = statistics.mean(s.elapsed_time(e) for s, e in ev)
    if gla.gla_last_device_status(dev) != 0:
        raise RuntimeError("device status word reports an expired wait during the benchmark")
    ms_per_step = total_ms / args.steps
    tokens_all = job_tokens(cfg, world)
    value = tokens_all / (ms_per_step / 1e3)
    byts = chunk_bytes(cfg, n_states, gate_per_head=args.gate == "head")
    achieved_gbs = byts / (per_launch_ms / 1e3) / 1e9
    clocks = clk.summary()

    # ---- end to end through the public API: gla_chunk_fwd_host on pinned host
    # buffers; every call copies its inputs in and its outputs out (pipelined
    # over groups of heads), all inside the timed region
    e2e = None
    if not args.no_e2e and not args.varlen and args.gate == "channel":
        hq, hk, hv, ha = (t.cpu().pin_memory() for t in (q, k, v, a))
        hh0 = None if h0 is None else h0.cpu().pin_memory()
        ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        hhT = torch.empty(hT.shape, dtype=hT.dtype).pin_memory()

        def e2e_step():
            gla.gla_chunk_fwd_host(hq, hk, hv, ha, cfg.scale, hh0, out=ho, final_state=hhT,
                                   device=dev.index)

        e2e_steps = max(2, min(args.steps, 5))
        for _ in range(2):
            e2e_step()
        barrier()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        s1.record(stream)
        barrier()
        e2e_ms = max_over_ranks(s0.elapsed_time(s1)) / e2e_steps
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, ha)) + (
            0 if hh0 is None else hh0.numel() * 4)
        d2h = ho.numel() * 2 + hhT.numel() * 4
        e2e = {"value": tokens_all / (e2e_ms / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e2e_ms, "api": "gla_chunk_fwd_host"}
        del hq, hk, hv, ha, hh0, ho, hhT

    del q, k, v, a, h0, o, hT
    torch.cuda.empty_cache()

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": cfg.name + (f"-packed{args.varlen}" if args.varlen else "") +
                   ("-gate-per-head" if args.gate == "head" else ""),
                   "B": cfg.B, "H": cfg.H, "T": cfg.T, "dk": cfg.dk,
                   "dv": cfg.dv, "chunk": 128, "replicas": world,
                   "l2": "inputs (%.2f GB) larger than L2; no flush" % (byts / 1e9)},
        "roofline": roofline(byts, chunk_flops(cfg), per_launch_ms / 1e3, pk, pk_kind) | {
            "traffic": None if (args.varlen or args.gate == "head") else measured_traffic(cfg),
            "traffic_unit": "bytes per call", "kernel": "chunk_fwd_kernel",
            "flops_chunk": KERNEL_CHUNK},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if packed is not None:
        line["config"]["packed"] = packed
    return line


def bwd_leg(args, cfg, world, rank, dev, gla, barrier, max_over_ranks, pk, pk_kind):
    """The chunkwise backward (gla_chunk_bwd) on the workload, its own JSON line."""
    import torch
    from synth import make_backward_grads
    stream = torch.cuda.current_stream(dev)
    plan = gla.gla_chunk_bwd_plan(cfg.B, cfg.H, cfg.T, cfg.dk, cfg.dv)
    packed = None
    if args.varlen:
        # the same tokens per head packed into --varlen sequences of mixed lengths
        from synth import make_chunk_inputs
        per_head = cfg.B * cfg.T
        lens = packed_lengths(per_head, args.varlen, seed=1234 + rank)
        cu = [0]
        for m in lens:
            cu.append(cu[-1] + m)
        q, k, v, a, _ = make_chunk_inputs(1, cfg.H, per_head, cfg.dk, cfg.dv, sigma_z=cfg.sigma_z,
                                          tau=cfg.tau, seed=rank, device=dev)
        q, k, v, a = (t[0] for t in (q, k, v, a))
        d_o, _ = make_backward_grads(1, cfg.H, per_head, cfg.dk, cfg.dv, seed=rank, device=dev)
        d_o = d_o[0]
        h0 = dhT = None
        if cfg.sigma_h0 is not None:
            g = torch.Generator(device=dev)
            g.manual_seed(5678 + rank)
            h0 = torch.randn(len(lens), cfg.H, cfg.dk, cfg.dv, generator=g, device=dev).mul_(0.1)
            dhT = torch.randn(len(lens), cfg.H, cfg.dk, cfg.dv, generator=g, device=dev).mul_(0.1)
        srt = sorted(lens)
        packed = {"sequences": len(lens), "min_len": srt[0], "median_len": srt[len(srt) // 2],
                  "max_len": srt[-1], "lengths": "log-normal weights (sigma 1), seed 1234"}

        def step():
            return gla.gla_chunk_bwd_varlen(q, k, v, a, d_o, cu, cfg.scale, h0, dhT)
    else:
        q, k, v, a, h0 = replica_inputs(cfg, rank, dev)
        d_o, dhT = make_backward_grads(cfg.B, cfg.H, cfg.T, cfg.dk, cfg.dv,
                                       sigma_dhT=0.1 if h0 is not None else None, seed=rank,
                                       device=dev)

        def step():
            return gla.gla_chunk_bwd(q, k, v, a, d_o, cfg.scale, h0, dhT)

    for _ in range(args.warmup):
        step()
    barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with ClockSampler(dev.index) as clk:
        barrier()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for s0, e0 in ev:
            s0.record(stream)
            step()
            e0.record(stream)
        t_end.record(stream)
        barrier()
    total_ms = max_over_ranks(t_start.elapsed_time(t_end))
    per_call_ms = statistics.mean(s0.elapsed_time(e0) for s0, e0 in ev)
    ms_per_step = total_ms / args.steps
    tokens_all = job_tokens(cfg, world)
    byts = bwd_bytes(cfg, None if packed is None else packed["sequences"] * cfg.H)
    achieved = byts / (per_call_ms / 1e3) / 1e9

    # end to end: pinned host inputs copied in and gradients copied out every call
    e2e = None
    if not args.no_e2e and not args.varlen:
        host_in = [t.cpu().pin_memory() for t in (q, k, v, a, d_o, h0, dhT) if t is not None]
        dev_in = [torch.empty_like(t, device=dev) for t in host_in]
        outs = step()
        host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]
        st = 3 if h0 is not None else None

        def e2e_step():
            for hsrc, dst in zip(host_in, dev_in):
                dst.copy_(hsrc, non_blocking=True)
            di = dev_in
            res = gla.gla_chunk_bwd(di[0], di[1], di[2], di[3], di[4], cfg.scale,
                                    di[5] if st else None, di[6] if st else None)
            for src, hdst in zip(res, host_out):
                hdst.copy_(src, non_blocking=True)

        for _ in range(2):
            e2e_step()
        barrier()
        x0 = torch.cuda.Event(enable_timing=True)
        x1 = torch.cuda.Event(enable_timing=True)
        n_e2e = max(2, min(args.steps, 5))
        x0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        x1.record(stream)
        barrier()
        e2e_ms = max_over_ranks(x0.elapsed_time(x1)) / n_e2e
        e2e = {"value": tokens_all / (e2e_ms / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in host_in)),
               "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in host_out)),
               "ms_per_step": e2e_ms, "api": "gla_chunk_bwd with pinned-host copies"}
        del host_in, dev_in, host_out, outs
    del q, k, v, a, h0, d_o, dhT
    torch.cuda.empty_cache()
    line = {
        "metric": BWD_METRIC,
        "value": tokens_all / (ms_per_step / 1e3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        # bf16 tensor-core products (hi/lo pairs), fp32 accumulation and scans
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": cfg.name + (f"-packed{args.varlen}" if args.varlen else "") +
                   "-backward", "B": cfg.B, "H": cfg.H, "T": cfg.T,
                   "dk": cfg.dk, "dv": cfg.dv, "chunk": plan["chunk"], "replicas": world,
                   "l2": "inputs (%.2f GB) larger than L2; no flush" % (byts / 1e9)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / pk["hbm_gbs"],
                     "traffic": None if packed is not None else measured_bwd_traffic(cfg),
                     "traffic_unit": "bytes per call",
                     "peak_kind": pk_kind, "kernel": "gla_chunk_bwd (whole call, %d launches)"
                     % plan["launches"], "algorithmic_bytes_per_launch": byts,
                     "scratch_bytes": plan["scratch_bytes"]},
        "gpu_launches": plan["launches"] * args.steps,
        "clocks": clk.summary(),
    }
    if e2e is not None:
        line["e2e"] = e2e
    if packed is not None:
        line["config"]["packed"] = packed
    return line


def gdn_flops(cfg) -> int:
    """Per token, head and value column: k.S, the rank-1 update and q.S, dk FMAs each."""
    return 6 * cfg.B * cfg.H * cfg.T * cfg.dk * cfg.dv


def gdn_chunk_flops(cfg, C: int = 64) -> int:
    """Tensor-core flops of the chunk algorithm (chunk C), per token: K K^T, W = T(beta gamma K)
    and Q K^T (2 C dk each), U = T(beta V) and P D (2 C dv each), W S, Q S and K~^T D
    (2 dk dv each)."""
    return cfg.B * cfg.H * cfg.T * (3 * 2 * C * cfg.dk + 2 * 2 * C * cfg.dv
                                    + 3 * 2 * cfg.dk * cfg.dv)


def gdn_bytes(cfg) -> int:
    """q, k, v, o in bf16; g, beta in fp32; h0 and hT in fp32."""
    tok = cfg.B * cfg.H * cfg.T
    return tok * (2 * cfg.dk * 2 + 2 * cfg.dv * 2 + 2 * 4) + 2 * cfg.B * cfg.H * cfg.dk * cfg.dv * 4


def gdn_leg(args, cfg, world, rank, dev, gla, barrier, max_over_ranks, pk, pk_kind):
    """The gated delta rule forward on the workload's shape: by chunks on the tensor cores
    (gla_gdn_chunk_fwd, dk = 128) unless --gdn-impl token, or dk != 128 (gla_gdn_fwd)."""
    import torch
    from synth import make_gdn_inputs
    stream = torch.cuda.current_stream(dev)
    chunked = args.gdn_impl == "chunk" and cfg.dk == 128
    q, k, v, g, b, h0 = make_gdn_inputs(cfg.B, cfg.H, cfg.T, cfg.dk, cfg.dv, sigma_h0=0.1,
                                        seed=rank, device=dev)

    def step():
        return gla.gla_gdn_fwd(q, k, v, g, b, cfg.scale, h0, chunked=chunked)

    for _ in range(args.warmup):
        step()
    barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with ClockSampler(dev.index) as clk:
        barrier()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for s0, e0 in ev:
            s0.record(stream)
            step()
            e0.record(stream)
        t_end.record(stream)
        barrier()
    ms_per_step = max_over_ranks(t_start.elapsed_time(t_end)) / args.steps
    per_call_ms = statistics.mean(s0.elapsed_time(e0) for s0, e0 in ev)
    tokens_all = job_tokens(cfg, world)
    flops, byts = gdn_flops(cfg), gdn_bytes(cfg)
    achieved = flops / (per_call_ms / 1e3) / 1e12

    e2e = None
    if not args.no_e2e:
        host_in = [t.cpu().pin_memory() for t in (q, k, v, g, b, h0)]
        dev_in = [torch.empty_like(t, device=dev) for t in host_in]
        outs = step()
        host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]

        def e2e_step():
            for hsrc, dst in zip(host_in, dev_in):
                dst.copy_(hsrc, non_blocking=True)
            res = gla.gla_gdn_fwd(*dev_in[:5], cfg.scale, dev_in[5], chunked=chunked)
            for src, hdst in zip(res, host_out):
                hdst.copy_(src, non_blocking=True)

        for _ in range(2):
            e2e_step()
        barrier()
        x0 = torch.cuda.Event(enable_timing=True)
        x1 = torch.cuda.Event(enable_timing=True)
        n_e2e = max(2, min(args.steps, 5))
        x0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        x1.record(stream)
        barrier()
        e2e_ms = max_over_ranks(x0.elapsed_time(x1)) / n_e2e
        e2e = {"value": tokens_all / (e2e_ms / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in host_in)),
               "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in host_out)),
               "ms_per_step": e2e_ms,
               "api": ("gla_gdn_chunk_fwd" if chunked else "gla_gdn_fwd") + " with pinned-host copies"}
        del host_in, dev_in, host_out, outs
    del q, k, v, g, b, h0
    torch.cuda.empty_cache()
    line = {
        "metric": GDN_METRIC,
        "value": tokens_all / (ms_per_step / 1e3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        # chunked: bf16 tensor-core products (hi/lo pairs) with fp32 accumulation;
        # token recurrence: fp32 on the CUDA cores
        "dtype": "bf16" if chunked else "f32",
        "data": "synthetic",
        "config": {"workload": cfg.name + "-gated-delta-rule", "B": cfg.B, "H": cfg.H,
                   "T": cfg.T, "dk": cfg.dk, "dv": cfg.dv, "replicas": world,
                   "l2": "inputs (%.2f GB) larger than L2; no flush" % (byts / 1e9)},
        "roofline": (roofline(byts, gdn_chunk_flops(cfg), per_call_ms / 1e3, pk, pk_kind) | {
            "traffic": measured_gdn_chunk_traffic(cfg), "traffic_unit": "DRAM bytes per call",
            "kernel": "gdn_wy_kernel + gdn_seq_kernel (chunked, two launches)",
            "note": "algorithmic bytes count the contract's inputs and outputs once; the WY "
                    "pre-pass scratch (W and (T - I) diag(beta), written once and read by "
                    "each value-column tile) is extra traffic"}) if chunked else
        {"bound": "alu", "achieved": achieved, "peak": FP32_SIMT_TFLOPS,
                     "unit": "TFLOP/s", "frac": achieved / FP32_SIMT_TFLOPS,
                     "traffic": measured_gdn_traffic(cfg), "traffic_unit": "DRAM bytes per launch",
                     "peak_kind": "derived: 152 SMs x 128 fp32 FMA lanes x 2 x 2070 MHz",
                     "kernel": "gdn_recurrent_kernel (token-recurrent, one launch)",
                     "algorithmic_flops_per_launch": flops,
                     "hbm_gbs": byts / (per_call_ms / 1e3) / 1e9,
                     "hbm_frac": byts / (per_call_ms / 1e3) / 1e9 / pk["hbm_gbs"],
                     "hbm_peak_kind": pk_kind},
        "gpu_launches": args.steps * (2 if chunked else 1),
        "clocks": clk.summary(),
    }
    if e2e is not None:
        line["e2e"] = e2e
    return line


def gdn_oracle_sample(cfg, target_s: float, threads: int) -> dict:
    """Time the fp64 gated-delta-rule oracle on whole heads and a prefix of tokens."""
    from oracle import gdn_oracle
    from synth import make_gdn_inputs
    gdn_oracle.build()

    def inputs(heads, T):
        q, k, v, g, b, h0 = make_gdn_inputs(1, heads, T, cfg.dk, cfg.dv, sigma_h0=0.1, seed=0)
        return [q.float().numpy(), k.float().numpy(), v.float().numpy(), g.numpy(), b.numpy(),
                h0.double().numpy()]

    def run(ins):
        t0 = time.perf_counter()
        gdn_oracle.forward(*ins[:5], cfg.scale, ins[5], nthreads=threads)
        return time.perf_counter() - t0

    heads = max(1, min(cfg.B * cfg.H, threads))
    probe = inputs(heads, min(cfg.T, 256))
    run(probe)
    # host-seconds per token with every thread busy
    per_token = run(probe) / (heads * probe[0].shape[-2]) * min(heads, threads) / threads
    budget = target_s / per_token                        # tokens that fill target_s
    T = int(min(cfg.T, max(256, budget / heads)))
    if T == cfg.T:                                       # whole sequences: widen to more heads
        heads = int(min(cfg.B * cfg.H, max(heads, budget / T)))
    repeat = max(1, int(budget / (heads * T))) if (heads == cfg.B * cfg.H and T == cfg.T) else 1
    ins = inputs(heads, T)
    dt = sum(run(ins) for _ in range(repeat))
    return {"value": repeat * heads * T / dt, "unit": "tokens/s", "cores": min(threads, heads),
            "kind": "oracle", "seconds": dt,
            "sample": f"{repeat} x {heads} heads x {T} tokens of {cfg.name} (dk={cfg.dk}, "
                      f"dv={cfg.dv}), fp64 gated-delta-rule recurrence, {dt:.1f} s"}


def decode_leg(args, world, rank, dev, gla, barrier, max_over_ranks, pk):
    """Decode steps at B=256, H=32, dk=dv=128 (secondary numbers on the same JSON line)."""
    import torch
    from synth import DECODE_CONFIG, make_decode_inputs
    stream = torch.cuda.current_stream(dev)
    dc = DECODE_CONFIG
    nsteps = args.decode_steps
    dh0, dqs, dks, dvs, das = make_decode_inputs(dc.B, dc.H, dc.dk, dc.dv, nsteps,
                                                 sigma_z=dc.sigma_z, tau=dc.tau,
                                                 sigma_h0=dc.sigma_h0, seed=rank, device=dev)
    h = dh0.clone()
    do = torch.empty(dc.B, dc.H, dc.dv, dtype=torch.bfloat16, device=dev)
    for s in range(min(3, nsteps)):
        gla.gla_recurrent_step(dqs[s], dks[s], dvs[s], das[s], h, dc.scale, out=do)
    barrier()
    d0 = torch.cuda.Event(enable_timing=True)
    d1 = torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for s in range(nsteps):
        gla.gla_recurrent_step(dqs[s], dks[s], dvs[s], das[s], h, dc.scale, out=do)
    d1.record(stream)
    barrier()
    dms = max_over_ranks(d0.elapsed_time(d1)) / nsteps
    dbytes = decode_bytes(dc)
    dgbs = dbytes / (dms / 1e3) / 1e9
    # DRAM bytes per step as ncu measured them (null once the kernel source changed):
    # the algorithmic rate can read above the copy peak because part of the state hits
    # in L2; the DRAM rate cannot
    try:
        fresh = kernel_sources_hash(DECODE_TRAFFIC_SOURCES) == MEASURED_DECODE_TRAFFIC["sources"]
    except OSError:
        fresh = False
    traffic = MEASURED_DECODE_TRAFFIC["bytes_per_step"] if fresh else None
    decode = {"workload": dc.name, "steps_per_s": 1e3 / dms, "replicas": world,
              "ms_per_step": dms, "hbm_gbs": dgbs, "bytes_per_step": dbytes,
              "frac_of_hbm_peak": dgbs / pk["hbm_gbs"], "timed_steps": nsteps,
              "traffic": traffic, "traffic_unit": "DRAM bytes per step (ncu)",
              "dram_gbs": None if traffic is None else traffic / (dms / 1e3) / 1e9,
              "dram_frac_of_hbm_peak": None if traffic is None
              else traffic / (dms / 1e3) / 1e9 / pk["hbm_gbs"],
              "gpu_launches": nsteps}
    del dh0, dqs, dks, dvs, das, h, do
    torch.cuda.empty_cache()
    return decode


# --------------------------------------------------------------------------- CPU baseline

class OracleSample:
    """A bounded sample of the workload for timing the fp64 CPU oracle.

    The sample takes whole heads of the workload (up to all B*H of them) and a
    prefix of T tokens, sized from a short probe so that one pass costs about
    target_s seconds of host time; a workload smaller than that is run whole,
    repeated to fill the time.
    """

    def __init__(self, cfg, target_s: float, threads: int, backward: bool = False):
        from oracle import gla_oracle
        gla_oracle.build()
        self.oracle, self.cfg, self.threads = gla_oracle, cfg, threads
        self.backward = backward
        heads = max(1, min(cfg.B * cfg.H, threads))
        t_probe = min(cfg.T, 2048)
        probe = self._inputs(heads, t_probe)
        self._pass(heads, t_probe, probe)          # first call pays for thread start-up
        dt = self._pass(heads, t_probe, probe)
        per_token = dt / (heads * t_probe) * min(heads, threads)   # host-seconds per token
        budget = target_s * threads / per_token                     # tokens that fill target_s
        T = int(min(cfg.T, max(t_probe, budget / heads)))
        if T == cfg.T:
            heads = int(min(cfg.B * cfg.H, max(heads, budget / T)))
        self.heads, self.T = heads, T
        self.repeat = max(1, int(budget / (heads * T))) if (heads == cfg.B * cfg.H and T == cfg.T) else 1
        self.inputs = self._inputs(heads, T)

    def _inputs(self, heads, T):
        from synth import make_chunk_inputs
        c = self.cfg
        q, k, v, a, h0 = make_chunk_inputs(1, heads, T, c.dk, c.dv, sigma_z=c.sigma_z, tau=c.tau,
                                           sigma_h0=c.sigma_h0, seed=0)
        f = lambda t: t.float().numpy()  # noqa: E731
        ins = [f(q), f(k), f(v), a.numpy(), None if h0 is None else h0.double().numpy()]
        if self.backward:
            from synth import make_backward_grads
            d_o, dhT = make_backward_grads(1, heads, T, c.dk, c.dv,
                                           sigma_dhT=0.1 if h0 is not None else None, seed=0)
            ins += [f(d_o), None if dhT is None else dhT.double().numpy()]
        return ins

    def _pass(self, heads, T, inputs=None):
        ins = inputs if inputs is not None else self._inputs(heads, T)
        q, k, v, a, h0 = ins[:5]
        t0 = time.perf_counter()
        if self.backward:
            self.oracle.backward(q, k, v, a, self.cfg.scale, ins[5], h0, ins[6],
                                 nthreads=self.threads)
        else:
            self.oracle.forward(q, k, v, a, self.cfg.scale, h0, nthreads=self.threads)
        return time.perf_counter() - t0

    def run(self) -> dict:
        dt = sum(self._pass(self.heads, self.T, self.inputs) for _ in range(self.repeat))
        tokens = self.repeat * self.heads * self.T
        c = self.cfg
        return {"value": tokens / dt, "unit": "tokens/s", "cores": min(self.threads, self.heads),
                "kind": "oracle",
                "sample": f"{self.repeat} x {self.heads} heads x {self.T} tokens of {c.name} "
                          f"(dk={c.dk}, dv={c.dv}), fp64 recurrence"
                          f"{' and its reverse-mode backward' if self.backward else ''}, {dt:.1f} s"}


def oracle_sample(cfg, target_s: float, threads: int, backward: bool = False) -> dict:
    """Time the fp64 oracle on a bounded sample of the workload; returns a cpu_baseline dict."""
    return OracleSample(cfg, target_s, threads, backward).run()


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args):
    """The reference arm: the fp64 CPU oracle on the host cores, one bounded sample per step."""
    cfg = chunk_config(args)
    threads = host_threads()
    per_step_s = max(0.5, min(args.ref_seconds, 150.0 / max(1, args.steps + args.warmup)))
    if args.only == "gdn":
        per = [gdn_oracle_sample(cfg, per_step_s, threads) for _ in range(args.warmup + args.steps)]
        per = per[args.warmup:]
        value = statistics.median(p["value"] for p in per)
        base = dict(per[-1], value=value)
        return {
            "impl": "reference", "metric": GDN_METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.median(p["seconds"] for p in per),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": cfg.name + "-gated-delta-rule", "B": cfg.B, "H": cfg.H,
                       "T": cfg.T, "dk": cfg.dk, "dv": cfg.dv},
            "cpu_baseline": base,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0,
        }
    sample = OracleSample(cfg, per_step_s, threads, backward=args.only == "bwd")
    for _ in range(args.warmup):
        sample.run()
    per = [sample.run() for _ in range(args.steps)]
    base = dict(per[-1])
    value = statistics.median(p["value"] for p in per)
    base["value"] = value
    return {
        "impl": "reference", "metric": BWD_METRIC if args.only == "bwd" else METRIC,
        "value": value, "unit": "tokens/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sample.repeat * sample.heads * sample.T / value,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": cfg.name + ("-backward" if args.only == "bwd"
                                                                else ""), "B": cfg.B, "H": cfg.H, "T": cfg.T,
                                        "dk": cfg.dk, "dv": cfg.dv},
        "cpu_baseline": base,
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="long", choices=["small", "medium", "long", "very_long"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--decode-steps", type=int, default=1024)
    ap.add_argument("--only", default="both", choices=["both", "chunk", "decode", "bwd", "gdn"],
                    help="run only the chunked forward, only the decode step, only the "
                         "chunkwise backward, or only the gated delta rule forward (the last "
                         "two on their own JSON line)")
    ap.add_argument("--no-decode", action="store_true", help="same as --only chunk")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's B")
    ap.add_argument("--heads", type=int, default=0, help="override the workload's H")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--gdn-impl", default="chunk", choices=["chunk", "token"],
                    help="gated delta rule leg: the chunk algorithm on the tensor cores "
                         "(gla_gdn_chunk_fwd, dk = 128) or the token recurrence (gla_gdn_fwd)")
    ap.add_argument("--gate", default="channel", choices=["channel", "head"],
                    help="log_alpha per key channel [B,H,T,dk] (the workloads') or per head "
                         "[B,H,T] (no e2e leg)")
    ap.add_argument("--varlen", type=int, default=0,
                    help="pack each head's tokens into this many sequences of mixed lengths "
                         "(gla_chunk_fwd_varlen; no e2e leg)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-seconds", type=float, default=15.0,
                    help="CPU seconds per oracle sample")
    args = ap.parse_args()
    if args.no_decode:
        args.only = "chunk"
    if args.warmup < 3 and args.impl == "ours":
        log("warning: fewer than 3 warm-up steps")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline and args.only == "gdn":
            line["cpu_baseline"] = gdn_oracle_sample(chunk_config(args), args.ref_seconds,
                                                     host_threads())
        elif not args.no_cpu_baseline:
            line["cpu_baseline"] = oracle_sample(chunk_config(args), args.ref_seconds,
                                                 host_threads(), backward=args.only == "bwd")
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
