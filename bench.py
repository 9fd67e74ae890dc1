"""Benchmark of the routed MoE-LoRA expert layer on GB300.

One step = one forward of the whole layer (routing, permute, gate_up GEMM, LoRA gate_up
chain, activation, down GEMM, down LoRA, finalize) over one batch of seeded synthetic
input already resident in HBM.  Default workload: decode, T=64 tokens, H=2048, I=768,
E=128 experts, top_k=8, one rank-16 adapter (Qwen3-30B-A3B-like experts).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0).  For N > 1 it runs under torchrun with one independent
replica per GPU (the layer has no data-path exchange on one GPU): value = tokens of all
ranks / max-over-ranks time.  `--impl reference` times the CPU oracle on the host cores
(the only other arm there is: the pages ship no code) on a bounded sample of the same
workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-LoRA layer tokens/s (decode T<=256, prefill 8K); % of HBM/bf16 roofline"
UNIT = "tokens/s"
EV_EVERY = 16   # gate_up GEMM events on every 16th timed step


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(value: float, world: int) -> float:
    """Max of a float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(tokens_per_rank: int, steps: int, world: int, seconds_max: float) -> dict:
    """Whole-job throughput from the per-rank work and the slowest rank's time."""
    total_tokens = tokens_per_rank * steps * world
    return dict(value=total_tokens / seconds_max, ms_per_step=1e3 * seconds_max / steps)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def gemm_source_hash():
    with open(os.path.join(ROOT, "routed_moe_expert_gb300", "csrc", "grouped_gemm.cu"), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(name: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current GEMM source (else None)."""
    p = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m_src = re.search(r"grouped_gemm\.cu sha256\[:16\]:\s*([0-9a-f]{16})", txt)
    m_val = re.search(r"dram bytes per launch \(read\+write\):\s*([0-9.eE+]+)", txt)
    if not m_src or not m_val or m_src.group(1) != gemm_source_hash():
        return None
    return float(m_val.group(1))


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"])
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return dict(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=smax, reasons=sorted(reasons),
                    samples=len(sm))


# ------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------

def _touched_and_lora(cfg, fwd, pkg, ws, T, E, k, I, H, g, torch):
    """Touched experts and touched (slot, expert) LoRA bytes of the drawn routing."""
    offsets = torch.empty((E + 1,), dtype=torch.int32, device="cuda")
    fwd(outputs=dict(expert_offsets=offsets))
    torch.cuda.synchronize()
    loads = np.diff(offsets.cpu().numpy())
    touched = int((loads > 0).sum())
    st, word = pkg.moe_lora_check_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {word:#x}")
    lora_blocks = 0
    slots = g["slot_idx"].cpu().numpy()
    if cfg.S > 0:
        ids_out = torch.empty((T, k), dtype=torch.int32, device="cuda")
        fwd(outputs=dict(topk_ids=ids_out))
        ids_np = ids_out.cpu().numpy()
        pairs = {(int(slots[t]), int(e)) for t in range(T) for e in ids_np[t] if slots[t] >= 0}
        if cfg.shared_outer:   # per (slot, expert): B_gu and A_dn; per slot: A_gu and B_dn
            lora_blocks = sum(2 * cfg.ranks[s] * (2 * I + I) for s, _ in pairs) + \
                sum(2 * cfg.ranks[s] * (H + H) for s in {s for s, _ in pairs})
        else:
            lora_blocks = sum(2 * cfg.ranks[s] * (2 * H + 3 * I) for s, _ in pairs)
    return touched, lora_blocks, loads


def _act_in_gate_up(P, E):
    """True where the library runs the activation in the gate_up GEMM's epilogue (token
    tiles of 32 or more: twice the mean pairs per expert above 16), so that GEMM writes the
    [P, I] activation instead of the [P, 2I] gate_up output."""
    return 2 * ((P + E - 1) // E) > 16


def _gemm_roofline(name, flops, nbytes, avg_s, peaks, tc_peak, tc_src):
    """Roofline block of one GEMM launch: tensor-bound when its flops at the tensor peak take
    longer than its algorithmic bytes at the HBM peak, else HBM-bound."""
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (tc_peak * 1e12)
    if t_tc > t_hbm:
        ach = flops / avg_s / 1e12
        return {"kernel": name, "bound": "tensor", "achieved": ach, "peak": tc_peak, "unit": "TFLOP/s",
                "frac": ach / tc_peak, "peak_source": tc_src, "algorithmic_flops_per_launch": flops,
                "algorithmic_bytes_per_launch": nbytes, "avg_launch_us": avg_s * 1e6}
    ach = nbytes / avg_s / 1e9
    return {"kernel": name, "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": ach / peaks["hbm_gbs"], "peak_source": f"{peaks['source']} hbm_gbs",
            "algorithmic_bytes_per_launch": nbytes, "algorithmic_flops_per_launch": flops,
            "avg_launch_us": avg_s * 1e6}


def _timed_steps(fwd, stream, steps, torch, pkg, clock_index=None, world=1):
    """Time `steps` forwards between CUDA events on `stream`.  On every EV_EVERY-th step the
    gate_up and down GEMMs are bracketed by events on their stream (an event between two
    kernels holds the second one back from starting early, so not on every step).
    Returns (seconds, mean gate_up GEMM seconds, mean down GEMM seconds, clocks)."""
    n_ev = 2 * pkg.NUM_STAGES
    gu = pkg.STAGES.index("gate_up_gemm")
    dn = pkg.STAGES.index("down_gemm")
    ev_sets = []
    for _ in range((steps + EV_EVERY - 1) // EV_EVERY):
        evs = [None] * n_ev
        for i in (2 * gu, 2 * gu + 1, 2 * dn, 2 * dn + 1):
            evs[i] = torch.cuda.Event(enable_timing=True)
            evs[i].record(stream)          # materialise the CUDA event handle
        ev_sets.append(evs)
    torch.cuda.synchronize()
    clocks = ClockSampler(clock_index) if clock_index is not None else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        fwd(prof=ev_sets[i // EV_EVERY] if i % EV_EVERY == 0 else None)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if clocks else None
    sec = t0.elapsed_time(t1) / 1e3
    gu_s = statistics.mean(ev[2 * gu].elapsed_time(ev[2 * gu + 1]) for ev in ev_sets) / 1e3
    dn_s = statistics.mean(ev[2 * dn].elapsed_time(ev[2 * dn + 1]) for ev in ev_sets) / 1e3
    return sec, gu_s, dn_s, clk


def _lora_off_ms(fwd, stream, steps, warmup, torch, pkg):
    for _ in range(warmup):
        fwd(flags=pkg.FLAG_LORA_OFF)
    torch.cuda.synchronize()
    o0 = torch.cuda.Event(enable_timing=True)
    o1 = torch.cuda.Event(enable_timing=True)
    o0.record(stream)
    for _ in range(steps):
        fwd(flags=pkg.FLAG_LORA_OFF)
    o1.record(stream)
    torch.cuda.synchronize()
    return o0.elapsed_time(o1) / steps


def _make_fwd(pkg, h, cfg, g, ws, out, k, args, w8=None, w4=None):
    # The expand-ready LoRA B copies are made once, like the weights (a weight-load step of the
    # library); the bf16 layer's fused LoRA stages read them.
    packed = {}
    if w4 is None and cfg.S > 0 and not args.per_slot_lora:
        packed = dict(lora_B_gu_packed=pkg.moe_lora_pack_lora_b(h, g["lora_B_gu"], cfg.ranks, 1),
                      lora_B_dn_packed=pkg.moe_lora_pack_lora_b(h, g["lora_B_dn"], cfg.ranks, 0),
                      lora_A_gu_packed=pkg.moe_lora_pack_lora_a(h, g["lora_A_gu"], cfg.ranks),
                      lora_A_dn_packed=pkg.moe_lora_pack_lora_a(h, g["lora_A_dn"], cfg.ranks))

    def fwd(flags=0, prof=None, hidden=None, logits=None, slot=None, o=out, outputs=None):
        flags |= args.flags | (pkg.FLAG_SHARED_OUTER if cfg.shared_outer else 0)
        hid = g["hidden"] if hidden is None else hidden
        lg = g["router_logits"] if logits is None else logits
        kw = dict(routing_method=cfg.method, correction_bias=g["correction_bias"],
                  routed_scaling_factor=cfg.rsf, lora_A_gu=g["lora_A_gu"], lora_B_gu=g["lora_B_gu"],
                  lora_A_dn=g["lora_A_dn"], lora_B_dn=g["lora_B_dn"],
                  slot_idx=g["slot_idx"] if slot is None else slot, ranks=cfg.ranks, scalings=cfg.scalings,
                  flags=flags, out=o, workspace=ws, prof_events=prof, outputs=outputs)
        if w8 is not None:
            return pkg.moe_lora_forward_fp8(h, hid, lg, *w8, k, **kw, **packed)
        if w4 is not None:
            return pkg.moe_lora_forward_nvfp4(h, hid, lg, *w4, k, **kw)
        return pkg.moe_lora_forward(h, hid, lg, g["w1"], g["w2"], k, **kw, **packed)
    return fwd


# the benchmark's other configurations (multi-slot, skewed prefill, Kimi-like decode and
# prefill), timed beside the headline decode workload, in this order
SIDE_WORKLOADS = ["multi_slot", "prefill_zipf", "kimi_decode", "kimi_prefill"]
SIDE_BUDGET_S = 4.0   # timed seconds per side workload (LoRA on); steps are capped to fit


def measure_side_workload(name, args, h, local, peaks):
    """One entry of the line's `workloads` object: the same measurements as the headline
    (device-timed steps with inputs resident in HBM, LoRA-on / LoRA-off, the step's roofline
    fraction and both GEMMs' roofline blocks) on another configuration.  Steps are the run's
    --steps, capped so the timed region stays near SIDE_BUDGET_S; warm-up is the run's."""
    import torch
    import routed_moe_expert_gb300 as pkg
    from routed_moe_expert_gb300 import workloads as wl

    cfg = wl.CONFIGS[name]
    g = wl.make_inputs(cfg, seed=args.seed, device="cuda")
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k
    P = T * k
    ws = pkg.alloc_workspace(T, H, I, E, k, cfg.S, cfg.R)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    fwd = _make_fwd(pkg, h, cfg, g, ws, out, k, args)
    touched, lora_blocks, loads = _touched_and_lora(cfg, fwd, pkg, ws, T, E, k, I, H, g, torch)
    slots = g["slot_idx"].cpu().numpy()
    w_bytes_expert = 3 * H * I * 2
    io_bytes = T * H * 2 * 2 + T * E * 2
    step_bytes = touched * w_bytes_expert + lora_blocks + io_bytes
    step_flops = 2 * 3 * H * I * P + sum(2 * cfg.ranks[int(slots[t])] * (2 * H + 3 * I) * k
                                         for t in range(T) if cfg.S > 0 and slots[t] >= 0)
    act_fused = _act_in_gate_up(P, E)
    gu_bytes = touched * (2 * I * H * 2) + P * H * 2 + (P * I * 2 if act_fused else P * 2 * I * 2)
    gu_flops = 2 * 2 * I * H * P
    dn_bytes = touched * (H * I * 2) + P * I * 2 + P * H * 4
    dn_flops = 2 * H * I * P

    for _ in range(args.warmup):
        fwd()
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    for _ in range(3):
        fwd()
    torch.cuda.synchronize()
    est = (time.perf_counter() - w0) / 3
    steps = int(max(args.warmup, min(args.steps, SIDE_BUDGET_S / max(est, 1e-6))))
    sec, gu_s, dn_s, clk = _timed_steps(fwd, stream, steps, torch, pkg, clock_index=local)
    ms = 1e3 * sec / steps
    tc_peak = peaks["bf16_tflops_sustained"]
    tc_src = f"{peaks['source']} bf16_tflops_sustained (kernel timed inside a long loop)"
    t_hbm = step_bytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = step_flops / (tc_peak * 1e12)
    entry = {
        "workload": cfg.describe(), "T": T, "H": H, "I": I, "E": E, "top_k": k,
        "lora_ranks": list(cfg.ranks), "routing": "DeepSeekV3" if cfg.method else "Renormalize",
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms, "tokens_per_s": T / (ms / 1e3),
        "touched_experts": touched, "max_over_mean_expert_load": float(loads.max() / max(loads.mean(), 1e-9)),
        "step_bytes": step_bytes, "step_flops": step_flops,
        "step_bound": "tensor" if t_tc > t_hbm else "hbm",
        "step_roofline_frac": max(t_hbm, t_tc) / (ms / 1e3),
        "step_roofline_peak": (f"{tc_peak} TFLOP/s ({tc_src})" if t_tc > t_hbm
                               else f"{peaks['hbm_gbs']} GB/s ({peaks['source']} hbm_gbs)"),
        "l2": f"inputs larger than L2: {touched} touched experts = {touched * w_bytes_expert / 1e9:.2f} GB "
              f"of weights per step",
        "gate_up_gemm": _gemm_roofline("grouped_gemm (gate_up)", gu_flops, gu_bytes, gu_s, peaks, tc_peak, tc_src),
        "down_gemm": _gemm_roofline("grouped_gemm (down)", dn_flops, dn_bytes, dn_s, peaks, tc_peak, tc_src),
        "clocks": clk,
    }
    if cfg.S > 0:
        off_ms = _lora_off_ms(fwd, stream, max(1, steps // 2), args.warmup, torch, pkg)
        entry["lora_off_ms_per_step"] = off_ms
        entry["lora_on_over_off"] = off_ms / ms
    st, word = pkg.moe_lora_check_status(ws)
    if st != 0:
        raise RuntimeError(f"{name}: device status {word:#x}")
    del g, ws, out, fwd
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry


def run_gpu(args):
    import torch
    import torch.distributed as dist
    import routed_moe_expert_gb300 as pkg
    from routed_moe_expert_gb300 import _build
    from routed_moe_expert_gb300 import workloads as wl

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    if rank == 0 or world > 1:
        _build.build()
    cfg = wl.CONFIGS[args.workload]
    inp = wl.make_inputs(cfg, seed=args.seed, device="cuda")
    g = inp
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k
    # --fp8: the same layer with block-FP8 expert weights quantised from the drawn ones
    w8 = None
    if args.fp8:
        w1q, w1s = wl.quantize_weights_fp8(g["w1"])
        w2q, w2s = wl.quantize_weights_fp8(g["w2"])
        w8 = (w1q, w1s, w2q, w2s)
    # --nvfp4: the same layer with NVFP4 expert weights quantised from the drawn ones
    w4 = None
    if args.nvfp4:
        w4 = wl.quantize_weights_nvfp4(g["w1"]) + wl.quantize_weights_nvfp4(g["w2"])
    quant = w8 is not None or w4 is not None
    P = T * k
    h = pkg.Handle(local)
    ws = pkg.alloc_workspace(T, H, I, E, k, cfg.S, cfg.R)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    fwd = _make_fwd(pkg, h, cfg, g, ws, out, k, args, w8, w4)

    # touched experts (routing is fixed for the fixed input)
    touched, lora_blocks, _ = _touched_and_lora(cfg, fwd, pkg, ws, T, E, k, I, H, g, torch)
    slots = g["slot_idx"].cpu().numpy()

    # algorithmic bytes / flops (FP8: one byte per weight plus a float per 128 x 128 block,
    # the permuted hidden rows as codes plus a float per 128 values; NVFP4: half a byte per
    # weight plus a byte per 16 and two floats per expert, the permuted hidden rows as the
    # f16 values the GEMM reads plus a float per row)
    if w4 is not None:
        w_bytes_expert = 3 * H * I // 2 + 3 * H * I // 16 + 8
    else:
        wb = 1 if w8 is not None else 2
        w_bytes_expert = 3 * H * I * wb + (3 * H * I // (128 * 128) * 4 if w8 is not None else 0)
    io_bytes = T * H * 2 * 2 + T * E * 2
    step_bytes = touched * w_bytes_expert + lora_blocks + io_bytes
    step_flops = 2 * 3 * H * I * P + sum(2 * cfg.ranks[max(int(slots[t]), 0)] * (2 * H + 3 * I) * k
                                         for t in range(T) if cfg.S > 0 and slots[t] >= 0)
    act_fused = not quant and _act_in_gate_up(P, E)
    g_out = P * I * 2 if act_fused else P * 2 * I * 2
    if w4 is not None:
        gu_bytes = touched * (2 * I * H // 2 + 2 * I * H // 16 + 4) + P * H * 2 + P * 4 + P * 2 * I * 2
    elif w8 is None:
        gu_bytes = touched * (2 * I * H * 2) + P * H * 2 + g_out   # weights + xp read + g (or a) write
    else:
        gu_bytes = touched * (2 * I * H + 2 * I * H // (128 * 128) * 4) + P * H + P * H // 128 * 4 + P * 2 * I * 2
    gu_flops = 2 * 2 * I * H * P

    for _ in range(args.warmup):
        fwd()
    torch.cuda.synchronize()

    # ---- device-timed region: K steps (gate_up and down GEMM events on every 16th step)
    launches0 = h.launch_count()
    sec, gu_avg_s, dn_avg_s, clk = _timed_steps(fwd, stream, args.steps, torch, pkg, clock_index=local,
                                                world=world)
    launches = h.launch_count() - launches0
    sec_max = max_over_ranks(sec, world)
    agg = aggregate(T, args.steps, world, sec_max)

    # ---- end-to-end: inputs from pinned host memory each step, result back to host
    h_hidden = g["hidden"].cpu().pin_memory()
    h_logits = g["router_logits"].cpu().pin_memory()
    h_slot = g["slot_idx"].cpu().pin_memory()
    h_out = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    h2d = h_hidden.numel() * 2 + h_logits.numel() * 2 + h_slot.numel() * 4
    d2h = h_out.numel() * 2
    e2e_steps = max(1, args.steps // 4)
    # Each step copies its inputs in and its output back.  The copies run on two copy
    # streams against double-buffered device inputs and outputs, so step i's copies overlap
    # the neighbouring steps' forwards (which stay in order on the compute stream, sharing
    # one workspace), as a serving loop would run them.
    bufs = [dict(hidden=torch.empty_like(g["hidden"]), logits=torch.empty_like(g["router_logits"]),
                 slot=torch.empty_like(g["slot_idx"]), out=torch.empty_like(out)) for _ in range(2)]
    cs_in, cs_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in, ev_fwd, ev_d2h = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def e2e_step(i):
        b, j = bufs[i % 2], i % 2
        with torch.cuda.stream(cs_in):
            cs_in.wait_event(ev_fwd[j])        # the forward that last read these inputs is done
            b["hidden"].copy_(h_hidden, non_blocking=True)
            b["logits"].copy_(h_logits, non_blocking=True)
            b["slot"].copy_(h_slot, non_blocking=True)
            ev_in[j].record(cs_in)
        stream.wait_event(ev_in[j])
        stream.wait_event(ev_d2h[j])           # this output buffer has been read back
        fwd(hidden=b["hidden"], logits=b["logits"], slot=b["slot"], o=b["out"])
        ev_fwd[j].record(stream)
        with torch.cuda.stream(cs_out):
            cs_out.wait_event(ev_fwd[j])
            h_out.copy_(b["out"], non_blocking=True)
            ev_d2h[j].record(cs_out)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    cs_in.wait_event(e0)                       # the first copy starts inside the timed region
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_event(ev_d2h[(e2e_steps - 1) % 2])   # ... and the last read-back ends in it
    e1.record(stream)
    torch.cuda.synchronize()
    e_sec = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    e2e_val = aggregate(T, e2e_steps, world, e_sec)["value"]

    peaks = load_peaks()
    # the gate_up GEMM is HBM-bound when its bytes take longer than its flops at peak
    t_hbm = gu_bytes / (peaks["hbm_gbs"] * 1e9)
    # the ncu summaries cover the bf16 GEMM only
    traffic = profiled_traffic(f"gate_up_gemm_{args.workload}.md") if not quant else None
    kname = ("grouped_gemm_fp8 (gate_up)" if w8 is not None else
             "grouped_gemm_nvfp4 (gate_up)" if w4 is not None else "grouped_gemm (gate_up)")
    # an e4m3 contraction's peak: the measured bf16 peak times the nominal fp8 / bf16 ratio (2)
    tc_peak = peaks["bf16_tflops_sustained"] * (2 if w8 is not None else 1)
    tc_src = (f"{peaks['source']} bf16_tflops_sustained x 2 (nominal e4m3 / bf16 ratio)" if w8 is not None
              else f"{peaks['source']} bf16_tflops_sustained (kernel timed inside a long loop)")
    t_tc = gu_flops / (tc_peak * 1e12)
    tensor_bound = t_tc > t_hbm
    line = {
        "metric": METRIC, "value": agg["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": agg["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": ("e4m3 expert weights and GEMM inputs, bf16 LoRA" if w8 is not None else
                  "NVFP4 (e2m1, e4m3 per 16 values) expert weights and GEMM inputs, f16 tensor-core products, "
                  "bf16 LoRA" if w4 is not None else "bf16"), "data": "synthetic",
        "config": {
            "workload": cfg.describe(), "T": T, "H": H, "I": I, "E": E, "top_k": k,
            "lora_ranks": list(cfg.ranks), "routing": "DeepSeekV3" if cfg.method else "Renormalize",
            "l2": f"inputs larger than L2: {touched} touched experts = {touched * w_bytes_expert / 1e9:.2f} GB of weights per step",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "forward_flags": args.flags,
            "lora_b": ("per slot" if (args.per_slot_lora or w4 is not None)
                       else "expand- and shrink-ready copies (moe_lora_pack_lora_b / _a, made once at set-up)"),
            "step_bytes": step_bytes, "step_flops": step_flops,
            "step_roofline_frac": max(step_bytes / (peaks["hbm_gbs"] * 1e9),
                                      step_flops / (tc_peak * 1e12)) / (agg["ms_per_step"] / 1e3),
        },
        "roofline": ({
            "kernel": kname, "bound": "tensor", "achieved": gu_flops / gu_avg_s / 1e12,
            "peak": tc_peak, "unit": "TFLOP/s",
            "frac": gu_flops / gu_avg_s / 1e12 / tc_peak, "traffic": traffic,
            "peak_source": tc_src,
            "algorithmic_flops_per_launch": gu_flops, "algorithmic_bytes_per_launch": gu_bytes,
            "avg_launch_us": gu_avg_s * 1e6,
        } if tensor_bound else {
            "kernel": kname, "bound": "hbm", "achieved": gu_bytes / gu_avg_s / 1e9,
            "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gu_bytes / gu_avg_s / 1e9 / peaks["hbm_gbs"],
            "traffic": traffic, "peak_source": f"{peaks['source']} hbm_gbs",
            "algorithmic_bytes_per_launch": gu_bytes, "avg_launch_us": gu_avg_s * 1e6,
        }),
        "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if cfg.S > 0:
        # LoRA-off throughput of the same kernels, for the on/off ratio
        off_ms = _lora_off_ms(fwd, stream, max(1, args.steps // 4), args.warmup, torch, pkg)
        line["config"]["lora_off_ms_per_step"] = off_ms
        line["config"]["lora_on_over_off"] = off_ms / agg["ms_per_step"]
    if args.stage_times:
        # average device time of every stage of the forward (events on the stream that runs
        # each stage), LoRA on and LoRA off
        n_ev = 2 * pkg.NUM_STAGES
        for label, fl in (("lora_on", 0), ("lora_off", pkg.FLAG_LORA_OFF)):
            n = 50
            evsets = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(n)]
            for evs in evsets:
                for e_ in evs:
                    e_.record(stream)
            torch.cuda.synchronize()
            for i in range(n):
                fwd(flags=fl, prof=evsets[i])
            torch.cuda.synchronize()
            st_ms = {}
            for si, name in enumerate(pkg.STAGES):
                vals = []
                for evs in evsets:
                    try:
                        v_ = evs[2 * si].elapsed_time(evs[2 * si + 1])
                    except RuntimeError:
                        continue
                    if v_ > 0:
                        vals.append(v_)
                if vals:
                    st_ms[name] = round(1e3 * statistics.median(vals), 2)
            line.setdefault("stage_us", {})[label] = st_ms
    # the other benchmark configurations, one after another on the same GPU (rank 0 of a
    # single-GPU run only: replicas would repeat the same numbers), each freed before the next
    side = [] if (quant or world > 1 or args.workload != "decode" or args.no_workloads) else \
        [w for w in SIDE_WORKLOADS if args.only_workloads is None or w in args.only_workloads.split(",")]
    if side:
        del fwd, ws, out, bufs
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        line["workloads"] = {}
        for name in side:
            line["workloads"][name] = measure_side_workload(name, args, h, local, peaks)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, inp, args, w8=w8, w4=w4)
    if rank == 0:
        print(json.dumps(line), flush=True)
    h.close()
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------------------------------------
# CPU oracle (baseline leg / reference arm)
# ------------------------------------------------------------------------------------

def _oracle_inputs(cfg, inp):
    f = lambda t: None if t is None else (t.float().cpu().numpy() if t.dtype.is_floating_point else t.cpu().numpy())
    return {k: (f(v) if hasattr(v, "dtype") and hasattr(v, "cpu") else v) for k, v in inp.items()}


def _oracle_call(cfg, o, tokens):
    from oracle import moe_lora_oracle as orc
    if "w1nv" in o:   # NVFP4 expert weights
        return orc.moe_lora_forward_nvfp4(o["hidden"], o["router_logits"], o["w1nv"], o["w2nv"], cfg.top_k,
                                          cfg.method, o["correction_bias"], cfg.rsf, o["lora_A_gu"], o["lora_B_gu"],
                                          o["lora_A_dn"], o["lora_B_dn"], o["slot_idx"], cfg.ranks, cfg.scalings,
                                          tokens=tokens, shared_outer=cfg.shared_outer)
    if "w1q" in o:   # block-FP8 expert weights
        return orc.moe_lora_forward_fp8(o["hidden"], o["router_logits"], o["w1q"], o["w1s"], o["w2q"], o["w2s"],
                                        cfg.top_k, cfg.method, o["correction_bias"], cfg.rsf, o["lora_A_gu"],
                                        o["lora_B_gu"], o["lora_A_dn"], o["lora_B_dn"], o["slot_idx"], cfg.ranks,
                                        cfg.scalings, tokens=tokens, shared_outer=cfg.shared_outer)
    return orc.moe_lora_forward(o["hidden"], o["router_logits"], o["w1"], o["w2"], cfg.top_k, cfg.method,
                                o["correction_bias"], cfg.rsf, o["lora_A_gu"], o["lora_B_gu"], o["lora_A_dn"],
                                o["lora_B_dn"], o["slot_idx"], cfg.ranks, cfg.scalings, tokens=tokens,
                                shared_outer=cfg.shared_outer)


def cpu_baseline(cfg, inp, args, budget_s: float = None, w8=None, w4=None) -> dict:
    """Time the oracle, as it stands, on a bounded sample of the workload: a token subset
    that grows until one call takes a good part of the budget, then repeated calls until
    about `budget_s` seconds of CPU work are done (tokens/s over all of them).  With w8
    (block-FP8 weights) the oracle's FP8 layer runs on those codes and scales, with w4 (NVFP4
    weights) its NVFP4 layer."""
    budget_s = args.cpu_budget if budget_s is None else budget_s
    if w8 is not None or w4 is not None:
        inp = {k_: v for k_, v in inp.items() if k_ not in ("w1", "w2")}
    o = _oracle_inputs(cfg, inp)
    if w8 is not None:
        o.update(w1q=w8[0].cpu().numpy(), w1s=w8[1].cpu().numpy(), w2q=w8[2].cpu().numpy(), w2s=w8[3].cpu().numpy())
    if w4 is not None:
        c = [t.cpu().numpy() for t in w4]
        o.update(w1nv=tuple(c[:3]), w2nv=tuple(c[3:]))
    n_tok = min(cfg.T, 8)
    t0 = time.perf_counter()
    _oracle_call(cfg, o, np.arange(n_tok))
    dt = time.perf_counter() - t0
    # grow the token subset while one call stays well inside the budget
    while dt * 4 < budget_s and n_tok < cfg.T:
        n_tok = min(cfg.T, n_tok * 2)
        t0 = time.perf_counter()
        _oracle_call(cfg, o, np.arange(n_tok))
        dt = time.perf_counter() - t0
    # repeat that call until the budget is spent
    done, spent, calls = 0, 0.0, 0
    while calls == 0 or spent + dt <= budget_s:
        t0 = time.perf_counter()
        _oracle_call(cfg, o, np.arange(n_tok))
        dt = time.perf_counter() - t0
        done, spent, calls = done + n_tok, spent + dt, calls + 1
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return dict(value=done / spent, unit=UNIT, cores=cores, kind="oracle",
                sample=f"{calls} calls on the first {n_tok} of {cfg.T} tokens of the {cfg.name} workload (full "
                       f"routing of all tokens each call), {spent:.1f} s, numpy float64 with its default BLAS threads")


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return
    import torch
    from routed_moe_expert_gb300 import workloads as wl
    cfg = wl.CONFIGS[args.workload]
    inp = wl.make_inputs(cfg, seed=args.seed, device="cpu")
    o = _oracle_inputs(cfg, inp)
    n_tok = max(1, min(cfg.T, args.ref_tokens))
    for _ in range(min(args.warmup, 1)):
        _oracle_call(cfg, o, np.arange(n_tok))
    steps = max(1, min(args.steps, args.ref_steps))
    t0 = time.perf_counter()
    for _ in range(steps):
        _oracle_call(cfg, o, np.arange(n_tok))
    dt = time.perf_counter() - t0
    val = n_tok * steps / dt
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sample = f"{n_tok} of {cfg.T} tokens per step, {steps} steps, CPU oracle (numpy float64)"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * dt / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.describe()},
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_routed(args):
    """Auxiliary line: the externally routed entry on the same workload, with the routing
    given as packed top-k words (seeded, every expert local) and do_finalize as asked.
    Not the headline metric: it times the layer without its router."""
    import torch
    import routed_moe_expert_gb300 as pkg
    from routed_moe_expert_gb300 import _build
    from routed_moe_expert_gb300 import workloads as wl

    _build.build()
    cfg = wl.CONFIGS[args.workload]
    g = wl.make_inputs(cfg, seed=args.seed, device="cuda")
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k
    ids, w = wl.make_routing(T, E, k, seed=args.seed + 1)
    packed = wl.packed_routing_words(ids, w).cuda()
    h = pkg.Handle(0)
    ws = pkg.alloc_workspace(T, H, I, E, k, cfg.S, cfg.R)
    fin = args.routed == "finalize"
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    extra = {} if fin else dict(gemm2_output=torch.empty((T * k, H), dtype=torch.float32, device="cuda"),
                                activation_output=torch.empty((T * k, I), dtype=torch.bfloat16, device="cuda"))

    def fwd():
        pkg.moe_lora_forward_routed(h, g["hidden"], packed, g["w1"], g["w2"], k, E, do_finalize=fin,
                                    lora_A_gu=g["lora_A_gu"], lora_B_gu=g["lora_B_gu"], lora_A_dn=g["lora_A_dn"],
                                    lora_B_dn=g["lora_B_dn"], slot_idx=g["slot_idx"], ranks=cfg.ranks,
                                    scalings=cfg.scalings, out=out, workspace=ws, **extra,
                                    flags=args.flags | (pkg.FLAG_SHARED_OUTER if cfg.shared_outer else 0))

    for _ in range(args.warmup):
        fwd()
    torch.cuda.synchronize()
    st, word = pkg.moe_lora_check_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {word:#x}")
    stream = torch.cuda.current_stream()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        fwd()
    t1.record(stream)
    torch.cuda.synchronize()
    sec = t0.elapsed_time(t1) / 1e3
    print(json.dumps({
        "metric": METRIC, "value": T * args.steps / sec, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sec * 1e3 / args.steps, "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{cfg.name} through moe_lora_forward_routed (packed top-k, every expert "
                               f"local, do_finalize={int(fin)})", "T": T, "H": H, "I": I, "E": E, "top_k": k},
        "entry": "routed"}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-tokens", type=int, default=16)
    ap.add_argument("--ref-steps", type=int, default=5)
    ap.add_argument("--flags", type=int, default=0, help="extra moe_lora_forward flags (e.g. 8: unfused LoRA)")
    ap.add_argument("--per-slot-lora", action="store_true",
                    help="no expand-ready LoRA B copies: the fused LoRA stages read B per slot")
    ap.add_argument("--stage-times", action="store_true", help="add per-stage device times (us) to the line")
    ap.add_argument("--fp8", action="store_true",
                    help="block-FP8 expert weights (e4m3, 128x128 scales) quantised from the drawn bf16 ones")
    ap.add_argument("--nvfp4", action="store_true",
                    help="NVFP4 expert weights (e2m1, e4m3 scale per 16, float32 per expert) quantised from the "
                         "drawn bf16 ones")
    ap.add_argument("--routed", choices=["finalize", "unfinalized"], default=None,
                    help="time the externally routed entry instead (auxiliary line, not the headline)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="time the decode headline only (no `workloads` object for the other configurations)")
    ap.add_argument("--only-workloads", default=None,
                    help="comma-separated subset of the other configurations to time")
    args = ap.parse_args()
    if (args.fp8 or args.nvfp4) and (args.routed or args.impl == "reference"):
        ap.error("--fp8 / --nvfp4 time the quantised layers through moe_lora_forward_fp8 / _nvfp4; they do not "
                 "combine with --routed or --impl reference")
    if args.fp8 and args.nvfp4:
        ap.error("choose one of --fp8 and --nvfp4")
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.routed:
        run_routed(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
