#!/usr/bin/env python
"""Benchmark of the routed-expert MoE layer (one GB300 per rank).

A step is one full layer call -- router logits, top-8 + weights, bucketing,
shared expert, grouped routed experts, weighted combine -- on one decode batch
of synthetic tokens.  The default workload is decode batch 8 with 4-bit g64
experts, a 4-bit shared expert with an 8-bit sigmoid gate, an fp32 router and
Zipf(1.1)-skewed routing (hidden 2048, 256 experts, top-8, intermediate 512).

Timing: the K timed steps run as CUDA-graph replays on one stream, bracketed by
CUDA events; steps rotate over 8 independent layer-weight banks (~3.6 GB,
far larger than the 129 MB L2) and 16 token batches, so every step streams its
experts from HBM.  `value` is whole-job tokens/s (max time over ranks).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gpu|reference]
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "decode8_affine4_shared_zipf"
E, K_TOP, H, I = 256, 8, 2048, 512


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--banks", type=int, default=8)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    return p.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only: no data-path collective)

def dist_init(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, ws: int) -> float:
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# byte accounting (algorithmic bytes: what the step must read or write once)

BITS = {"affine8_g64": 8, "affine4_g64": 4, "affine3_g64": 3, "w4a16_g128": 4}
GROUP = {"affine8_g64": 64, "affine4_g64": 64, "affine3_g64": 64, "w4a16_g128": 128}


def kernel_source_hash(read=None) -> str:
    """sha256 over the library's kernel sources and public header (file names
    and contents, sorted), used to tell whether an ncu capture still matches."""
    import hashlib
    csrc = os.path.join(ROOT, "bit_affine_quantized_fp32_gb300", "csrc")
    names = sorted(f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h")))
    files = [("bit_affine_quantized_fp32_gb300/csrc/" + f) for f in names] + ["include/moe_gb300.h"]
    h = hashlib.sha256()
    for rel in files:
        data = read(rel) if read else open(os.path.join(ROOT, rel), "rb").read()
        h.update(rel.encode() + b"\0" + data + b"\0")
    return h.hexdigest()


def captured_traffic():
    """DRAM bytes per launch of the fused kernel from the committed ncu
    summary, or None when the kernel sources changed since that capture."""
    p = os.path.join(ROOT, "profiles", "k_decode_traffic.json")
    try:
        rec = json.load(open(p))
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != kernel_source_hash():
        return None
    return int(rec["dram_bytes_per_launch"])


def matrix_bytes(fmt: str | None, rows: int, cols: int) -> int:
    if fmt is None:
        return 0
    if fmt == "f32":
        return rows * cols * 4
    if fmt in ("bf16", "f16"):
        return rows * cols * 2
    n = rows * cols
    b = n * BITS[fmt] // 8
    groups = n // GROUP[fmt]
    return b + groups * 2 * (1 if fmt == "w4a16_g128" else 2)


def expert_bytes(fmt: str) -> int:
    return matrix_bytes(fmt, 2 * I, H) + matrix_bytes(fmt, H, I)


# ---------------------------------------------------------------------------
# clocks sampled during the timed region

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.15)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        return parse_clock_lines(self.lines)


def parse_clock_lines(lines) -> dict:
    """Median SM clock, maximum SM clock and the throttle reasons seen, from
    `nvidia-smi --query-gpu=<ClockSampler.FIELDS> --format=csv,noheader,nounits`
    lines (a reason counts when its column reads Active)."""
    sm, smax, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for ln in lines:
        parts = [p.strip() for p in ln.split(",")]
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
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# GPU arm

class RawBank:
    """Weight bank b of a workload in its canonical stored form (the seeded
    generators' tensors on `device`); the oracle reads these.  No library
    call is made here."""
    def __init__(self, cfg: dict, b: int, device):
        from bit_affine_quantized_fp32_gb300 import synth
        seed = 1000 + 97 * b + cfg["seed"]
        self.cfg = cfg
        self.raw = {"router": synth.device_matrix(cfg["router_fmt"], E, H, seed, device),
                    "experts": synth.device_bank(cfg["expert_fmt"], E, I, H, seed + 2, device)}
        self.bias = synth.device_zipf_bias(E, seed + 1, device) if cfg["zipf"] else None
        if cfg["shared_fmt"]:
            self.raw["shared"] = synth.device_bank(cfg["shared_fmt"], 1, I, H, seed + 3, device)
        if cfg["gate_fmt"]:
            self.raw["gate"] = synth.device_matrix(cfg["gate_fmt"], 1, H, seed + 4, device)


class Bank(RawBank):
    """The same bank as the library's handles, experts repacked to the tiled
    layout on the GPU."""
    def __init__(self, cfg: dict, b: int, device):
        import torch
        from bit_affine_quantized_fp32_gb300 import capi
        super().__init__(cfg, b, device)
        r, ex = self.raw["router"], self.raw["experts"]
        self.router = capi.QMatrix(cfg["router_fmt"], E, H, r["q"], r["s"], r["b"])
        self.experts = capi.ExpertBank(cfg["expert_fmt"], E, I, H, ex["w13"], ex["s13"], ex["b13"],
                                       ex["w2"], ex["s2"], ex["b2"]).tiled()
        self.shared = self.gate = None
        if cfg["shared_fmt"]:
            sh = self.raw["shared"]
            self.shared = capi.ExpertBank(cfg["shared_fmt"], 1, I, H, sh["w13"], sh["s13"],
                                          sh["b13"], sh["w2"], sh["s2"], sh["b2"]).tiled()
        if cfg["gate_fmt"]:
            g = self.raw["gate"]
            self.gate = capi.QMatrix(cfg["gate_fmt"], 1, H, g["q"], g["s"], g["b"])
        torch.cuda.synchronize()


def run_gpu(args, ws_world, rank, local):
    import torch
    from bit_affine_quantized_fp32_gb300 import build as B
    B.build()
    from bit_affine_quantized_fp32_gb300 import capi, synth

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    cfg = dict(synth.WORKLOADS[args.workload])
    T = cfg["T"]
    act = cfg["act"]
    banks = [Bank(cfg, b, device) for b in range(args.banks)]
    n_in = 16
    xs = [synth.device_x(T, H, act, 500 + 31 * i + rank, device) for i in range(n_in)]
    wsb = capi.moe_workspace_bytes(T, E, K_TOP, H, I)
    ws = torch.empty(wsb, dtype=torch.uint8, device=device)
    capi.moe_workspace_init(ws)
    out = torch.empty((T, H), dtype=xs[0].dtype, device=device)

    def step(i, x=None, o=None):
        bk = banks[i % len(banks)]
        capi.moe_layer_forward(bk.router, bk.bias, bk.gate, bk.experts, bk.shared,
                               xs[i % n_in] if x is None else x, K_TOP,
                               out if o is None else o, None, None, 0, ws)

    # experts touched per (bank, batch): from the library's own routing
    pairs = math.lcm(len(banks), n_in)
    U = []
    offs = torch.empty(E + 1, dtype=torch.int32, device=device)
    perm = torch.empty(T * K_TOP, dtype=torch.int32, device=device)
    idx = torch.empty((T, K_TOP), dtype=torch.int32, device=device)
    wt = torch.empty((T, K_TOP), dtype=torch.float32, device=device)
    for i in range(pairs):
        bk = banks[i % len(banks)]
        capi.moe_route(bk.router, bk.bias, bk.gate, xs[i % n_in], K_TOP, None, idx, wt, None,
                       offs, perm, ws)
        U.append(int((offs[1:] - offs[:-1] > 0).sum().item()))
    eb = expert_bytes(cfg["expert_fmt"])
    fixed = (matrix_bytes(cfg["router_fmt"], E, H) + matrix_bytes(cfg["gate_fmt"], 1, H) +
             (expert_bytes(cfg["shared_fmt"]) if cfg["shared_fmt"] else 0) + 2 * T * H * 2)
    step_bytes = [u * eb + fixed for u in U]

    def bytes_for(steps):
        return sum(step_bytes[i % pairs] for i in range(steps))

    # eager warm-up (sets kernel attributes outside capture)
    for i in range(3):
        step(i)
    torch.cuda.synchronize()

    G = 64

    def capture(n, start):
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=device)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for j in range(n):
                    step(start + j)
        torch.cuda.current_stream().wait_stream(s)
        return g

    g_main = capture(G, 0)
    rem = args.steps % G
    g_rem = capture(rem, 0) if rem else None
    wrem = args.warmup % G
    g_wrem = capture(wrem, 0) if wrem else None

    def run_steps(n, main, remg):
        for _ in range(n // G):
            main.replay()
        if n % G:
            remg.replay()

    # warm-up steps (untimed)
    run_steps(args.warmup, g_main, g_wrem)
    torch.cuda.synchronize()
    barrier(ws_world)

    clocks = ClockSampler(local)
    clocks.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws_world)
    torch.cuda.synchronize()
    ev0.record()
    run_steps(args.steps, g_main, g_rem)
    ev1.record()
    torch.cuda.synchronize()
    barrier(ws_world)
    ms = ev0.elapsed_time(ev1)
    clk = clocks.stop()
    ms_max = max_over_ranks(ms, ws_world)
    tokens = T * args.steps * ws_world
    value = tokens / (ms_max / 1e3)
    step_ms = ms_max / args.steps
    gbs = bytes_for(args.steps) / (ms / 1e3) / 1e9

    # end to end through the C ABI with host buffers: pinned x in, out back, every step
    x_host = [xs[i].cpu().pin_memory() for i in range(n_in)]
    out_host = torch.empty((T, H), dtype=out.dtype).pin_memory()
    x_dev = torch.empty_like(xs[0])

    def e2e_step(i):
        x_dev.copy_(x_host[i % n_in], non_blocking=True)
        step(i, x=x_dev)
        out_host.copy_(out, non_blocking=True)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    ge = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device=device)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(ge, stream=s):
            for j in range(G):
                e2e_step(j)
    torch.cuda.current_stream().wait_stream(s)
    ge.replay()
    torch.cuda.synchronize()
    n_e2e = max(G, (args.steps // G) * G)
    barrier(ws_world)
    ev0.record()
    for _ in range(n_e2e // G):
        ge.replay()
    ev1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(ev0.elapsed_time(ev1), ws_world)
    e2e_value = T * n_e2e * ws_world / (e2e_ms / 1e3)

    # correctness of the timed configuration: the last step's output is finite
    assert torch.isfinite(out.float()).all()
    assert capi.moe_get_device_status(ws) == 0

    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    peak = float(peaks.get("hbm_gbs", 6800.0))
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"

    # one persistent launch per layer call for decode batches (<= 32 tokens);
    # the prefill form: routing (3), shared expert (2), tiles and sub-slots
    # (2), tensor-core gate/up and down (2), activation sums, decode units for
    # the light experts (2), combine
    launches_per_step = 1 if T <= 32 else 3 + (2 if cfg["shared_fmt"] else 0) + 8
    line = {
        "metric": "MoE-layer tokens/s (%s %d, %s)" % (
            "decode batch" if T <= 32 else "prefill window", T, cfg["expert_fmt"]),
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": ws_world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": act,
        "arith": (("%s activations times the exact integer codes (mma.sync), fp32 "
                   "accumulation, per-group scale and bias in fp32" % act) if T <= 32 else
                  "dequantised weights and h as 16-bit hi + lo parts (tcgen05), fp32 "
                  "accumulation in tensor memory"),
        "data": "synthetic (seeded; random-init weights of the layer's shapes)",
        "config": {"workload": args.workload, "tokens": T, "experts": E, "top_k": K_TOP,
                   "hidden": H, "inter": I, "expert_fmt": cfg["expert_fmt"],
                   "router_fmt": cfg["router_fmt"], "shared_fmt": cfg["shared_fmt"],
                   "gate_fmt": cfg["gate_fmt"], "zipf": cfg["zipf"],
                   "parallelism": f"replicas{ws_world}", "weight_banks": len(banks),
                   "l2": "inputs larger than L2 (%d rotating weight banks, %.1f GB)" % (
                       len(banks), len(banks) * (E * eb + fixed) / 1e9),
                   "experts_touched_mean": round(float(np.mean(U)), 2)},
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4),
                     "traffic": captured_traffic() if T <= 32 else None,
                     "kernel": ("k_decode: the whole layer in one persistent launch" if T <= 32
                                else "whole step (all launches of one layer call)"),
                     "peak_source": peak_src,
                     "algorithmic_bytes_per_step": round(float(np.mean(step_bytes)))},
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 2},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    return line, banks, xs, cfg


# ---------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)

def oracle_inputs(bank, cfg):
    """Host copies of one bank in the oracle's containers."""
    def m(d, fmt, rows, cols):
        if fmt == "f32":
            return {"fmt": fmt, "q": d["q"].cpu().numpy(), "rows": rows, "cols": cols}
        if fmt in ("bf16", "f16"):
            return {"fmt": fmt, "q": d["q"].cpu().view(__import__("torch").int16).numpy().view(np.uint16),
                    "rows": rows, "cols": cols}
        return {"fmt": fmt, "q": d["q"].cpu().numpy().view(np.uint32),
                "s": d["s"].cpu().numpy().view(np.uint16),
                "b": None if d["b"] is None else d["b"].cpu().numpy().view(np.uint16),
                "rows": rows, "cols": cols}

    def bank_np(d, fmt, n):
        out = {"fmt": fmt, "E": n, "I": I,
               "w13": d["w13"].cpu().numpy().view(np.uint32), "w2": d["w2"].cpu().numpy().view(np.uint32),
               "s13": d["s13"].cpu().numpy().view(np.uint16), "s2": d["s2"].cpu().numpy().view(np.uint16)}
        if d["b13"] is not None:
            out["b13"] = d["b13"].cpu().numpy().view(np.uint16)
            out["b2"] = d["b2"].cpu().numpy().view(np.uint16)
        return out

    r = m(bank.raw["router"], cfg["router_fmt"], E, H)
    ex = bank_np(bank.raw["experts"], cfg["expert_fmt"], E)
    sh = None
    if cfg["shared_fmt"]:
        sh = bank_np(bank.raw["shared"], cfg["shared_fmt"], 1)
        sh = {k: (v[0] if isinstance(v, np.ndarray) else v) for k, v in sh.items()}
    g = m(bank.raw["gate"], cfg["gate_fmt"], 1, H) if cfg["gate_fmt"] else None
    bias = bank.bias.cpu().numpy() if bank.bias is not None else None
    return r, ex, sh, g, bias


def time_oracle(bank, cfg, xs_np, seconds: float, max_steps: int | None = None,
                tokens_per_step: int = 1):
    from oracle import oracle as O
    O.build()
    cores = O.set_threads(0)
    r, ex, sh, g, bias = oracle_inputs(bank, cfg)
    done_tokens, steps = 0, 0
    t0 = time.perf_counter()
    i = 0
    while True:
        x = xs_np[i % len(xs_np)][:tokens_per_step]
        O.moe_layer(x, K_TOP, r, ex, sh, g, bias)
        done_tokens += x.shape[0]
        steps += 1
        i += 1
        el = time.perf_counter() - t0
        if max_steps is not None and steps >= max_steps:
            break
        if max_steps is None and el >= seconds:
            break
    el = time.perf_counter() - t0
    return done_tokens / el, cores, steps, el


def xs_to_np(xs, act):
    from oracle import oracle as O
    import torch
    out = []
    for x in xs:
        bits = x.cpu().view(torch.int16).numpy().view(np.uint16)
        out.append(O.act_to_double(act, bits))
    return out


def run_reference(args, ws_world, rank, local):
    """The oracle as it stands on the host cores, on the GPU arm's workload:
    each step is one token of the batch through the whole layer.  The inputs
    come from the same seeded generators as the GPU arm's, on the GPU when
    there is one (the same values), else on the CPU (same laws); the library
    is not used."""
    import torch
    from bit_affine_quantized_fp32_gb300 import synth
    cfg = dict(synth.WORKLOADS[args.workload])
    T = cfg["T"]
    have_gpu = torch.cuda.is_available()
    device = torch.device("cuda", local) if have_gpu else torch.device("cpu")
    if have_gpu:
        torch.cuda.set_device(local)
    bank = RawBank(cfg, 0, device)
    xs = [synth.device_x(T, H, cfg["act"], 500 + 31 * i, device) for i in range(16)]
    xs_np = xs_to_np(xs, cfg["act"])
    time_oracle(bank, cfg, xs_np, 0, max_steps=max(0, args.warmup))
    tps, cores, steps, el = time_oracle(bank, cfg, xs_np, 0, max_steps=args.steps)
    line = {
        "impl": "reference",
        "metric": "MoE-layer tokens/s (%s %d, %s)" % (
            "decode batch" if T <= 32 else "prefill window", T, cfg["expert_fmt"]),
        "value": round(tps, 3), "unit": "tokens/s", "n_gpus": ws_world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(el * 1e3 / max(1, steps), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; generated on the %s)" % ("GPU" if have_gpu else "CPU"),
        "config": {"workload": args.workload, "tokens": T, "experts": E, "top_k": K_TOP,
                   "hidden": H, "inter": I, "parallelism": "host cores"},
        "cpu_baseline": {"value": round(tps, 3), "unit": "tokens/s", "cores": cores,
                         "kind": "oracle",
                         "sample": "each step: one token of the batch through the whole layer "
                                   "(fp64 C++ oracle, OpenMP over experts)"},
        "e2e": {"value": round(tps, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    ws_world, rank, local = dist_init(args)
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, ws_world, rank, local)
        return
    line, banks, xs, cfg = run_gpu(args, ws_world, rank, local)
    if rank == 0 and ws_world == 1 and not args.no_cpu_baseline:
        xs_np = xs_to_np(xs, cfg["act"])
        tps, cores, steps, el = time_oracle(banks[0], cfg, xs_np, args.cpu_seconds,
                                            tokens_per_step=cfg["T"])
        line["cpu_baseline"] = {"value": round(tps, 3), "unit": "tokens/s", "cores": cores,
                                "kind": "oracle",
                                "sample": f"{steps} full decode batches of {cfg['T']} tokens "
                                          f"on weight bank 0 ({el:.1f} s, fp64 C++ oracle)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws_world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
