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
# A sweep runs a prompt of `windows` x T tokens of a base workload as that
# many consecutive layer calls of T tokens (one step = the whole prompt).
SWEEPS = {"prefill4096_affine4_zipf_sweep": ("prefill512_affine4_zipf", 8)}
OTHER_WORKLOADS = ["decode1_affine4", "decode4_affine3", "decode32_w4a16",
                   "prefill512_affine4_zipf", "prefill4096_affine4_zipf_sweep"]
E, K_TOP, H, I = 256, 8, 2048, 512


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--also", default=",".join(OTHER_WORKLOADS),
                   help="comma list of further workloads measured in the same run "
                        "(summarised under 'workloads'), or 'none'")
    p.add_argument("--other-steps", type=int, default=2000)
    p.add_argument("--banks", type=int, default=8)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=8.0,
                   help="seconds of oracle work at all threads, and again at one thread")
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


def captured_traffic(workload: str = DEFAULT_WORKLOAD):
    """DRAM bytes per layer call of `workload` from the committed ncu record
    (profiles/traffic_<workload>.json), or None when there is none or the
    kernel sources changed since that capture."""
    p = os.path.join(ROOT, "profiles", f"traffic_{workload}.json")
    try:
        rec = json.load(open(p))
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != kernel_source_hash():
        return None
    return int(rec["dram_bytes_per_step"])


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


def load_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def step_flops(cfg: dict, T: int) -> float:
    """Algorithmic FLOPs of one layer call: every routed (token, expert) pair
    and the shared expert run three I x H matrix-vector products (2 flops per
    weight), the router one E x H."""
    per_pair = 2.0 * 3 * I * H
    return (T * K_TOP * per_pair + (T * per_pair if cfg["shared_fmt"] else 0.0)
            + 2.0 * E * H * T + (2.0 * H * T if cfg["gate_fmt"] else 0.0))


def launches_per_step(cfg: dict, T: int) -> int:
    # one persistent launch per decode call (T <= 32); the prefill form:
    # routing (weight split, tensor-core router, top-k, bucket sort with the
    # tile and sub-slot tables), activation sums with the fp16 copy (1, on the
    # side stream), the tensor-core gate/up and down GEMMs (2, the shared
    # expert folded in), the decode units of the light experts (2) and the
    # combine (1); a shared expert of another format runs its own conversion
    # and two GEMMs, and the tables then take a launch of their own
    if T <= 32:
        return 1
    if cfg["shared_fmt"] and cfg["shared_fmt"] != cfg["expert_fmt"]:
        return 4 + 3 + 1 + 1 + 2 + 2 + 1
    return 4 + 1 + 2 + 2 + 1


def workload_cfg(name: str):
    """(config of one layer call, tokens per call, calls per step) of a
    workload or a sweep."""
    from bit_affine_quantized_fp32_gb300 import synth
    base, nwin = SWEEPS.get(name, (name, 1))
    cfg = dict(synth.WORKLOADS[base])
    return cfg, cfg["T"], nwin


def measure(name: str, steps: int, warmup: int, nbanks: int, ws_world: int, rank: int,
            device, keep: bool = False) -> dict:
    """Time `steps` steps of workload `name` (after `warmup`), device-only and
    end to end; a step is one layer call, or for a sweep the prompt's
    consecutive calls.  Returns the figures of one JSON line (and, with keep,
    the banks and inputs for the CPU baseline)."""
    import torch
    from bit_affine_quantized_fp32_gb300 import capi, synth

    cfg, Tw, nwin = workload_cfg(name)
    T = Tw * nwin                     # tokens per step
    act = cfg["act"]
    banks = [Bank(cfg, b, device) for b in range(nbanks)]
    n_in = 16
    xs = [synth.device_x(T, H, act, 500 + 31 * i + rank, device) for i in range(n_in)]
    wsb = capi.moe_workspace_bytes(Tw, E, K_TOP, H, I)
    ws = torch.empty(wsb, dtype=torch.uint8, device=device)
    capi.moe_workspace_init(ws)
    out = torch.empty((T, H), dtype=xs[0].dtype, device=device)

    def step(i, x=None, o=None):
        bk = banks[i % len(banks)]
        xx = xs[i % n_in] if x is None else x
        oo = out if o is None else o
        for w in range(nwin):  # consecutive windows of the prompt, one workspace
            capi.moe_layer_forward(bk.router, bk.bias, bk.gate, bk.experts, bk.shared,
                                   xx[w * Tw:(w + 1) * Tw], K_TOP, oo[w * Tw:(w + 1) * Tw],
                                   None, None, 0, ws)

    # experts touched per (bank, batch, window): from the library's own routing
    pairs = math.lcm(len(banks), n_in)
    eb = expert_bytes(cfg["expert_fmt"])
    fixed = (matrix_bytes(cfg["router_fmt"], E, H) + matrix_bytes(cfg["gate_fmt"], 1, H) +
             (expert_bytes(cfg["shared_fmt"]) if cfg["shared_fmt"] else 0) + 2 * Tw * H * 2)
    U = []
    step_bytes = []
    offs = torch.empty(E + 1, dtype=torch.int32, device=device)
    perm = torch.empty(Tw * K_TOP, dtype=torch.int32, device=device)
    idx = torch.empty((Tw, K_TOP), dtype=torch.int32, device=device)
    wt = torch.empty((Tw, K_TOP), dtype=torch.float32, device=device)
    for i in range(pairs):
        bk = banks[i % len(banks)]
        sb = 0
        for w in range(nwin):
            capi.moe_route(bk.router, bk.bias, bk.gate, xs[i % n_in][w * Tw:(w + 1) * Tw], K_TOP,
                           None, idx, wt, None, offs, perm, ws)
            u = int((offs[1:] - offs[:-1] > 0).sum().item())
            U.append(u)
            sb += u * eb + fixed
        step_bytes.append(sb)

    def bytes_for(n):
        return sum(step_bytes[i % pairs] for i in range(n))

    for i in range(3):  # eager warm-up (sets kernel attributes outside capture)
        step(i)
    torch.cuda.synchronize()

    G = 64

    def capture(fn, n):
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=device)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                fn(n)
        torch.cuda.current_stream().wait_stream(s)
        return g

    def plain(n):
        for j in range(n):
            step(j)

    graphs = {}

    def graph(fn, n):
        if (fn, n) not in graphs:  # capture once, outside any timed region
            graphs[(fn, n)] = capture(fn, n)
        return graphs[(fn, n)]

    def run_steps(fn, n):
        for _ in range(n // G):
            graph(fn, G).replay()
        if n % G:
            graph(fn, n % G).replay()

    # bring clocks and memory out of their idle states with ~0.3 s of untimed
    # calls before the counted warm-up steps
    t_pre = time.perf_counter()
    while time.perf_counter() - t_pre < 0.3:
        run_steps(plain, G)
        torch.cuda.synchronize()
    run_steps(plain, warmup)
    torch.cuda.synchronize()
    barrier(ws_world)

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    graph(plain, G)
    if steps % G:
        graph(plain, steps % G).replay()  # first replay (upload) outside the timed region
        torch.cuda.synchronize()
    clocks = ClockSampler(device.index or 0)
    clocks.start()
    barrier(ws_world)
    torch.cuda.synchronize()
    ev0.record()
    run_steps(plain, steps)
    ev1.record()
    torch.cuda.synchronize()
    barrier(ws_world)
    ms = ev0.elapsed_time(ev1)
    clk = clocks.stop()
    ms_max = max_over_ranks(ms, ws_world)
    value = T * steps * ws_world / (ms_max / 1e3)

    # End to end through the C ABI with host buffers, every step: x from
    # pinned host memory in, the output back to pinned host memory.  The
    # copies of step j + 1 (in) and j (out) run on two copy streams while the
    # layer call of step j runs, double-buffered on the device.
    x_host = [xs[i].cpu().pin_memory() for i in range(n_in)]
    out_host = [torch.empty((T, H), dtype=out.dtype).pin_memory() for _ in range(2)]
    xd = [torch.empty_like(xs[0]) for _ in range(2)]
    od = [torch.empty_like(out) for _ in range(2)]

    def e2e(n):
        main = torch.cuda.current_stream()
        cin, cout = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
        cin.wait_stream(main)
        cout.wait_stream(main)
        k_done = [None] * n
        h_done = [None] * (n + 1)
        d_done = [None] * n

        def h2d(j):
            with torch.cuda.stream(cin):
                if j >= 2:
                    cin.wait_event(k_done[j - 2])
                xd[j % 2].copy_(x_host[j % n_in], non_blocking=True)
                h_done[j] = torch.cuda.Event()
                h_done[j].record(cin)

        h2d(0)
        for j in range(n):
            if j + 1 < n:
                h2d(j + 1)
            main.wait_event(h_done[j])
            if j >= 2:
                main.wait_event(d_done[j - 2])
            step(j, x=xd[j % 2], o=od[j % 2])
            k_done[j] = torch.cuda.Event()
            k_done[j].record(main)
            with torch.cuda.stream(cout):
                cout.wait_event(k_done[j])
                out_host[j % 2].copy_(od[j % 2], non_blocking=True)
                d_done[j] = torch.cuda.Event()
                d_done[j].record(cout)
        main.wait_stream(cin)
        main.wait_stream(cout)

    n_e2e = max(G, (steps // G) * G)
    ge = capture(e2e, G)
    ge.replay()
    torch.cuda.synchronize()
    barrier(ws_world)
    ev0.record()
    for _ in range(n_e2e // G):
        ge.replay()
    ev1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(ev0.elapsed_time(ev1), ws_world)
    e2e_value = T * n_e2e * ws_world / (e2e_ms / 1e3)

    # the timed configuration ran cleanly: the last outputs are finite and the
    # workspace reports no timeout
    assert torch.isfinite(out.float()).all() and torch.isfinite(od[0].float()).all()
    assert capi.moe_get_device_status(ws) == 0

    peaks = load_peaks()
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    hbm_src = "measured" if "hbm_gbs" in peaks else "fallback"
    gbs = bytes_for(steps) / (ms / 1e3) / 1e9
    step_ms = ms_max / steps
    if T <= 32:
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(gbs / hbm, 4), "traffic": captured_traffic(name),
                "kernel": "k_decode: the whole layer in one persistent launch",
                "peak_source": hbm_src, "target_frac": 0.70,
                "algorithmic_bytes_per_step": round(float(np.mean(step_bytes)))}
    else:
        tf = float(peaks.get("bf16_tflops", 1900.0))
        tf_sus = float(peaks.get("bf16_tflops_sustained", tf))
        fl = step_flops(cfg, Tw) * nwin
        tfs = fl / (step_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": round(tfs, 2), "peak": tf, "unit": "TFLOP/s",
                "frac": round(tfs / tf, 4), "frac_of_sustained": round(tfs / tf_sus, 4),
                "traffic": captured_traffic(name),
                "kernel": "whole step (all launches of the step's layer calls; the tcgen05 "
                          "expert GEMMs lead)",
                "peak_source": "measured" if "bf16_tflops" in peaks else "fallback",
                "target_frac": 0.50, "algorithmic_flops_per_step": fl,
                "hbm": {"achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                        "frac": round(gbs / hbm, 4),
                        "algorithmic_bytes_per_step": round(float(np.mean(step_bytes)))}}
    res = {
        "name": name, "cfg": cfg, "T": T, "value": value, "ms_per_step": step_ms,
        "roofline": roof,
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 2,
                "copies": "pinned host x in and out back every step, on two copy streams "
                          "overlapping the neighbouring steps' layer calls"},
        "gpu_launches": launches_per_step(cfg, Tw) * nwin * steps,
        "clocks": clk,
        "config": {"workload": name, "tokens": T, "experts": E, "top_k": K_TOP,
                   "hidden": H, "inter": I, "expert_fmt": cfg["expert_fmt"],
                   "router_fmt": cfg["router_fmt"], "shared_fmt": cfg["shared_fmt"],
                   "gate_fmt": cfg["gate_fmt"], "zipf": cfg["zipf"],
                   "parallelism": f"replicas{ws_world}", "weight_banks": len(banks),
                   "l2": "inputs larger than L2 (%d rotating weight banks, %.1f GB)" % (
                       len(banks), len(banks) * (E * eb + fixed) / 1e9),
                   "experts_touched_mean": round(float(np.mean(U)), 2)},
    }
    if nwin > 1:
        res["config"]["tokens_per_call"] = Tw
        res["config"]["calls_per_step"] = nwin
    if keep:
        res["banks"], res["xs"] = banks, xs
    else:
        del banks, xs
        graphs.clear()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return res


def metric_name(T: int, fmt: str, name: str = "") -> str:
    if name in SWEEPS:
        _, nwin = SWEEPS[name]
        return "MoE-layer tokens/s (prefill sweep of %d tokens in %d-token windows, %s)" % (
            T, T // nwin, fmt)
    return "MoE-layer tokens/s (%s %d, %s)" % ("decode batch" if T <= 32 else "prefill window",
                                               T, fmt)


def dtype_of(T: int, act: str) -> str:
    # the decode form multiplies the activations as given; the prefill GEMMs
    # take fp16 operands
    return act if T <= 32 else "f16"


def arith_note(T: int, act: str) -> str:
    if T <= 32:
        return ("%s activations times the exact integer codes (mma.sync), fp32 accumulation, "
                "per-group scale and bias in fp32" % act)
    return ("fp16 operands (weights fp16(s*q+b) rounded once, x and h in fp16) on tcgen05 "
            "with fp32 accumulation in tensor memory; exact-product bf16-split router")


def run_gpu(args, ws_world, rank, local):
    import torch
    from bit_affine_quantized_fp32_gb300 import build as B
    B.build()

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    head = measure(args.workload, args.steps, args.warmup, args.banks, ws_world, rank, device,
                   keep=True)
    others = {}
    for name in ([] if args.also == "none" else args.also.split(",")):
        if name == args.workload or not name:
            continue
        _, Tw, nwin = workload_cfg(name)
        n = args.other_steps if Tw <= 32 else max(64, args.other_steps // (4 * nwin))
        r = measure(name, n, args.warmup, args.banks, ws_world, rank, device)
        others[name] = {"metric": metric_name(r["T"], r["cfg"]["expert_fmt"], name),
                        "value": round(r["value"], 1), "unit": "tokens/s",
                        "ms_per_step": round(r["ms_per_step"], 6), "steps": n,
                        "dtype": dtype_of(r["T"], r["cfg"]["act"]),
                        "arith": arith_note(r["T"], r["cfg"]["act"]),
                        "roofline": r["roofline"], "e2e": r["e2e"],
                        "gpu_launches": r["gpu_launches"], "clocks": r["clocks"],
                        "config": r["config"]}
    line = {
        "metric": metric_name(head["T"], head["cfg"]["expert_fmt"], head["name"]),
        "value": round(head["value"], 1),
        "unit": "tokens/s",
        "n_gpus": ws_world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(head["ms_per_step"], 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_of(head["T"], head["cfg"]["act"]),
        "arith": arith_note(head["T"], head["cfg"]["act"]),
        "data": "synthetic (seeded; random-init weights of the layer's shapes)",
        "config": head["config"],
        "roofline": head["roofline"],
        "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
    }
    if others:
        line["workloads"] = others
    return line, head["banks"], head["xs"], head["cfg"]


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
                tokens_per_step: int = 1, threads: int = 0):
    from oracle import oracle as O
    O.build()
    cores = O.set_threads(threads)
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
    cfg, T, _ = workload_cfg(args.workload)  # a sweep's oracle sample: tokens of one window
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
        tps1, _, steps1, el1 = time_oracle(banks[0], cfg, xs_np, args.cpu_seconds,
                                           tokens_per_step=cfg["T"], threads=1)
        line["cpu_baseline"] = {"value": round(tps, 3), "unit": "tokens/s", "cores": cores,
                                "kind": "oracle",
                                "sample": f"{steps} full decode batches of {cfg['T']} tokens "
                                          f"on weight bank 0 ({el:.1f} s, fp64 C++ oracle, "
                                          f"OpenMP over the batch's experts)",
                                "single_thread": {"value": round(tps1, 3), "cores": 1,
                                                  "sample": f"{steps1} batches ({el1:.1f} s)"}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws_world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
