"""Seeded synthetic inputs for the MoE layer (shared by the tests, bench and smoke).

This module only draws random numbers and stores them in the formats' raw
containers (integer codes, fp16/bf16 bit patterns, fp32 arrays).  It holds none
of the layer's arithmetic (no packing, dequantisation, routing or expert math):
the CUDA path and the CPU oracle each do that on their own.

The distributions follow the workload descriptions of the routed-expert layer
of the qwen3_5 MoE 35B-A3B family (hidden 2048, 256 experts, top-8, expert
intermediate 512):

* activations  ``x = round(z / rms(z))``, z ~ N(0, 1) per token row, stored
  as bf16 (fp16 for the W4A16 workload);
* fp32 router  ``N(0, 0.02)``;
* affine 4-bit ``q ~ U{0..15}``, ``scale = fp16(|N(0, 0.004)|)``,
  ``bias = fp16(-8 * scale + N(0, 1e-4))``;
* affine 3-bit ``q ~ U{0..7}``, ``scale = fp16(|N(0, 0.008)|)``,
  ``bias = fp16(-4 * scale)``;
* affine 8-bit ``q ~ U{0..255}``, ``scale = fp16(|N(0, 2.7e-4)|)``,
  ``bias = fp16(-128 * scale + N(0, 1e-4))`` (chosen so the weights spread
  like the N(0, 0.02) fp32 router);
* W4A16        ``q ~ U{-8..7}``, ``scale = fp16(|N(0, 0.004)|)``, no bias;
* bf16 shared-gate row ``N(0, 0.02)``;
* Zipf(1.1) logit bias: ``bias_e = -1.1 * ln(rank_e)``, ranks a seeded
  permutation of 1..E.

Uniform codes packed densely are uniform random bits, so the device-side
generators (for full-size banks) draw packed words directly as random bytes.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BITS = {"affine8_g64": 8, "affine4_g64": 4, "affine3_g64": 3, "w4a16_g128": 4,
        "affine2_g64": 2, "affine5_g64": 5, "affine6_g64": 6}
GROUP = {"affine8_g64": 64, "affine4_g64": 64, "affine3_g64": 64, "w4a16_g128": 128,
         "affine2_g64": 64, "affine5_g64": 64, "affine6_g64": 64}
# scale laws |N(0, sigma)|: the 3- and 4-bit values of the workloads; the other
# widths keep the weights' spread of the 4-bit law (sigma = 0.064 / 2^bits)
SCALE_SIGMA = {"affine8_g64": 2.7e-4, "affine4_g64": 0.004, "affine3_g64": 0.008,
               "w4a16_g128": 0.004, "affine2_g64": 0.016, "affine5_g64": 0.002,
               "affine6_g64": 0.001}
BIAS_NOISE = {"affine8_g64": 1e-4, "affine4_g64": 1e-4, "affine3_g64": 0.0,
              "affine2_g64": 1e-4, "affine5_g64": 1e-4, "affine6_g64": 1e-4}


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round fp32 values to bfloat16 (nearest, ties to even); return the bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def f32_to_f16_bits(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64).astype(np.float16).view(np.uint16)


def gen_codes(rng: np.random.Generator, fmt: str, rows: int, cols: int) -> np.ndarray:
    """Uniform integer codes [rows, cols]: uint8 for affine, int8 in -8..7 for W4A16."""
    if fmt == "w4a16_g128":
        return rng.integers(-8, 8, size=(rows, cols), dtype=np.int8)
    return rng.integers(0, 1 << BITS[fmt], size=(rows, cols), dtype=np.uint8)


def gen_scales(rng, fmt: str, rows: int, cols: int, sigma: float | None = None) -> np.ndarray:
    s = SCALE_SIGMA[fmt] if sigma is None else sigma
    return f32_to_f16_bits(np.abs(rng.normal(0.0, s, size=(rows, cols // GROUP[fmt]))))


def gen_biases(rng, fmt: str, scales_bits: np.ndarray) -> np.ndarray | None:
    if fmt == "w4a16_g128":
        return None
    s = scales_bits.view(np.float16).astype(np.float64)
    mid = float(1 << (BITS[fmt] - 1))
    noise = BIAS_NOISE[fmt]
    extra = rng.normal(0.0, noise, size=s.shape) if noise > 0 else 0.0
    return f32_to_f16_bits(-mid * s + extra)


def gen_x(rng, T: int, H: int, act: str = "bf16") -> np.ndarray:
    z = rng.standard_normal((T, H))
    if T > 0:
        z = z / np.sqrt(np.mean(z * z, axis=1, keepdims=True))
    if act == "bf16":
        return f32_to_bf16_bits(z.astype(np.float32))
    if act == "f16":
        return f32_to_f16_bits(z)
    raise ValueError(act)


def zipf_bias(rng, E: int, alpha: float = 1.1) -> np.ndarray:
    ranks = rng.permutation(E) + 1
    return (-alpha * np.log(ranks.astype(np.float64))).astype(np.float32)


@dataclass
class QMatrix:
    """One matrix in its stored form; ``codes`` is the unpacked integer form."""
    fmt: str
    rows: int
    cols: int
    codes: np.ndarray | None = None      # uint8/int8 [rows, cols] for quantised formats
    values: np.ndarray | None = None     # float32 (f32) or uint16 bits (bf16/f16)
    scales: np.ndarray | None = None     # uint16 fp16 bits [rows, cols/G]
    biases: np.ndarray | None = None     # uint16 fp16 bits [rows, cols/G] or None


def gen_qmatrix(rng, fmt: str, rows: int, cols: int) -> QMatrix:
    if fmt == "f32":
        return QMatrix(fmt, rows, cols, values=rng.normal(0.0, 0.02, (rows, cols)).astype(np.float32))
    if fmt == "bf16":
        return QMatrix(fmt, rows, cols,
                       values=f32_to_bf16_bits(rng.normal(0.0, 0.02, (rows, cols)).astype(np.float32)))
    codes = gen_codes(rng, fmt, rows, cols)
    s = gen_scales(rng, fmt, rows, cols)
    b = gen_biases(rng, fmt, s)
    return QMatrix(fmt, rows, cols, codes=codes, scales=s, biases=b)


@dataclass
class ExpertBank:
    """E experts: w13 = [gate rows; up rows] of [2I, H] and w2 = [H, I] per expert."""
    fmt: str
    E: int
    I: int
    H: int
    w13: list = field(default_factory=list)   # list of QMatrix [2I, H]
    w2: list = field(default_factory=list)    # list of QMatrix [H, I]


def gen_bank(rng, fmt: str, E: int, I: int, H: int) -> ExpertBank:
    bank = ExpertBank(fmt, E, I, H)
    for _ in range(E):
        bank.w13.append(gen_qmatrix(rng, fmt, 2 * I, H))
        bank.w2.append(gen_qmatrix(rng, fmt, H, I))
    return bank


@dataclass
class LayerInputs:
    name: str
    T: int
    E: int
    k: int
    H: int
    I: int
    act: str
    x: np.ndarray
    router: QMatrix
    experts: ExpertBank
    shared: ExpertBank | None
    gate: QMatrix | None
    logit_bias: np.ndarray | None


# The five workloads of the layer (tokens, formats, skew), by name.
WORKLOADS = {
    "decode1_affine4": dict(T=1, expert_fmt="affine4_g64", router_fmt="f32", shared_fmt=None,
                            gate_fmt=None, act="bf16", zipf=False, seed=0),
    "decode8_affine4_shared_zipf": dict(T=8, expert_fmt="affine4_g64", router_fmt="f32",
                                        shared_fmt="affine4_g64", gate_fmt="affine8_g64",
                                        act="bf16", zipf=True, seed=1),
    "decode4_affine3": dict(T=4, expert_fmt="affine3_g64", router_fmt="affine8_g64",
                            shared_fmt="affine4_g64", gate_fmt="affine8_g64", act="bf16",
                            zipf=False, seed=2),
    "decode32_w4a16": dict(T=32, expert_fmt="w4a16_g128", router_fmt="f32",
                           shared_fmt="w4a16_g128", gate_fmt="bf16", act="f16", zipf=False,
                           seed=3),
    "prefill512_affine4_zipf": dict(T=512, expert_fmt="affine4_g64", router_fmt="f32",
                                    shared_fmt="affine4_g64", gate_fmt="affine8_g64",
                                    act="bf16", zipf=True, seed=4),
}


def gen_layer(name: str = "custom", *, T: int, E: int = 256, k: int = 8, H: int = 2048,
              I: int = 512, expert_fmt: str = "affine4_g64", router_fmt: str = "f32",
              shared_fmt: str | None = None, gate_fmt: str | None = None, act: str = "bf16",
              zipf: bool = False, seed: int = 0) -> LayerInputs:
    """Draw every input of one layer call, in a fixed order, from one seed."""
    rng = np.random.default_rng(seed)
    x = gen_x(rng, T, H, act)
    router = gen_qmatrix(rng, router_fmt, E, H)
    bias = zipf_bias(rng, E) if zipf else None
    experts = gen_bank(rng, expert_fmt, E, I, H)
    shared = gen_bank(rng, shared_fmt, 1, I, H) if shared_fmt else None
    gate = gen_qmatrix(rng, gate_fmt, 1, H) if gate_fmt else None
    return LayerInputs(name, T, E, k, H, I, act, x, router, experts, shared, gate, bias)


def workload(name: str, **over) -> LayerInputs:
    cfg = dict(WORKLOADS[name])
    cfg.update(over)
    return gen_layer(name, **cfg)


# ---------------------------------------------------------------------------
# Device-side generators for full-size banks (torch; imported lazily).

def _torch():
    import torch
    return torch


def words_per_row(fmt: str, cols: int) -> int:
    return cols * BITS[fmt] // 32


def device_bank(fmt: str, E: int, I: int, H: int, seed: int, device="cuda") -> dict:
    """A full bank as packed random words + fp16 scales/biases on the device.

    Uniform codes packed densely are uniform random bits, so the packed words
    are drawn directly as random bytes.  Scales/biases follow the same laws as
    the numpy generators.  Returns torch tensors keyed w13,s13,b13,w2,s2,b2.
    """
    torch = _torch()
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    G = GROUP[fmt]
    out = {}
    for name, rows, cols in (("13", 2 * I, H), ("2", H, I)):
        nbytes = E * rows * words_per_row(fmt, cols) * 4
        w = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=device, generator=g)
        out["w" + name] = w.view(torch.int32).view(E, rows, words_per_row(fmt, cols))
        s = torch.randn((E, rows, cols // G), device=device, generator=g, dtype=torch.float32)
        s = (s * SCALE_SIGMA[fmt]).abs().to(torch.float16)
        out["s" + name] = s
        if fmt == "w4a16_g128":
            out["b" + name] = None
        else:
            mid = float(1 << (BITS[fmt] - 1))
            noise = BIAS_NOISE[fmt]
            b = -mid * s.float()
            if noise > 0:
                b = b + noise * torch.randn(b.shape, device=device, generator=g)
            out["b" + name] = b.to(torch.float16)
    return out


def device_matrix(fmt: str, rows: int, cols: int, seed: int, device="cuda") -> dict:
    """One router / gate matrix on the device: {'q','s','b'} torch tensors."""
    torch = _torch()
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    if fmt == "f32":
        return {"q": 0.02 * torch.randn((rows, cols), device=device, generator=g), "s": None, "b": None}
    if fmt == "bf16":
        return {"q": (0.02 * torch.randn((rows, cols), device=device, generator=g)).to(torch.bfloat16),
                "s": None, "b": None}
    G = GROUP[fmt]
    nbytes = rows * words_per_row(fmt, cols) * 4
    q = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=device, generator=g)
    s = (SCALE_SIGMA[fmt] * torch.randn((rows, cols // G), device=device, generator=g)).abs().to(torch.float16)
    b = None
    if fmt != "w4a16_g128":
        mid = float(1 << (BITS[fmt] - 1))
        b = -mid * s.float()
        if BIAS_NOISE[fmt] > 0:
            b = b + BIAS_NOISE[fmt] * torch.randn(b.shape, device=device, generator=g)
        b = b.to(torch.float16)
    return {"q": q.view(torch.int32).view(rows, words_per_row(fmt, cols)), "s": s, "b": b}


def device_x(T: int, H: int, act: str, seed: int, device="cuda"):
    torch = _torch()
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    z = torch.randn((T, H), device=device, generator=g)
    if T > 0:
        z = z / torch.sqrt((z * z).mean(dim=1, keepdim=True))
    return z.to(torch.bfloat16 if act == "bf16" else torch.float16)


def device_zipf_bias(E: int, seed: int, device="cuda", alpha: float = 1.1):
    rng = np.random.default_rng(seed)
    torch = _torch()
    return torch.from_numpy(zipf_bias(rng, E, alpha)).to(device)


def layer_bytes(fmt: str, I: int, H: int) -> int:
    """Stored bytes of one expert (codes + fp16 scales (+ biases))."""
    n_w = 3 * I * H
    b = n_w * BITS[fmt] // 8
    groups = n_w // GROUP[fmt]
    b += groups * 2 * (1 if fmt == "w4a16_g128" else 2)
    return b


assert math.isclose(layer_bytes("affine4_g64", 512, 2048), 1769472)
