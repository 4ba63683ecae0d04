"""Shared helpers of the GPU parity tests: move seeded inputs to the device,
run the library through its C ABI, and run the fp64 oracle on the same data.

The tolerance is the one stated for the layer's outputs:
    |gpu - oracle| <= 1e-2 * rms(oracle) + 1e-3   per element,
against the fp64 oracle; packed bytes, dequantised weights, top-k indices and
bucket layouts must match exactly.  The layer's output is rounded once to the
activation type, so for bf16/fp16 outputs the bound is taken before that
rounding: half an ulp of the output type at the element's magnitude is
allowed on top (fp32 results get no allowance).  Without it the exactly
computed sum itself misses the bound wherever |out| >= 1 and rms(out) is
about 0.13 (bf16's half ulp there is 2^-8 = 3.9e-3 against 2.3e-3).
"""

from __future__ import annotations

import numpy as np

from bit_affine_quantized_fp32_gb300 import synth
from oracle import oracle as O

RTOL_RMS = 1e-2
ATOL = 1e-3


def torch():
    import torch as _t
    return _t


def dev(a, dtype=None):
    t = torch()
    x = t.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        x = x.view(dtype)
    return x.cuda()


def bits16(a, act):
    """uint16 bit patterns -> torch bf16/f16 tensor on the device."""
    t = torch()
    return dev(a.astype(np.uint16)).view(t.bfloat16 if act == "bf16" else t.float16)


# significand bits + 1 of each rounded output type: half an ulp of v is
# 2^(e - HALF_ULP_SHIFT) where v = m * 2^e, 0.5 <= m < 1
HALF_ULP_SHIFT = {"bf16": 9, "f16": 12}


def output_rounding(ref: np.ndarray, tol: float, out_type: str | None) -> np.ndarray | float:
    """Half an ulp of the output type at |ref| + tol (the rounded value may sit
    one binade above ref), elementwise; 0 for unrounded (fp32) results."""
    if out_type is None:
        return 0.0
    _, e = np.frexp(np.abs(np.asarray(ref, np.float64)) + tol)
    half = np.ldexp(1.0, e - HALF_ULP_SHIFT[out_type])
    if out_type == "f16":
        half = np.maximum(half, 2.0 ** -25)  # subnormal spacing 2^-24
    return half


def assert_layer_close(gpu: np.ndarray, ref: np.ndarray, what: str = "out",
                       out_type: str | None = None):
    """gpu within the stated bound of ref; out_type ('bf16' / 'f16') when gpu
    is the layer's output rounded to that type, None for fp32 results."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    tol = RTOL_RMS * rms + ATOL
    err = np.abs(gpu - ref)
    bad = ~(err <= tol + output_rounding(ref, tol, out_type))
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {err.size} elements off; max err "
                           f"{float(err.max()):.3e} > tol {tol:.3e} (rms {rms:.3e})")
    return float(err.max()), tol


def projection_errors(gpu: np.ndarray, ref: np.ndarray) -> dict:
    """Worst-column and aggregate error of one projection (columns = outputs)."""
    e = np.abs(np.asarray(gpu, np.float64) - ref)
    scale = np.sqrt(np.mean(ref * ref, axis=0)) + 1e-30
    col = e.max(axis=0) / scale
    agg = float(np.sqrt(np.mean(e * e)) / (np.sqrt(np.mean(ref * ref)) + 1e-30))
    return {"worst_column_rel": float(col.max()), "aggregate_rel": agg}


def assert_routing_near_ties(L: synth.LayerInputs, idx_gpu: np.ndarray, ref_logits: np.ndarray,
                             what: str = "routing"):
    """The GPU's top-k equals the oracle's fp64 top-k on every token, except
    where the fp64 logits hold a near tie: the GPU's fp32 logits may order two
    experts differently only when the fp64 gap between two of the k + 1
    largest logits is within twice the fp32 dot-product error bound
    H * 2^-24 * sum_h |W[e, h] x[t, h]| of the token (max over experts)."""
    idx_gpu = np.asarray(idx_gpu)
    idx64, _ = O.topk(ref_logits, L.k)
    differ = np.nonzero(np.any(idx64 != idx_gpu, axis=1))[0]
    if differ.size == 0:
        return 0
    r = oracle_matrix(L.router)
    W = np.abs(O.dequant(L.router.fmt, r["q"], r.get("s"), r.get("b"), L.E, L.H))
    x = np.abs(O.act_to_double(L.act, L.x[differ]))
    bound = L.H * 2.0 ** -24 * (x @ W.T).max(axis=1) + 1e-6
    for n, t in enumerate(differ):
        srt = np.sort(ref_logits[t])[::-1]
        gaps = np.abs(np.diff(srt[: L.k + 1]))
        assert gaps.min() <= 2 * bound[n], (
            f"{what}: token {t} routes differently from fp64 without a near tie "
            f"(smallest gap {gaps.min():.3e}, bound {2 * bound[n]:.3e})")
    return int(differ.size)


# ---------------------------------------------------------------------------
# numpy (oracle-side) containers

def oracle_matrix(m: synth.QMatrix) -> dict:
    if m.fmt in ("f32", "bf16", "f16"):
        return {"fmt": m.fmt, "q": m.values, "rows": m.rows, "cols": m.cols}
    return {"fmt": m.fmt, "q": O.pack(m.fmt, m.codes), "s": m.scales, "b": m.biases,
            "rows": m.rows, "cols": m.cols}


def oracle_bank(b: synth.ExpertBank) -> dict:
    d = {"fmt": b.fmt, "E": b.E, "I": b.I,
         "w13": np.stack([O.pack(b.fmt, m.codes) for m in b.w13]),
         "w2": np.stack([O.pack(b.fmt, m.codes) for m in b.w2]),
         "s13": np.stack([m.scales for m in b.w13]), "s2": np.stack([m.scales for m in b.w2])}
    if b.fmt != "w4a16_g128":
        d["b13"] = np.stack([m.biases for m in b.w13])
        d["b2"] = np.stack([m.biases for m in b.w2])
    return d


def oracle_expert(bank: dict, e: int) -> dict:
    return {k: (v[e] if isinstance(v, np.ndarray) else v) for k, v in bank.items()}


def oracle_layer(L: synth.LayerInputs, **kw) -> dict:
    x = O.act_to_double(L.act, L.x)
    return O.moe_layer(x, L.k, oracle_matrix(L.router), oracle_bank(L.experts),
                       oracle_expert(oracle_bank(L.shared), 0) if L.shared else None,
                       oracle_matrix(L.gate) if L.gate else None, L.logit_bias, **kw)


# ---------------------------------------------------------------------------
# device containers (packed by the library's own pack kernels)

def gpu_pack(fmt: str, codes: np.ndarray):
    """Pack int codes [rows, cols] on the GPU; returns int32 words."""
    from bit_affine_quantized_fp32_gb300 import capi
    t = torch()
    rows, cols = codes.shape
    if fmt == "w4a16_g128":
        c = dev(codes.astype(np.int8))
    else:
        c = dev(codes.astype(np.uint8))
    out = t.empty((rows, cols * synth.BITS[fmt] // 32), dtype=t.int32, device="cuda")
    capi.moe_pack(fmt, c, out)
    return out


def gpu_matrix(m: synth.QMatrix):
    from bit_affine_quantized_fp32_gb300 import capi
    t = torch()
    if m.fmt == "f32":
        return capi.QMatrix("f32", m.rows, m.cols, dev(m.values))
    if m.fmt in ("bf16", "f16"):
        return capi.QMatrix(m.fmt, m.rows, m.cols, bits16(m.values, m.fmt))
    q = gpu_pack(m.fmt, m.codes)
    s = dev(m.scales).view(t.float16)
    b = dev(m.biases).view(t.float16) if m.biases is not None else None
    return capi.QMatrix(m.fmt, m.rows, m.cols, q, s, b)


def gpu_bank(b: synth.ExpertBank):
    """The bank in the TILED layout the expert kernels read."""
    return gpu_bank_canonical(b).tiled()


def gpu_bank_canonical(b: synth.ExpertBank):
    from bit_affine_quantized_fp32_gb300 import capi
    t = torch()
    E, I, H = b.E, b.I, b.H
    w13 = gpu_pack(b.fmt, np.concatenate([m.codes for m in b.w13])).view(E, 2 * I, -1)
    w2 = gpu_pack(b.fmt, np.concatenate([m.codes for m in b.w2])).view(E, H, -1)
    s13 = dev(np.stack([m.scales for m in b.w13])).view(t.float16)
    s2 = dev(np.stack([m.scales for m in b.w2])).view(t.float16)
    b13 = b2 = None
    if b.fmt != "w4a16_g128":
        b13 = dev(np.stack([m.biases for m in b.w13])).view(t.float16)
        b2 = dev(np.stack([m.biases for m in b.w2])).view(t.float16)
    return capi.ExpertBank(b.fmt, E, I, H, w13, s13, b13, w2, s2, b2)


def workspace(T, E, k, H, I):
    from bit_affine_quantized_fp32_gb300 import capi
    t = torch()
    n = capi.moe_workspace_bytes(max(T, 1), E, k, H, I)
    ws = t.empty(n, dtype=t.uint8, device="cuda")
    capi.moe_workspace_init(ws)
    return ws


class GpuLayer:
    """A layer's inputs on the device plus a ready workspace."""

    def __init__(self, L: synth.LayerInputs, max_tokens: int | None = None):
        self.L = L
        self.router = gpu_matrix(L.router)
        self.gate = gpu_matrix(L.gate) if L.gate else None
        self.experts = gpu_bank(L.experts)
        self.shared = gpu_bank(L.shared) if L.shared else None
        self.bias = dev(L.logit_bias) if L.logit_bias is not None else None
        self.x = bits16(L.x, L.act)
        self.ws = workspace(max_tokens or L.T, L.E, L.k, L.H, L.I)

    def forward(self, x=None, flags: int = 0):
        from bit_affine_quantized_fp32_gb300 import capi
        t = torch()
        x = self.x if x is None else x
        T = x.shape[0]
        out = t.empty((T, self.L.H), dtype=x.dtype, device="cuda")
        idx = t.empty((T, self.L.k), dtype=t.int32, device="cuda")
        w = t.empty((T, self.L.k), dtype=t.float32, device="cuda")
        capi.moe_layer_forward(self.router, self.bias, self.gate, self.experts, self.shared, x,
                               self.L.k, out, idx, w, flags, self.ws)
        return out, idx, w

    def route(self, x=None, flags: int = 0):
        from bit_affine_quantized_fp32_gb300 import capi
        t = torch()
        x = self.x if x is None else x
        T, E, k = x.shape[0], self.L.E, self.L.k
        r = {"logits": t.empty((T, E), dtype=t.float32, device="cuda"),
             "idx": t.empty((T, k), dtype=t.int32, device="cuda"),
             "w": t.empty((T, k), dtype=t.float32, device="cuda"),
             "sg": t.empty((T,), dtype=t.float32, device="cuda"),
             "offsets": t.empty((E + 1,), dtype=t.int32, device="cuda"),
             "perm": t.empty((T * k,), dtype=t.int32, device="cuda")}
        capi.moe_route(self.router, self.bias, self.gate, x, k, r["logits"], r["idx"], r["w"],
                       r["sg"] if self.gate else None, r["offsets"], r["perm"], self.ws,
                       flags=flags)
        return r


def to_np(t):
    import torch as _t
    if t.dtype in (_t.bfloat16, _t.float16):
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy()
