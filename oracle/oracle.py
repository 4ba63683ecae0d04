"""ctypes wrapper around the fp64 CPU oracle (``moe_oracle.cpp``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline and reference legs of ``bench.py`` use it.  The library's GPU path never imports
this module, and this module imports nothing from the library.

Arrays are numpy.  Bit patterns of fp16 / bf16 values travel as ``uint16``
arrays; packed codes as ``uint32`` arrays.  Format names are the plain strings
``"f32" "bf16" "f16" "affine8_g64" "affine4_g64" "affine3_g64" "w4a16_g128"``
and the other MLX affine widths ``"affine2_g64" "affine5_g64" "affine6_g64"``
(oracle only: the library's kernels read 8/4/3-bit and W4A16).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SRC = HERE / "moe_oracle.cpp"
LIB = HERE / "libmoe_oracle.so"

FMT = {
    "f32": 0,
    "bf16": 1,
    "f16": 2,
    "affine8_g64": 3,
    "affine4_g64": 4,
    "affine3_g64": 5,
    "w4a16_g128": 6,
    "affine2_g64": 7,
    "affine5_g64": 8,
    "affine6_g64": 9,
}
BITS = {"affine8_g64": 8, "affine4_g64": 4, "affine3_g64": 3, "w4a16_g128": 4,
        "affine2_g64": 2, "affine5_g64": 5, "affine6_g64": 6}
GROUP = {"affine8_g64": 64, "affine4_g64": 64, "affine3_g64": 64, "w4a16_g128": 128,
         "affine2_g64": 64, "affine5_g64": 64, "affine6_g64": 64}


# Layout version of the structures passed by pointer (LayerArgs).
ABI_VERSION = 2


def build(force: bool = False) -> Path:
    """Compile the oracle into ``oracle/libmoe_oracle.so`` (g++, OpenMP when present)."""
    if LIB.exists() and not force and LIB.stat().st_mtime >= SRC.stat().st_mtime:
        return LIB
    base = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off"]
    tmp = LIB.with_suffix(f".so.tmp{os.getpid()}")
    for extra in (["-fopenmp"], []):
        r = subprocess.run(base + extra + [str(SRC), "-o", str(tmp)],
                           capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, LIB)
            return LIB
    raise RuntimeError("oracle build failed:\n" + r.stderr)


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(str(LIB))
        if L.oracle_abi_version() != ABI_VERSION:
            raise RuntimeError(f"{LIB} is ABI {L.oracle_abi_version()}, this module wants "
                               f"{ABI_VERSION}: rebuild it with oracle.build(force=True)")
        P = ctypes.c_void_p
        i64 = ctypes.c_long
        i32 = ctypes.c_int
        L.oracle_set_threads.argtypes = [i32]
        L.oracle_pack.argtypes = [i32, i64, i64, P, P]
        L.oracle_unpack.argtypes = [i32, i64, i64, P, P]
        L.oracle_dequant.argtypes = [i32, i64, i64, P, P, P, P]
        L.oracle_act_to_double.argtypes = [i32, i64, P, P]
        L.oracle_fp16_to_double.argtypes = [i64, P, P]
        L.oracle_router_logits.argtypes = [i32, i64, i64, P, P, P, P, i64, P, P]
        L.oracle_topk.argtypes = [i64, i64, i64, P, P, P]
        L.oracle_shared_gate.argtypes = [i32, i64, P, P, P, i64, P, P, P]
        L.oracle_expert_mlp.argtypes = [i32, i64, i64, P, P, P, P, P, P, i64, P, P, P]
        L.oracle_down.argtypes = [i32, i64, i64, P, P, P, i64, P, P]
        L.oracle_bucket.argtypes = [i64, i64, i64, P, P, P, P, P, P]
        L.oracle_moe_layer.argtypes = [P]
        L.oracle_round_bf16.argtypes = [i64, P, P]
        L.oracle_combine_f32.argtypes = [i64, i64, i64, P, P, P, P, P]
        L.oracle_chain_gate_weight.argtypes = [i64, P, P]
        L.oracle_value_bytes.restype = i64
        L.oracle_value_bytes.argtypes = [i32, i64, i64]
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def set_threads(n: int) -> int:
    return lib().oracle_set_threads(int(n))


def pack(fmt: str, codes: np.ndarray) -> np.ndarray:
    codes = _c(codes, np.int32)
    rows, cols = codes.shape
    out = np.zeros((rows, cols * BITS[fmt] // 32), np.uint32)
    _check(lib().oracle_pack(FMT[fmt], rows, cols, _p(codes), _p(out)), "pack")
    return out


def unpack(fmt: str, words: np.ndarray, cols: int) -> np.ndarray:
    words = _c(words, np.uint32)
    rows = words.shape[0]
    out = np.zeros((rows, cols), np.int32)
    _check(lib().oracle_unpack(FMT[fmt], rows, cols, _p(words), _p(out)), "unpack")
    return out


def dequant(fmt: str, q, scales, biases, rows: int, cols: int) -> np.ndarray:
    if fmt == "f32":
        q = _c(q, np.float32)
    elif fmt in ("bf16", "f16"):
        q = _c(q, np.uint16)
    else:
        q = _c(q, np.uint32)
    s = _c(scales, np.uint16)
    b = _c(biases, np.uint16)
    out = np.zeros((rows, cols), np.float64)
    _check(lib().oracle_dequant(FMT[fmt], rows, cols, _p(q), _p(s), _p(b), _p(out)), "dequant")
    return out


def act_to_double(fmt: str, x) -> np.ndarray:
    x = _c(x, np.float32 if fmt == "f32" else np.uint16)
    out = np.zeros(x.shape, np.float64)
    _check(lib().oracle_act_to_double(FMT[fmt], x.size, _p(x), _p(out)), "act_to_double")
    return out


def fp16_to_double(h) -> np.ndarray:
    h = _c(h, np.uint16)
    out = np.zeros(h.shape, np.float64)
    lib().oracle_fp16_to_double(h.size, _p(h), _p(out))
    return out


def _qm(m):
    """(fmt, q, s, b) of a matrix dict {'fmt','q','s','b'} with proper dtypes."""
    fmt = m["fmt"]
    if fmt == "f32":
        q = _c(m["q"], np.float32)
    elif fmt in ("bf16", "f16"):
        q = _c(m["q"], np.uint16)
    else:
        q = _c(m["q"], np.uint32)
    return fmt, q, _c(m.get("s"), np.uint16), _c(m.get("b"), np.uint16)


def router_logits(router: dict, x: np.ndarray, bias=None) -> np.ndarray:
    fmt, q, s, b = _qm(router)
    E, H = router["rows"], router["cols"]
    x = _c(x, np.float64)
    T = x.shape[0]
    bias = _c(bias, np.float32)
    out = np.zeros((T, E), np.float64)
    _check(lib().oracle_router_logits(FMT[fmt], E, H, _p(q), _p(s), _p(b), _p(bias), T,
                                      _p(x), _p(out)), "router_logits")
    return out


def topk(logits: np.ndarray, k: int):
    logits = _c(logits, np.float64)
    T, E = logits.shape
    idx = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    _check(lib().oracle_topk(T, E, k, _p(logits), _p(idx), _p(w)), "topk")
    return idx, w


def shared_gate(gate: dict, x: np.ndarray):
    fmt, q, s, b = _qm(gate)
    x = _c(x, np.float64)
    T, H = x.shape
    logit = np.zeros(T, np.float64)
    sg = np.zeros(T, np.float64)
    _check(lib().oracle_shared_gate(FMT[fmt], H, _p(q), _p(s), _p(b), T, _p(x), _p(logit),
                                    _p(sg)), "shared_gate")
    return logit, sg


def expert_mlp(fmt: str, I: int, H: int, e: dict, x: np.ndarray):
    """e = {'w13','s13','b13','w2','s2','b2'} for ONE expert. Returns (h, y)."""
    x = _c(x, np.float64)
    T = x.shape[0]
    h = np.zeros((T, I), np.float64)
    y = np.zeros((T, H), np.float64)
    arr = [_c(e["w13"], np.uint32), _c(e.get("s13"), np.uint16), _c(e.get("b13"), np.uint16),
           _c(e["w2"], np.uint32), _c(e.get("s2"), np.uint16), _c(e.get("b2"), np.uint16)]
    _check(lib().oracle_expert_mlp(FMT[fmt], I, H, *[_p(a) for a in arr], T, _p(x), _p(h),
                                   _p(y)), "expert_mlp")
    return h, y


def down(fmt: str, H: int, I: int, w2, s2, b2, h: np.ndarray) -> np.ndarray:
    h = _c(h, np.float64)
    T = h.shape[0]
    y = np.zeros((T, H), np.float64)
    arr = [_c(w2, np.uint32), _c(s2, np.uint16), _c(b2, np.uint16)]
    _check(lib().oracle_down(FMT[fmt], H, I, *[_p(a) for a in arr], T, _p(h), _p(y)), "down")
    return y


def bucket(idx: np.ndarray, E: int):
    idx = _c(idx, np.int32)
    T, k = idx.shape
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    perm = np.zeros(T * k, np.int32)
    active = np.zeros(E, np.int32)
    n = np.zeros(1, np.int32)
    _check(lib().oracle_bucket(T, k, E, _p(idx), _p(counts), _p(offsets), _p(perm),
                               _p(active), _p(n)), "bucket")
    return counts, offsets, perm, active[: n[0]]


class _LayerArgs(ctypes.Structure):
    P = ctypes.c_void_p
    _fields_ = [("T", ctypes.c_long), ("E", ctypes.c_long), ("k", ctypes.c_long),
                ("H", ctypes.c_long), ("I", ctypes.c_long), ("x", P),
                ("router_fmt", ctypes.c_int), ("router_q", P), ("router_s", P), ("router_b", P),
                ("logit_bias", P),
                ("expert_fmt", ctypes.c_int), ("w13", P), ("s13", P), ("b13", P),
                ("w2", P), ("s2", P), ("b2", P),
                ("shared_fmt", ctypes.c_int), ("sh_w13", P), ("sh_s13", P), ("sh_b13", P),
                ("sh_w2", P), ("sh_s2", P), ("sh_b2", P),
                ("gate_fmt", ctypes.c_int), ("gate_q", P), ("gate_s", P), ("gate_b", P),
                ("idx_override", P),
                ("logits", P), ("idx", P), ("w", P), ("sg", P), ("y_slots", P),
                ("y_shared", P), ("out", P),
                ("round_bf16", ctypes.c_int)]


def moe_layer(x: np.ndarray, k: int, router: dict, experts: dict, shared: dict | None = None,
              gate: dict | None = None, logit_bias=None, idx_override=None,
              want_slots: bool = False, round_bf16: bool = False) -> dict:
    """Whole layer in fp64.

    x: float64 [T, H] (already decoded activations).
    router: {'fmt','q','s','b','rows'=E,'cols'=H}.
    experts: {'fmt','E','I','w13','s13','b13','w2','s2','b2'} (per-expert blocks stacked).
    shared: same keys for one expert (or None); gate: matrix dict (or None).
    round_bf16: the engine's bf16 rounding chain for the routing inputs
    (router and gate rows rounded to bf16, w -> bf16(w), the shared weight
    bf16(sigmoid(bf16(g)))); logits, experts and the sum stay fp64.
    """
    x = _c(x, np.float64)
    T, H = x.shape
    E, I = experts["E"], experts["I"]
    keep = []

    def P(a):
        keep.append(a)
        return _p(a)

    a = _LayerArgs()
    a.T, a.E, a.k, a.H, a.I = T, E, k, H, I
    a.x = P(x)
    rf, rq, rs, rb = _qm(router)
    a.router_fmt, a.router_q, a.router_s, a.router_b = FMT[rf], P(rq), P(rs), P(rb)
    a.logit_bias = P(_c(logit_bias, np.float32))
    ef = experts["fmt"]
    a.expert_fmt = FMT[ef]
    a.w13, a.s13, a.b13 = P(_c(experts["w13"], np.uint32)), P(_c(experts.get("s13"), np.uint16)), \
        P(_c(experts.get("b13"), np.uint16))
    a.w2, a.s2, a.b2 = P(_c(experts["w2"], np.uint32)), P(_c(experts.get("s2"), np.uint16)), \
        P(_c(experts.get("b2"), np.uint16))
    if shared is not None:
        a.shared_fmt = FMT[shared["fmt"]]
        a.sh_w13, a.sh_s13, a.sh_b13 = P(_c(shared["w13"], np.uint32)), \
            P(_c(shared.get("s13"), np.uint16)), P(_c(shared.get("b13"), np.uint16))
        a.sh_w2, a.sh_s2, a.sh_b2 = P(_c(shared["w2"], np.uint32)), \
            P(_c(shared.get("s2"), np.uint16)), P(_c(shared.get("b2"), np.uint16))
    if gate is not None:
        gf, gq, gs, gb = _qm(gate)
        a.gate_fmt, a.gate_q, a.gate_s, a.gate_b = FMT[gf], P(gq), P(gs), P(gb)
    a.idx_override = P(_c(idx_override, np.int32))
    out = {"logits": np.zeros((T, E)), "idx": np.zeros((T, k), np.int32),
           "w": np.zeros((T, k)), "sg": np.zeros(T), "y_shared": np.zeros((T, H)),
           "out": np.zeros((T, H))}
    if want_slots:
        out["y_slots"] = np.zeros((T, k, H))
    a.logits, a.idx, a.w, a.sg = P(out["logits"]), P(out["idx"]), P(out["w"]), P(out["sg"])
    a.y_slots = P(out["y_slots"]) if want_slots else None
    a.y_shared, a.out = P(out["y_shared"]), P(out["out"])
    a.round_bf16 = int(bool(round_bf16))
    _check(lib().oracle_moe_layer(ctypes.byref(a)), "moe_layer")
    return out


# ---------------------------------------------------------------------------
# The engine's fp32 precision (byte-exact references)

def round_bf16(a) -> np.ndarray:
    """fp32 values rounded to bf16 (nearest, ties to even), returned as fp32."""
    a = _c(a, np.float32)
    out = np.empty_like(a)
    _check(lib().oracle_round_bf16(a.size, _p(a), _p(out)), "round_bf16")
    return out


def combine_f32(y, w, ysh=None, sg=None) -> np.ndarray:
    """The slots' fp32 fma sum (slot order, shared slot last), rounded once to
    bf16; y [T*k, H], w [T, k], ysh [T, H] or None, sg [T] or None.  Returns
    the bf16 bit patterns [T, H] as uint16."""
    w = _c(w, np.float32)
    T, k = w.shape
    y = _c(y, np.float32)
    H = y.shape[1]
    assert y.shape == (T * k, H)
    ysh = None if ysh is None else _c(ysh, np.float32)
    sg = None if sg is None else _c(sg, np.float32)
    out = np.empty((T, H), np.uint16)
    _check(lib().oracle_combine_f32(T, k, H, _p(y), _p(w), _p(ysh), _p(sg), _p(out)),
           "combine_f32")
    return out


def chain_gate_weight(g) -> np.ndarray:
    """bf16(sigmoid(bf16(g))) per token, as fp32."""
    g = _c(g, np.float32)
    out = np.empty_like(g)
    _check(lib().oracle_chain_gate_weight(g.size, _p(g), _p(out)), "chain_gate_weight")
    return out
