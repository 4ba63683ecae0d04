"""Thin ctypes binding of ``libmoe_gb300.so`` (the C ABI in ``include/moe_gb300.h``).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Tensors are torch tensors on the GPU (PyTorch supplies device memory
and streams); the functions keep the C names and pass ``data_ptr()``s and the
current CUDA stream.  Importing this module loads the library and fails loudly
if it is missing -- there is no CPU fallback.
"""

from __future__ import annotations

import ctypes
from ctypes import c_int, c_int32, c_size_t, c_void_p
from pathlib import Path

LIB_PATH = Path(__file__).resolve().parent / "libmoe_gb300.so"

FMT = {"f32": 0, "bf16": 1, "f16": 2, "affine8_g64": 3, "affine4_g64": 4,
       "affine3_g64": 5, "w4a16_g128": 6, "affine2_g64": 7, "affine5_g64": 8,
       "affine6_g64": 9}
PACKED = ("affine8_g64", "affine4_g64", "affine3_g64", "w4a16_g128", "affine2_g64",
          "affine5_g64", "affine6_g64")
MOE_FLAG_FORCE_DECODE = 1
MOE_FLAG_UNFUSED = 2
MOE_FLAG_ROUND_BF16 = 4
MOE_FLAG_FORCE_PREFILL = 8
MOE_DECODE_MAX_TOKENS = 32

EXPORTS = [
    "moe_status_string", "moe_last_error", "moe_workspace_bytes", "moe_workspace_init",
    "moe_workspace_set_wait_limit", "moe_get_device_status", "moe_route", "moe_route_static", "moe_topk_softmax", "moe_bucket",
    "moe_expert_mlp", "moe_shared_expert", "moe_experts_forward", "moe_layer_forward",
    "moe_pack_affine8_g64", "moe_unpack_affine8_g64", "moe_pack_affine4_g64",
    "moe_unpack_affine4_g64", "moe_pack_affine3_g64", "moe_unpack_affine3_g64",
    "moe_pack_w4a16_g128", "moe_unpack_w4a16_g128", "moe_pack_affine2_g64",
    "moe_unpack_affine2_g64", "moe_pack_affine5_g64", "moe_unpack_affine5_g64",
    "moe_pack_affine6_g64", "moe_unpack_affine6_g64", "moe_tiled_bytes", "moe_repack_bank",
    "moe_unrepack_bank", "moe_dequant",
]
LAYOUT_CANONICAL = 0
LAYOUT_TILED = 1


class MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


class QMatrixS(ctypes.Structure):
    _fields_ = [("fmt", c_int32), ("rows", c_int32), ("cols", c_int32), ("reserved", c_int32),
                ("qweight", c_void_p), ("scales", c_void_p), ("biases", c_void_p)]


class ExpertBankS(ctypes.Structure):
    _fields_ = [("fmt", c_int32), ("n_experts", c_int32), ("inter", c_int32), ("hidden", c_int32),
                ("layout", c_int32), ("reserved", c_int32), ("w13", c_void_p), ("s13", c_void_p), ("b13", c_void_p),
                ("w2", c_void_p), ("s2", c_void_p), ("b2", c_void_p)]


def _load():
    if not LIB_PATH.exists():
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "bit_affine_quantized_fp32_gb300.build.build() (nvcc, sm_103a)")
    L = ctypes.CDLL(str(LIB_PATH))
    P = c_void_p
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_status_string.argtypes = [c_int]
    L.moe_last_error.restype = ctypes.c_char_p
    L.moe_workspace_bytes.restype = c_size_t
    L.moe_workspace_bytes.argtypes = [c_int] * 5
    L.moe_workspace_init.argtypes = [P, c_size_t, P]
    L.moe_workspace_set_wait_limit.argtypes = [P, c_size_t, ctypes.c_uint, P]
    L.moe_get_device_status.argtypes = [P, c_size_t, P, P]
    L.moe_route.argtypes = [P, P, P, P, c_int, c_int, c_int, P, P, P, P, P, P, c_int, P, c_size_t,
                            P]
    L.moe_route_static.argtypes = [P, P, P, P, c_int, c_int, c_int, P, P, P, P, P, P]
    L.moe_topk_softmax.argtypes = [P, c_int, c_int, c_int, P, P, P]
    L.moe_bucket.argtypes = [P, c_int, c_int, c_int, P, P, P]
    L.moe_expert_mlp.argtypes = [P, c_int, P, c_int, c_int, P, P, P, c_size_t, P]
    L.moe_shared_expert.argtypes = [P, P, c_int, c_int, P, P, c_size_t, P]
    L.moe_experts_forward.argtypes = [P, P, c_int, c_int, c_int, P, P, P, P, P, P, P, c_int, P,
                                      c_size_t, P]
    L.moe_layer_forward.argtypes = [P, P, P, P, P, P, c_int, c_int, c_int, P, P, P, c_int, P,
                                    c_size_t, P]
    for n in PACKED:
        getattr(L, f"moe_pack_{n}").argtypes = [P, c_int, c_int, P, P]
        getattr(L, f"moe_unpack_{n}").argtypes = [P, c_int, c_int, P, P]
    L.moe_tiled_bytes.restype = c_size_t
    L.moe_tiled_bytes.argtypes = [c_int] * 5
    L.moe_repack_bank.argtypes = [P, P, P, P]
    L.moe_unrepack_bank.argtypes = [P] * 8
    L.moe_dequant.argtypes = [P, P, P]
    for name in EXPORTS:
        if name not in ("moe_status_string", "moe_last_error", "moe_workspace_bytes",
                        "moe_tiled_bytes"):
            getattr(L, name).restype = c_int
    return L


lib = _load()


def _check(rc: int):
    if rc != 0:
        raise MoeError(rc, f"{lib.moe_status_string(rc).decode()}: {lib.moe_last_error().decode()}")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def act_code(x) -> int:
    import torch
    if x.dtype == torch.bfloat16:
        return FMT["bf16"]
    if x.dtype == torch.float16:
        return FMT["f16"]
    raise MoeError(2, f"activation dtype {x.dtype} is not read (bf16 or f16)")


class QMatrix:
    """A matrix [rows, cols] in one format: values (F32/BF16/F16) or packed
    codes + fp16 scales (+ fp16 biases for affine)."""

    def __init__(self, fmt: str, rows: int, cols: int, q, s=None, b=None):
        self.fmt, self.rows, self.cols = fmt, rows, cols
        self.q, self.s, self.b = q, s, b
        self.struct = QMatrixS(FMT[fmt], rows, cols, 0, _ptr(q), _ptr(s), _ptr(b))

    def ref(self):
        return ctypes.byref(self.struct)


class ExpertBank:
    """E experts.  CANONICAL: w13 [E, 2I, *] (gate rows then up rows), w2 [E, H, *]
    packed words plus fp16 scales/biases.  TILED: w13 and w2 are the two
    kernel-tiled byte buffers (moe_repack_bank), scales/biases None."""

    def __init__(self, fmt: str, n_experts: int, inter: int, hidden: int, w13, s13, b13, w2, s2,
                 b2, layout: int = LAYOUT_CANONICAL):
        self.fmt, self.n_experts, self.inter, self.hidden = fmt, n_experts, inter, hidden
        self.layout = layout
        self.tensors = (w13, s13, b13, w2, s2, b2)
        self.struct = ExpertBankS(FMT[fmt], n_experts, inter, hidden, layout, 0, _ptr(w13),
                                  _ptr(s13), _ptr(b13), _ptr(w2), _ptr(s2), _ptr(b2))

    def ref(self):
        return ctypes.byref(self.struct)

    def tiled(self, stream=None) -> "ExpertBank":
        """The TILED copy of this CANONICAL bank (device buffers from torch)."""
        import torch
        dev = self.tensors[0].device
        b13 = moe_tiled_bytes(self.fmt, self.n_experts, self.inter, self.hidden, 0)
        b2 = moe_tiled_bytes(self.fmt, self.n_experts, self.inter, self.hidden, 1)
        t13 = torch.empty(b13, dtype=torch.uint8, device=dev)
        t2 = torch.empty(b2, dtype=torch.uint8, device=dev)
        moe_repack_bank(self, t13, t2, stream)
        return ExpertBank(self.fmt, self.n_experts, self.inter, self.hidden, t13, None, None, t2,
                          None, None, layout=LAYOUT_TILED)


def _ref(o):
    return None if o is None else o.ref()


def moe_workspace_bytes(max_tokens: int, n_experts: int, top_k: int, hidden: int,
                        inter: int) -> int:
    return int(lib.moe_workspace_bytes(max_tokens, n_experts, top_k, hidden, inter))


def moe_workspace_init(ws, stream=None):
    _check(lib.moe_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_workspace_set_wait_limit(ws, limit_us: int, stream=None):
    _check(lib.moe_workspace_set_wait_limit(_ptr(ws), ws.numel() * ws.element_size(),
                                            int(limit_us), _stream(stream)))


def moe_get_device_status(ws, stream=None) -> int:
    v = ctypes.c_int(-1)
    _check(lib.moe_get_device_status(_ptr(ws), ws.numel() * ws.element_size(), ctypes.byref(v),
                                     _stream(stream)))
    return v.value


def moe_route(router: QMatrix, logit_bias, shared_gate: QMatrix | None, x, top_k: int, logits,
              topk_idx, topk_w, shared_gate_w, bucket_offsets, bucket_perm, ws, stream=None,
              flags: int = 0):
    _check(lib.moe_route(router.ref(), _ptr(logit_bias), _ref(shared_gate), _ptr(x), act_code(x),
                         x.shape[0], top_k, _ptr(logits), _ptr(topk_idx), _ptr(topk_w),
                         _ptr(shared_gate_w), _ptr(bucket_offsets), _ptr(bucket_perm), flags,
                         _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_route_static(router: QMatrix, logit_bias, shared_gate: QMatrix | None, x, top_k: int,
                     topk_idx, topk_w, shared_gate_w, bucket_offsets, bucket_perm, stream=None):
    _check(lib.moe_route_static(router.ref(), _ptr(logit_bias), _ref(shared_gate), _ptr(x),
                                act_code(x), x.shape[0], top_k, _ptr(topk_idx), _ptr(topk_w),
                                _ptr(shared_gate_w), _ptr(bucket_offsets), _ptr(bucket_perm),
                                _stream(stream)))


def moe_topk_softmax(logits, top_k: int, topk_idx, topk_w, stream=None):
    T, E = logits.shape
    _check(lib.moe_topk_softmax(_ptr(logits), T, E, top_k, _ptr(topk_idx), _ptr(topk_w),
                                _stream(stream)))


def moe_bucket(topk_idx, n_experts: int, bucket_offsets, bucket_perm, stream=None):
    T, k = topk_idx.shape
    _check(lib.moe_bucket(_ptr(topk_idx), T, k, n_experts, _ptr(bucket_offsets),
                          _ptr(bucket_perm), _stream(stream)))


def moe_expert_mlp(bank: ExpertBank, expert: int, x, h_out, y_out, ws, stream=None):
    _check(lib.moe_expert_mlp(bank.ref(), expert, _ptr(x), act_code(x), x.shape[0], _ptr(h_out),
                              _ptr(y_out), _ptr(ws), ws.numel() * ws.element_size(),
                              _stream(stream)))


def moe_shared_expert(shared: ExpertBank, x, y_shared, ws, stream=None):
    _check(lib.moe_shared_expert(shared.ref(), _ptr(x), act_code(x), x.shape[0], _ptr(y_shared),
                                 _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_experts_forward(experts: ExpertBank, x, top_k: int, topk_idx, topk_w, bucket_offsets,
                        bucket_perm, y_shared, shared_gate_w, out, flags: int, ws, stream=None):
    _check(lib.moe_experts_forward(experts.ref(), _ptr(x), act_code(x), x.shape[0], top_k,
                                   _ptr(topk_idx), _ptr(topk_w), _ptr(bucket_offsets),
                                   _ptr(bucket_perm), _ptr(y_shared), _ptr(shared_gate_w),
                                   _ptr(out), flags, _ptr(ws), ws.numel() * ws.element_size(),
                                   _stream(stream)))


def moe_layer_forward(router: QMatrix, logit_bias, shared_gate: QMatrix | None,
                      experts: ExpertBank, shared: ExpertBank | None, x, top_k: int, out,
                      topk_idx=None, topk_w=None, flags: int = 0, ws=None, stream=None):
    _check(lib.moe_layer_forward(router.ref(), _ptr(logit_bias), _ref(shared_gate), experts.ref(),
                                 _ref(shared), _ptr(x), act_code(x), x.shape[0], top_k, _ptr(out),
                                 _ptr(topk_idx), _ptr(topk_w), flags, _ptr(ws),
                                 ws.numel() * ws.element_size(), _stream(stream)))


def moe_pack(fmt: str, codes, packed, stream=None):
    rows, cols = codes.shape
    _check(getattr(lib, f"moe_pack_{fmt}")(_ptr(codes), rows, cols, _ptr(packed),
                                           _stream(stream)))


def moe_unpack(fmt: str, packed, rows: int, cols: int, codes, stream=None):
    _check(getattr(lib, f"moe_unpack_{fmt}")(_ptr(packed), rows, cols, _ptr(codes),
                                             _stream(stream)))


def moe_tiled_bytes(fmt: str, n_experts: int, inter: int, hidden: int, which: int) -> int:
    n = lib.moe_tiled_bytes(FMT[fmt], n_experts, inter, hidden, which)
    if n == 0:
        raise MoeError(1, lib.moe_last_error().decode())
    return n


def moe_repack_bank(canonical: ExpertBank, w13_tiled, w2_tiled, stream=None):
    _check(lib.moe_repack_bank(canonical.ref(), _ptr(w13_tiled), _ptr(w2_tiled),
                               _stream(stream)))


def moe_unrepack_bank(tiled: ExpertBank, w13, s13, b13, w2, s2, b2, stream=None):
    _check(lib.moe_unrepack_bank(tiled.ref(), _ptr(w13), _ptr(s13), _ptr(b13), _ptr(w2),
                                 _ptr(s2), _ptr(b2), _stream(stream)))


def moe_dequant(m: QMatrix, w, stream=None):
    _check(lib.moe_dequant(m.ref(), _ptr(w), _stream(stream)))
