"""Child process of tests/test_zz_no_alloc.py: moe_route_static in more than
one CUDA context of the same device.

The static scratch array belongs to the library's module as loaded into one
context, so its address has to be looked up per context.  This process owns
its contexts through the driver API (no torch): it routes the same inputs in
the device's primary context, then in a context it creates, then in the
primary context again, each time checking moe_route_static against moe_route
(with a workspace) bit for bit.  Prints "route_static contexts ok".
"""

from __future__ import annotations

import ctypes
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from bit_affine_quantized_fp32_gb300 import capi, synth  # noqa: E402  (no torch needed)

cu = ctypes.CDLL("libcuda.so.1")
U64 = ctypes.c_uint64


def ck(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what}: CUresult {rc}")


def alloc(nbytes: int) -> int:
    p = U64()
    ck(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(max(nbytes, 256))), "cuMemAlloc")
    return p.value


def h2d(dst: int, a: np.ndarray):
    a = np.ascontiguousarray(a)
    ck(cu.cuMemcpyHtoD_v2(U64(dst), a.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(a.nbytes)),
       "cuMemcpyHtoD")


def d2h(src: int, shape, dtype) -> np.ndarray:
    a = np.empty(shape, dtype)
    ck(cu.cuMemcpyDtoH_v2(a.ctypes.data_as(ctypes.c_void_p), U64(src), ctypes.c_size_t(a.nbytes)),
       "cuMemcpyDtoH")
    return a


def route_once(L) -> None:
    T, E, k, H = L.T, L.E, L.k, L.H
    bufs = []

    def dev(a):
        p = alloc(a.nbytes)
        h2d(p, a)
        bufs.append(p)
        return p

    router = capi.QMatrixS(capi.FMT["f32"], E, H, 0, dev(L.router.values), None, None)
    gate = capi.QMatrixS(capi.FMT["bf16"], 1, H, 0, dev(L.gate.values.astype(np.uint16)), None,
                         None)
    bias = dev(L.logit_bias.astype(np.float32))
    x = dev(L.x.astype(np.uint16))
    outs = {}
    for which in ("ws", "static"):
        o = {"idx": alloc(4 * T * k), "w": alloc(4 * T * k), "sg": alloc(4 * T),
             "off": alloc(4 * (E + 1)), "perm": alloc(4 * T * k)}
        bufs.extend(o.values())
        if which == "ws":
            wsb = capi.lib.moe_workspace_bytes(T, E, k, H, 128)
            ws = alloc(wsb)
            bufs.append(ws)
            rc = capi.lib.moe_route(ctypes.byref(router), bias, ctypes.byref(gate), x,
                                    capi.FMT["bf16"], T, k, None, o["idx"], o["w"], o["sg"],
                                    o["off"], o["perm"], 0, ws, wsb, None)
        else:
            rc = capi.lib.moe_route_static(ctypes.byref(router), bias, ctypes.byref(gate), x,
                                           capi.FMT["bf16"], T, k, o["idx"], o["w"], o["sg"],
                                           o["off"], o["perm"], None)
        if rc != 0:
            raise RuntimeError(f"{which}: {capi.lib.moe_last_error().decode()}")
        ck(cu.cuCtxSynchronize(), "cuCtxSynchronize")
        outs[which] = {"idx": d2h(o["idx"], (T, k), np.int32), "w": d2h(o["w"], (T, k), np.uint32),
                       "sg": d2h(o["sg"], (T,), np.uint32), "off": d2h(o["off"], (E + 1,), np.int32),
                       "perm": d2h(o["perm"], (T * k,), np.int32)}
    for key in outs["ws"]:
        if not np.array_equal(outs["ws"][key], outs["static"][key]):
            raise AssertionError(f"moe_route_static differs from moe_route in {key}")
    for p in bufs:
        ck(cu.cuMemFree_v2(U64(p)), "cuMemFree")


def main():
    L = synth.gen_layer(T=8, E=256, k=8, H=2048, I=128, expert_fmt="affine4_g64",
                        router_fmt="f32", shared_fmt="affine4_g64", gate_fmt="bf16", zipf=True,
                        seed=75)
    ck(cu.cuInit(0), "cuInit")
    dev = ctypes.c_int()
    ck(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")
    primary = ctypes.c_void_p()
    ck(cu.cuDevicePrimaryCtxRetain(ctypes.byref(primary), dev), "cuDevicePrimaryCtxRetain")
    ck(cu.cuCtxSetCurrent(primary), "cuCtxSetCurrent")
    route_once(L)                       # primary context: the address is looked up and cached
    own = ctypes.c_void_p()
    ck(cu.cuCtxCreate_v2(ctypes.byref(own), 0, dev), "cuCtxCreate")   # becomes current
    route_once(L)                       # a second context: its own copy of the array
    ck(cu.cuCtxSetCurrent(primary), "cuCtxSetCurrent")
    route_once(L)                       # the primary context again: the cached address
    ck(cu.cuCtxDestroy_v2(own), "cuCtxDestroy")
    ck(cu.cuDevicePrimaryCtxRelease_v2(dev), "cuDevicePrimaryCtxRelease")
    print("route_static contexts ok")


if __name__ == "__main__":
    main()
