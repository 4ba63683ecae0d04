"""moe_route_static (routing with its scratch in a static device array, no
caller workspace) against moe_route on the same inputs, two calls in a row.

Collected last on purpose: it must pass both alone in a fresh process and
after every other GPU test.
"""

import os
import subprocess
import sys

import numpy as np
import pytest

from bit_affine_quantized_fp32_gb300 import synth

from . import _harness as Hn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def capi():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_affine_quantized_fp32_gb300 import build
    build.build()
    from bit_affine_quantized_fp32_gb300 import capi as C
    return C


CASES = [
    dict(T=8, E=256, k=8, H=2048, rfmt="f32", gfmt="affine8_g64", zipf=True, seed=71),
    dict(T=32, E=256, k=8, H=1024, rfmt="affine8_g64", gfmt=None, zipf=False, seed=72),
    dict(T=1, E=64, k=4, H=512, rfmt="bf16", gfmt="bf16", zipf=False, seed=73),
]


def _outputs(torch, T, E, k):
    return {"idx": torch.empty((T, k), dtype=torch.int32, device="cuda"),
            "w": torch.empty((T, k), dtype=torch.float32, device="cuda"),
            "sg": torch.empty((T,), dtype=torch.float32, device="cuda"),
            "offsets": torch.empty((E + 1,), dtype=torch.int32, device="cuda"),
            "perm": torch.empty((T * k,), dtype=torch.int32, device="cuda")}


@pytest.mark.parametrize("c", CASES, ids=lambda c: f"T{c['T']}_E{c['E']}_{c['rfmt']}")
def test_route_static_equals_route(capi, c):
    torch = Hn.torch()
    L = synth.gen_layer(T=c["T"], E=c["E"], k=c["k"], H=c["H"], I=128,
                        expert_fmt="affine4_g64", router_fmt=c["rfmt"],
                        shared_fmt="affine4_g64" if c["gfmt"] else None,
                        gate_fmt=c["gfmt"], zipf=c["zipf"], seed=c["seed"])
    router = Hn.gpu_matrix(L.router)
    gate = Hn.gpu_matrix(L.gate) if L.gate else None
    bias = Hn.dev(L.logit_bias) if L.logit_bias is not None else None
    x = Hn.bits16(L.x, L.act)
    T, E, k = c["T"], c["E"], c["k"]
    ws = Hn.workspace(T, E, k, c["H"], 128)
    ref = _outputs(torch, T, E, k)
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    capi.moe_route(router, bias, gate, x, k, logits, ref["idx"], ref["w"],
                   ref["sg"] if gate else None, ref["offsets"], ref["perm"], ws)
    for _ in range(2):   # two calls in a row reuse the same static scratch
        got = _outputs(torch, T, E, k)
        capi.moe_route_static(router, bias, gate, x, k, got["idx"], got["w"],
                              got["sg"] if gate else None, got["offsets"], got["perm"])
        torch.cuda.synchronize()
        assert torch.equal(got["idx"], ref["idx"])
        assert torch.equal(got["offsets"], ref["offsets"])
        assert torch.equal(got["perm"], ref["perm"])
        # same kernels and arithmetic: the same bits
        assert torch.equal(got["w"], ref["w"])
        if gate:
            assert torch.equal(got["sg"], ref["sg"])


def test_route_static_refuses_oversize(capi):
    torch = Hn.torch()
    L = synth.gen_layer(T=33, E=64, k=4, H=512, I=128, expert_fmt="affine4_g64", seed=74)
    router = Hn.gpu_matrix(L.router)
    x = Hn.bits16(L.x, L.act)
    o = _outputs(torch, 33, 64, 4)
    with pytest.raises(capi.MoeError) as e:
        capi.moe_route_static(router, None, None, x, 4, o["idx"], o["w"], None, o["offsets"],
                              o["perm"])
    assert e.value.status == 3 and "static scratch" in str(e.value)


def test_route_static_per_context(capi):
    """The static array belongs to the module as loaded into one CUDA context:
    a child process (driver-API contexts, no torch) routes in the primary
    context, in a context of its own and in the primary context again, and
    moe_route_static equals moe_route bit for bit in each."""
    script = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_ctx_route_static.py")
    r = subprocess.run([sys.executable, script], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "route_static contexts ok" in r.stdout
