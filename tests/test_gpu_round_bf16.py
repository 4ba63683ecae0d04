"""The engine's bf16 rounding chain on the device (MOE_FLAG_ROUND_BF16)
against the oracle's references for it.

"qwen3_5_moe on native CUDA with 3-bit routed experts ... #803", comment
"Progress on the 4-bit gate", paragraph "What is in it": the router and the
combine are checked byte-equal against a host reference, the weights within
a bf16 step.  Read here as: router and gate rows rounded to bf16, slot weights
stored as bf16(w), the shared weight as bf16(sigmoid(bf16(g))), the slots'
fp32 fma sum rounded once.

Exact where IEEE arithmetic fixes every bit (the combine given fp32 inputs);
bf16-exact up to near ties where an fp32 transcendental sits under the
rounding (a weight or gate value within 2^-19 relative of a bf16 rounding
boundary may land on either neighbour); within the layer's tolerance for the
outputs against the oracle's fp64 layer under the same chain.
"""

import numpy as np
import pytest

from bit_affine_quantized_fp32_gb300 import synth
from oracle import oracle as O

from . import _harness as Hn

pytestmark = pytest.mark.gpu

NEAR = 2.0 ** -19   # relative distance to a bf16 rounding boundary that counts as a tie


@pytest.fixture(scope="module")
def capi():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_affine_quantized_fp32_gb300 import build
    build.build()
    from bit_affine_quantized_fp32_gb300 import capi as C
    return C


def _bf16_boundary_distance(v: np.ndarray) -> np.ndarray:
    """Relative distance of each fp64 value to the nearest bf16 rounding
    boundary (the midpoint between its two bf16 neighbours)."""
    v = np.asarray(v, np.float64)
    f = v.astype(np.float32)
    bits = f.view(np.uint32)
    lo = (bits & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)
    hi = ((bits & np.uint32(0xFFFF0000)) + np.uint32(0x10000)).view(np.float32).astype(np.float64)
    mid = 0.5 * (lo + hi)
    return np.abs(v - mid) / np.maximum(np.abs(v), 1e-300)


def assert_bf16_exact_up_to_ties(gpu: np.ndarray, exact: np.ndarray, what: str,
                                 also_tie=None):
    """gpu (fp32 holding bf16 values) equals bf16(fp32(exact)) bit for bit,
    except where exact lies within NEAR of a bf16 rounding boundary (or where
    also_tie marks a tie of an earlier rounding); there it may be either
    neighbour."""
    gpu = np.asarray(gpu, np.float32)
    ref = O.round_bf16(np.asarray(exact, np.float64).astype(np.float32))
    assert np.all((gpu.view(np.uint32) & 0xFFFF) == 0), f"{what}: not bf16 values"
    same = gpu.view(np.uint32) == ref.view(np.uint32)
    tie = _bf16_boundary_distance(exact) <= NEAR
    if also_tie is not None:
        tie = tie | also_tie
    step = np.abs(gpu.astype(np.float64) - ref) <= np.abs(ref) * 2.0 ** -7 * 1.01
    bad = ~(same | (tie & step))
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} differ from the bf16 "
                           f"rounding of the exact value")
    return int((~same).sum())


ROUTE_CASES = ["decode8_affine4_shared_zipf", "decode4_affine3", "decode32_w4a16"]


@pytest.mark.parametrize("name", ROUTE_CASES)
def test_route_chain(capi, name):
    """moe_route with the chain: logits from bf16-rounded rows within the fp32
    dot-product bound of the oracle's chain logits; indices exact on the GPU's
    own logits; slot weights and the shared weight bf16-exact (up to ties)."""
    L = synth.workload(name)
    g = Hn.GpuLayer(L)
    r = g.route(flags=capi.MOE_FLAG_ROUND_BF16)
    ref = Hn.oracle_layer(L, round_bf16=True)
    lg = r["logits"].cpu().numpy().astype(np.float64)
    x = O.act_to_double(L.act, L.x)
    om = Hn.oracle_matrix(L.router)
    Wb = O.round_bf16(O.dequant(L.router.fmt, om["q"], om.get("s"), om.get("b"), L.E,
                                L.H).astype(np.float32)).astype(np.float64)
    bound = L.H * 2.0 ** -24 * (np.abs(x) @ np.abs(Wb).T) + 1e-6
    assert np.all(np.abs(lg - ref["logits"]) <= bound), "chain logits beyond the fp32 bound"
    idx_ref, w_exact = O.topk(lg, L.k)
    assert np.array_equal(r["idx"].cpu().numpy(), idx_ref)
    assert_bf16_exact_up_to_ties(r["w"].cpu().numpy(), w_exact, "slot weights")
    if L.gate is not None:
        gm = Hn.oracle_matrix(L.gate)
        gb = O.round_bf16(O.dequant(L.gate.fmt, gm["q"], gm.get("s"), gm.get("b"), 1,
                                    L.H).astype(np.float32)).astype(np.float64)[0]
        g64 = x @ gb
        gbound = L.H * 2.0 ** -24 * (np.abs(x) @ np.abs(gb)) + 1e-6
        # the gate logit is rounded to bf16 before the sigmoid: a logit within
        # the fp32 bound of a bf16 boundary may round either way
        g_tie = _bf16_boundary_distance(g64) * np.abs(g64) <= 2 * gbound
        s_exact = O.chain_gate_weight(g64.astype(np.float32)).astype(np.float64)
        # the sigmoid of the bf16 logit, in fp64, is what is rounded last
        gbf = O.round_bf16(g64.astype(np.float32)).astype(np.float64)
        sig = 1.0 / (1.0 + np.exp(-gbf))
        assert np.array_equal(O.round_bf16(sig.astype(np.float32)), s_exact)
        assert_bf16_exact_up_to_ties(r["sg"].cpu().numpy(), sig, "shared weight", also_tie=g_tie)


@pytest.mark.parametrize("name", ["decode8_affine4_shared_zipf", "decode1_affine4"])
def test_combine_byte_equal(capi, name):
    """The layer's output under the chain is, byte for byte, the fp32 fma sum
    (slot order, shared slot last, one bf16 rounding) of the GPU's own slot
    outputs with the GPU's own bf16 weights (oracle combine_f32)."""
    torch = Hn.torch()
    L = synth.workload(name)
    g = Hn.GpuLayer(L)
    flags = capi.MOE_FLAG_ROUND_BF16
    out, idx, w = g.forward(flags=flags)
    r = g.route(flags=flags)
    assert torch.equal(r["idx"], idx) and torch.equal(r["w"], w)
    T, H, k = L.T, L.H, L.k
    ws = Hn.workspace(T, L.E, 1, H, L.I)
    idx_np = idx.cpu().numpy()
    y = np.zeros((T * k, H), np.float32)
    yt = torch.empty((T, H), dtype=torch.float32, device="cuda")
    for e in np.unique(idx_np):
        capi.moe_expert_mlp(g.experts, int(e), g.x, None, yt, ws)
        ye = yt.cpu().numpy()
        for t, j in zip(*np.nonzero(idx_np == e)):
            y[t * k + j] = ye[t]
    ysh = sg = None
    if g.shared is not None:
        ysht = torch.empty((T, H), dtype=torch.float32, device="cuda")
        capi.moe_shared_expert(g.shared, g.x, ysht, ws)
        ysh = ysht.cpu().numpy()
        sg = r["sg"].cpu().numpy() if g.gate is not None else None
    ref_bits = O.combine_f32(y, w.cpu().numpy(), ysh, sg)
    got_bits = out.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got_bits, ref_bits)


LAYER_CASES = [
    ("decode8_affine4_shared_zipf", {}),
    ("decode4_affine3", {}),
    ("decode32_w4a16", {}),
    ("prefill", dict(T=300, E=16, k=4, H=256, I=128, expert_fmt="affine4_g64",
                     shared_fmt="affine4_g64", gate_fmt="affine8_g64", zipf=True, seed=51)),
]


@pytest.mark.parametrize("name,cfg", LAYER_CASES, ids=[c[0] for c in LAYER_CASES])
def test_layer_chain_vs_oracle(capi, name, cfg):
    """The whole layer under the chain against the oracle's fp64 layer under
    the same chain (moe_layer(..., round_bf16=True)), within the layer's
    tolerance; the fused decode launch and the launch-per-step path agree bit
    for bit."""
    torch = Hn.torch()
    L = synth.gen_layer(**cfg) if cfg else synth.workload(name)
    g = Hn.GpuLayer(L)
    flags = capi.MOE_FLAG_ROUND_BF16
    out, idx, w = g.forward(flags=flags)
    if L.T <= capi.MOE_DECODE_MAX_TOKENS:
        out_u, idx_u, w_u = g.forward(flags=flags | capi.MOE_FLAG_UNFUSED)
        assert torch.equal(idx, idx_u) and torch.equal(w, w_u) and torch.equal(out, out_u)
    ref = Hn.oracle_layer(L, idx_override=idx.cpu().numpy(), round_bf16=True)
    Hn.assert_layer_close(Hn.to_np(out), ref["out"], out_type=L.act)
    # the chain's weights are bf16 values within one bf16 step of the oracle's
    wg = w.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(wg - ref["w"]) <= np.abs(ref["w"]) * 2.0 ** -7 * 1.01 + 1e-7)
    assert capi.moe_get_device_status(g.ws) == 0
