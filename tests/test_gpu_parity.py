"""GPU parity of the CUDA path against the fp64 CPU oracle (calls go through the C ABI).

Exact: packed bytes, unpacked codes, dequantised weights (fp32 rounding of the
exact value), top-k indices (given the GPU's own fp32 logits), bucket layouts,
3-bit vs widened 4-bit outputs, batch invariance.  Within tolerance
(|gpu - oracle| <= 1e-2 rms(oracle) + 1e-3): logits, routing weights, expert
projections, layer outputs.
"""

import math

import numpy as np
import pytest

from bit_affine_quantized_fp32_gb300 import synth
from oracle import oracle as O

from . import _harness as Hn

pytestmark = pytest.mark.gpu

FMTS = ["affine8_g64", "affine4_g64", "affine3_g64", "w4a16_g128", "affine2_g64", "affine5_g64",
        "affine6_g64"]


@pytest.fixture(scope="module")
def capi():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_affine_quantized_fp32_gb300 import build
    build.build()
    from bit_affine_quantized_fp32_gb300 import capi as C
    return C


# --------------------------------------------------------------------------
# formats

@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(1, 128), (7, 256), (33, 2048), (512, 640)])
def test_pack_unpack_bitexact(capi, fmt, shape):
    rng = np.random.default_rng(100 + shape[0])
    codes = synth.gen_codes(rng, fmt, *shape)
    gpu = Hn.gpu_pack(fmt, codes)
    ref = O.pack(fmt, codes)
    assert np.array_equal(gpu.cpu().numpy().view(np.uint32), ref)
    torch = Hn.torch()
    out = torch.empty(shape, dtype=torch.int8 if fmt == "w4a16_g128" else torch.uint8,
                      device="cuda")
    capi.moe_unpack(fmt, gpu, shape[0], shape[1], out)
    assert np.array_equal(out.cpu().numpy().astype(np.int32), codes)


EXPERT_FMTS = ["affine4_g64", "affine3_g64", "w4a16_g128", "affine2_g64", "affine5_g64",
               "affine6_g64", "affine8_g64"]
BITS_OF = {"affine2_g64": 2, "affine3_g64": 3, "affine4_g64": 4, "affine5_g64": 5,
           "affine6_g64": 6, "affine8_g64": 8, "w4a16_g128": 4}


def _tiled_reference(fmt, mats, I, H, which):
    """The tiled buffer of one matrix family written out in numpy from the
    layout's definition (blocks, chunks, (w, G) code blocks, lanes, planes,
    scale entries), independent of the repack kernel."""
    rows, K = (H, I) if which else (2 * I, H)
    CK = 512 if K % 512 == 0 else (256 if K % 256 == 0 else 128)
    ng, nch = CK // 64, K // CK
    nblk = H // 128 if which else I // 64
    w4 = fmt == "w4a16_g128"
    bits = BITS_OF[fmt]
    out = bytearray()
    for m in mats:
        codes = m.codes.astype(np.int64) + (8 if w4 else 0)          # stored values
        words = np.zeros((rows, K // 8), dtype=np.uint64)            # low 4 bits
        hiwords = np.zeros((rows, K // 8), dtype=np.uint64)          # bits 4..7
        for i in range(8):   # code i of a word in nibble (i & 1) * 4 + i // 2
            nib = (i & 1) * 4 + i // 2
            words |= ((codes[:, i::8] & 15).astype(np.uint64) << np.uint64(4 * nib))
            hiwords |= ((codes[:, i::8] >> 4).astype(np.uint64) << np.uint64(4 * nib))
        words = words.astype(np.uint32)
        hiwords = hiwords.astype(np.uint32)
        sc = m.scales.view(np.uint16) if m.scales.dtype != np.uint16 else m.scales
        bi = None if w4 else (m.biases.view(np.uint16) if m.biases.dtype != np.uint16 else m.biases)
        for blk in range(nblk):
            for c in range(nch):
                item = bytearray()
                for w in range(8):
                    if which:
                        base = blk * 128 + 16 * w
                    else:
                        base = blk * 64 + 16 * w if w < 4 else I + blk * 64 + 16 * (w - 4)
                    for G in range(ng):
                        lw = np.zeros((32, 4), dtype=np.uint32)
                        hw = np.zeros((32, 4), dtype=np.uint32)
                        for lane in range(32):
                            g, t = lane // 4, lane % 4
                            k0 = c * CK + 64 * G + 16 * t
                            for j in range(4):
                                r = base + g + 8 * (j >> 1)
                                lw[lane, j] = words[r, (k0 + 8 * (j & 1)) // 8]
                                hw[lane, j] = hiwords[r, (k0 + 8 * (j & 1)) // 8]
                        if bits in (2, 3):
                            m3 = np.uint32(0x33333333)
                            L01 = (lw[:, 0] & m3) | ((lw[:, 1] & m3) << np.uint32(2))
                            L23 = (lw[:, 2] & m3) | ((lw[:, 3] & m3) << np.uint32(2))
                            planes = [L01, L23]
                            if bits == 3:
                                planes.append(
                                    ((lw[:, 0] >> np.uint32(2)) & np.uint32(0x11111111))
                                    | ((lw[:, 1] >> np.uint32(1)) & np.uint32(0x22222222))
                                    | (lw[:, 2] & np.uint32(0x44444444))
                                    | ((lw[:, 3] << np.uint32(1)) & np.uint32(0x88888888)))
                            item += np.concatenate(planes).astype("<u4").tobytes()
                        else:
                            item += lw.astype("<u4").tobytes()
                            # the bits above the low nibble, by the written
                            # definitions of the 5-bit and 6-bit planes
                            if bits in (5, 6):
                                P = np.zeros((2, 32), dtype=np.uint64)
                                for x in range(4):
                                    for n in range(8):
                                        hb = (hw[:, x] >> np.uint32(4 * n)).astype(np.uint64)
                                        if bits == 5:
                                            pos = 4 * x + (n & 3) + 16 * (n >> 2)
                                            P[0] |= (hb & np.uint64(1)) << np.uint64(pos)
                                        else:
                                            pos = 2 * (4 * (x & 1) + (n & 3)) + 16 * (n >> 2)
                                            P[x >> 1] |= (hb & np.uint64(3)) << np.uint64(pos)
                                item += P[: 1 if bits == 5 else 2].astype("<u4").tobytes()
                            if bits == 8:
                                item += hw.astype("<u4").tobytes()
                gs = 128 if w4 else 64
                nsg = CK // gs
                for w in range(8):
                    if which:
                        base = blk * 128 + 16 * w
                    else:
                        base = blk * 64 + 16 * w if w < 4 else I + blk * 64 + 16 * (w - 4)
                    for g in range(8):
                        for G in range(nsg):
                            gi = c * nsg + G
                            r0, r1 = base + g, base + g + 8
                            if w4:
                                ent = [sc[r0, gi], sc[r1, gi]]
                            else:
                                ent = [sc[r0, gi], bi[r0, gi], sc[r1, gi], bi[r1, gi]]
                            item += np.array(ent, dtype="<u2").tobytes()
                out += item
    return np.frombuffer(bytes(out), dtype=np.uint8)


@pytest.mark.parametrize("fmt", EXPERT_FMTS)
def test_tiled_layout_matches_definition(capi, fmt):
    I, H = (256, 512) if fmt == "w4a16_g128" else (128, 640)   # chunks 256/512 and 128/128
    if fmt in ("affine5_g64", "affine6_g64", "affine8_g64"):
        I, H = 128, 256
    bank = synth.gen_bank(np.random.default_rng(41), fmt, 2, I, H)
    tb = Hn.gpu_bank(bank)
    got13 = tb.tensors[0].cpu().numpy()
    got2 = tb.tensors[3].cpu().numpy()
    assert np.array_equal(got13, _tiled_reference(fmt, bank.w13, I, H, 0))
    assert np.array_equal(got2, _tiled_reference(fmt, bank.w2, I, H, 1))


@pytest.mark.parametrize("fmt", EXPERT_FMTS)
@pytest.mark.parametrize("E,I,H", [(3, 256, 768), (2, 512, 2048), (1, 256, 1280)])
def test_repack_roundtrip_bitexact(capi, fmt, E, I, H):
    if fmt == "w4a16_g128" and (H % 256 or I % 256):
        pytest.skip("W4A16 shapes are multiples of 256")
    bank = synth.gen_bank(np.random.default_rng(42 + E), fmt, E, I, H)
    canon = Hn.gpu_bank_canonical(bank)
    tiled = canon.tiled()
    torch = Hn.torch()
    outs = [torch.zeros_like(t) if t is not None else None for t in canon.tensors]
    capi.moe_unrepack_bank(tiled, *outs)
    for a, b in zip(canon.tensors, outs):
        if a is not None:
            assert torch.equal(a, b)


@pytest.mark.parametrize("fmt", FMTS + ["f32", "bf16"])
def test_dequant_bitexact(capi, fmt):
    rng = np.random.default_rng(7)
    rows, cols = 24, 512
    m = synth.gen_qmatrix(rng, fmt, rows, cols)
    gm = Hn.gpu_matrix(m)
    torch = Hn.torch()
    w = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
    capi.moe_dequant(gm, w)
    om = Hn.oracle_matrix(m)
    ref = O.dequant(fmt, om["q"], om.get("s"), om.get("b"), rows, cols).astype(np.float32)
    assert np.array_equal(w.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_dequant_special_scales(capi):
    # zero, subnormal, negative and maximal fp16 scales/biases
    fmt = "affine4_g64"
    rows, cols = 8, 128
    codes = np.tile(np.arange(16, dtype=np.int32), (rows, cols // 16))
    special = np.array([0x0000, 0x8000, 0x0001, 0x03FF, 0x7BFF, 0xFBFF, 0x3C00, 0xB555], np.uint16)
    s = np.stack([special, special[::-1]], axis=1)
    b = np.stack([special[::-1], special], axis=1)
    m = synth.QMatrix(fmt, rows, cols, codes=codes, scales=s, biases=b)
    gm = Hn.gpu_matrix(m)
    torch = Hn.torch()
    w = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
    capi.moe_dequant(gm, w)
    om = Hn.oracle_matrix(m)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = O.dequant(fmt, om["q"], s, b, rows, cols).astype(np.float32)
    got = w.cpu().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok].view(np.uint32), ref[ok].view(np.uint32))


# --------------------------------------------------------------------------
# routing

def _route_case(T, E, k, H, rfmt, gfmt, zipf, seed):
    L = synth.gen_layer(T=T, E=E, k=k, H=H, I=128, expert_fmt="affine4_g64", router_fmt=rfmt,
                        shared_fmt="affine4_g64" if gfmt else None, gate_fmt=gfmt, zipf=zipf,
                        seed=seed)
    return L


@pytest.mark.parametrize("T,E,k,H,rfmt,gfmt,zipf", [
    (1, 256, 8, 2048, "f32", None, False),
    (8, 256, 8, 2048, "f32", "affine8_g64", True),
    (4, 256, 8, 2048, "affine8_g64", "affine8_g64", False),
    (32, 256, 8, 2048, "f32", "bf16", False),
    (37, 16, 4, 384, "bf16", "bf16", True),
    (200, 64, 8, 256, "f32", None, True),
])
def test_route_parity(capi, T, E, k, H, rfmt, gfmt, zipf):
    L = _route_case(T, E, k, H, rfmt, gfmt, zipf, seed=T + E)
    g = Hn.GpuLayer(L)
    r = g.route()
    lg = r["logits"].cpu().numpy().astype(np.float64)
    x = O.act_to_double(L.act, L.x)
    ref = O.router_logits(Hn.oracle_matrix(L.router), x, L.logit_bias)
    # fp32 dot product of H terms: error bound ~ H * 2^-24 * sum |w x|
    W = np.abs(O.dequant(rfmt, Hn.oracle_matrix(L.router)["q"], Hn.oracle_matrix(L.router).get("s"),
                         Hn.oracle_matrix(L.router).get("b"), E, H))
    bound = H * 2.0 ** -24 * (np.abs(x) @ W.T) + 1e-6
    assert np.all(np.abs(lg - ref) <= bound)
    # top-k on the GPU's own fp32 logits: indices exact, weights close
    idx_ref, w_ref = O.topk(lg, k)
    idx = r["idx"].cpu().numpy()
    assert np.array_equal(idx, idx_ref)
    assert np.allclose(r["w"].cpu().numpy(), w_ref, rtol=2e-6, atol=1e-7)
    # against fp64 logits: equal except at near ties (within the bound)
    idx64, _ = O.topk(ref, k)
    for t in np.nonzero(np.any(idx64 != idx, axis=1))[0]:
        srt = np.sort(ref[t])[::-1]
        gaps = np.abs(np.diff(srt[: k + 1]))
        assert gaps.min() <= 2 * bound[t].max(), f"token {t}: routing differs without a near tie"
    # shared gate
    if gfmt:
        _, sg_ref = O.shared_gate(Hn.oracle_matrix(L.gate), x)
        assert np.allclose(r["sg"].cpu().numpy(), sg_ref, rtol=1e-5, atol=1e-6)
    # bucketing: exact against the oracle's counting sort of the GPU's picks
    counts, offs, perm, active = O.bucket(idx, E)
    assert np.array_equal(r["offsets"].cpu().numpy(), offs)
    assert np.array_equal(r["perm"].cpu().numpy(), perm)


def test_topk_edge_rows(capi):
    torch = Hn.torch()
    E, k = 256, 8
    rows = []
    rows.append(np.zeros(E))                             # flat row
    r = np.zeros(E); r[[200, 3, 77]] = 5.0; rows.append(r)  # ties -> lower id first
    rows.append(np.full(E, np.nan))                      # all NaN -> ids 0..7
    r = np.arange(E, dtype=np.float64); r[255] = np.nan; r[254] = -np.inf; rows.append(r)
    r = np.full(E, -np.inf); r[9] = 1.0; rows.append(r)
    r = -np.arange(E, dtype=np.float64); r[[0, 1]] = np.nan; rows.append(r)
    rng = np.random.default_rng(3)
    rows.append(rng.integers(-2, 3, E).astype(np.float64))  # many ties
    r = np.full(E, -1.0); r[5] = -0.0; r[3] = 0.0; r[200] = -0.0; rows.append(r)  # -0 == +0
    r = np.full(E, np.inf); r[[7, 9]] = np.nan; rows.append(r)  # +inf ties
    lg = np.stack(rows).astype(np.float32)
    T = lg.shape[0]
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    capi.moe_topk_softmax(Hn.dev(lg), k, idx, w)
    idx_ref, w_ref = O.topk(lg.astype(np.float64), k)
    assert np.array_equal(idx.cpu().numpy(), idx_ref)
    wg = w.cpu().numpy()
    assert np.array_equal(np.isnan(wg), np.isnan(w_ref))
    ok = ~np.isnan(w_ref)
    assert np.allclose(wg[ok], w_ref[ok], rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("T,k,E", [(0, 8, 16), (1, 8, 256), (32, 8, 256), (512, 8, 256),
                                   (4096, 8, 256), (3, 1, 1), (100, 3, 5)])
def test_bucket_bitexact(capi, T, k, E):
    torch = Hn.torch()
    rng = np.random.default_rng(T + k + E)
    if T:
        p = np.exp(-1.1 * np.log(np.arange(1, E + 1)))
        idx = np.stack([rng.choice(E, size=k, replace=False, p=p / p.sum()) for _ in range(T)])
    else:
        idx = np.zeros((0, k), np.int64)
    idx = idx.astype(np.int32)
    offs = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    perm = torch.full((max(T * k, 1),), -1, dtype=torch.int32, device="cuda")
    capi.moe_bucket(Hn.dev(idx) if T else torch.zeros((0, k), dtype=torch.int32, device="cuda"),
                    E, offs, perm)
    _, offs_ref, perm_ref, _ = O.bucket(idx, E)
    assert np.array_equal(offs.cpu().numpy(), offs_ref)
    assert np.array_equal(perm.cpu().numpy()[: T * k], perm_ref)


# --------------------------------------------------------------------------
# experts

@pytest.mark.parametrize("fmt,act,T,H,I", [
    ("affine4_g64", "bf16", 1, 2048, 512),
    ("affine4_g64", "bf16", 13, 256, 128),
    ("affine3_g64", "bf16", 5, 2048, 512),
    ("affine3_g64", "bf16", 40, 384, 256),
    ("w4a16_g128", "f16", 32, 2048, 512),
    ("w4a16_g128", "bf16", 3, 512, 256),
    ("affine4_g64", "f16", 9, 512, 128),
    ("affine2_g64", "bf16", 6, 512, 256),
    ("affine5_g64", "bf16", 11, 2048, 512),
    ("affine6_g64", "f16", 7, 384, 128),
    ("affine8_g64", "bf16", 8, 512, 128),
    ("affine8_g64", "f16", 3, 256, 256),
])
def test_expert_mlp_per_projection(capi, fmt, act, T, H, I):
    torch = Hn.torch()
    rng = np.random.default_rng(T * 7 + H)
    bank = synth.gen_bank(rng, fmt, 2, I, H)
    x = synth.gen_x(rng, T, H, act)
    gb = Hn.gpu_bank(bank)
    ws = Hn.workspace(T, 2, 1, H, I)
    h = torch.empty((T, I), dtype=torch.float32, device="cuda")
    y = torch.empty((T, H), dtype=torch.float32, device="cuda")
    capi.moe_expert_mlp(gb, 1, Hn.bits16(x, act), h, y, ws)
    xd = O.act_to_double(act, x)
    ob = Hn.oracle_bank(bank)
    h_ref, y_ref = O.expert_mlp(fmt, I, H, Hn.oracle_expert(ob, 1), xd)
    hg = h.cpu().numpy().astype(np.float64)
    Hn.assert_layer_close(hg, h_ref, "h (gate/up projection)")
    # gate/up sums are exact-product fp32 sums: far inside the tolerance
    assert Hn.projection_errors(hg, h_ref)["aggregate_rel"] < 1e-5
    # down alone, on the GPU's own h
    y_down = O.down(fmt, H, I, ob["w2"][1], ob["s2"][1], ob.get("b2", [None, None])[1], hg)
    yg = y.cpu().numpy().astype(np.float64)
    Hn.assert_layer_close(yg, y_down, "y (down projection)")
    assert Hn.projection_errors(yg, y_down)["aggregate_rel"] < 1e-4
    Hn.assert_layer_close(yg, y_ref, "y (expert)")


# --------------------------------------------------------------------------
# the layer

SMALL = [
    # (name-like, overrides)
    dict(T=1, E=16, k=8, H=256, I=128, expert_fmt="affine4_g64", seed=1),
    dict(T=8, E=32, k=8, H=512, I=128, expert_fmt="affine4_g64", shared_fmt="affine4_g64",
         gate_fmt="affine8_g64", zipf=True, seed=2),
    dict(T=4, E=16, k=8, H=512, I=256, expert_fmt="affine3_g64", router_fmt="affine8_g64",
         shared_fmt="affine4_g64", gate_fmt="affine8_g64", seed=3),
    dict(T=32, E=64, k=8, H=512, I=256, expert_fmt="w4a16_g128", shared_fmt="w4a16_g128",
         gate_fmt="bf16", act="f16", seed=4),
    dict(T=19, E=12, k=3, H=384, I=128, expert_fmt="affine4_g64", shared_fmt="affine3_g64",
         gate_fmt="f32", seed=5),
    dict(T=70, E=16, k=4, H=256, I=128, expert_fmt="affine4_g64", shared_fmt="affine4_g64",
         gate_fmt="affine8_g64", zipf=True, seed=6),
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: f"T{c['T']}_{c['expert_fmt']}")
def test_layer_small(capi, cfg):
    L = synth.gen_layer(**cfg)
    g = Hn.GpuLayer(L)
    out, idx, w = g.forward()
    idx = idx.cpu().numpy()
    ref = Hn.oracle_layer(L, idx_override=idx)
    Hn.assert_layer_close(Hn.to_np(out), ref["out"], out_type=L.act)


@pytest.mark.parametrize("name", ["decode1_affine4", "decode8_affine4_shared_zipf",
                                  "decode4_affine3", "decode32_w4a16"])
def test_layer_full_size(capi, name):
    """Every output of the workload at its full size (E=256, hidden 2048,
    inter 512), from the seeded synthetic inputs, against the oracle."""
    L = synth.workload(name)
    g = Hn.GpuLayer(L)
    out, idx, w = g.forward()
    idx = idx.cpu().numpy()
    ref = Hn.oracle_layer(L, idx_override=idx)
    Hn.assert_layer_close(Hn.to_np(out), ref["out"], out_type=L.act)
    # routing matched the oracle's own fp64 routing except at near ties
    Hn.assert_routing_near_ties(L, idx, ref["logits"])


def test_batch_invariance(capi):
    """Row r of a T-token call is bit-identical to the same token alone, in
    any batch composition and order."""
    L = synth.gen_layer(T=32, E=64, k=8, H=512, I=256, expert_fmt="affine4_g64",
                        shared_fmt="affine4_g64", gate_fmt="affine8_g64", zipf=True, seed=21)
    g = Hn.GpuLayer(L, max_tokens=32)
    full, _, _ = g.forward()
    full = full.cpu()
    torch = Hn.torch()
    for t in [0, 5, 31]:
        one, _, _ = g.forward(g.x[t:t + 1])
        assert torch.equal(one.cpu()[0], full[t])
    for lo, hi in [(0, 4), (8, 16), (3, 30)]:
        part, _, _ = g.forward(g.x[lo:hi].contiguous())
        assert torch.equal(part.cpu(), full[lo:hi])
    p = torch.randperm(32, generator=torch.Generator().manual_seed(0))
    perm_out, _, _ = g.forward(g.x[p.cuda()].contiguous())
    assert torch.equal(perm_out.cpu(), full[p])


def test_3bit_widened_to_4bit_bitexact(capi):
    """The same 3-bit codes stored as 4-bit words give bit-identical outputs."""
    L3 = synth.gen_layer(T=6, E=16, k=8, H=512, I=256, expert_fmt="affine3_g64",
                         shared_fmt="affine3_g64", gate_fmt="affine8_g64", seed=22)
    g3 = Hn.GpuLayer(L3)
    out3, _, _ = g3.forward()

    def widen(b):
        nb = synth.ExpertBank("affine4_g64", b.E, b.I, b.H)
        nb.w13 = [synth.QMatrix("affine4_g64", m.rows, m.cols, codes=m.codes, scales=m.scales,
                                biases=m.biases) for m in b.w13]
        nb.w2 = [synth.QMatrix("affine4_g64", m.rows, m.cols, codes=m.codes, scales=m.scales,
                               biases=m.biases) for m in b.w2]
        return nb

    L3.experts = widen(L3.experts)
    L3.shared = widen(L3.shared)
    g4 = Hn.GpuLayer(L3)
    out4, _, _ = g4.forward()
    assert Hn.torch().equal(out3, out4)


def _rewidth(b, fmt):
    """The same codes, scales and biases stored at another affine width."""
    nb = synth.ExpertBank(fmt, b.E, b.I, b.H)
    nb.w13 = [synth.QMatrix(fmt, m.rows, m.cols, codes=m.codes, scales=m.scales,
                            biases=m.biases) for m in b.w13]
    nb.w2 = [synth.QMatrix(fmt, m.rows, m.cols, codes=m.codes, scales=m.scales,
                           biases=m.biases) for m in b.w2]
    return nb


@pytest.mark.parametrize("T", [5, 40])
def test_codes_widened_across_all_widths_bitexact(capi, T):
    """The widening control of "qwen3_5_moe on native CUDA with 3-bit routed
    experts ... #803" (comment "The 3-bit width is up as #972") at every width
    the expert kernels read: 2-bit codes stored as 2-, 3-, 4-, 5-, 6- and
    8-bit banks give bit-identical layers (one accumulation order on the
    exact integer codes), in the fused and the launch-per-step decode forms
    (T=5) and in the decode form of a prefill-sized call (T=40)."""
    torch = Hn.torch()
    L = synth.gen_layer(T=T, E=16, k=8, H=512, I=256, expert_fmt="affine2_g64",
                        shared_fmt="affine2_g64", gate_fmt="affine8_g64", seed=27)
    flags = capi.MOE_FLAG_FORCE_DECODE
    ref = None
    for fmt in ["affine2_g64", "affine3_g64", "affine4_g64", "affine5_g64", "affine6_g64",
                "affine8_g64"]:
        L.experts = _rewidth(L.experts, fmt)
        L.shared = _rewidth(L.shared, fmt)
        g = Hn.GpuLayer(L)
        outs = [g.forward(flags=flags)[0], g.forward(flags=flags | capi.MOE_FLAG_UNFUSED)[0]]
        for o in outs:
            if ref is None:
                ref = o
            assert torch.equal(o, ref), fmt
    ref_o = Hn.oracle_layer(L, idx_override=g.forward(flags=flags)[1].cpu().numpy())
    Hn.assert_layer_close(Hn.to_np(ref), ref_o["out"], out_type=L.act)


@pytest.mark.parametrize("fmt", ["affine2_g64", "affine5_g64", "affine6_g64", "affine8_g64"])
def test_other_widths_full_size(capi, fmt):
    """MLX affine experts at the other widths the pages' loader reads
    ("Affine experts at other widths"), at full size: decode batch 8 (E=256,
    hidden 2048, inter 512, Zipf routing, a shared expert of the same width),
    every output against the oracle, the routing against its fp64 routing up
    to near ties."""
    L = synth.workload("decode8_affine4_shared_zipf", expert_fmt=fmt, shared_fmt=fmt)
    g = Hn.GpuLayer(L)
    out, idx, _ = g.forward()
    assert capi.moe_get_device_status(g.ws) == 0
    idx = idx.cpu().numpy()
    ref = Hn.oracle_layer(L, idx_override=idx)
    Hn.assert_layer_close(Hn.to_np(out), ref["out"], out_type=L.act)
    Hn.assert_routing_near_ties(L, idx, ref["logits"])


def test_zero_tokens_and_zero_input(capi):
    L = synth.gen_layer(T=3, E=8, k=2, H=256, I=128, expert_fmt="affine4_g64",
                        shared_fmt="affine4_g64", gate_fmt="affine8_g64", seed=23)
    g = Hn.GpuLayer(L)
    torch = Hn.torch()
    out, _, _ = g.forward(g.x[:0])
    assert out.shape == (0, 256)
    z = torch.zeros_like(g.x)
    out, _, _ = g.forward(z)
    assert torch.count_nonzero(out.float()) == 0


def test_decode_path_large_T(capi):
    """The grouped-GEMV path at a prefill-sized T (more than 4 n-tiles per
    expert) on sampled rows."""
    L = synth.gen_layer(T=300, E=16, k=4, H=256, I=128, expert_fmt="affine4_g64",
                        shared_fmt="affine4_g64", gate_fmt="affine8_g64", zipf=True, seed=24)
    g = Hn.GpuLayer(L)
    out, idx, _ = g.forward(flags=1)
    ref = Hn.oracle_layer(L, idx_override=idx.cpu().numpy())
    Hn.assert_layer_close(Hn.to_np(out), ref["out"], out_type=L.act)


def test_validation_errors(capi):
    torch = Hn.torch()
    L = synth.gen_layer(T=2, E=8, k=2, H=256, I=128, expert_fmt="affine4_g64", seed=25)
    g = Hn.GpuLayer(L)
    out = torch.empty((2, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(capi.MoeError) as e:
        capi.moe_layer_forward(g.router, None, None, g.experts, None, g.x, 9, out, ws=g.ws)
    assert e.value.status == 1
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(capi.MoeError) as e:
        capi.moe_layer_forward(g.router, None, None, g.experts, None, g.x, 2, out, ws=small)
    assert e.value.status == 3
    bad = capi.ExpertBank("bf16", 8, 128, 256, *g.experts.tensors)
    with pytest.raises(capi.MoeError) as e:
        capi.moe_layer_forward(g.router, None, None, bad, None, g.x, 2, out, ws=g.ws)
    assert e.value.status == 2 and "BF16" in str(e.value)
    assert capi.moe_get_device_status(g.ws) == 0


FUSED_CASES = [
    dict(T=1, E=256, k=8, H=2048, I=512, expert_fmt="affine4_g64", seed=31),
    dict(T=8, E=256, k=8, H=2048, I=512, expert_fmt="affine4_g64", shared_fmt="affine4_g64",
         gate_fmt="affine8_g64", zipf=True, seed=32),
    dict(T=4, E=64, k=8, H=1024, I=256, expert_fmt="affine3_g64", router_fmt="affine8_g64",
         shared_fmt="affine4_g64", gate_fmt="affine8_g64", seed=33),
    dict(T=32, E=128, k=8, H=1024, I=512, expert_fmt="w4a16_g128", shared_fmt="w4a16_g128",
         gate_fmt="bf16", act="f16", seed=34),
    dict(T=13, E=12, k=3, H=384, I=128, expert_fmt="affine4_g64", shared_fmt="affine3_g64",
         seed=35),
]


@pytest.mark.parametrize("cfg", FUSED_CASES, ids=lambda c: f"T{c['T']}_{c['expert_fmt']}")
def test_fused_layer_equals_unfused_and_oracle(capi, cfg):
    """The single persistent launch gives the same bits as the launch-per-step
    path, repeatably (its counters reset themselves), and matches the oracle."""
    L = synth.gen_layer(**cfg)
    g = Hn.GpuLayer(L)
    torch = Hn.torch()
    outs = []
    for _ in range(3):
        out, idx, w = g.forward()
        outs.append((out.clone(), idx.clone(), w.clone()))
    ref_out, ref_idx, ref_w = g.forward(flags=capi.MOE_FLAG_UNFUSED)
    for out, idx, w in outs:
        assert torch.equal(idx, ref_idx)
        assert torch.equal(w, ref_w)
        assert torch.equal(out, ref_out)
    assert capi.moe_get_device_status(g.ws) == 0
    ref = Hn.oracle_layer(L, idx_override=ref_idx.cpu().numpy())
    Hn.assert_layer_close(Hn.to_np(outs[0][0]), ref["out"], out_type=L.act)


def test_fused_alternating_shapes(capi):
    """Fused calls of different token counts on one workspace."""
    L = synth.gen_layer(T=32, E=64, k=8, H=512, I=256, expert_fmt="affine4_g64",
                        shared_fmt="affine4_g64", gate_fmt="affine8_g64", zipf=True, seed=36)
    g = Hn.GpuLayer(L, max_tokens=32)
    torch = Hn.torch()
    full, _, _ = g.forward()
    for T in [1, 7, 32, 3, 16]:
        part, _, _ = g.forward(g.x[:T].contiguous())
        assert torch.equal(part, full[:T])
    assert capi.moe_get_device_status(g.ws) == 0


# ---------------------------------------------------------------------------
# Prefill form (T > 32): the tcgen05 expert GEMMs with single fp16 operands
# (weights fp16(s*q + b) rounded once, x and h in fp16) and fp32
# accumulation; the tolerance is the layer's (a CPU emulation of the
# full-size window puts the operands' rounding at about a fifth of it).

PREFILL_CASES = [
    # Zipf routing: the busiest experts take more than one 128-token tile
    dict(T=300, E=16, k=4, H=256, I=128, expert_fmt="affine4_g64", shared_fmt="affine4_g64",
         gate_fmt="affine8_g64", zipf=True, seed=41),
    dict(T=200, E=8, k=2, H=512, I=256, expert_fmt="affine3_g64", router_fmt="affine8_g64",
         shared_fmt="affine4_g64", gate_fmt="affine8_g64", seed=42),
    dict(T=160, E=16, k=8, H=512, I=256, expert_fmt="w4a16_g128", shared_fmt="w4a16_g128",
         gate_fmt="bf16", act="f16", seed=43),
    # the smallest prefill call; four experts hold every token (tiles of 33)
    dict(T=33, E=4, k=4, H=256, I=128, expert_fmt="affine4_g64", seed=44),
    # 300 tokens per expert: three tiles each, the last one ragged
    dict(T=600, E=4, k=2, H=256, I=128, expert_fmt="affine4_g64", shared_fmt="affine4_g64",
         seed=45),
]


@pytest.mark.parametrize("cfg", PREFILL_CASES,
                         ids=lambda c: f"T{c['T']}_E{c['E']}_{c['expert_fmt']}")
def test_prefill_layer(capi, cfg):
    L = synth.gen_layer(**cfg)
    g = Hn.GpuLayer(L)
    out, idx, _ = g.forward()
    ref = Hn.oracle_layer(L, idx_override=idx.cpu().numpy())
    Hn.assert_layer_close(Hn.to_np(out), ref["out"], out_type=L.act)
    # the decode form of the same call agrees with the oracle too
    out_d, idx_d, _ = g.forward(flags=1)
    assert Hn.torch().equal(idx, idx_d)
    Hn.assert_layer_close(Hn.to_np(out_d), ref["out"], out_type=L.act)


def test_prefill_graph_capture_with_side_stream(capi):
    """The prefill form forks the light experts' decode units onto a side
    stream and joins them before the combine: captured into a CUDA graph on
    the caller's stream and replayed, the call gives the eager call's bits
    (and the oracle's values), the light experts included."""
    torch = Hn.torch()
    L = synth.gen_layer(T=300, E=64, k=4, H=256, I=128, expert_fmt="affine4_g64",
                        shared_fmt="affine4_g64", gate_fmt="affine8_g64", zipf=True, seed=46)
    g = Hn.GpuLayer(L)
    out, idx, w = g.forward()
    counts = np.bincount(idx.cpu().numpy().ravel(), minlength=L.E)
    assert ((counts > 0) & (counts <= 16)).any() and (counts > 16).any()  # both kinds
    out_g = torch.empty_like(out)
    idx_g = torch.empty_like(idx)
    w_g = torch.empty_like(w)
    from bit_affine_quantized_fp32_gb300 import capi as C

    def call():
        C.moe_layer_forward(g.router, g.bias, g.gate, g.experts, g.shared, g.x, L.k, out_g,
                            idx_g, w_g, 0, g.ws)

    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):  # the library's per-stream state is made outside capture
        call()
    cap.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        call()
    for _ in range(3):
        out_g.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_g, out) and torch.equal(idx_g, idx) and torch.equal(w_g, w)
    ref = Hn.oracle_layer(L, idx_override=idx.cpu().numpy())
    Hn.assert_layer_close(Hn.to_np(out_g), ref["out"], out_type=L.act)
    assert capi.moe_get_device_status(g.ws) == 0


def test_prefill_standalone_calls_equal_the_layer(capi):
    """moe_route, moe_shared_expert and moe_experts_forward above 32 tokens
    (the standalone prefill flow: its own tables launch and activation pass,
    the light experts on the side stream) give the layer's bits; the layer
    builds its tables in the bucket launch and folds the shared expert into
    the routed experts' GEMM launches."""
    torch = Hn.torch()
    L = synth.gen_layer(T=300, E=64, k=4, H=256, I=128, expert_fmt="affine4_g64",
                        shared_fmt="affine4_g64", gate_fmt="affine8_g64", zipf=True, seed=47)
    g = Hn.GpuLayer(L)
    out, idx, w = g.forward()
    r = g.route()
    assert torch.equal(r["idx"], idx) and torch.equal(r["w"], w)
    ysh = torch.empty((L.T, L.H), dtype=torch.float32, device="cuda")
    capi.moe_shared_expert(g.shared, g.x, ysh, g.ws)
    out2 = torch.empty_like(out)
    capi.moe_experts_forward(g.experts, g.x, L.k, r["idx"], r["w"], r["offsets"], r["perm"], ysh,
                             r["sg"], out2, 0, g.ws)
    torch.cuda.synchronize()
    assert torch.equal(out2, out)
    ref = Hn.oracle_layer(L, idx_override=idx.cpu().numpy())
    Hn.assert_layer_close(Hn.to_np(out2), ref["out"], out_type=L.act)
    assert capi.moe_get_device_status(g.ws) == 0


def test_prefill_range_status(capi):
    """The prefill form's operands are fp16: a bf16 activation beyond fp16's
    range (2^17 here) sets MOE_ERR_RANGE in the workspace status word; the
    decode form of the same tokens does not, and after the workspace is
    re-initialised an in-range call reads 0."""
    torch = Hn.torch()
    L = synth.gen_layer(T=40, E=8, k=2, H=256, I=128, expert_fmt="affine4_g64", seed=48)
    g = Hn.GpuLayer(L)
    out, _, _ = g.forward()
    assert capi.moe_get_device_status(g.ws) == 0
    xbig = g.x.clone()
    xbig[3, 5] = 131072.0
    g.forward(xbig)
    torch.cuda.synchronize()
    assert capi.moe_get_device_status(g.ws) == 7  # MOE_ERR_RANGE
    capi.moe_workspace_init(g.ws)
    g.forward(xbig[:32].contiguous())  # the decode form (T <= 32): no fp16 operands
    assert capi.moe_get_device_status(g.ws) == 0
    out2, _, _ = g.forward()
    assert capi.moe_get_device_status(g.ws) == 0
    assert torch.equal(out2, out)


@pytest.mark.parametrize("name", ["decode8_affine4_shared_zipf", "decode4_affine3",
                                  "decode32_w4a16"])
def test_force_prefill_at_decode_sizes(capi, name):
    """MOE_FLAG_FORCE_PREFILL runs the prefill form (tensor-core GEMMs for the
    experts above the light threshold, the shared expert folded in) at a
    decode batch: every output against the oracle at full size, the routing
    equal to the decode form's."""
    torch = Hn.torch()
    L = synth.workload(name)
    g = Hn.GpuLayer(L)
    out_d, idx_d, w_d = g.forward()
    out, idx, w = g.forward(flags=capi.MOE_FLAG_FORCE_PREFILL)
    assert torch.equal(idx, idx_d) and torch.equal(w, w_d)
    ref = Hn.oracle_layer(L, idx_override=idx.cpu().numpy())
    Hn.assert_layer_close(Hn.to_np(out), ref["out"], out_type=L.act)
    assert capi.moe_get_device_status(g.ws) == 0


def test_prefill_full_size(capi):
    """The 512-token prefill window at full size (E=256, hidden 2048, inter
    512, Zipf routing, shared expert): every output of every token against the
    oracle, the routing against the oracle's fp64 routing up to near ties."""
    L = synth.workload("prefill512_affine4_zipf")
    g = Hn.GpuLayer(L)
    out, idx, _ = g.forward()
    assert capi.moe_get_device_status(g.ws) == 0
    idx = idx.cpu().numpy()
    ref = Hn.oracle_layer(L, idx_override=idx)
    Hn.assert_layer_close(Hn.to_np(out), ref["out"], out_type=L.act)
    Hn.assert_routing_near_ties(L, idx, ref["logits"])


def test_prefill_sweep_4096_in_512_windows(capi):
    """A 4096-token prompt as eight consecutive 512-row windows through the
    layer (the chunking of "Native server: --backend xpu for Nemotron on Intel
    Arc", update comment), one workspace, every window compared in full with
    the oracle's layer over all 4096 tokens."""
    torch = Hn.torch()
    L = synth.workload("prefill512_affine4_zipf", T=4096)
    g = Hn.GpuLayer(L, max_tokens=512)
    outs, idxs = [], []
    for w in range(8):
        o, i, _ = g.forward(g.x[512 * w: 512 * (w + 1)])
        outs.append(o)
        idxs.append(i)
    assert capi.moe_get_device_status(g.ws) == 0
    out = torch.cat(outs).cpu()
    idx = torch.cat(idxs).cpu().numpy()
    ref = Hn.oracle_layer(L, idx_override=idx)
    got = Hn.to_np(out)
    for w in range(8):
        rows = slice(512 * w, 512 * (w + 1))
        Hn.assert_layer_close(got[rows], ref["out"][rows], f"window {w}", out_type=L.act)
    Hn.assert_routing_near_ties(L, idx, ref["logits"])


def test_wait_timeout_reported_and_recovered(capi):
    """A bounded device-side wait that runs out (the engine's counterpart of
    the serving loop's wall-clock guard in "Native server: --backend xpu for
    Nemotron on Intel Arc", update comment): with the workspace's wait limit
    set to 1 us, the fused decode launch -- whose CTAs wait microseconds for
    each other's router rows and h rows -- records MOE_ERR_TIMEOUT and still
    ends; after moe_workspace_init the next call gives the same bits as before
    and matches the oracle."""
    torch = Hn.torch()
    L = synth.workload("decode8_affine4_shared_zipf")
    g = Hn.GpuLayer(L)
    ref_out, ref_idx, _ = g.forward()
    assert capi.moe_get_device_status(g.ws) == 0
    capi.moe_workspace_set_wait_limit(g.ws, 1)
    g.forward()
    torch.cuda.synchronize()  # the launch ended
    assert capi.moe_get_device_status(g.ws) == 5  # MOE_ERR_TIMEOUT
    capi.moe_workspace_init(g.ws)
    out, idx, _ = g.forward()
    assert capi.moe_get_device_status(g.ws) == 0
    assert torch.equal(idx, ref_idx) and torch.equal(out, ref_out)
    ref = Hn.oracle_layer(L, idx_override=idx.cpu().numpy())
    Hn.assert_layer_close(Hn.to_np(out), ref["out"], out_type=L.act)
    with pytest.raises(capi.MoeError) as e:
        capi.moe_workspace_set_wait_limit(g.ws, 1 << 31)
    assert e.value.status == 1
