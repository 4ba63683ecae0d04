"""Pins of the fp64 CPU oracle against what the format definitions and the
mathematics fix (no GPU).  Every oracle function is checked here against
something other than itself: hand-derived words, a big-integer bit stream,
numpy's own fp16/bf16 decoding, exact rational arithmetic, brute force over
orderings, closed-form softmax values, and a dense SwiGLU MLP written with
numpy matrix products.

Sources (page title, section):
  * "qwen3_5_moe on native CUDA with 3-bit routed experts ... #803":
    Description (MLX affine, groups of 64, 3/4/8-bit); comment "Progress on
    the 4-bit gate" (routing, weights, shared slot, SwiGLU epilogue, host
    reference checks with a tie, a flat row and a NaN); comment "The 3-bit
    width is up as #972" (3-bit codes rewritten as 4-bit words).
  * "Sage-1.5-W4A16", Model details / Recipe: int4 symmetric, group 128.
"""

import itertools
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import oracle as O
from bit_affine_quantized_fp32_gb300 import synth


def stream_int(words: np.ndarray) -> int:
    """The packed row as one little-endian integer (bit 0 = bit 0 of word 0)."""
    return int.from_bytes(np.ascontiguousarray(words, dtype="<u4").tobytes(), "little")


# --------------------------------------------------------------------------
# Formats: bit layout

def test_pack_affine4_hand_word():
    # codes 1..8 then 15,0,... : code i sits at bits [4i, 4i+4) of a word
    codes = np.zeros((1, 64), np.int32)
    codes[0, :8] = [1, 2, 3, 4, 5, 6, 7, 8]
    codes[0, 8] = 15
    w = O.pack("affine4_g64", codes)
    assert w[0, 0] == 0x87654321
    assert w[0, 1] == 0x0000000F
    assert np.all(w[0, 2:] == 0)


def test_pack_affine8_hand_word():
    codes = np.zeros((1, 64), np.int32)
    codes[0, :4] = [0x11, 0x22, 0x33, 0xFE]
    w = O.pack("affine8_g64", codes)
    assert w[0, 0] == 0xFE332211


def test_pack_affine3_hand_words():
    # codes c_i = 7 for i = 10 (straddles words 0/1: stream bits 30..32) and
    # c_21 = 5 (stream bits 63..65, straddles words 1/2), all others 0.
    codes = np.zeros((1, 64), np.int32)
    codes[0, 10] = 7
    codes[0, 21] = 5
    w = O.pack("affine3_g64", codes)
    # bits 30,31 of word 0 set; bit 0 of word 1 set (7 = 0b111)
    assert w[0, 0] == 0xC0000000
    # c_21 = 0b101: stream bit 63 (word 1 bit 31) = 1, bit 64 (word 2 bit 0) = 0,
    # bit 65 (word 2 bit 1) = 1
    assert w[0, 1] == 0x80000001
    assert w[0, 2] == 0x00000002
    assert w.shape == (1, 6)   # 64 codes * 3 bits = 192 bits = 6 words


def test_pack_w4a16_offset_binary():
    # compressed-tensors stores q + 8: q = -8 -> 0, q = 7 -> 15, q = -1 -> 7
    codes = np.zeros((1, 128), np.int32) - 8
    codes[0, 0] = 7
    codes[0, 1] = -1
    codes[0, 2] = 0
    w = O.pack("w4a16_g128", codes)
    assert w[0, 0] == 0x0000087F
    assert np.all(w[0, 1:] == 0)


@pytest.mark.parametrize("fmt", ["affine8_g64", "affine4_g64", "affine3_g64", "w4a16_g128",
                                 "affine2_g64", "affine5_g64", "affine6_g64"])
def test_pack_every_code_every_position_bitstream(fmt):
    """A single code v at column c lands at stream bits [b*c, b*c + b) as v
    (offset-binary for W4A16), for every v and every position of a 64/128 group."""
    bits = O.BITS[fmt]
    cols = O.GROUP[fmt] * 2
    lo = -8 if fmt == "w4a16_g128" else 0
    hi = 7 if fmt == "w4a16_g128" else (1 << bits) - 1
    zero = -8 if fmt == "w4a16_g128" else 0
    rows = []
    expect = []
    for c in range(cols):
        for v in range(lo, hi + 1):
            row = np.full(cols, zero, np.int32)
            row[c] = v
            rows.append(row)
            stored = v + 8 if fmt == "w4a16_g128" else v
            expect.append(stored << (bits * c))
    codes = np.stack(rows)
    words = O.pack(fmt, codes)
    for r in range(len(rows)):
        assert stream_int(words[r]) == expect[r]
    assert np.array_equal(O.unpack(fmt, words, cols), codes)


@pytest.mark.parametrize("fmt", ["affine8_g64", "affine4_g64", "affine3_g64", "w4a16_g128"])
def test_pack_random_rows_bitstream(fmt):
    rng = np.random.default_rng(11)
    cols = 256
    codes = synth.gen_codes(rng, fmt, 9, cols)
    words = O.pack(fmt, codes)
    bits = O.BITS[fmt]
    for r in range(codes.shape[0]):
        acc = 0
        for c in range(cols):
            v = int(codes[r, c]) + (8 if fmt == "w4a16_g128" else 0)
            acc |= v << (bits * c)
        assert stream_int(words[r]) == acc
    assert np.array_equal(O.unpack(fmt, words, cols), codes)


def test_pack_rejects_out_of_range():
    with pytest.raises(ValueError):
        O.pack("affine4_g64", np.full((1, 64), 16, np.int32))
    with pytest.raises(ValueError):
        O.pack("w4a16_g128", np.full((1, 128), 8, np.int32))
    with pytest.raises(ValueError):
        O.pack("affine3_g64", np.full((1, 64), 8, np.int32))


# --------------------------------------------------------------------------
# fp16 / bf16 decoding: all 65536 patterns against numpy's conversions

def test_fp16_decoder_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = O.fp16_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.array_equal(np.signbit(mine[~nan]), np.signbit(ref[~nan]))


def test_bf16_decoder_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = O.act_to_double("bf16", bits)
    with np.errstate(invalid="ignore"):
        ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


# --------------------------------------------------------------------------
# Dequantisation

def _np_dequant(fmt, codes, s_bits, b_bits):
    G = O.GROUP[fmt]
    s = np.repeat(s_bits.view(np.float16).astype(np.float64), G, axis=1)
    if fmt == "w4a16_g128":
        return s * codes
    b = np.repeat(b_bits.view(np.float16).astype(np.float64), G, axis=1)
    return s * codes + b


@pytest.mark.parametrize("fmt", ["affine8_g64", "affine4_g64", "affine3_g64", "w4a16_g128"])
def test_dequant_matches_definition(fmt):
    rng = np.random.default_rng(5)
    m = synth.gen_qmatrix(rng, fmt, 16, 256)
    words = O.pack(fmt, m.codes)
    got = O.dequant(fmt, words, m.scales, m.biases, 16, 256)
    assert np.array_equal(got, _np_dequant(fmt, m.codes, m.scales, m.biases))


def test_dequant_group_index():
    # every (row, group) gets its own power-of-two scale; a wrong group index
    # or a transposed scale table changes the result
    fmt = "affine4_g64"
    rows, cols = 4, 256
    codes = np.ones((rows, cols), np.int32)
    s = np.zeros((rows, cols // 64), np.float16)
    for r in range(rows):
        for g in range(cols // 64):
            s[r, g] = 2.0 ** -(r * 4 + g)
    b = np.zeros_like(s)
    got = O.dequant(fmt, O.pack(fmt, codes), s.view(np.uint16), b.view(np.uint16), rows, cols)
    for r in range(rows):
        for c in range(cols):
            assert got[r, c] == 2.0 ** -(r * 4 + c // 64)


def test_dequant_exact_rational_sweep():
    # w = s*q + b is exact in fp64 for fp16 s, b and 8-bit q: compare with Fractions,
    # including subnormal, zero, negative-zero and maximal fp16 values.
    special = np.array([0x0000, 0x8000, 0x0001, 0x03FF, 0x0400, 0x3C00, 0x7BFF, 0xFBFF,
                        0x8001, 0x1234, 0xB0F0], np.uint16)
    fmt = "affine8_g64"
    for sb in special:
        for bb in special:
            codes = np.arange(256, dtype=np.int32)[None, :].repeat(1, 0)
            codes = np.concatenate([codes, codes], axis=1)[:, :256]
            s = np.full((1, 4), sb, np.uint16)
            b = np.full((1, 4), bb, np.uint16)
            got = O.dequant(fmt, O.pack(fmt, codes), s, b, 1, 256)
            fs = Fraction(float(s.view(np.float16)[0, 0]))
            fb = Fraction(float(b.view(np.float16)[0, 0]))
            for c in range(256):
                assert Fraction(got[0, c]) == fs * int(codes[0, c]) + fb


def test_dequant_w4a16_symmetric():
    codes = np.arange(-8, 8, dtype=np.int32).repeat(8)[None, :]
    s = np.array([[0x3800]], np.uint16)  # 0.5
    got = O.dequant("w4a16_g128", O.pack("w4a16_g128", codes), s, None, 1, 128)
    assert np.array_equal(got[0], codes[0] * 0.5)


# --------------------------------------------------------------------------
# Top-k and weights

def _brute_topk(l, k):
    """The unique k-sequence that is ordered by (logit desc, id asc; NaN last)
    and ranks ahead of every unselected expert -- checked by enumeration."""
    E = len(l)

    def before(a, b):
        na, nb = math.isnan(l[a]), math.isnan(l[b])
        if na != nb:
            return nb
        if not na and l[a] != l[b]:
            return l[a] > l[b]
        return a < b

    found = []
    for seq in itertools.permutations(range(E), k):
        if not all(before(seq[i], seq[i + 1]) for i in range(k - 1)):
            continue
        rest = [e for e in range(E) if e not in seq]
        if all(before(seq[-1], r) for r in rest):
            found.append(seq)
    assert len(found) == 1
    return list(found[0])


def test_topk_brute_force_with_ties_and_nan():
    rng = np.random.default_rng(3)
    for trial in range(300):
        E = int(rng.integers(2, 7))
        k = int(rng.integers(1, E + 1))
        l = rng.integers(-2, 3, size=E).astype(np.float64)  # many ties
        if trial % 5 == 0:
            l[rng.integers(0, E)] = np.nan
        if trial % 7 == 0:
            l[rng.integers(0, E)] = -np.inf
        if trial % 11 == 0:
            l[:] = np.nan
        idx, _ = O.topk(l[None, :], k)
        assert list(idx[0]) == _brute_topk(list(l), k), (l, k)


def test_topk_flat_row_and_nan_row():
    idx, w = O.topk(np.zeros((1, 16)), 8)
    assert list(idx[0]) == list(range(8))
    assert np.allclose(w[0], 1 / 8, rtol=0, atol=1e-15)
    l = np.full((1, 16), np.nan)
    idx, _ = O.topk(l, 8)
    assert list(idx[0]) == list(range(8))
    l = np.zeros((1, 16))
    l[0, 5] = np.nan
    l[0, 9] = 1.0
    idx, _ = O.topk(l, 16)
    assert idx[0, 0] == 9 and idx[0, -1] == 5


def test_topk_tie_goes_to_lower_id():
    l = np.zeros((1, 8))
    l[0, [6, 2, 4]] = 3.0
    idx, w = O.topk(l, 2)
    assert list(idx[0]) == [2, 4]
    assert np.allclose(w[0], [0.5, 0.5], atol=1e-15)


def test_softmax_closed_forms():
    # logits ln3 and 0 over k=2 -> 3/4, 1/4; ln1..ln4 over k=4 -> i/10
    l = np.full((1, 6), -50.0)
    l[0, 1] = math.log(3.0)
    l[0, 4] = 0.0
    idx, w = O.topk(l, 2)
    assert list(idx[0]) == [1, 4]
    assert abs(w[0, 0] - 0.75) < 1e-15 and abs(w[0, 1] - 0.25) < 1e-15
    l = np.log(np.array([[1.0, 2.0, 3.0, 4.0, 0.5]]))
    idx, w = O.topk(l, 4)
    assert list(idx[0]) == [3, 2, 1, 0]
    assert np.allclose(w[0], [0.4, 0.3, 0.2, 0.1], rtol=0, atol=1e-15)


def test_weights_sum_to_one_and_descend():
    rng = np.random.default_rng(8)
    l = rng.normal(0, 1, size=(64, 256))
    idx, w = O.topk(l, 8)
    assert np.all(np.abs(w.sum(1) - 1.0) < 8 * 2.0 ** -52)
    assert np.all(np.diff(w, axis=1) <= 0)
    ref = np.argsort(-l, axis=1, kind="stable")[:, :8]
    assert np.array_equal(idx, ref)


# --------------------------------------------------------------------------
# Router, shared gate

@pytest.mark.parametrize("rfmt", ["f32", "bf16", "affine8_g64"])
def test_router_logits_are_matmul(rfmt):
    rng = np.random.default_rng(21)
    E, H, T = 16, 256, 5
    r = synth.gen_qmatrix(rng, rfmt, E, H)
    rd = _mat(r)
    x = O.act_to_double("bf16", synth.gen_x(rng, T, H))
    bias = synth.zipf_bias(rng, E)
    got = O.router_logits(rd, x, bias)
    W = _dense(r)
    ref = x @ W.T + bias.astype(np.float64)[None, :]
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-13)


def test_shared_gate_sigmoid():
    H = 128
    zero = {"fmt": "bf16", "q": np.zeros((1, H), np.uint16)}
    x = np.ones((3, H))
    logit, sg = O.shared_gate(zero, x)
    assert np.all(logit == 0) and np.all(sg == 0.5)
    rng = np.random.default_rng(2)
    g = synth.gen_qmatrix(rng, "affine8_g64", 1, H)
    x = O.act_to_double("bf16", synth.gen_x(rng, 4, H))
    logit, sg = O.shared_gate(_mat(g), x)
    ref = x @ _dense(g)[0]
    assert np.allclose(logit, ref, rtol=1e-13, atol=1e-14)
    assert np.allclose(sg, 1 / (1 + np.exp(-ref)), rtol=1e-14)


# --------------------------------------------------------------------------
# Experts and the layer

def _mat(m: synth.QMatrix) -> dict:
    if m.fmt in ("f32", "bf16", "f16"):
        return {"fmt": m.fmt, "q": m.values, "rows": m.rows, "cols": m.cols}
    return {"fmt": m.fmt, "q": O.pack(m.fmt, m.codes), "s": m.scales, "b": m.biases,
            "rows": m.rows, "cols": m.cols}


def _dense(m: synth.QMatrix) -> np.ndarray:
    """Dequantised matrix built with numpy alone (independent of the oracle)."""
    if m.fmt == "f32":
        return m.values.astype(np.float64)
    if m.fmt == "bf16":
        return (m.values.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return _np_dequant(m.fmt, m.codes, m.scales, m.biases)


def _bank(b: synth.ExpertBank) -> dict:
    w13 = np.stack([O.pack(b.fmt, m.codes) for m in b.w13])
    w2 = np.stack([O.pack(b.fmt, m.codes) for m in b.w2])
    d = {"fmt": b.fmt, "E": b.E, "I": b.I, "w13": w13, "w2": w2,
         "s13": np.stack([m.scales for m in b.w13]), "s2": np.stack([m.scales for m in b.w2])}
    if b.fmt != "w4a16_g128":
        d["b13"] = np.stack([m.biases for m in b.w13])
        d["b2"] = np.stack([m.biases for m in b.w2])
    return d


def _expert(bank: dict, e: int) -> dict:
    return {k: (v[e] if isinstance(v, np.ndarray) else v) for k, v in bank.items()}


def _np_swiglu(W13, W2, x):
    I = W13.shape[0] // 2
    ab = x @ W13.T
    a, b = ab[:, :I], ab[:, I:]
    h = a / (1 + np.exp(-a)) * b
    return h, h @ W2.T


@pytest.mark.parametrize("fmt", ["affine4_g64", "affine3_g64", "w4a16_g128", "affine8_g64"])
def test_expert_mlp_is_dense_swiglu(fmt):
    rng = np.random.default_rng(31)
    I, H, T = (128 if fmt == "w4a16_g128" else 64), 256, 3
    bank = synth.gen_bank(rng, fmt, 1, I, H)
    x = O.act_to_double("bf16", synth.gen_x(rng, T, H))
    h, y = O.expert_mlp(fmt, I, H, _expert(_bank(bank), 0), x)
    h_ref, y_ref = _np_swiglu(_dense(bank.w13[0]), _dense(bank.w2[0]), x)
    assert np.allclose(h, h_ref, rtol=1e-12, atol=1e-14)
    assert np.allclose(y, y_ref, rtol=1e-12, atol=1e-14)
    # the gate rows come first: swapping gate and up changes the result
    W13 = _dense(bank.w13[0])
    swapped = np.concatenate([W13[I:], W13[:I]])
    _, y_bad = _np_swiglu(swapped, _dense(bank.w2[0]), x)
    assert not np.allclose(y, y_bad, rtol=1e-3)
    y2 = O.down(fmt, H, I, O.pack(fmt, bank.w2[0].codes), bank.w2[0].scales,
                bank.w2[0].biases, h_ref)
    assert np.allclose(y2, y_ref, rtol=1e-12, atol=1e-14)


def _layer(L: synth.LayerInputs, **kw):
    x = O.act_to_double(L.act, L.x)
    return O.moe_layer(x, L.k, _mat(L.router), _bank(L.experts),
                       _expert(_bank(L.shared), 0) if L.shared else None,
                       _mat(L.gate) if L.gate else None, L.logit_bias, **kw)


def test_layer_one_expert_equals_dense_mlp():
    L = synth.gen_layer(T=4, E=1, k=1, H=256, I=64, expert_fmt="affine4_g64", seed=9)
    out = _layer(L)["out"]
    x = O.act_to_double("bf16", L.x)
    _, y = _np_swiglu(_dense(L.experts.w13[0]), _dense(L.experts.w2[0]), x)
    assert np.allclose(out, y, rtol=1e-12, atol=1e-14)


def test_layer_identical_experts_and_shared_slot():
    # all E experts are the same MLP M, so sum_k w_k M(x) = M(x) when the
    # weights sum to one; the shared expert adds sigmoid(g . x) * S(x)
    L = synth.gen_layer(T=5, E=12, k=4, H=256, I=64, expert_fmt="affine4_g64",
                        shared_fmt="affine4_g64", gate_fmt="affine8_g64", seed=10)
    for e in range(1, L.E):
        L.experts.w13[e] = L.experts.w13[0]
        L.experts.w2[e] = L.experts.w2[0]
    out = _layer(L)["out"]
    x = O.act_to_double("bf16", L.x)
    _, M = _np_swiglu(_dense(L.experts.w13[0]), _dense(L.experts.w2[0]), x)
    _, S = _np_swiglu(_dense(L.shared.w13[0]), _dense(L.shared.w2[0]), x)
    g = x @ _dense(L.gate)[0]
    ref = M + (1 / (1 + np.exp(-g)))[:, None] * S
    assert np.allclose(out, ref, rtol=1e-11, atol=1e-13)


def test_layer_weights_in_slot_order_closed_form():
    # router rows designed so logits are exactly [0, ln3] on experts 0 and 1
    # (one-hot x); expert 0 is all-zero, expert 1 is an MLP M:
    # out = 3/4 * M(x) exactly up to the fp32 rounding of ln3.
    rng = np.random.default_rng(12)
    H, I, E = 128, 64, 4
    L = synth.gen_layer(T=1, E=E, k=2, H=H, I=I, expert_fmt="affine4_g64", seed=12)
    x_bits = np.zeros((1, H), np.uint16)
    x_bits[0, 0] = 0x3F80  # 1.0 in bf16
    L.x = x_bits
    W = np.zeros((E, H), np.float32)
    W[:, 0] = [0.0, math.log(3.0), -30.0, -40.0]
    L.router = synth.QMatrix("f32", E, H, values=W)
    z = L.experts.w13[0]
    L.experts.w13[0] = synth.QMatrix(z.fmt, z.rows, z.cols, codes=np.zeros_like(z.codes),
                                     scales=np.zeros_like(z.scales), biases=np.zeros_like(z.biases))
    r = _layer(L)
    x = O.act_to_double("bf16", L.x)
    _, M = _np_swiglu(_dense(L.experts.w13[1]), _dense(L.experts.w2[1]), x)
    l1 = float(np.float32(math.log(3.0)))
    w1 = math.exp(l1) / (math.exp(l1) + 1.0)
    assert list(r["idx"][0]) == [1, 0]
    assert np.allclose(r["out"], w1 * M, rtol=1e-12, atol=1e-15)


def test_layer_zero_input_gives_zero():
    L = synth.gen_layer(T=3, E=8, k=2, H=128, I=64, expert_fmt="affine4_g64",
                        shared_fmt="affine4_g64", gate_fmt="affine8_g64", seed=13)
    L.x = np.zeros_like(L.x)
    assert np.all(_layer(L)["out"] == 0.0)


def test_layer_3bit_codes_widened_to_4bit_equal():
    # the same 3-bit codes stored as 4-bit words, same scales/biases, give the
    # same layer output
    L3 = synth.gen_layer(T=4, E=8, k=3, H=256, I=128, expert_fmt="affine3_g64", seed=14)
    out3 = _layer(L3)["out"]
    bank4 = synth.ExpertBank("affine4_g64", L3.E, L3.I, L3.H)
    for m in L3.experts.w13:
        bank4.w13.append(synth.QMatrix("affine4_g64", m.rows, m.cols, codes=m.codes,
                                       scales=m.scales, biases=m.biases))
    for m in L3.experts.w2:
        bank4.w2.append(synth.QMatrix("affine4_g64", m.rows, m.cols, codes=m.codes,
                                      scales=m.scales, biases=m.biases))
    L3.experts = bank4
    out4 = _layer(L3)["out"]
    assert np.array_equal(out3, out4)


def test_layer_token_permutation_equivariant():
    L = synth.gen_layer(T=6, E=16, k=4, H=128, I=64, expert_fmt="affine4_g64",
                        shared_fmt="affine4_g64", gate_fmt="affine8_g64", zipf=True, seed=15)
    out = _layer(L)["out"]
    p = np.array([3, 0, 5, 1, 4, 2])
    L.x = L.x[p]
    out_p = _layer(L)["out"]
    assert np.array_equal(out_p, out[p])


def test_layer_idx_override_reproduces_own_routing():
    L = synth.gen_layer(T=4, E=16, k=4, H=128, I=64, expert_fmt="affine4_g64", seed=16)
    r = _layer(L)
    r2 = _layer(L, idx_override=r["idx"])
    assert np.array_equal(r["out"], r2["out"])


# --------------------------------------------------------------------------
# Bucketing

def test_bucket_invariants():
    rng = np.random.default_rng(17)
    for T, k, E in [(1, 8, 256), (8, 8, 256), (33, 4, 16), (512, 8, 256), (0, 8, 16)]:
        idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]) \
            if T else np.zeros((0, k), np.int32)
        counts, offsets, perm, active = O.bucket(idx, E)
        flat = idx.reshape(-1)
        assert np.array_equal(np.sort(perm), np.arange(T * k))
        assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
        assert np.array_equal(counts, np.bincount(flat, minlength=E))
        for e in range(E):
            seg = perm[offsets[e]:offsets[e + 1]]
            assert np.all(flat[seg] == e)
            assert np.all(np.diff(seg) > 0)
        assert np.array_equal(active, np.unique(flat))


# --------------------------------------------------------------------------
# The engine's own precision: bf16 rounding and the fp32 combine
# ("Progress on the 4-bit gate": the slots' fma sum rounded once to bf16; the
# routing's bf16 rounding chain)

def test_round_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.standard_normal(4096).astype(np.float32) * np.float32(1e3),
        np.array([0.0, -0.0, np.inf, -np.inf, 1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8,
                  -(1 + 2 ** -8), 2 ** -126, 2 ** -133, 3.3895e38, 65504.0], np.float32)])
    ours = O.round_bf16(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))
    # ties go to the even neighbour
    assert O.round_bf16(np.array([1 + 2 ** -8], np.float32))[0] == 1.0
    assert O.round_bf16(np.array([1 + 3 * 2 ** -8], np.float32))[0] == 1 + 2 ** -6
    # NaN stays NaN
    assert np.isnan(O.round_bf16(np.array([np.nan], np.float32))[0])


def bf16_bits(x: float) -> int:
    return int(np.array([x], np.float32).view(np.uint32)[0] >> 16)


def test_combine_f32_single_slot_is_rounding():
    y = np.array([[1.0, 1 + 2 ** -8, -3.25, 1e-3]], np.float32)
    out = O.combine_f32(y, np.array([[1.0]], np.float32))
    expect = O.round_bf16(y[0]).view(np.uint32) >> 16
    assert np.array_equal(out[0].astype(np.uint32), expect)


def test_combine_f32_uses_fused_multiply_add():
    # w1*y1 = 1 + 2^-11 + 2^-24 exactly; a rounded product loses the 2^-24,
    # which the fused multiply-add keeps after the first slot cancels 1 + 2^-11
    a = 1 + 2 ** -12
    y = np.array([[-(1 + 2 ** -11)], [a]], np.float32)
    w = np.array([[1.0, a]], np.float32)
    out = O.combine_f32(y, w)
    assert int(out[0, 0]) == bf16_bits(2 ** -24)


def test_combine_f32_slot_order_and_shared_last():
    # fp32 sums do not associate: (1e8 + 1) - 1e8 = 0 in slot order, while
    # 1e8 - 1e8 + 1 would give 1
    y = np.array([[1e8], [1.0], [-1e8]], np.float32)
    out = O.combine_f32(y, np.ones((1, 3), np.float32))
    assert int(out[0, 0]) == bf16_bits(0.0)
    # the shared slot comes after every routed slot: (1e8 - 1e8) + 1 = 1
    y2 = np.array([[1e8], [-1e8]], np.float32)
    out = O.combine_f32(y2, np.ones((1, 2), np.float32), ysh=np.array([[1.0]], np.float32),
                        sg=np.array([1.0], np.float32))
    assert int(out[0, 0]) == bf16_bits(1.0)
    # without sg the shared slot has weight 1
    out = O.combine_f32(y2, np.ones((1, 2), np.float32), ysh=np.array([[1.0]], np.float32))
    assert int(out[0, 0]) == bf16_bits(1.0)


def test_combine_f32_agrees_with_fp64_layer_combine():
    # on random data the fp32 chain is the fp64 sum to within the bf16 step
    rng = np.random.default_rng(11)
    T, k, H = 3, 8, 64
    y = rng.standard_normal((T * k, H)).astype(np.float32)
    w = rng.dirichlet(np.ones(k), size=T).astype(np.float32)
    ysh = rng.standard_normal((T, H)).astype(np.float32)
    sg = rng.uniform(0, 1, T).astype(np.float32)
    out = O.combine_f32(y, w, ysh, sg).astype(np.uint32) << 16
    got = out.view(np.float32)
    ref = np.einsum("tk,tkh->th", w.astype(np.float64), y.reshape(T, k, H).astype(np.float64))
    ref += sg[:, None].astype(np.float64) * ysh
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2 ** -8 + 1e-6)


def test_chain_gate_weight_closed_forms():
    s = O.chain_gate_weight(np.array([0.0, 40.0, -40.0, 1.0], np.float32))
    assert s[0] == 0.5
    assert s[1] == 1.0
    assert 0.0 <= s[2] < 2 ** -50
    # sigmoid(1) = 0.7310585786... -> bf16 0.73046875 (0x3F3B)
    assert int(np.array([s[3]], np.float32).view(np.uint32)[0] >> 16) == 0x3F3B



# --------------------------------------------------------------------------
# The layer under the engine's bf16 rounding chain (round_bf16=True): router
# and gate rows rounded to bf16, slot weights bf16(w), shared weight
# bf16(sigmoid(bf16(g))).  Values below are worked by hand from the bf16
# encoding (8 significant bits, round to nearest even).

def _is_bf16(v) -> bool:
    f = np.asarray(v, np.float64).astype(np.float32)
    return bool(np.all(f.astype(np.float64) == np.asarray(v, np.float64))
                and np.all((f.view(np.uint32) & 0xFFFF) == 0))


def test_layer_round_bf16_closed_form():
    # the slot-order case above under the chain: the router entry ln 3
    # (fp32 0x3F8C9F54) is stored as bf16 0x3F8D = 1 + 13/128, so the
    # weights are sigmoid(+-141/128) = 0.750554.. and 0.249446.., which round
    # to 0.75 (0x3F40) and 255/1024 (0x3E7F); expert 0 is zero, so
    # out = 0.75 * M(x) exactly
    H, I, E = 128, 64, 4
    L = synth.gen_layer(T=1, E=E, k=2, H=H, I=I, expert_fmt="affine4_g64", seed=12)
    x_bits = np.zeros((1, H), np.uint16)
    x_bits[0, 0] = 0x3F80
    L.x = x_bits
    W = np.zeros((E, H), np.float32)
    W[:, 0] = [0.0, math.log(3.0), -30.0, -40.0]
    L.router = synth.QMatrix("f32", E, H, values=W)
    z = L.experts.w13[0]
    L.experts.w13[0] = synth.QMatrix(z.fmt, z.rows, z.cols, codes=np.zeros_like(z.codes),
                                     scales=np.zeros_like(z.scales), biases=np.zeros_like(z.biases))
    r = _layer(L, round_bf16=True)
    assert list(r["idx"][0]) == [1, 0]
    assert r["logits"][0, 1] == 1 + 13 / 128
    assert list(r["w"][0]) == [0.75, 255 / 1024]
    x = O.act_to_double("bf16", L.x)
    _, M = _np_swiglu(_dense(L.experts.w13[1]), _dense(L.experts.w2[1]), x)
    assert np.allclose(r["out"], 0.75 * M, rtol=1e-12, atol=1e-15)
    # without the chain slot 1 keeps 1 / (exp(l1) + 1) ~ 1/4, l1 = fp32(ln 3):
    # the 255/1024 above comes from the router row's rounding
    r0 = _layer(L)
    assert abs(r0["w"][0, 1] - 0.25) < 1e-8


def test_layer_round_bf16_flat_row_thirds():
    # a zero router gives a flat row: ids 0..k-1 and weights 1/3, stored as
    # bf16 0x3EAB = 171/512 (1/3 = fp32 0x3EAAAAAB rounds up)
    L = synth.gen_layer(T=3, E=6, k=3, H=128, I=64, expert_fmt="affine4_g64", seed=21)
    L.router = synth.QMatrix("f32", 6, 128, values=np.zeros((6, 128), np.float32))
    r = _layer(L, round_bf16=True)
    assert np.all(r["idx"] == np.array([0, 1, 2], np.int32))
    assert np.all(r["w"] == 171 / 512)
    assert np.all(_layer(L)["w"] == 1 / 3)


def test_layer_round_bf16_gate_closed_forms():
    # gate row (1, 3 * 2^-9, 0, ...) in bf16: s_t = bf16(sigmoid(bf16(g_t)));
    # x = 0 -> g = 0 -> 1/2; x = e_0 -> g = 1 -> sigmoid 0.73106.. -> 187/256;
    # x = e_0 + e_1 -> g = 1 + 3 * 2^-9, which bf16 holds only as 1 + 2^-7
    # (0.75 ulp rounds up), sigmoid 0.73259.. -> 188/256 (rounding after the
    # sigmoid alone would give sigmoid(g) = 0.73220.. -> 187/256)
    H = 128
    L = synth.gen_layer(T=3, E=4, k=2, H=H, I=64, expert_fmt="affine4_g64",
                        shared_fmt="affine4_g64", gate_fmt="bf16", seed=22)
    g_row = np.zeros((1, H), np.uint16)
    g_row[0, :2] = [0x3F80, 0x3BC0]
    L.gate = synth.QMatrix("bf16", 1, H, values=g_row)
    x_bits = np.zeros((3, H), np.uint16)
    x_bits[1, 0] = 0x3F80
    x_bits[2, :2] = 0x3F80
    L.x = x_bits
    r = _layer(L, round_bf16=True)
    assert list(r["sg"]) == [0.5, 187 / 256, 188 / 256]
    r0 = _layer(L)
    assert r0["sg"][0] == 0.5
    assert abs(r0["sg"][1] - 1 / (1 + math.exp(-1.0))) < 1e-15


def test_layer_round_bf16_gate_row_rounded():
    # gate row (1 + 2^-8 + 2^-10, -1, 0, ...) in fp32 and x = (8, 8, 0, ...):
    # the chain stores the first entry as bf16 1 + 2^-7 (0.625 ulp rounds up),
    # so g = 8 * 2^-7 = 1/16 and s = bf16(sigmoid(1/16)) = bf16(0.515620..)
    # = 132/256; the exact row gives g = 2^-5 + 2^-7 and s = sigmoid(g)
    H = 128
    L = synth.gen_layer(T=1, E=4, k=2, H=H, I=64, expert_fmt="affine4_g64",
                        shared_fmt="affine4_g64", gate_fmt="f32", seed=23)
    g_row = np.zeros((1, H), np.float32)
    g_row[0, :2] = [1 + 2 ** -8 + 2 ** -10, -1.0]
    L.gate = synth.QMatrix("f32", 1, H, values=g_row)
    x_bits = np.zeros((1, H), np.uint16)
    x_bits[0, :2] = 0x4100  # 8.0
    L.x = x_bits
    assert _layer(L, round_bf16=True)["sg"][0] == 132 / 256
    assert abs(_layer(L)["sg"][0] - 1 / (1 + math.exp(-(2 ** -5 + 2 ** -7)))) < 1e-15


def test_layer_round_bf16_weights_are_bf16_and_used_in_out():
    L = synth.gen_layer(T=6, E=16, k=4, H=256, I=64, expert_fmt="affine4_g64",
                        shared_fmt="affine4_g64", gate_fmt="affine8_g64", seed=24)
    r = _layer(L, round_bf16=True, want_slots=True)
    assert _is_bf16(r["w"]) and _is_bf16(r["sg"])
    # the chain moves each weight by at most half a bf16 ulp of the exact one
    # when the picks agree (the router rows differ by their own rounding)
    r0 = _layer(L)
    if np.array_equal(r["idx"], r0["idx"]):
        assert np.all(np.abs(r["w"] - r0["w"]) <= 2 ** -8 * r0["w"] + 2 ** -8 * 0.02)
    ref = np.einsum("tk,tkh->th", r["w"], r["y_slots"]) + r["sg"][:, None] * r["y_shared"]
    assert np.allclose(r["out"], ref, rtol=1e-12, atol=1e-14)


def test_layer_round_bf16_is_identity_on_bf16_exact_routing():
    # a zero router (flat row, k = 8: weights 1/8) and a zero gate row
    # (weight 1/2) are bf16 values already: the chain changes nothing
    L = synth.gen_layer(T=2, E=8, k=8, H=128, I=64, expert_fmt="affine4_g64",
                        shared_fmt="affine4_g64", gate_fmt="affine8_g64", seed=25)
    L.router = synth.QMatrix("bf16", 8, 128, values=np.zeros((8, 128), np.uint16))
    L.gate = synth.QMatrix("bf16", 1, 128, values=np.zeros((1, 128), np.uint16))
    a, b = _layer(L, round_bf16=True), _layer(L)
    assert np.all(a["w"] == 0.125) and np.all(a["sg"] == 0.5)
    assert np.array_equal(a["out"], b["out"])


# --------------------------------------------------------------------------
# MLX affine at the other widths the pages' loader reads (2/5/6-bit; oracle
# only for now): one LSB-first bit stream per row, as for 3-bit

WIDE = ["affine2_g64", "affine5_g64", "affine6_g64"]


@pytest.mark.parametrize("fmt", WIDE)
def test_pack_random_rows_bitstream_other_widths(fmt):
    rng = np.random.default_rng(21)
    bits, cols = O.BITS[fmt], 192
    codes = rng.integers(0, 1 << bits, size=(7, cols), dtype=np.int32)
    words = O.pack(fmt, codes)
    assert words.shape == (7, cols * bits // 32)
    for r in range(codes.shape[0]):
        acc = 0
        for c in range(cols):
            acc |= int(codes[r, c]) << (bits * c)
        assert stream_int(words[r]) == acc
    assert np.array_equal(O.unpack(fmt, words, cols), codes)
    with pytest.raises(ValueError):
        O.pack(fmt, np.full((1, 64), 1 << bits, np.int32))


@pytest.mark.parametrize("fmt", WIDE)
def test_dequant_other_widths_exact(fmt):
    rng = np.random.default_rng(22)
    bits, rows, cols = O.BITS[fmt], 6, 256
    codes = rng.integers(0, 1 << bits, size=(rows, cols), dtype=np.int32)
    s = (np.abs(rng.standard_normal((rows, cols // 64))) * 0.01).astype(np.float16)
    b = (rng.standard_normal((rows, cols // 64)) * 0.1).astype(np.float16)
    got = O.dequant(fmt, O.pack(fmt, codes), s.view(np.uint16), b.view(np.uint16), rows, cols)
    for r in range(rows):
        for c in range(0, cols, 37):
            want = Fraction(float(s[r, c // 64])) * codes[r, c] + Fraction(float(b[r, c // 64]))
            assert Fraction(got[r, c]) == want


def test_same_codes_at_every_width_dequantise_equally():
    # codes 0..3 stored at every width from 2 to 8 bits decode to the same
    # weights (the widening control, across all widths)
    rng = np.random.default_rng(23)
    rows, cols = 3, 128
    codes = rng.integers(0, 4, size=(rows, cols), dtype=np.int32)
    s = (np.abs(rng.standard_normal((rows, cols // 64))) * 0.01).astype(np.float16).view(np.uint16)
    b = (rng.standard_normal((rows, cols // 64)) * 0.1).astype(np.float16).view(np.uint16)
    ref = O.dequant("affine2_g64", O.pack("affine2_g64", codes), s, b, rows, cols)
    for fmt in ["affine3_g64", "affine4_g64", "affine5_g64", "affine6_g64", "affine8_g64"]:
        got = O.dequant(fmt, O.pack(fmt, codes), s, b, rows, cols)
        assert np.array_equal(got, ref), fmt


def test_layer_codes_widened_across_widths_equal():
    # the same 2-bit codes as 2-, 5- and 6-bit experts give the same layer output
    L = synth.gen_layer(T=3, E=6, k=2, H=128, I=64, expert_fmt="affine3_g64", seed=24)
    outs = []
    for fmt in ["affine2_g64", "affine5_g64", "affine6_g64"]:
        bank = synth.ExpertBank(fmt, L.E, L.I, L.H)
        for src, dst in ((L.experts.w13, bank.w13), (L.experts.w2, bank.w2)):
            for m in src:
                dst.append(synth.QMatrix(fmt, m.rows, m.cols, codes=m.codes & 3,
                                         scales=m.scales, biases=m.biases))
        L2 = synth.LayerInputs(**{**L.__dict__, "experts": bank})
        outs.append(_layer(L2)["out"])
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
