"""The seeded input generators against the stated input recipe (no GPU): value
laws of activations, router, codes, scales and biases, the Zipf routing bias,
and the device-side generators (run here on the CPU device) following the
same laws.  Statistical checks use sample sizes that put the bounds many
standard errors away from the expected values."""
import math

import numpy as np
import pytest
import torch

from bit_affine_quantized_fp32_gb300 import synth

HALF_NORMAL_MEAN = math.sqrt(2.0 / math.pi)  # E|N(0, 1)|


def _f16(bits):
    return np.asarray(bits).view(np.float16).astype(np.float64)


def test_activations_rms_normalised_per_row():
    rng = np.random.default_rng(0)
    x = synth.gen_x(rng, 64, 2048, "bf16")
    v = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    rms = np.sqrt(np.mean(v * v, axis=1))
    assert np.all(np.abs(rms - 1.0) < 2.0 ** -8)  # bf16 rounding only
    assert abs(v.mean()) < 0.01
    xf = _f16(synth.gen_x(rng, 16, 2048, "f16"))
    assert np.all(np.abs(np.sqrt(np.mean(xf * xf, axis=1)) - 1.0) < 2.0 ** -10)


def test_router_rows_normal_002():
    rng = np.random.default_rng(1)
    m = synth.gen_qmatrix(rng, "f32", 256, 2048)
    assert m.values.dtype == np.float32
    assert abs(float(m.values.std()) - 0.02) < 2e-4
    assert abs(float(m.values.mean())) < 1e-4


@pytest.mark.parametrize("fmt,bits,G,sigma,mid,noise", [
    ("affine4_g64", 4, 64, 0.004, 8, 1e-4),
    ("affine3_g64", 3, 64, 0.008, 4, 0.0),
    ("affine8_g64", 8, 64, 2.7e-4, 128, 1e-4),
])
def test_affine_matrix_laws(fmt, bits, G, sigma, mid, noise):
    rng = np.random.default_rng(2)
    m = synth.gen_qmatrix(rng, fmt, 512, 2048)
    c = m.codes.astype(np.int64)
    assert c.min() == 0 and c.max() == (1 << bits) - 1
    freq = np.bincount(c.ravel(), minlength=1 << bits) / c.size
    # each bin within 6 standard errors of uniform
    assert np.all(np.abs(freq * (1 << bits) - 1.0) < 6 * math.sqrt((1 << bits) / c.size))
    s, b = _f16(m.scales), _f16(m.biases)
    assert m.scales.shape == (512, 2048 // G)
    assert np.all(s >= 0)
    assert abs(s.mean() / (sigma * HALF_NORMAL_MEAN) - 1.0) < 0.02
    resid = b + mid * s
    if noise == 0.0:
        assert np.all(resid == 0.0)  # bias = -mid * scale exactly (a power of two)
    else:
        assert abs(resid.std() / noise - 1.0) < 0.05


def test_w4a16_laws():
    rng = np.random.default_rng(3)
    m = synth.gen_qmatrix(rng, "w4a16_g128", 512, 2048)
    c = m.codes.astype(np.int64)
    assert c.min() == -8 and c.max() == 7
    assert m.biases is None
    assert m.scales.shape == (512, 16)
    assert abs(_f16(m.scales).mean() / (0.004 * HALF_NORMAL_MEAN) - 1.0) < 0.03


def test_zipf_bias_is_minus_alpha_log_rank():
    rng = np.random.default_rng(4)
    b = synth.zipf_bias(rng, 256, 1.1)
    expect = (-1.1 * np.log(np.arange(1, 257, dtype=np.float64))).astype(np.float32)
    assert np.array_equal(np.sort(b)[::-1], expect)
    assert len(set(np.argsort(b).tolist())) == 256


def test_gen_layer_is_seeded():
    a = synth.gen_layer(T=3, E=4, k=2, H=128, I=64, shared_fmt="affine4_g64",
                        gate_fmt="affine8_g64", zipf=True, seed=11)
    b = synth.gen_layer(T=3, E=4, k=2, H=128, I=64, shared_fmt="affine4_g64",
                        gate_fmt="affine8_g64", zipf=True, seed=11)
    c = synth.gen_layer(T=3, E=4, k=2, H=128, I=64, shared_fmt="affine4_g64",
                        gate_fmt="affine8_g64", zipf=True, seed=12)
    assert np.array_equal(a.x, b.x) and np.array_equal(a.experts.w13[3].codes,
                                                       b.experts.w13[3].codes)
    assert not np.array_equal(a.x, c.x)


def test_device_generators_follow_the_same_laws():
    # run on the CPU device: packed words are uniform random bits (uniform
    # codes packed densely), scales and biases follow the numpy laws
    d = synth.device_bank("affine4_g64", 4, 128, 512, seed=5, device="cpu")
    w = d["w13"].numpy().view(np.uint32).ravel()
    bits = np.unpackbits(w.view(np.uint8))
    assert abs(bits.mean() - 0.5) < 0.005
    nib = np.concatenate([(w >> (4 * j)) & 15 for j in range(8)])
    freq = np.bincount(nib.astype(np.int64), minlength=16) / nib.size
    assert np.all(np.abs(freq * 16 - 1.0) < 0.03)
    s = d["s13"].float().numpy().astype(np.float64)
    b = d["b13"].float().numpy().astype(np.float64)
    assert abs(s.mean() / (0.004 * HALF_NORMAL_MEAN) - 1.0) < 0.03
    assert abs((b + 8 * s).std() / 1e-4 - 1.0) < 0.06
    assert d["w13"].shape == (4, 256, 512 * 4 // 32)
    assert d["w2"].shape == (4, 512, 128 * 4 // 32)
    x = synth.device_x(8, 2048, "bf16", seed=6, device="cpu").float().numpy()
    assert np.all(np.abs(np.sqrt(np.mean(x.astype(np.float64) ** 2, axis=1)) - 1.0) < 2.0 ** -8)
    r = synth.device_matrix("f32", 256, 2048, seed=7, device="cpu")["q"].numpy()
    assert abs(float(r.std()) - 0.02) < 2e-4
    g = synth.device_matrix("affine8_g64", 1, 2048, seed=8, device="cpu")
    assert g["q"].dtype == torch.int32 and g["s"].dtype == torch.float16
