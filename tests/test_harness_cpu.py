"""The parity tolerance itself (no GPU): the layer's output is rounded once to
its activation type, and the check allows exactly that rounding on top of the
stated bound."""
import numpy as np
import pytest
import torch

from tests import _harness as Hn


def _round(v: np.ndarray, out_type: str) -> np.ndarray:
    dt = torch.bfloat16 if out_type == "bf16" else torch.float16
    return torch.from_numpy(np.asarray(v, np.float64)).to(dt).double().numpy()


def test_half_ulp_values():
    r = Hn.output_rounding(np.array([1.0, 0.75, 1.5, 2.0, 0.001]), 0.0, "bf16")
    assert list(r) == [2.0 ** -8, 2.0 ** -9, 2.0 ** -8, 2.0 ** -7, 2.0 ** -18]
    r = Hn.output_rounding(np.array([1.0, 0.75, 1e-7]), 0.0, "f16")
    assert list(r) == [2.0 ** -11, 2.0 ** -12, 2.0 ** -25]
    assert Hn.output_rounding(np.array([1.0]), 0.0, None) == 0.0
    # a value just below a power of two is judged in the binade above it
    assert Hn.output_rounding(np.array([1.0 - 1e-6]), 1e-3, "bf16")[0] == 2.0 ** -8


def test_exact_sum_rounded_to_bf16_needs_the_allowance():
    # rms ~ 0.13 (tol 2.3e-3) and one output of 1 + 2^-8, which bf16 rounds
    # to 1 (ties to even): the correctly rounded result misses the bare bound
    rng = np.random.default_rng(0)
    ref = rng.normal(0.0, 0.13, 4096)
    ref[7] = 1.0 + 2.0 ** -8
    got = _round(ref, "bf16")
    assert got[7] == 1.0
    with pytest.raises(AssertionError):
        Hn.assert_layer_close(got, ref)
    Hn.assert_layer_close(got, ref, out_type="bf16")


@pytest.mark.parametrize("out_type", ["bf16", "f16"])
def test_rounded_results_pass_and_real_errors_fail(out_type):
    rng = np.random.default_rng(1)
    ref = rng.normal(0.0, 1.0, 20000) * np.exp(rng.normal(0.0, 1.5, 20000))
    rms = float(np.sqrt(np.mean(ref * ref)))
    tol = Hn.RTOL_RMS * rms + Hn.ATOL
    # any arithmetic error inside the bound, then the output rounding
    noisy = ref + rng.uniform(-0.99, 0.99, ref.size) * tol
    Hn.assert_layer_close(_round(noisy, out_type), ref, out_type=out_type)
    # one element off by more than the bound plus a whole ulp fails
    bad = _round(noisy, out_type)
    bad[123] = ref[123] + tol + 2.5 * Hn.output_rounding(ref[123:124], tol, out_type)[0]
    with pytest.raises(AssertionError):
        Hn.assert_layer_close(bad, ref, out_type=out_type)
    # fp32 results get no allowance
    with pytest.raises(AssertionError):
        Hn.assert_layer_close(ref + 1.01 * tol, ref)
