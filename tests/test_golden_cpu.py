"""Pins of the oracle's storage formats against weight totals the pages print
(``tests/golden/model_storage.txt``, each figure with its page and section).

The pages print no worked example of a packed word or of a layer output.
They do print the stored size of two checkpoints of this layer's family.  The
bytes of one expert matrix are taken from the oracle itself: the words its
packer writes per row, plus the scale and bias words of each group (one
16-bit scale and one 16-bit bias per MLX affine group of 64, one fp16 scale
per W4A16 group of 128).  The routed experts of every layer are then counted
at the checkpoint's stated width.  They must fit inside the printed total and
make up most of it, since routed experts hold over 90 % of a 35B-A3B's
parameters.

The check catches three mistakes:
  * a wrong code width: 4-bit codes stored for the 3-bit experts come to
    18.1 GB, more than 15;
  * scales and biases left out of the storage: 12.2 GB, too little of 15;
  * an expert width other than 512: 768 gives 21 GB.  The pages do not print
    the width, so these totals are the pages' only check on it.

"GB" is read generously: anything up to the printed figure plus a half,
in GiB.
"""

from pathlib import Path

import numpy as np
import pytest

from oracle import oracle as O

GOLDEN = Path(__file__).resolve().parent / "golden" / "model_storage.txt"
I_EXPERT = 512  # expert intermediate width of the layer under test


def golden() -> dict:
    vals = {}
    for line in GOLDEN.read_text().splitlines():
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = int(v)
    return vals


def matrix_bytes(fmt: str, rows: int, cols: int) -> int:
    """Stored bytes of a rows x cols matrix in `fmt`, from the oracle's packer
    (words per row) and the format's group words (checked against the
    oracle's dequantisation in test_oracle_pins)."""
    words = O.pack(fmt, np.zeros((1, cols), np.int32)).nbytes
    if fmt == "w4a16_g128":
        group_words = (cols // 128) * 2          # fp16 scale
    else:
        group_words = (cols // 64) * (2 + 2)     # bf16 scale + bf16 bias
    return rows * (words + group_words)


def expert_bytes(fmt: str, H: int, I: int) -> int:
    return matrix_bytes(fmt, 2 * I, H) + matrix_bytes(fmt, H, I)


def bounds(gb: int):
    return 0.85 * gb * 1e9, (gb + 0.5) * 2**30


def test_golden_file_is_complete():
    g = golden()
    assert set(g) == {"layers", "experts", "top_k", "hidden", "mlx_3bit_experts_total_gb",
                      "w4a16_shards_gb"}


def test_mlx_mix_fits_the_printed_total():
    g = golden()
    L, E, H = g["layers"], g["experts"], g["hidden"]
    routed = L * E * expert_bytes("affine3_g64", H, I_EXPERT)
    rest = L * (expert_bytes("affine4_g64", H, I_EXPERT)       # shared expert
                + matrix_bytes("affine8_g64", E, H)             # router
                + matrix_bytes("affine8_g64", 1, H))            # shared-expert gate
    lo, hi = bounds(g["mlx_3bit_experts_total_gb"])
    assert lo <= routed and routed + rest <= hi, (routed, rest, lo, hi)


def test_w4a16_experts_fit_the_printed_shards():
    g = golden()
    routed = g["layers"] * g["experts"] * expert_bytes("w4a16_g128", g["hidden"], I_EXPERT)
    lo, hi = (0.7 * g["w4a16_shards_gb"] * 1e9, (g["w4a16_shards_gb"] + 0.5) * 2**30)
    assert lo <= routed <= hi, (routed, lo, hi)


@pytest.mark.parametrize("mistake", ["4-bit codes", "no group words", "width 768"])
def test_the_pin_rejects_plausible_mistakes(mistake):
    """Each mistake, planted in the byte count on the CPU, leaves the 15 GB
    bounds."""
    g = golden()
    L, E, H = g["layers"], g["experts"], g["hidden"]
    if mistake == "4-bit codes":
        routed = L * E * expert_bytes("affine4_g64", H, I_EXPERT)
    elif mistake == "no group words":
        n = 3 * H * I_EXPERT
        routed = L * E * (O.pack("affine3_g64", np.zeros((1, n), np.int32)).nbytes)
    else:
        routed = L * E * expert_bytes("affine3_g64", H, 768)
    lo, hi = bounds(g["mlx_3bit_experts_total_gb"])
    assert not (lo <= routed <= hi), (mistake, routed, lo, hi)
