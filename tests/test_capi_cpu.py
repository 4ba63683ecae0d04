"""Host-side checks of the C-ABI library (no GPU needed): it builds for
sm_103a, loads, exports every function include/moe_gb300.h declares, and
refuses bad arguments by name before touching the device."""

import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def capi():
    from bit_affine_quantized_fp32_gb300 import build
    build.build()
    from bit_affine_quantized_fp32_gb300 import capi as C
    return C


def declared_functions():
    text = (ROOT / "include" / "moe_gb300.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ["moe_route", "moe_experts_forward", "moe_shared_expert", "moe_pack_affine4_g64",
                 "moe_unpack_affine3_g64", "moe_pack_w4a16_g128", "moe_dequant"]:
        assert must in names


def test_library_exports_every_declared_symbol(capi):
    lib = ctypes.CDLL(str(capi.LIB_PATH))
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(capi.EXPORTS) == declared_functions()


def test_status_strings(capi):
    assert capi.lib.moe_status_string(0) == b"MOE_OK"
    assert capi.lib.moe_status_string(2) == b"MOE_ERR_UNSUPPORTED_FORMAT"
    assert capi.lib.moe_status_string(99) == b"MOE_ERR_UNKNOWN"


def test_workspace_bytes(capi):
    n1 = capi.moe_workspace_bytes(1, 256, 8, 2048, 512)
    n32 = capi.moe_workspace_bytes(32, 256, 8, 2048, 512)
    assert 0 < n1 < n32
    assert capi.moe_workspace_bytes(-1, 256, 8, 2048, 512) == 0
    assert capi.moe_workspace_bytes(4, 256, 8, 2000, 512) == 0


def _bank(fmt, E=8, I=128, H=256, base=1 << 20, layout=1):
    S = capi_mod().ExpertBankS
    p = [base + 4096 * i for i in range(6)]
    return S(capi_mod().FMT[fmt], E, I, H, layout, 0, *p)


def capi_mod():
    from bit_affine_quantized_fp32_gb300 import capi as C
    return C


def _call_experts(capi, bank, T=2, k=2, ws=1 << 24, wsb=1 << 30):
    P = 1 << 21
    return capi.lib.moe_experts_forward(ctypes.byref(bank), P, 1, T, k, P, P, P, P, None, None,
                                        P, 0, ws, wsb, None)


def test_refuses_unread_width_by_name(capi):
    rc = _call_experts(capi, _bank("bf16"))         # a dense type is not an expert format
    assert rc == 2
    assert b"BF16" in capi.lib.moe_last_error()
    S = capi.ExpertBankS
    rc = _call_experts(capi, S(42, 8, 128, 256, 1, 0, *[1 << 20] * 6))
    assert rc == 2


def test_refuses_bad_shapes_and_pointers(capi):
    assert _call_experts(capi, _bank("affine4_g64", I=100)) == 1          # inter % 128
    assert _call_experts(capi, _bank("w4a16_g128", I=128)) == 1           # w4a16 needs 256
    assert _call_experts(capi, _bank("affine4_g64"), k=9) == 1            # k > 8
    assert _call_experts(capi, _bank("affine4_g64", E=4), k=5) == 1       # k > E
    assert _call_experts(capi, _bank("affine4_g64", base=(1 << 20) + 4)) == 6  # misaligned
    assert _call_experts(capi, _bank("affine4_g64"), ws=None) == 3        # no workspace
    assert _call_experts(capi, _bank("affine4_g64"), wsb=1024) == 3       # too small
    S = capi.ExpertBankS
    nul = S(capi.FMT["affine4_g64"], 8, 128, 256, 1, 0, None, 1 << 20, 1 << 20, 1 << 20, 1 << 20,
            1 << 20)
    assert _call_experts(capi, nul) == 1
    # the expert kernels read the tiled layout only
    assert _call_experts(capi, _bank("affine4_g64", layout=0)) == 1
    assert b"TILED" in capi.lib.moe_last_error()


@pytest.mark.parametrize("fmt,bits,G,bias", [("affine4_g64", 4, 64, True),
                                             ("affine3_g64", 3, 64, True),
                                             ("w4a16_g128", 4, 128, False)])
@pytest.mark.parametrize("E,I,H", [(256, 512, 2048), (3, 256, 768), (1, 512, 1024)])
def test_tiled_bytes_equal_canonical_bytes(capi, fmt, bits, G, bias, E, I, H):
    """The tiled layout only rearranges: codes at exactly `bits` bits each plus
    one fp16 scale (and bias) per group, nothing padded."""
    if fmt == "w4a16_g128" and (I % 256 or H % 256):
        pytest.skip("W4A16 shapes are multiples of 256")
    for which, rows, cols in ((0, 2 * I, H), (1, H, I)):
        want = E * rows * (cols * bits // 8 + (cols // G) * 2 * (2 if bias else 1))
        assert capi.lib.moe_tiled_bytes(capi.FMT[fmt], E, I, H, which) == want


def test_tiled_bytes_refuses_bad_shapes(capi):
    assert capi.lib.moe_tiled_bytes(capi.FMT["affine4_g64"], 8, 100, 256, 0) == 0
    assert capi.lib.moe_tiled_bytes(capi.FMT["bf16"], 8, 128, 256, 0) == 0
    assert capi.lib.moe_tiled_bytes(capi.FMT["affine4_g64"], 8, 128, 256, 2) == 0


def test_repack_validation(capi):
    S = capi.ExpertBankS
    P = 1 << 21
    canon = _bank("affine4_g64", layout=0)
    assert capi.lib.moe_repack_bank(ctypes.byref(canon), None, P, None) == 1
    assert capi.lib.moe_repack_bank(ctypes.byref(canon), P + 4, P, None) == 6
    tiled = _bank("affine4_g64", layout=1)
    assert capi.lib.moe_repack_bank(ctypes.byref(tiled), P, P, None) == 1
    nob = S(capi.FMT["affine4_g64"], 8, 128, 256, 0, 0, P, P, None, P, P, None)
    assert capi.lib.moe_repack_bank(ctypes.byref(nob), P, P, None) == 1
    assert capi.lib.moe_unrepack_bank(ctypes.byref(canon), P, P, P, P, P, P, None) == 1
    assert capi.lib.moe_unrepack_bank(ctypes.byref(tiled), P, P, None, P, P, P, None) == 1


def test_route_validation(capi):
    Q = capi.QMatrixS
    P = 1 << 21
    r = Q(capi.FMT["affine4_g64"], 256, 2048, 0, P, P, P)   # 4-bit router is not read
    rc = capi.lib.moe_route(ctypes.byref(r), None, None, P, 1, 4, 8, None, P, P, None, P, P,
                            0, P, 1 << 30, None)
    assert rc == 2 and b"router" in capi.lib.moe_last_error()
    r = Q(capi.FMT["f32"], 300, 2048, 0, P, None, None)     # > 256 experts
    rc = capi.lib.moe_route(ctypes.byref(r), None, None, P, 1, 4, 8, None, P, P, None, P, P,
                            0, P, 1 << 30, None)
    assert rc == 1
    r = Q(capi.FMT["f32"], 256, 2048, 0, P, None, None)
    rc = capi.lib.moe_route(ctypes.byref(r), None, None, P, 7, 4, 8, None, P, P, None, P, P,
                            0, P, 1 << 30, None)                # activation format 7
    assert rc == 2
    rc = capi.lib.moe_route(ctypes.byref(r), None, None, P, 1, 4, 8, None, P, P, None, P, P,
                            8, P, 1 << 30, None)                # unknown flag
    assert rc == 1 and b"flags" in capi.lib.moe_last_error()


def test_force_prefill_flag_validation(capi):
    # MOE_FLAG_FORCE_PREFILL with MOE_FLAG_FORCE_DECODE is refused, and so is
    # a format the tensor-core GEMMs do not read (checked before any launch)
    P = 1 << 21

    def call(bank, flags):
        return capi.lib.moe_experts_forward(ctypes.byref(bank), P, 1, 4, 2, P, P, P, P, None,
                                            None, P, flags, 1 << 24, 1 << 30, None)

    rc = call(_bank("affine4_g64"), capi.MOE_FLAG_FORCE_PREFILL | capi.MOE_FLAG_FORCE_DECODE)
    assert rc == 1 and b"FORCE_DECODE" in capi.lib.moe_last_error()
    rc = call(_bank("affine2_g64"), capi.MOE_FLAG_FORCE_PREFILL)
    assert rc == 2 and b"AFFINE2" in capi.lib.moe_last_error()
    rc = call(_bank("affine4_g64"), 16)  # unknown flag
    assert rc == 1 and b"flags" in capi.lib.moe_last_error()


def test_wait_limit_validation(capi):
    assert capi.lib.moe_workspace_set_wait_limit(None, 1 << 20, 5, None) == 3
    assert capi.lib.moe_workspace_set_wait_limit(1 << 21, 1 << 20, 1 << 31, None) == 1


def test_pack_validation(capi):
    assert capi.lib.moe_pack_affine4_g64(1 << 20, 4, 33, 1 << 21, None) == 1
    assert capi.lib.moe_pack_affine3_g64(None, 4, 64, 1 << 21, None) == 1


def test_route_static_limits(capi):
    """moe_route_static refuses shapes beyond its static scratch before any
    launch (no device needed)."""
    Q = capi.QMatrixS
    P = 1 << 21
    r = Q(capi.FMT["f32"], 256, 2048, 0, P, None, None)
    rc = capi.lib.moe_route_static(ctypes.byref(r), None, None, P, 1, 33, 8, P, P, None, P, P,
                                   None)
    assert rc == 3 and b"static scratch" in capi.lib.moe_last_error()
    r = Q(capi.FMT["f32"], 256, 2048, 0, P, None, None)
    rc = capi.lib.moe_route_static(ctypes.byref(r), None, None, P, 1, 32, 8, None, P, None, P,
                                   P, None)
    assert rc == 1   # NULL topk_idx, caught before the scratch is looked up


@pytest.mark.parametrize("fmt,bits", [("affine2_g64", 2), ("affine3_g64", 3), ("affine4_g64", 4),
                                      ("affine5_g64", 5), ("affine6_g64", 6), ("affine8_g64", 8)])
def test_tiled_bytes_hold_exactly_the_canonical_bytes(capi, fmt, bits):
    """A tiled bank at any affine width holds the codes at their width plus the
    fp16 scale and bias of every 64-group, nothing more (no padding)."""
    E, I, H = 3, 256, 512
    for which, (rows, cols) in enumerate([(2 * I, H), (H, I)]):
        n = rows * cols
        assert capi.lib.moe_tiled_bytes(capi.FMT[fmt], E, I, H, which) == \
            E * (n * bits // 8 + n // 64 * 4)
