"""bench.py without a GPU: the algorithmic bytes behind the roofline figure,
the guard that drops a stale DRAM-traffic record, and the oracle (reference)
arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


# bytes per quantisation group, from the formats' definitions: codes at their
# width, then one fp16 scale (and one fp16 bias for the affine formats)
@pytest.mark.parametrize("fmt,per_group,G", [
    ("affine8_g64", 64 + 4, 64),
    ("affine4_g64", 32 + 4, 64),
    ("affine3_g64", 24 + 4, 64),
    ("w4a16_g128", 64 + 2, 128),
])
def test_matrix_bytes_per_group(fmt, per_group, G):
    for rows, cols in [(1, 2048), (256, 2048), (2048, 512), (1024, 256)]:
        assert bench.matrix_bytes(fmt, rows, cols) == rows * cols // G * per_group


def test_matrix_bytes_dense_and_absent():
    assert bench.matrix_bytes("f32", 256, 2048) == 2 * 1024 * 1024
    assert bench.matrix_bytes("bf16", 1, 2048) == 4096
    assert bench.matrix_bytes("f16", 3, 8) == 48
    assert bench.matrix_bytes(None, 256, 2048) == 0


def test_expert_bytes_at_layer_shape():
    # gate, up and down of one expert: 3 * 512 * 2048 = 3,145,728 weights
    n = 3 * 512 * 2048
    assert bench.expert_bytes("affine4_g64") == n // 64 * 36 == 1_769_472
    assert bench.expert_bytes("affine3_g64") == n // 64 * 28 == 1_376_256
    assert bench.expert_bytes("w4a16_g128") == n // 128 * 66 == 1_622_016


def test_kernel_source_hash_tracks_every_source():
    base = bench.kernel_source_hash()
    assert base == bench.kernel_source_hash()
    real = lambda rel: open(os.path.join(ROOT, rel), "rb").read()  # noqa: E731
    for target in ("include/moe_gb300.h", "bit_affine_quantized_fp32_gb300/csrc/decode.cu"):
        changed = lambda rel, t=target: real(rel) + (b" " if rel == t else b"")  # noqa: E731
        assert bench.kernel_source_hash(changed) != base


def test_captured_traffic_needs_matching_sources(tmp_path, monkeypatch):
    rec = {"source_sha256": "0" * 64, "dram_bytes_per_step": 123}
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic_decode1_affine4.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda read=None: "f" * 64)
    assert bench.captured_traffic("decode1_affine4") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda read=None: "0" * 64)
    assert bench.captured_traffic("decode1_affine4") == 123
    assert bench.captured_traffic("decode4_affine3") is None      # no record


def test_step_flops_of_the_prefill_window():
    # 512 tokens x 8 routed experts and the shared expert, three 512 x 2048
    # products each at 2 flops per weight, plus the 256 x 2048 router and the
    # gate row: 29.5 GFLOP
    from bit_affine_quantized_fp32_gb300 import synth
    cfg = synth.WORKLOADS["prefill512_affine4_zipf"]
    per = 2 * 3 * 512 * 2048
    assert bench.step_flops(cfg, 512) == 512 * 8 * per + 512 * per + 2 * 256 * 2048 * 512 + \
        2 * 2048 * 512
    assert abs(bench.step_flops(cfg, 512) / 1e9 - 29.5) < 0.1
    # routing 4 (the bucket launch builds the tables), sums + fp16 copy 1,
    # GEMMs 2 (shared expert folded in), light-expert units 2, combine 1; a
    # shared expert of another format adds its conversion, two GEMMs and a
    # separate tables launch
    assert bench.launches_per_step(cfg, 512) == 10
    assert bench.launches_per_step(dict(cfg, shared_fmt="affine3_g64"), 512) == 14
    assert bench.launches_per_step(synth.WORKLOADS["decode8_affine4_shared_zipf"], 8) == 1


def test_reference_arm_line_on_cpu():
    # the oracle arm needs no GPU and no library: inputs from the seeded
    # generators on the CPU, one token per step through the whole layer
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in rec, key
    assert rec["impl"] == "reference" and rec["n_gpus"] == 1 and rec["steps"] == 2
    assert rec["value"] > 0 and rec["unit"] == "tokens/s" and rec["higher_is_better"] is True
    cb = rec["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == rec["value"]
    assert cb["sample"]
    assert rec["e2e"] == {"value": rec["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}
    assert rec["config"]["workload"] == bench.DEFAULT_WORKLOAD


def test_clock_record_parsing():
    idle = "0, 2070, 2070, 150.00, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"
    capped = "0, 1965, 2070, 1398.20, 0x0000000000000004, Not Active, Not Active, Not Active, Active"
    hot = "0, 1500, 2070, 900.00, 0x0000000000000020, Not Active, Not Active, Active, Not Active"
    r = bench.parse_clock_lines([idle, capped, idle, "garbage", "", "0, [N/A], 2070"])
    assert r == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                 "samples": 3}
    r = bench.parse_clock_lines([hot, idle])
    assert r["reasons"] == ["sw_thermal_slowdown"] and r["sm_mhz"] == (1500 + 2070) / 2
    assert bench.parse_clock_lines([]) == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                                           "samples": 0}


def test_sweep_workload_is_consecutive_windows():
    # the 4096-token prompt of the prefill configuration: eight consecutive
    # 512-token layer calls per step, reported beside the other workloads
    cfg, Tw, nwin = bench.workload_cfg("prefill4096_affine4_zipf_sweep")
    assert (Tw, nwin) == (512, 8) and cfg["expert_fmt"] == "affine4_g64" and cfg["zipf"]
    assert "prefill4096_affine4_zipf_sweep" in bench.OTHER_WORKLOADS
    assert bench.workload_cfg("decode8_affine4_shared_zipf")[1:] == (8, 1)
    assert bench.metric_name(4096, "affine4_g64", "prefill4096_affine4_zipf_sweep") == (
        "MoE-layer tokens/s (prefill sweep of 4096 tokens in 512-token windows, affine4_g64)")

