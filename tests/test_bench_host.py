"""The bench's host-side accounting, on the CPU: the algorithmic bytes and FLOPs its roofline
lines divide by, and the rule that a stored DRAM-traffic figure is reported only for the
kernel source it was captured on.

The expected numbers are worked out by hand below from the definition of one step (x, W
and y once; each distinct adapter's A and B once at its true rank; the ids; the fp32
intermediate of the low-rank term once), not by calling the bench's formulas."""
import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

bench = pytest.importorskip("bench")
from segmented_rank_gemm_gb300 import workloads  # noqa: E402


def _tiny():
    # T=4 rows, K=8, N=16, two slots of ranks 2 and 3, bf16; the seeded ids are [0, 1, 1, 1]
    wl = workloads.synthetic(1, 4, 8, 16, S=2, ranks=[2, 3], R=4)
    assert wl.token_slot.tolist() == [0, 1, 1, 1]
    return wl


def test_step_bytes_and_flops_delta_mode():
    w = bench.algorithmic(_tiny())
    # x 4*8*2 = 64, W 8*16*2 = 256, y 4*16*2 = 128, ids 4*4 = 16;
    # A: 8*2*2 + 8*3*2 = 80, B: 2*16*2 + 3*16*2 = 160
    assert w["step_bytes"] == 64 + 256 + 128 + 16 + 80 + 160 == 704
    # GEMM: x, W, y, ids and the fp32 delta of the 4 adapted rows (4*16*4 = 256)
    assert w["gemm_bytes"] == 64 + 256 + 128 + 16 + 256 == 720
    # low-rank kernel: x, A, B, the delta it writes, ids
    assert w["lowrank_bytes"] == 64 + 80 + 160 + 256 + 16 == 576
    # 2 T K N; 2 * sum over rows of r (K + N) = 2 * (2 + 3 + 3 + 3) * 24
    assert w["base_flops"] == 1024 and w["lora_flops"] == 528
    assert w["distinct_slots"] == 2 and w["adapted_rows"] == 4 and w["mode"] == "delta"


def test_step_bytes_v_mode():
    w = bench.algorithmic(_tiny(), delta_mode=False)
    # v: the rows' ranks (2 + 3 + 3 + 3 = 11) fp32 values = 44 bytes
    assert w["gemm_bytes"] == 64 + 256 + 128 + 160 + 44 + 16 == 668
    assert w["lowrank_bytes"] == 64 + 80 + 44 == 188
    assert w["mode"] == "v"


def test_step_bytes_e4m3_base():
    w = bench.algorithmic(_tiny(), fp8=True)
    # W one byte an element (128); xq (4*8 = 32 bytes) written once and read once
    assert w["step_bytes"] == 64 + 128 + 128 + 16 + 2 * 32 + 80 + 160 == 640
    # the GEMM reads xq instead of x
    assert w["gemm_bytes"] == 32 + 128 + 128 + 256 + 16 == 560


def test_stack_pass_work():
    flops, base_bytes, ad_bytes, act_bytes = bench._stack_flops_bytes(512, 32, 100)
    # sum of K N over q, k, v, o, gate, up, down of the 8B-class layer
    kn = 2 * 4096 * 4096 + 2 * 4096 * 1024 + 3 * 4096 * 14336
    assert kn == 218103808
    assert flops == 2 * 512 * kn * 32 == 7146825580544  # 7.15 TFLOP a pass
    assert base_bytes == kn * 2 * 32
    k_plus_n = 8192 + 5120 + 5120 + 8192 + 3 * 18432
    assert ad_bytes == 16 * k_plus_n * 2 * 32 * 100  # rank 16, every resident slot once
    assert act_bytes == 512 * k_plus_n * 2 * 32
    _, base8, _, _ = bench._stack_flops_bytes(512, 32, 100, fp8=True)
    assert base8 == kn * 32


def test_traffic_reported_only_for_its_kernel_source(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_bytes(b"// one kernel source\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({
        "decode_bgmv": {"dram_bytes_per_launch": 1234.0, "kernel_sha256_16": sha},
        "prefill_sgmv": {"dram_bytes_per_launch": 99.0, "kernel_sha256_16": "0" * 16}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profile(str(src), "decode_bgmv") == 1234.0
    assert bench.traffic_from_profile(str(src), "prefill_sgmv") is None  # another source
    assert bench.traffic_from_profile(str(src), "mixed_continuous") is None  # not captured
    src.write_bytes(b"// the source edited since the capture\n")
    assert bench.traffic_from_profile(str(src), "decode_bgmv") is None
