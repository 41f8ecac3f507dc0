"""bench.py's host-side arithmetic (no GPU): the algorithmic work of a layer call as the measurement
plan defines it, and the choice of the binding roofline from the measured peaks."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from nvfp4_w4a4_mixture_gb300 import workloads as wl  # noqa: E402


def test_expert_bytes_flash_shape():
    # gate + up + down of H 2048 x I 768: 3 * 2048 * 768 E2M1 codes (1/2 byte) + UE4M3 scales per 16
    # (1/16 byte) + three FP32 tensor scales
    assert bench.expert_bytes(2048, 768) == 3 * 2048 * 768 // 2 + 3 * 2048 * 768 // 16 + 12 == 2_654_220


def test_algorithmic_work_prefill16k():
    c = wl.CONFIGS["prefill16k"]
    w = bench.algorithmic_work(c, 512)
    assert w["weights"] == 513 * 2_654_220
    assert w["io"] == 2 * 16384 * 2048 * 2  # x in, out
    assert w["router"] == 513 * 2048 * 2
    assert w["kernel_bytes"] == w["weights"] + w["io"]
    assert w["layer_bytes"] == w["weights"] + w["router"] + w["io"]
    assert w["flops_fp4"] == 2.0 * 16384 * 11 * 3 * 2048 * 768
    # the intermediates are not algorithmic bytes
    assert w["overhead_bytes"]["y_written_read"] == 2 * 16384 * 11 * 2048 * 2


def test_algorithmic_work_stack_counts_the_residual():
    c = wl.CONFIGS["stack48"]
    w = bench.algorithmic_work(c, 512)
    assert w["io"] == 3 * 2048 * 2048 * 2


def test_roofline_picks_the_longer_time():
    hbm, fp4 = 6663.2, 11415.6
    # 16k chunk: 1.50 GB at 6.66 TB/s (225 us) outlasts 1.70 TFLOP at 11.4 PF/s (149 us)
    w = bench.algorithmic_work(wl.CONFIGS["prefill16k"], 512)
    r = bench.roofline(w["kernel_bytes"], w["flops_fp4"], 1e-3, hbm, fp4)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["frac"] - w["kernel_bytes"] / 1e-3 / 1e9 / hbm) < 1e-12
    # the same FLOPs over a tenth of the bytes: the tensor cores bind
    r = bench.roofline(w["kernel_bytes"] / 10, w["flops_fp4"], 1e-3, hbm, fp4)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["frac"] - w["flops_fp4"] / 1e-3 / 1e12 / fp4) < 1e-12


def test_default_workload_is_the_largest_single_layer_config():
    assert bench.DEFAULT_CONFIG == "prefill16k"
    assert set(bench.EXTRA_CONFIGS) == {"decode", "decode_stack48", "stack48"}


def test_traffic_hash_ignores_comments_but_not_code(tmp_path):
    src = os.path.join(ROOT, "nvfp4_w4a4_mixture_gb300", "csrc")
    for f in bench.GEMM_SOURCES:
        with open(os.path.join(src, f), encoding="utf-8") as fh:
            (tmp_path / f).write_text(fh.read(), encoding="utf-8")
    base = bench.gemm_sources_hash(str(tmp_path))
    assert base == bench.gemm_sources_hash()
    k = tmp_path / "grouped_gemm.cu"
    text = k.read_text(encoding="utf-8")
    k.write_text("// a new comment line\n/* and a block\n   comment */\n" + text.replace(";", ";   ", 3), encoding="utf-8")
    assert bench.gemm_sources_hash(str(tmp_path)) == base
    k.write_text(text.replace("STAGES = 4", "STAGES = 3", 1), encoding="utf-8")
    assert bench.gemm_sources_hash(str(tmp_path)) != base

