"""The bench's work counts (host arithmetic, no GPU), pinned to the
algorithmic bytes and flops that the workload's shapes fix: Qwen3-8B layer
matrices and Qwen3-30B-A3B experts as the FP8-RL pages name them ("Results":
the dense and MoE models), each byte counted once (bf16 in, E4M3 out, fp32
scales; a GEMM's weights once).  A formula that drops a term or mixes up N and
K moves one of these figures."""
import pytest

import bench
from fp8_w8a8_rollout_gb300 import synth


def test_weight_sync_bytes_of_a_layer_the_model_and_the_experts():
    layer = sum(bench.wq_bytes(n, k) for _, n, k in synth.QWEN3_8B_LAYER)
    assert layer == 578_861_056
    assert layer * synth.QWEN3_8B_LAYERS == pytest.approx(20.839e9, rel=1e-4)
    moe = synth.MOE_LAYERS * synth.MOE_EXPERTS * (bench.wq_bytes(2 * synth.MOE_INTER, synth.MOE_HIDDEN) +
                                                  bench.wq_bytes(synth.MOE_HIDDEN, synth.MOE_INTER))
    assert moe == pytest.approx(86.98e9, rel=1e-3)
    # UE8M0: one byte per block scale instead of four
    assert bench.wq_bytes(4096, 4096, 1) == 3 * 4096 * 4096 + 32 * 32


def test_activation_quant_bytes():
    assert bench.aq_bytes(8192, 12288) == 3 * 8192 * 12288 + 4 * 8192 * 96
    assert bench.aq_bytes(8192, 12288) == pytest.approx(305.1e6, rel=1e-3)
    assert bench.aq_bytes(3, 200) == 3 * 3 * 200 + 4 * 3 * 2  # a partial last group has a scale


def test_gemm_flops_and_bytes():
    assert bench.gemm_flops(8192, 24576, 4096) == pytest.approx(1.649e12, rel=1e-3)
    assert bench.gemm_bytes(8192, 24576, 4096) == pytest.approx(538.0e6, rel=1e-3)
    assert bench.gemm_bytes(16, 6144, 4096) == pytest.approx(25.44e6, rel=1e-3)
    # at decode sizes the weights are 98 % of the bytes
    assert bench.gemm_bytes(16, 6144, 4096) - 6144 * 4096 < 0.02 * 6144 * 4096


def test_grouped_gemm_bytes_and_flops():
    rows = synth.MOE_TOKENS * synth.MOE_TOPK
    e, h, i = synth.MOE_EXPERTS, synth.MOE_HIDDEN, synth.MOE_INTER
    assert bench.gemm_flops(rows, 2 * i, h) == pytest.approx(206.2e9, rel=1e-3)
    assert bench.grouped_gemm_bytes(e, rows, 2 * i, h) == pytest.approx(572.6e6, rel=1e-3)
    assert bench.gemm_flops(rows, h, i) == pytest.approx(103.1e9, rel=1e-3)
    assert bench.grouped_gemm_bytes(e, rows, h, i) == pytest.approx(361.5e6, rel=1e-3)
    # one expert holding every row is the dense GEMM
    assert bench.grouped_gemm_bytes(1, 1024, 2048, 768) == bench.gemm_bytes(1024, 2048, 768)


def test_roofline_picks_the_lower_roof():
    hbm, fp8 = 6789.0, 3748.6
    small = bench.gemm_roof(bench.gemm_flops(16, 6144, 4096), bench.gemm_bytes(16, 6144, 4096), 0.01, hbm, fp8)
    assert small["bound"] == "hbm" and small["unit"] == "GB/s"
    assert small["frac"] == pytest.approx(bench.gemm_bytes(16, 6144, 4096) / 1e-5 / 1e9 / hbm)
    big = bench.gemm_roof(bench.gemm_flops(8192, 24576, 4096), bench.gemm_bytes(8192, 24576, 4096), 0.67, hbm, fp8)
    assert big["bound"] == "tensor" and big["unit"] == "TFLOP/s"
    assert big["frac"] == pytest.approx(1.649267e12 / 0.67e-3 / 1e12 / fp8, rel=1e-5)
    # the grouped MoE GEMMs at T = 4096 sit below the ridge: HBM-bound
    rows = synth.MOE_TOKENS * synth.MOE_TOPK
    g = bench.gemm_roof(bench.gemm_flops(rows, 1536, 2048), bench.grouped_gemm_bytes(128, rows, 1536, 2048), 0.14,
                        hbm, fp8)
    assert g["bound"] == "hbm"


def test_fp8_peak_is_twice_the_burst_bf16_rate():
    assert bench.fp8_peak({"bf16_tflops": 1874.3, "bf16_tflops_sustained": 1722.0}) == pytest.approx(3748.6)


def test_traffic_record_matches_the_committed_gemm_sources():
    """The dominant GEMM's captured DRAM bytes are reported only while its
    sources are those the capture was taken with; the record in bench.py
    must describe the sources as committed."""
    t = bench.captured_traffic("gemm_gate_up")
    assert t is not None, "gemm.cu / ptx.cuh / common.cuh changed since the ncu capture: re-capture"
    assert 0.9 * bench.gemm_bytes(8192, 24576, 4096) < t < 1.1 * bench.gemm_bytes(8192, 24576, 4096)
    assert bench.captured_traffic("no_such_kernel") is None
