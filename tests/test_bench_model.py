"""The bench's roofline accounting (bench.work_model, bench.t_roof) against
figures worked out by hand from the workload's shapes: the Qwen3-8B weight
sync, the four linears at M = 8192, the Qwen3-30B-A3B MoE layer and the
KV recalibration.  CPU only."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def phases():
    return {name: (flops, nbytes) for name, flops, nbytes in bench.work_model()}


def test_weight_sync_bytes():
    # 36 layers x (qkv 6144x4096 + o 4096x4096 + gate_up 24576x4096 + down
    # 4096x12288) = 6,945,767,424 weights, 2 B read + 1 B written each, plus
    # one FP32 scale per 128x128 block (423,936 blocks)
    elems = 36 * (6144 * 4096 + 4096 * 4096 + 24576 * 4096 + 4096 * 12288)
    blocks = 36 * (48 * 32 + 32 * 32 + 192 * 32 + 32 * 96)
    assert elems == 6_945_767_424 and blocks == 423_936
    flops, nbytes = phases()["weight_quant"]
    assert flops == 0 and nbytes == 3 * elems + 4 * blocks == 20_838_998_016


def test_linear_flops_and_bytes():
    M = 8192
    shapes = [(6144, 4096), (4096, 4096), (24576, 4096), (4096, 12288)]
    flops, nbytes = phases()["gemm_linears"]
    assert flops == sum(2 * M * n * k for n, k in shapes) == 16384 * 192_937_984 == 3_161_095_929_856
    # codes of X and W read once, the scale grids, the BF16 output written once
    want = sum(M * k + n * k + 4 * (M * (k // 128) + (n // 128) * (k // 128)) + 2 * M * n
               for n, k in shapes)
    assert nbytes == want
    aq_flops, aq_bytes = phases()["act_quant_linears"]
    assert aq_flops == 0 and aq_bytes == sum(3 * M * k + 4 * M * (k // 128) for _, k in shapes)


def test_moe_layer():
    T, H, I, E, R = 4096, 2048, 768, 128, 4096 * 8
    flops, _ = phases()["grouped_gemm_moe"]
    # gate_up: [R, H] x [2I, H]^T; down: [R, I] x [H, I]^T
    assert flops == 2 * R * (2 * I) * H + 2 * R * H * I
    _, qbytes = phases()["act_quant_moe"]
    # the token activations and the down input, each read once and coded once
    assert qbytes == 3 * T * H + 4 * T * (H // 128) + 3 * R * I + 4 * R * (I // 128)


def test_kv_recalibration_bytes():
    n = 32 * 8192 * 8 * 128
    assert n == 268_435_456
    flops, nbytes = phases()["kv_quant"]
    # K and V: the amax pass reads 2 B, the code pass reads 2 B and writes 1 B
    assert flops == 0 and nbytes == 2 * 5 * n


def test_decode_passes():
    # every layer's 4 linears at M tokens: the GEMM's codes, scale grids and
    # BF16 output, plus the activation quantizer's 3 B per element and scales
    shapes = [(6144, 4096), (4096, 4096), (24576, 4096), (4096, 12288)]
    for M in bench.DECODE_MS:
        flops, nbytes = phases()[f"decode_m{M}"]
        assert flops == 36 * sum(2 * M * n * k for n, k in shapes)
        want = 36 * sum(M * k + n * k + 4 * (M * (k // 128) + (n // 128) * (k // 128)) + 2 * M * n
                        + 3 * M * k + 4 * M * (k // 128) for n, k in shapes)
        assert nbytes == want
        # the weights dominate: 36 x 176 MB of FP8 codes per pass
        assert 36 * sum(n * k for n, k in shapes) == 6_945_767_424


def test_roofline_time_takes_the_binding_resource():
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 500.0, "bf16_tflops_sustained": 400.0}
    # 1 GB at 1 TB/s = 1 ms; 1 TFLOP at 2 x 500 TF/s (the burst figure) = 1 ms;
    # 2 TFLOP = 2 ms
    assert bench.t_roof(0, 1e9, peaks) == pytest.approx(1e-3)
    assert bench.t_roof(2e12, 1e9, peaks) == pytest.approx(2e12 / (bench.FP8_OVER_BF16 * 500e12))
    assert bench.t_roof(1e11, 1e9, peaks) == pytest.approx(1e-3)
    assert bench.fp8_peak_tflops(peaks) == pytest.approx(1000.0)


def test_single_linear_work():
    """X [128, 512], W [256, 512]: 2 m n k FLOPs; the bytes of both
    quantizers (2 B read + 1 B written per element + scales) and of the
    GEMM (codes, scales, BF16 output)."""
    f, b = bench.single_linear_work()
    assert f == 2 * 128 * 256 * 512
    q_x = 131072 + 65536 + 4 * 128 * 4
    q_w = 262144 + 131072 + 4 * 2 * 4
    gemm = 65536 + 131072 + 4 * (128 * 4 + 2 * 4) + 65536
    assert b == q_x + q_w + gemm


def test_prefill_attention_flops():
    """Causal: query token i meets i + 1 keys, 4 D FLOPs per (query, key,
    head): S (S + 1) / 2 pairs per sequence and head."""
    assert bench.prefill_attention_flops(1, 1, 1) == 4 * 128
    assert bench.prefill_attention_flops(2, 3, 4) == 4 * 128 * 4 * 2 * 6

