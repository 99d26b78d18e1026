"""The benchmark's roofline arithmetic (counted FLOPs and algorithmic bytes)
against figures derived by hand from the workloads' shapes, so that a slip in
a formula (a dropped term, a wrong width, a factor of two) shows up here and
not as a wrong roofline fraction.  CPU only."""
import pytest

import bench


def test_counted_prefill_flops_per_chunk():
    # C^2 (6 dk + 4 dv) + 6 C dk dv + C^3 / 3 at C = 64, dk = dv = 256:
    # 4096 * 2560 + 6 * 64 * 65536 + 262144 / 3
    f_chunk = 10_485_760 + 25_165_824 + 262_144 / 3
    assert bench.prefill_flops([64], H=1) == pytest.approx(f_chunk, rel=1e-15)
    assert round(f_chunk) == 35_738_965
    # per token-head and per token at H = 6
    assert bench.prefill_flops([64], H=1) / 64 == pytest.approx(558_421.33, abs=0.01)
    assert bench.prefill_flops([64]) / 64 == pytest.approx(3.3505e6, rel=1e-4)
    # partial chunks count whole: 65 tokens are two chunks
    assert bench.prefill_flops([65], H=1) == pytest.approx(2 * f_chunk)
    # the 8K workload: 4 x 128 chunks x 6 heads
    assert bench.prefill_flops([8192] * 4) == pytest.approx(3072 * f_chunk)
    assert bench.prefill_flops([8192] * 4) == pytest.approx(1.098e11, rel=1e-3)


def test_prefill_algorithmic_bytes():
    # per token: q, k, v, out bf16 at 256 wide (4 x 512 B) and alpha, beta
    # fp32, times 6 heads = 12,336 B; per sequence S0 and S_final, 1.5 MiB each
    assert bench.prefill_bytes([1], s0=False, s_final=False) == 12_336
    assert bench.prefill_bytes([0]) == 2 * 6 * 256 * 256 * 4
    assert bench.prefill_bytes([8192] * 4) == 32_768 * 12_336 + 4 * 2 * 1_572_864
    assert bench.prefill_bytes([8192] * 4) == 416_808_960
    # fp32 I/O doubles the token bytes but not alpha, beta or the states
    assert bench.prefill_bytes([1], io_bytes=4, s0=False, s_final=False) == 6 * (4 * 1024 + 8)


def test_decode_algorithmic_bytes():
    # per (sequence, head, step): state read + write 2 x 256 KiB, q, k, v,
    # out 4 x 512 B, alpha + beta 8 B
    assert bench.decode_bytes(1) == 6 * 526_344
    assert bench.decode_bytes(256) == 808_464_384
    assert bench.decode_bytes(1, dv=512) == 6 * (2 * 512 * 1024 + 2 * 512 + 2 * 1024 + 8)


def test_layer_step_bytes():
    # gdn_prepare on 4 x 8192 tokens: C = 6 x 768 = 4608 channels read and
    # written at bf16, 4 fp32 gate values a head read or written, the carried
    # state in and out per sequence, taps and per-head parameters once
    C = 4608
    expect = 32_768 * (2 * C * 2 + 16 * 6) + 2 * 4 * 3 * C * 2 + C * 16 + 2 * 6 * 4
    assert bench.prepare_bytes(32_768, 4) == expect == 607_420_464
    # gated RMSNorm: read o and g, write y, per (token, head) row, plus the weight
    assert bench.norm_gate_bytes(32_768 * 6) == 32_768 * 6 * 256 * 2 * 3 + 1024 == 301_990_912


def test_backward_executed_flops():
    # per (chunk, head) at C = 64, dk = dv = 256: one C x d x d product is
    # 8,388,608 FLOP, one C x C x d product 2,097,152, one C^3 product 524,288
    big, small, cube = 8_388_608, 2_097_152, 524_288
    fwd = 4 * small + 2 * big            # KK^T, QK^T, W, U~ (C x C x d); U, S' (C x d x d)
    rev = 3 * big + small                # K dS'^T, dO^T Qh, dU^T W; Ph^T dO
    # U, dO S, dU S, U dS', K dS'^T (C x d x d); dPh, dT (two), T^T dW, T^T dU,
    # (M + M^T) K, FG^T Q, FG K (C x C x d); dA = -T^T dT T^T (two C^3)
    local = 5 * big + 8 * small + 2 * cube
    per = fwd + rev + local
    assert (fwd, rev, local) == (25_165_824, 27_262_976, 59_768_832)
    assert bench.backward_flops([64], H=1) == per == 112_197_632
    assert bench.backward_flops([8192] * 4) == 3072 * per == 344_671_125_504


def test_fp32_fma_peak():
    assert bench.FP32_FMA_TFLOPS == pytest.approx(152 * 128 * 2 * 2.07e-3)
    assert bench.FP32_FMA_TFLOPS == pytest.approx(80.5, abs=0.05)
    # the dense tf32 tensor peak scales the bf16 one by the nominal 1.1 / 2.25
    assert bench.TF32_TFLOPS({"bf16": 2250.0}) == pytest.approx(1100.0)
