"""Pins for the oracle's dequantisation and verify GEMMs (CPU only).

Each check is independent of the oracle's own code path: hand-computed
values, a special case that reduces to the raw integer codes, and a
pure-Python brute force that reads the packed bytes element by element.
"""
import numpy as np
import pytest

import oracle
from bit_qgemm_w4_gb300 import inputs


def _f16(vals):
    return np.asarray(vals, dtype=np.float16)


def test_w4_dequant_hand_example():
    # N=2 rows, K=8, groups of 4 along k.  The 4 bytes of a row's word carry
    # (k0|k2<<4), (k4|k6<<4), (k1|k3<<4), (k5|k7<<4).
    # row 0 codes [10, 3, 15, 0, 1, 2, 3, 4] -> bytes 0xFA, 0x31, 0x03, 0x42
    # row 1 codes [1, 2, 7, 8, 9, 10, 11, 12] -> bytes 0x71, 0xB9, 0x82, 0xCA
    qcodes = np.array([[0xFA, 0x31, 0x03, 0x42], [0x71, 0xB9, 0x82, 0xCA]], dtype=np.uint8)
    # zeros [G=2][N/2=1]: group 0 -> (n0=5, n1=1) = 0x15 ; group 1 -> (n0=0, n1=9) = 0x90
    zeros = np.array([[0x15], [0x90]], dtype=np.uint8)
    scales = _f16([[0.5, 2.0], [0.25, 1.0]])   # [G][N]
    w = oracle.dequant_w4(qcodes, scales, zeros, 4, 2, 8)
    expected = np.array([[2.5, -1.0, 5.0, -2.5, 0.25, 0.5, 0.75, 1.0],
                         [0.0, 2.0, 12.0, 14.0, 0.0, 1.0, 2.0, 3.0]])
    np.testing.assert_array_equal(w, expected)


def test_w4_generator_packing_matches_layout():
    codes = np.arange(16, dtype=np.uint8)[None, :] % 16   # k = 0..15
    packed = inputs.pack_w4_codes(codes)
    assert list(packed[0]) == [0x20, 0x64, 0x31, 0x75, 0xA8, 0xEC, 0xB9, 0xFD]


def test_w4_zero_points_zero_scales_one_gives_codes():
    rng = np.random.default_rng(1)
    W = inputs.w4_weights(rng, 64, 256, 64)
    zeros = np.zeros_like(W.zeros)
    scales = np.ones_like(W.scales)
    w = oracle.dequant_w4(W.qcodes, scales, zeros, 64, 64, 256)
    np.testing.assert_array_equal(w, W.raw_codes.astype(np.float64))


def test_w4_dequant_is_exact_in_fp32():
    # (code - zero) is a 5-bit integer and the scale an 11-bit fp16 significand,
    # so the product needs at most 16 significant bits: float32 holds it exactly.
    rng = np.random.default_rng(2)
    W = inputs.w4_weights(rng, 32, 512, 64)
    w64 = oracle.dequant_w4(W.qcodes, W.scales, W.zeros, 64, 32, 512)
    np.testing.assert_array_equal(w64.astype(np.float32).astype(np.float64), w64)


def test_w8_dequant_hand_example():
    codes = np.array([[-127, 0, 5, 127], [1, -1, 64, -64]], dtype=np.int8)
    w = oracle.dequant_w8(codes, _f16([0.5, 0.125]), 0, 2, 4)
    np.testing.assert_array_equal(w, np.array([[-63.5, 0, 2.5, 63.5], [0.125, -0.125, 8, -8]]))
    wg = oracle.dequant_w8(codes, _f16([[1.0, 2.0], [0.5, 4.0]]), 2, 2, 4)
    np.testing.assert_array_equal(wg, np.array([[-127, 0, 2.5, 63.5], [2, -2, 256, -256]]))


def _brute_w4(qcodes, scales, zeros, g, xbits, T, N, K):
    x = oracle.bf16_bits_to_f64(xbits)  # widening only
    y = [[0.0] * N for _ in range(T)]
    for n in range(N):
        for k in range(K):
            r = k % 8
            pos = 4 * (r % 2) + r // 2          # nibble position inside the word
            byte = int(qcodes[n, (k // 8) * 4 + pos // 2])
            code = (byte >> 4) if pos % 2 else (byte & 0xF)
            zb = int(zeros[k // g, n // 2])
            zero = (zb >> 4) if (n & 1) else (zb & 0xF)
            w = (code - zero) * float(scales[k // g, n])
            for t in range(T):
                y[t][n] += float(x[t, k]) * w
    return np.array(y)


@pytest.mark.parametrize("T,N,K,g", [(3, 6, 16, 4), (2, 4, 128, 64), (1, 2, 64, 64)])
def test_w4_gemm_brute_force(T, N, K, g):
    rng = np.random.default_rng(10 + T + N)
    W = inputs.w4_weights(rng, N, K, g)
    xb = inputs.activations(rng, T, K)
    y = oracle.qgemm_w4a16(W.qcodes, W.scales, W.zeros, g, xb, T, N, K)
    yb = _brute_w4(W.qcodes, W.scales, W.zeros, g, xb, T, N, K)
    np.testing.assert_allclose(y, yb, rtol=1e-12, atol=1e-12)


def test_w4_gemm_integer_special_case_exact():
    # zero points 0, scales 1, integer activations: the GEMM is an exact integer product.
    rng = np.random.default_rng(3)
    T, N, K = 4, 16, 128
    W = inputs.w4_weights(rng, N, K, 64)
    xi = rng.integers(-8, 9, size=(T, K)).astype(np.float32)
    xb = inputs.f32_to_bf16_bits(xi)
    y = oracle.qgemm_w4a16(W.qcodes, np.ones_like(W.scales), np.zeros_like(W.zeros), 64, xb, T, N, K)
    exact = xi.astype(np.int64) @ W.raw_codes.astype(np.int64).T
    np.testing.assert_array_equal(y, exact.astype(np.float64))


def test_w8_gemm_brute_force():
    rng = np.random.default_rng(4)
    T, N, K = 2, 5, 16
    W = inputs.w8_weights(rng, N, K, 0)
    xb = inputs.activations(rng, T, K)
    x = oracle.bf16_bits_to_f64(xb)
    y = oracle.qgemm_w8a16(W.qcodes, W.scales, 0, xb, T, N, K)
    for t in range(T):
        for n in range(N):
            ref = sum(float(x[t, k]) * int(W.qcodes[n, k]) for k in range(K)) * float(W.scales[n])
            assert abs(y[t, n] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_w8_grouped_gemm_brute_force():
    rng = np.random.default_rng(5)
    T, N, K, g = 2, 4, 32, 8
    W = inputs.w8_weights(rng, N, K, g)
    xb = inputs.activations(rng, T, K)
    x = oracle.bf16_bits_to_f64(xb)
    y = oracle.qgemm_w8a16(W.qcodes, W.scales, g, xb, T, N, K)
    for t in range(T):
        for n in range(N):
            ref = sum(float(x[t, k]) * int(W.qcodes[n, k]) * float(W.scales[k // g, n])
                      for k in range(K))
            assert abs(y[t, n] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_gemm_transposed_operand_would_fail():
    # N != K/g so a transposed scale or zero layout cannot pass the brute force above;
    # here check that the layouts are not interchangeable on a non-square case.
    rng = np.random.default_rng(6)
    W = inputs.w4_weights(rng, 6, 16, 4)
    a = oracle.dequant_w4(W.qcodes, W.scales, W.zeros, 4, 6, 16)
    assert a.shape == (6, 16)
    assert not np.array_equal(a[:, :4], a[:, 4:8])
