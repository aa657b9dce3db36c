"""Pins for the oracle's random Hadamard transform (CPU only).

The source ("Karpathy's Trick for Faster Local LLMs Finally Has Proper
Tooling", section "How Uzu optimizes bytes and tokens per pass") fixes: +1/-1
entries with one overall scale, random sign flips before the mixing, block
diagonal, exactly reversible.  Checked here against orthogonality, scipy's
Sylvester construction, unit vectors, norm preservation, the inverse and the
weight-rotation invariance.
"""
import math

import numpy as np
import pytest
import scipy.linalg

import oracle
from bit_qgemm_w4_gb300 import inputs


@pytest.mark.parametrize("B", [1, 2, 4, 8, 32, 64, 256, 1024])
def test_hadamard_orthogonal_and_sylvester(B):
    H = oracle.hadamard(B)
    assert set(np.unique(H)) <= {-1.0, 1.0}
    np.testing.assert_array_equal(H @ H.T, B * np.eye(B))
    np.testing.assert_array_equal(H, scipy.linalg.hadamard(B).astype(np.float64))


@pytest.mark.parametrize("B", [2, 8, 32])
def test_hadamard_entries_by_popcount(B):
    H = oracle.hadamard(B)
    for i in range(B):
        for j in range(B):
            assert H[i, j] == (-1.0) ** bin(i & j).count("1")


@pytest.mark.parametrize("B", [32, 64])
def test_rht_unit_vectors_give_signed_columns(B):
    rng = np.random.default_rng(0)
    s = inputs.hadamard_signs(rng, 2 * B)
    H = scipy.linalg.hadamard(B)
    for j in [0, 1, B - 1, B, 2 * B - 1]:
        e = np.zeros((1, 2 * B))
        e[0, j] = 1.0
        out = oracle.rht(e, s, B)
        expect = np.zeros(2 * B)
        blk = j // B
        expect[blk * B:(blk + 1) * B] = H[:, j % B] * s[j] / math.sqrt(B)
        np.testing.assert_allclose(out[0], expect, atol=1e-15)


def test_rht_norm_inverse_and_invariance():
    rng = np.random.default_rng(1)
    T, K, B, N = 3, 5 * 64, 64, 7
    s = inputs.hadamard_signs(rng, K)
    x = rng.standard_normal((T, K))
    xr = oracle.rht(x, s, B)
    np.testing.assert_allclose(np.linalg.norm(xr, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    # inverse: x = diag(s) H^T xr / sqrt(B) per block
    H = scipy.linalg.hadamard(B) / math.sqrt(B)
    back = np.empty_like(xr)
    for b in range(K // B):
        c = slice(b * B, (b + 1) * B)
        back[:, c] = (xr[:, c] @ H) * s[c]
    np.testing.assert_allclose(back, x, atol=1e-12)
    # (W R^T)(R x) = W x
    W = rng.standard_normal((N, K))
    WRt = oracle.rht(W, s, B)  # rows of W rotated = W R^T
    np.testing.assert_allclose(xr @ WRt.T, x @ W.T, atol=1e-10)


def test_rht_signs_applied_before_mixing():
    # Block of 2: H = [[1,1],[1,-1]]/sqrt2.  x = (1, 0), s = (-1, +1):
    # signs first -> (-1, 0) -> (-1, -1)/sqrt2.  Mixing first would give
    # (1, 1)/sqrt2 * s = (-1, 1)/sqrt2.
    out = oracle.rht(np.array([[1.0, 0.0]]), np.array([-1, 1], dtype=np.int8), 2)
    np.testing.assert_allclose(out[0], np.array([-1.0, -1.0]) / math.sqrt(2), atol=1e-15)


def test_rht_gemm_matches_rotated_activations():
    rng = np.random.default_rng(2)
    T, N, K, B = 2, 4, 128, 64
    W = inputs.w8_weights(rng, N, K, 0)
    xb = inputs.activations(rng, T, K)
    s = inputs.hadamard_signs(rng, K)
    y = oracle.qgemm_w8a16(W.qcodes, W.scales, 0, xb, T, N, K, s, B)
    x = oracle.bf16_bits_to_f64(xb)
    xr = oracle.rht(x, s, B)
    ref = xr @ (W.qcodes.astype(np.float64) * W.scales.astype(np.float64)[:, None]).T
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
