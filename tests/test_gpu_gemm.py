"""GPU parity of the verify GEMMs against the fp64 oracle, through the C ABI.

Bar: max |y_gpu - y_oracle| <= 1e-2 * RMS(y_oracle) for fp32 outputs; bf16
outputs may additionally differ by their own rounding (half a bf16 ulp,
<= 2^-8 |y|).  Dequantised weights (fp32 export) are bit-exact.
"""
import numpy as np
import pytest

import oracle
import bit_qgemm_w4_gb300 as sv
from bit_qgemm_w4_gb300 import inputs
from tests.gpu_util import bf16_dev, dev, gemm_error_ratio, host

pytestmark = pytest.mark.gpu


# every test runs under both GEMM engines: one launch per GEMM (split) and
# the persistent launch (stack)
@pytest.fixture(scope="module", params=[sv.SPEC_GEMM_ENGINE_SPLIT, sv.SPEC_GEMM_ENGINE_STACK],
                ids=["split", "stack"])
def ctx(request):
    import torch  # noqa: F401
    from bit_qgemm_w4_gb300 import build
    build.build()
    c = sv.Context(0)
    sv.spec_set_gemm_engine(c, request.param)
    c.engine = request.param
    yield c
    c.close()


def _run_w4(ctx, W, xb, T, f32=True, signs=None, block=0):
    import torch
    y = torch.empty((T, W.N), dtype=torch.float32 if f32 else torch.bfloat16, device="cuda")
    sv.qgemm_w4a16(ctx, dev(W.qcodes), dev(W.scales), dev(W.zeros), W.group_size, bf16_dev(xb), y,
                   T, W.N, W.K, None if signs is None else dev(signs), block)
    sv.spec_sync_status(ctx)
    return host(y)


def _run_w8(ctx, W, xb, T, f32=True, signs=None, block=0):
    import torch
    y = torch.empty((T, W.N), dtype=torch.float32 if f32 else torch.bfloat16, device="cuda")
    sv.qgemm_w8a16(ctx, dev(W.qcodes), dev(W.scales), W.group_size, bf16_dev(xb), y, T, W.N, W.K,
                   None if signs is None else dev(signs), block)
    sv.spec_sync_status(ctx)
    return host(y)


W4_CASES = [
    # (T, N, K, g) -- Tiny config, ragged T, N not a multiple of 128, one stage, groups
    (16, 1024, 512, 64),
    (1, 1056, 768, 64),
    (5, 1056, 768, 64),
    (17, 1056, 768, 128),
    (32, 2048, 1024, 64),
    (33, 224, 1024, 256),
    (48, 512, 512, 64),
    (64, 1056, 640, 64),
    (16, 32, 64, 64),
    (16, 4096, 4096, 64),
]


@pytest.mark.parametrize("T,N,K,g", W4_CASES)
@pytest.mark.parametrize("f32", [True, False])
def test_w4_parity(ctx, T, N, K, g, f32):
    rng = np.random.default_rng(1000 + T * 7 + N + K + g)
    W = inputs.w4_weights(rng, N, K, g)
    xb = inputs.activations(rng, T, K)
    y = _run_w4(ctx, W, xb, T, f32)
    ref = oracle.qgemm_w4a16(W.qcodes, W.scales, W.zeros, g, xb, T, N, K)
    assert gemm_error_ratio(y, ref, not f32) <= 1.0


@pytest.mark.parametrize("T,N,K,g", [(32, 1024, 1024, 0), (16, 1064, 512, 0), (7, 256, 768, 128),
                                     (64, 128, 320, 64)])
@pytest.mark.parametrize("f32", [True, False])
def test_w8_parity(ctx, T, N, K, g, f32):
    rng = np.random.default_rng(2000 + T + N + K + g)
    W = inputs.w8_weights(rng, N, K, g)
    xb = inputs.activations(rng, T, K)
    y = _run_w8(ctx, W, xb, T, f32)
    ref = oracle.qgemm_w8a16(W.qcodes, W.scales, g, xb, T, N, K)
    assert gemm_error_ratio(y, ref, not f32) <= 1.0


@pytest.mark.parametrize("B,K", [(32, 512), (64, 512), (1024, 5120)])
def test_w8_with_rotation_parity(ctx, B, K):
    rng = np.random.default_rng(3000 + B)
    T, N = 32, 256
    W = inputs.w8_weights(rng, N, K, 0)
    xb = inputs.activations(rng, T, K)
    s = inputs.hadamard_signs(rng, K)
    y = _run_w8(ctx, W, xb, T, True, s, B)
    ref = oracle.qgemm_w8a16(W.qcodes, W.scales, 0, xb, T, N, K, s, B)
    assert gemm_error_ratio(y, ref, False) <= 1.0


def test_w4_with_rotation_parity(ctx):
    rng = np.random.default_rng(3100)
    T, N, K, B = 16, 512, 1024, 256
    W = inputs.w4_weights(rng, N, K, 64)
    xb = inputs.activations(rng, T, K)
    s = inputs.hadamard_signs(rng, K)
    y = _run_w4(ctx, W, xb, T, True, s, B)
    ref = oracle.qgemm_w4a16(W.qcodes, W.scales, W.zeros, 64, xb, T, N, K, s, B)
    assert gemm_error_ratio(y, ref, False) <= 1.0


@pytest.mark.parametrize("T", [16, 32])
def test_w4_block32_rotation_parity(ctx, T):
    # the smallest Hadamard block (32): one warp lane per element, no
    # in-register butterfly levels; ragged N and several 256-k stages
    rng = np.random.default_rng(3200 + T)
    N, K, B = 1056, 4096, 32
    W = inputs.w4_weights(rng, N, K, 64)
    xb = inputs.activations(rng, T, K)
    s = inputs.hadamard_signs(rng, K)
    for f32 in (True, False):
        y = _run_w4(ctx, W, xb, T, f32, s, B)
        ref = oracle.qgemm_w4a16(W.qcodes, W.scales, W.zeros, 64, xb, T, N, K, s, B)
        assert gemm_error_ratio(y, ref, not f32) <= 1.0


def test_w4_block32_rotation_full_size_sampled(ctx):
    # the 9B-class fused gate/up projection with the block-32 rotation
    rng = np.random.default_rng(3300)
    T, N, K, B = 32, 24576, 4096, 32
    W = inputs.w4_weights(rng, N, K, 64, keep_raw=False)
    xb = inputs.activations(rng, T, K)
    s = inputs.hadamard_signs(rng, K)
    y = _run_w4(ctx, W, xb, T, True, s, B)
    rows = np.sort(rng.choice(N // 2, size=64, replace=False))
    rows = np.stack([2 * rows, 2 * rows + 1], axis=1).reshape(-1)
    pairs = rows[0::2] // 2
    ref = oracle.qgemm_w4a16(W.qcodes[rows], W.scales[:, rows], W.zeros[:, pairs], 64, xb, T, len(rows), K,
                             s, B)
    assert np.isfinite(y).all()
    assert gemm_error_ratio(y[:, rows], ref, False) <= 1.0


def test_w4_integer_special_case_is_exact(ctx):
    # zero points 0, scales 1, small integer activations: every partial sum
    # is an integer below 2^24, so the GPU result must be exact.
    rng = np.random.default_rng(5)
    T, N, K = 16, 256, 1024
    W = inputs.w4_weights(rng, N, K, 64)
    W.zeros[:] = 0
    W.scales[:] = 1.0
    xi = rng.integers(-8, 9, size=(T, K)).astype(np.float32)
    xb = inputs.f32_to_bf16_bits(xi)
    y = _run_w4(ctx, W, xb, T, True)
    exact = xi.astype(np.int64) @ W.raw_codes.astype(np.int64).T
    np.testing.assert_array_equal(y, exact.astype(np.float64))


def test_counters_and_slots_reset_between_calls(ctx):
    # Split tiles are summed in a shared fp32 slot that the CTA finishing the
    # tile clears; a different shape in between must not see stale sums.
    rng = np.random.default_rng(6)
    A = inputs.w4_weights(rng, 2048, 2048, 64)
    B = inputs.w4_weights(rng, 1056, 768, 64)
    xa = inputs.activations(rng, 16, 2048)
    xb = inputs.activations(rng, 32, 768)
    refa = oracle.qgemm_w4a16(A.qcodes, A.scales, A.zeros, 64, xa, 16, 2048, 2048)
    refb = oracle.qgemm_w4a16(B.qcodes, B.scales, B.zeros, 64, xb, 32, 1056, 768)
    for _ in range(3):
        assert gemm_error_ratio(_run_w4(ctx, A, xa, 16), refa, False) <= 1.0
        assert gemm_error_ratio(_run_w4(ctx, B, xb, 32), refb, False) <= 1.0


def test_dequant_export_bit_exact(ctx):
    import torch
    rng = np.random.default_rng(7)
    N, K = 96, 256
    W = inputs.w4_weights(rng, N, K, 64)
    w = torch.empty((N, K), dtype=torch.float32, device="cuda")
    sv.qdequant_w4(ctx, dev(W.qcodes), dev(W.scales), dev(W.zeros), 64, N, K, w)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(w), oracle.dequant_w4(W.qcodes, W.scales, W.zeros, 64, N, K))
    for g in (0, 64):
        W8 = inputs.w8_weights(rng, N, K, g)
        sv.qdequant_w8(ctx, dev(W8.qcodes), dev(W8.scales), g, N, K, w)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host(w), oracle.dequant_w8(W8.qcodes, W8.scales, g, N, K))


@pytest.mark.parametrize("T,N,K,g", [(0, 128, 64, 64), (65, 128, 64, 64), (16, 100, 64, 64),
                                     (16, 128, 96, 64), (16, 128, 128, 32)])
def test_bad_shapes_rejected(ctx, T, N, K, g):
    import torch
    buf = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(sv.SpecError) as e:
        sv.qgemm_w4a16(ctx, buf, buf, buf, g, buf, buf, T, N, K)
    assert e.value.status == -2


# ----------------------------------------------------------------------------
# full-size layers in the benchmark's launch configuration, sampled rows
# ----------------------------------------------------------------------------

def _w4_rows(W, rows):
    """Sub-checkpoint holding only output rows `rows` (even/odd pairs)."""
    pairs = rows[0::2] // 2
    sub = inputs.W4Weights(len(rows), W.K, W.group_size, W.qcodes[rows], W.scales[:, rows],
                           W.zeros[:, pairs], None, None)
    return sub


def _sample_pairs(rng, N, n_pairs=64):
    p = np.sort(rng.choice(N // 2, size=n_pairs, replace=False))
    return np.stack([2 * p, 2 * p + 1], axis=1).reshape(-1)


@pytest.mark.parametrize("T,N,K", [(16, 6144, 4096), (32, 24576, 4096), (16, 4096, 12288),
                                   (32, 4096, 12288), (32, 151936, 4096)])
@pytest.mark.parametrize("f32", [True, False])
def test_w4_full_size_sampled(ctx, T, N, K, f32):
    rng = np.random.default_rng(4000 + N + T)
    W = inputs.w4_weights(rng, N, K, 64, keep_raw=False)
    xb = inputs.activations(rng, T, K)
    y = _run_w4(ctx, W, xb, T, f32)
    rows = _sample_pairs(rng, N)
    S = _w4_rows(W, rows)
    ref = oracle.qgemm_w4a16(S.qcodes, S.scales, S.zeros, 64, xb, T, len(rows), K)
    assert gemm_error_ratio(y[:, rows], ref, not f32) <= 1.0


@pytest.mark.parametrize("N,K", [(34816, 5120), (5120, 17408)])
@pytest.mark.parametrize("f32", [True, False])
def test_w8_rotated_full_size_sampled(ctx, N, K, f32):
    # the 27B-class gate_up (K = 5 rotation blocks) and down projection
    # (K = 17408 = 17 blocks of 1024, the only odd block count)
    rng = np.random.default_rng(4500 + K)
    T, B = 32, 1024
    W = inputs.w8_weights(rng, N, K, 0)
    xb = inputs.activations(rng, T, K)
    s = inputs.hadamard_signs(rng, K)
    y = _run_w8(ctx, W, xb, T, f32, s, B)
    rows = np.sort(rng.choice(N, size=128, replace=False))
    ref = oracle.qgemm_w8a16(W.qcodes[rows], W.scales[rows], 0, xb, T, len(rows), K, s, B)
    assert gemm_error_ratio(y[:, rows], ref, not f32) <= 1.0
