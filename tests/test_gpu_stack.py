"""GPU parity of GEMM stacks (qgemm_stack_*, one persistent launch for a list
of GEMMs) against the fp64 oracle, through the C ABI.

Bar as for single GEMMs: max |y_gpu - y_oracle| <= 1e-2 * RMS(y_oracle) for
fp32 outputs, plus half a bf16 ulp of y for bf16 outputs.
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


def _w4_desc(W, x, y, T, wait_prev=1):
    return {"quant": sv.SPEC_QUANT_W4, "qcodes": dev(W.qcodes), "scales": dev(W.scales),
            "zeros": dev(W.zeros), "group_size": W.group_size, "x": x, "y": y, "T": T, "N": W.N,
            "K": W.K, "wait_prev": wait_prev}


def _w8_desc(W, x, y, T, signs=None, block=0, wait_prev=1):
    return {"quant": sv.SPEC_QUANT_W8, "qcodes": dev(W.qcodes), "scales": dev(W.scales),
            "zeros": None, "group_size": W.group_size, "x": x, "y": y, "T": T, "N": W.N, "K": W.K,
            "signs": None if signs is None else dev(signs), "hadamard_block": block,
            "wait_prev": wait_prev}


# (N, K, g, wait_prev): ragged N, one-stage K, partial last stage, grouped
# scales, independent neighbours (wait_prev = 0) and dependent ones
STACK_W4 = [(1056, 768, 64, 1), (2048, 1024, 64, 0), (224, 1024, 256, 0), (512, 512, 64, 1),
            (4096, 4096, 64, 1), (32, 64, 64, 0), (1024, 640, 64, 1)]


@pytest.mark.parametrize("T", [1, 16, 32, 33])
@pytest.mark.parametrize("f32", [True, False])
def test_w4_stack_parity(ctx, T, f32):
    import torch
    rng = np.random.default_rng(7000 + T)
    keep, descs = [], []
    for N, K, g, wp in STACK_W4:
        W = inputs.w4_weights(rng, N, K, g)
        xb = inputs.activations(rng, T, K)
        y = torch.full((T, N), float("nan"), dtype=torch.float32 if f32 else torch.bfloat16, device="cuda")
        d = _w4_desc(W, bf16_dev(xb), y, T, wp)
        keep.append((W, xb, y, d))
        descs.append(d)
    st = sv.GemmStack(ctx, descs)
    for _ in range(2):   # a second run reuses the counters the first one reset
        st.run()
        sv.spec_sync_status(ctx)
        for W, xb, y, _ in keep:
            ref = oracle.qgemm_w4a16(W.qcodes, W.scales, W.zeros, W.group_size, xb, T, W.N, W.K)
            assert gemm_error_ratio(host(y), ref, not f32) <= 1.0
    st.close()


def _gather_weights(rng, N, K):
    """int4 weights whose rows each hold one code in {1, 2} (zero points 0,
    scales 1): y[t][n] = c_n * x[t][k_n], exact in every format on the path."""
    W = inputs.w4_weights(rng, N, K, 64)
    codes = np.zeros((N, K), dtype=np.uint8)
    codes[np.arange(N), rng.integers(0, K, size=N)] = rng.integers(1, 3, size=N)
    W.raw_codes = codes
    W.qcodes[:] = inputs.pack_w4_codes(codes)
    W.zeros[:] = 0
    W.scales[:] = 1.0
    return W


def test_w4_stack_dependent_chain(ctx):
    # every GEMM reads the previous one's bf16 output: the stack must not
    # load a GEMM's activations before its predecessor has written all of
    # them.  The data keeps every value an exact small integer, so the chain
    # must equal the oracle's chain exactly.
    import torch
    rng = np.random.default_rng(7100)
    T, dims = 32, [1024, 2048, 512, 4096, 1024, 1536]
    Ws = [_gather_weights(rng, dims[i + 1], dims[i]) for i in range(len(dims) - 1)]
    x0 = inputs.f32_to_bf16_bits(rng.integers(-2, 3, size=(T, dims[0])).astype(np.float32))
    bufs = [bf16_dev(x0)] + [torch.full((T, n), float("nan"), dtype=torch.bfloat16, device="cuda")
                             for n in dims[1:]]
    descs = [_w4_desc(W, bufs[i], bufs[i + 1], T, 1) for i, W in enumerate(Ws)]
    st = sv.GemmStack(ctx, descs)
    for rep in range(3):
        for b in bufs[1:]:
            b.fill_(float("nan"))
        st.run()
        sv.spec_sync_status(ctx)
        xb = x0
        for i, W in enumerate(Ws):
            ref = oracle.qgemm_w4a16(W.qcodes, W.scales, W.zeros, 64, xb, T, W.N, W.K)
            assert np.abs(ref).max() <= 256          # exact in bf16
            np.testing.assert_array_equal(host(bufs[i + 1]), ref, err_msg=f"rep {rep} gemm {i}")
            xb = inputs.f32_to_bf16_bits(ref.astype(np.float32))
    st.close()


def test_w8_stack_rotated_chain(ctx):
    # rotated int8 GEMMs in a dependent chain share the rotation scratch;
    # each GEMM is held to the bar on the input it read (the previous
    # GEMM's bf16 output), so that one GEMM's allowed error is not charged
    # to the next
    import torch
    rng = np.random.default_rng(7200)
    T, B, dims = 32, 1024, [2048, 3072, 1024, 2048]
    Ws = [inputs.w8_weights(rng, dims[i + 1], dims[i], 0) for i in range(len(dims) - 1)]
    ss = [inputs.hadamard_signs(rng, dims[i]) for i in range(len(dims) - 1)]
    x0 = inputs.activations(rng, T, dims[0])
    bufs = [bf16_dev(x0)] + [torch.full((T, n), float("nan"), dtype=torch.bfloat16, device="cuda")
                             for n in dims[1:]]
    descs = [_w8_desc(W, bufs[i], bufs[i + 1], T, ss[i], B, 1) for i, W in enumerate(Ws)]
    st = sv.GemmStack(ctx, descs)
    for rep in range(2):
        st.run()
        sv.spec_sync_status(ctx)
        xb = x0
        for i, W in enumerate(Ws):
            ref = oracle.qgemm_w8a16(W.qcodes, W.scales, 0, xb, T, W.N, W.K, ss[i], B)
            y = host(bufs[i + 1])
            assert gemm_error_ratio(y, ref, True) <= 1.0, (rep, i)
            xb = inputs.f32_to_bf16_bits(y.astype(np.float32))
    st.close()


def _sample_pairs(rng, N, n_pairs=64):
    p = np.sort(rng.choice(N // 2, size=n_pairs, replace=False))
    return np.stack([2 * p, 2 * p + 1], axis=1).reshape(-1)


def _w4_rows(W, rows):
    pairs = rows[0::2] // 2
    return inputs.W4Weights(len(rows), W.K, W.group_size, W.qcodes[rows], W.scales[:, rows],
                            W.zeros[:, pairs], None, None)


@pytest.mark.parametrize("T", [16, 32])
def test_w4_stack_9b_layer_full_size_sampled(ctx, T):
    # one 9B-class layer (fused qkv, o, fused gate_up, down) plus the LM head
    # with fp32 logits, as the benchmark's verify step launches them
    import torch
    rng = np.random.default_rng(7300 + T)
    shapes = [(K, N) for _, K, N in inputs.LAYER_9B] + [(4096, inputs.VOCAB_9B)]
    keep, descs = [], []
    for i, (K, N) in enumerate(shapes):
        W = inputs.w4_weights(rng, N, K, 64, keep_raw=False)
        xb = inputs.activations(rng, T, K)
        f32 = i == len(shapes) - 1
        y = torch.full((T, N), float("nan"), dtype=torch.float32 if f32 else torch.bfloat16, device="cuda")
        d = _w4_desc(W, bf16_dev(xb), y, T, 1)
        keep.append((W, xb, y, f32))
        descs.append(d)
    st = sv.GemmStack(ctx, descs)
    st.run()
    sv.spec_sync_status(ctx)
    for W, xb, y, f32 in keep:
        rows = _sample_pairs(rng, W.N)
        S = _w4_rows(W, rows)
        ref = oracle.qgemm_w4a16(S.qcodes, S.scales, S.zeros, 64, xb, T, len(rows), W.K)
        got = host(y)
        assert np.isfinite(got).all()
        assert gemm_error_ratio(got[:, rows], ref, not f32) <= 1.0
    st.close()


def test_w8_stack_27b_layer_full_size_sampled(ctx):
    # one 27B-class int8 layer with the block-1024 rotation (K = 5120 and the
    # down projection's 17408 = 17 blocks)
    import torch
    rng = np.random.default_rng(7400)
    T, B = 32, 1024
    keep, descs = [], []
    for _, K, N in inputs.LAYER_27B:
        W = inputs.w8_weights(rng, N, K, 0)
        xb = inputs.activations(rng, T, K)
        s = inputs.hadamard_signs(rng, K)
        y = torch.full((T, N), float("nan"), dtype=torch.float32, device="cuda")
        descs.append(_w8_desc(W, bf16_dev(xb), y, T, s, B, 1))
        keep.append((W, xb, s, y))
    st = sv.GemmStack(ctx, descs)
    st.run()
    sv.spec_sync_status(ctx)
    for W, xb, s, y in keep:
        rows = np.sort(rng.choice(W.N, size=128, replace=False))
        ref = oracle.qgemm_w8a16(W.qcodes[rows], W.scales[rows], 0, xb, T, len(rows), W.K, s, B)
        got = host(y)
        assert np.isfinite(got).all()
        assert gemm_error_ratio(got[:, rows], ref, False) <= 1.0
    st.close()


def test_stack_rules_rejected(ctx):
    import torch
    rng = np.random.default_rng(7500)
    W = inputs.w4_weights(rng, 256, 512, 64)
    x = bf16_dev(inputs.activations(rng, 16, 512))
    y = torch.empty((16, 256), dtype=torch.bfloat16, device="cuda")
    # four consecutive entries without wait_prev after the first
    with pytest.raises(sv.SpecError) as e:
        sv.GemmStack(ctx, [_w4_desc(W, x, y, 16, 1)] + [_w4_desc(W, x, y, 16, 0)] * 4)
    assert e.value.status == -1
    # mixed quant
    W8 = inputs.w8_weights(rng, 256, 512, 0)
    with pytest.raises(sv.SpecError) as e:
        sv.GemmStack(ctx, [_w4_desc(W, x, y, 16), _w8_desc(W8, x, y, 16)])
    assert e.value.status == -1
    # a bad shape inside the list
    with pytest.raises(sv.SpecError) as e:
        sv.GemmStack(ctx, [_w4_desc(W, x, y, 16), dict(_w4_desc(W, x, y, 16), K=96)])
    assert e.value.status == -2
