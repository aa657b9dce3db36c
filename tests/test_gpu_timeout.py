"""The GEMMs' bounded-wait failure path on the GPU.

The test hook spec_test_stall makes CTA 0 of the next GEMM launch skip the
weight copy of one stage (nothing ever completes that stage's barrier) and
shortens every wait to a few milliseconds.  The kernel must record
SPEC_ERR_TIMEOUT, drain its copies and MMAs, free its tensor memory and
return; spec_sync_status reports the error and resets the workspace, and the
next GEMM on the same context must match the oracle again.
"""
import numpy as np
import pytest

import oracle
import bit_qgemm_w4_gb300 as sv
from bit_qgemm_w4_gb300 import inputs
from tests.gpu_util import bf16_dev, dev, gemm_error_ratio, host

pytestmark = pytest.mark.gpu

SPEC_ERR_TIMEOUT = -6


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


def _gemm(ctx, W, xb, T):
    import torch
    y = torch.empty((T, W.N), dtype=torch.float32, device="cuda")
    sv.qgemm_w4a16(ctx, dev(W.qcodes), dev(W.scales), dev(W.zeros), W.group_size, bf16_dev(xb), y,
                   T, W.N, W.K)
    return y


@pytest.mark.parametrize("skip_unit", [0, 3])
def test_single_gemm_wait_runs_out_and_context_recovers(ctx, skip_unit):
    rng = np.random.default_rng(8000 + skip_unit)
    # 1024 stages over at most 152 CTAs: CTA 0 owns at least six of them
    T, N, K = 32, 8192, 4096
    W = inputs.w4_weights(rng, N, K, 64)
    xb = inputs.activations(rng, T, K)
    ref = oracle.qgemm_w4a16(W.qcodes, W.scales, W.zeros, 64, xb, T, N, K)
    sv.spec_test_stall(ctx, skip_unit, 5_000_000)   # 5 ms
    _gemm(ctx, W, xb, T)
    with pytest.raises(sv.SpecError) as e:
        sv.spec_sync_status(ctx)
    assert e.value.status == SPEC_ERR_TIMEOUT
    # the hook applied to one launch only; the context works again
    for _ in range(2):
        y = _gemm(ctx, W, xb, T)
        sv.spec_sync_status(ctx)
        assert gemm_error_ratio(host(y), ref, False) <= 1.0


def test_stack_wait_runs_out_and_context_recovers(ctx):
    # stack engine: a stalled CTA also leaves the other CTAs waiting at the
    # next GEMM's dependency gate, and the grid-wide abort flag releases
    # them; split engine: the hook stalls the first GEMM's launch, the
    # later launches run to their end
    import torch
    rng = np.random.default_rng(8100)
    T, dims = 16, [1024, 2048, 1024, 2048]
    Ws = [inputs.w4_weights(rng, dims[i + 1], dims[i], 64) for i in range(3)]
    xs = [inputs.activations(rng, T, dims[i]) for i in range(3)]
    ys = [torch.empty((T, dims[i + 1]), dtype=torch.float32, device="cuda") for i in range(3)]
    descs = [{"quant": sv.SPEC_QUANT_W4, "qcodes": dev(W.qcodes), "scales": dev(W.scales),
              "zeros": dev(W.zeros), "group_size": 64, "x": bf16_dev(x), "y": y, "T": T, "N": W.N,
              "K": W.K, "wait_prev": 1} for W, x, y in zip(Ws, xs, ys)]
    st = sv.GemmStack(ctx, descs)
    # a stage CTA 0 owns: the split engine's first launch gives it one
    skip = 0 if ctx.engine == sv.SPEC_GEMM_ENGINE_SPLIT else 1
    sv.spec_test_stall(ctx, skip, 5_000_000)
    st.run()
    with pytest.raises(sv.SpecError) as e:
        sv.spec_sync_status(ctx)
    assert e.value.status == SPEC_ERR_TIMEOUT
    st.run()
    sv.spec_sync_status(ctx)
    for W, x, y in zip(Ws, xs, ys):
        ref = oracle.qgemm_w4a16(W.qcodes, W.scales, W.zeros, 64, x, T, W.N, W.K)
        assert gemm_error_ratio(host(y), ref, False) <= 1.0
    st.close()


def test_stall_hook_arguments_checked(ctx):
    with pytest.raises(sv.SpecError):
        sv.spec_test_stall(ctx, -2, 5_000_000)
    with pytest.raises(sv.SpecError):
        sv.spec_test_stall(ctx, 0, 10)
