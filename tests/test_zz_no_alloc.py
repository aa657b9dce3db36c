"""spec_accept_noalloc: the context-free acceptance entry point whose scratch is
static device memory.  Through the C ABI it must give exactly what spec_accept
gives (same kernels, same arithmetic) on two calls in a row, reject T beyond
its scratch, and report an out-of-range draft token in device_status.

This file is collected last on purpose: it must pass in a fresh process and
after every other GPU test.
"""
import numpy as np
import pytest

import bit_qgemm_w4_gb300 as sv
from bit_qgemm_w4_gb300 import inputs
from tests.gpu_util import dev, host

pytestmark = pytest.mark.gpu

SPEC_ERR_SHAPE = -2


@pytest.fixture(scope="module")
def ctx():
    from bit_qgemm_w4_gb300 import build
    build.build()
    c = sv.Context(0)
    yield c
    c.close()


def _buffers(T):
    import torch
    n = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    toks = torch.full((T + 1,), -1, dtype=torch.int32, device="cuda")
    flags = torch.full((T + 1,), -1, dtype=torch.int32, device="cuda")
    return n, toks, flags


def _device_inputs(a):
    T, V = a.T, a.V
    q = dev(a.q) if T > 0 else dev(np.zeros((1, V), np.float32))
    d = dev(a.drafts) if T > 0 else dev(np.zeros(1, np.int32))
    return dev(a.logits), q, d, dev(a.u)


def _result(n, toks, flags):
    k = int(host(n)[0])
    return k, list(host(toks)[:k + 1]), list(host(flags))


@pytest.mark.parametrize("T,V,alpha,noise", [(0, 1000, 1.0, 1.0), (16, 1000, 1.0, 0.5),
                                             (32, 151936, 1.0, 0.25), (64, 151936, 1.0, 0.1),
                                             (64, 4096, 0.2, 2.0)])
def test_matches_spec_accept_twice(ctx, T, V, alpha, noise):
    import torch
    rng = np.random.default_rng(7000 + T + V)
    a = inputs.accept_inputs(rng, T, V, logit_std=3.0, alpha=alpha, noise_std=noise)
    logits, q, d, u = _device_inputs(a)

    n0, t0, f0 = _buffers(T)
    sv.spec_accept(ctx, logits, q, d, u, T, V, n0, t0, f0)
    sv.spec_sync_status(ctx)
    ref = _result(n0, t0, f0)

    # two calls in a row on the same stream, no synchronisation between them
    bufs = [_buffers(T) for _ in range(2)]
    status = [torch.full((1,), -1, dtype=torch.int32, device="cuda") for _ in range(2)]
    for (n, t, f), st in zip(bufs, status):
        sv.spec_accept_noalloc(logits, q, d, u, T, V, n, t, f, st)
    torch.cuda.synchronize()
    for (n, t, f), st in zip(bufs, status):
        assert _result(n, t, f) == ref
        assert int(host(st)[0]) == 0


def test_rejects_t_beyond_static_scratch():
    import torch
    from bit_qgemm_w4_gb300 import build
    build.build()
    T, V = 65, 1000
    a = inputs.accept_inputs(np.random.default_rng(1), T, V)
    logits, q, d, u = _device_inputs(a)
    n, t, f = _buffers(T)
    with pytest.raises(sv.SpecError) as e:
        sv.spec_accept_noalloc(logits, q, d, u, T, V, n, t, f)
    assert e.value.status == SPEC_ERR_SHAPE
    assert "at most 64" in str(e.value)
    torch.cuda.synchronize()
    assert int(host(n)[0]) == -1          # nothing was launched


def test_out_of_range_draft_reported(ctx):
    import torch
    T, V = 8, 1000
    a = inputs.accept_inputs(np.random.default_rng(3), T, V, logit_std=3.0, alpha=1.0, noise_std=0.05)
    drafts = a.drafts.copy()
    drafts[0] = V + 5                      # rejected at position 0, recorded as error 2
    logits, q, _, u = _device_inputs(a)
    d = dev(drafts)

    n0, t0, f0 = _buffers(T)
    sv.spec_accept(ctx, logits, q, d, u, T, V, n0, t0, f0)
    with pytest.raises(sv.SpecError):
        sv.spec_sync_status(ctx)
    ref = _result(n0, t0, f0)
    assert ref[0] == 0

    n, t, f = _buffers(T)
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    sv.spec_accept_noalloc(logits, q, d, u, T, V, n, t, f, st)
    torch.cuda.synchronize()
    assert _result(n, t, f) == ref
    assert int(host(st)[0]) == 2

    # the next call starts from a cleared error word
    a2 = inputs.accept_inputs(np.random.default_rng(4), T, V)
    logits2, q2, d2, u2 = _device_inputs(a2)
    sv.spec_accept_noalloc(logits2, q2, d2, u2, T, V, n, t, f, st)
    torch.cuda.synchronize()
    assert int(host(st)[0]) == 0
