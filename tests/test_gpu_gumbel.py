"""GPU parity of shared-seed (Gumbel-max) sampling and acceptance against the
oracle, through the C ABI.

Bars (the kernel decides each argmax in fp32, the oracle in fp64):
* a row's token equals the oracle's wherever the oracle's margin (best value
  minus the runner-up) is at least 1e-4; below that, the GPU's token must be
  one whose oracle value lies within 1e-4 of the best;
* near-tie flags agree wherever the oracle's margin is not within 2e-5 of the
  1e-4 bound;
* accepted lengths and tokens are bit-exact unless a row up to the emitted one
  is a near tie (counted separately).
"""
import numpy as np
import pytest

import oracle
import bit_qgemm_w4_gb300 as sv
from tests.gpu_util import dev, host

pytestmark = pytest.mark.gpu
EPS = 1e-4
SPEC_ERR_SHAPE = -2


@pytest.fixture(scope="module")
def ctx():
    from bit_qgemm_w4_gb300 import build
    build.build()
    c = sv.Context(0)
    yield c
    c.close()


def _positions(pos, R):
    return [(pos + r) % (1 << 64) for r in range(R)]


def _gpu_sample(ctx, logits_dev, R, V, seed, pos):
    import torch
    toks = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    flags = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    sv.spec_gumbel_sample(ctx, logits_dev, R, V, seed, pos, toks, flags)
    sv.spec_sync_status(ctx)
    return host(toks).astype(np.int64), host(flags)


def _check_rows(logits, seed, pos, toks_g, flags_g):
    R, V = logits.shape
    toks_o, margins = oracle.gumbel_sample(logits, seed, _positions(pos, R))
    ties = 0
    for r in range(R):
        if margins[r] >= EPS:
            assert toks_g[r] == toks_o[r], (r, toks_g[r], toks_o[r], margins[r])
        else:
            ties += 1
            z = logits[r].astype(np.float64) - np.log(-np.log(
                oracle.gumbel_uniforms(seed, (pos + r) % (1 << 64), V)))
            assert z[toks_g[r]] >= z.max() - EPS
        if abs(margins[r] - EPS) > 2e-5:
            assert flags_g[r] == int(margins[r] < EPS), (r, flags_g[r], margins[r])
    return ties


@pytest.mark.parametrize("R,V", [(1, 1), (3, 10), (17, 1000), (33, 151936), (5, 4099), (257, 1000)])
def test_sample_parity(ctx, R, V):
    rng = np.random.default_rng(100 + R + V)
    logits = (rng.standard_normal((R, V)) * 3).astype(np.float32)
    seed, pos = 0xDEADBEEF12345678, (1 << 32) - 3       # positions cross into the high word
    toks, flags = _gpu_sample(ctx, dev(logits), R, V, seed, pos)
    assert _check_rows(logits, seed, pos, toks, flags) <= max(1, R // 50)


def test_sample_unaligned_rows_and_masked_tokens(ctx):
    import torch
    rng = np.random.default_rng(7)
    R, V = 6, 1000
    logits = (rng.standard_normal((R, V)) * 3).astype(np.float32)
    logits[:, ::2] = -np.inf                             # masked vocabulary entries
    buf = torch.zeros(R * V + 1, dtype=torch.float32, device="cuda")
    buf[1:] = torch.from_numpy(logits.reshape(-1)).cuda()
    toks, flags = _gpu_sample(ctx, buf[1:], R, V, 77, 5)   # rows 4 bytes off 16-byte alignment
    assert np.all(toks % 2 == 1)
    _check_rows(logits, 77, 5, toks, flags)


def _accept_case(rng, T, V, kind):
    logits = (rng.standard_normal((T + 1, V)) * 3).astype(np.float32)
    if kind == "match":
        draft_logits = logits[:T]
    else:
        draft_logits = (logits[:T] + rng.standard_normal((T, V)) * 0.5).astype(np.float32)
    return logits, draft_logits


@pytest.mark.parametrize("T,V,kind", [(0, 1000, "noisy"), (8, 1000, "noisy"), (16, 1000, "match"),
                                      (32, 151936, "noisy"), (32, 151936, "match"),
                                      (64, 4096, "noisy"), (256, 1000, "match")])
def test_accept_parity(ctx, T, V, kind):
    import torch
    rng = np.random.default_rng(900 + T + V)
    seed, pos = 31337 + T, 123456789 + 1000 * T
    logits, draft_logits = _accept_case(rng, T, V, kind)
    drafts = (oracle.gumbel_sample(draft_logits, seed, _positions(pos, T))[0]
              if T > 0 else np.zeros(0, np.int64)).astype(np.int32)
    n_o, toks_o, near_o = oracle.spec_accept_gumbel(logits, drafts, seed, pos)
    if kind == "match":
        assert n_o == T

    n = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    toks = torch.full((T + 1,), -1, dtype=torch.int32, device="cuda")
    flags = torch.full((T + 1,), -1, dtype=torch.int32, device="cuda")
    d = dev(drafts) if T > 0 else None
    sv.spec_accept_gumbel(ctx, dev(logits), d, T, V, seed, pos, n, toks, flags)
    sv.spec_sync_status(ctx)
    k = int(host(n)[0])
    if near_o[:n_o + 1].any():
        pytest.skip("near tie among the deciding rows")
    assert k == n_o
    assert list(host(toks)[:k + 1]) == list(toks_o)


def test_drafter_and_verifier_on_gpu_agree_when_distributions_match(ctx):
    import torch
    rng = np.random.default_rng(11)
    T, V, seed, pos = 32, 151936, 2024, 50
    logits = dev((rng.standard_normal((T + 1, V)) * 3).astype(np.float32))
    drafts = torch.full((T,), -1, dtype=torch.int32, device="cuda")
    sv.spec_gumbel_sample(ctx, logits, T, V, seed, pos, drafts)
    n = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    toks = torch.full((T + 1,), -1, dtype=torch.int32, device="cuda")
    sv.spec_accept_gumbel(ctx, logits, drafts, T, V, seed, pos, n, toks)
    sv.spec_sync_status(ctx)
    assert int(host(n)[0]) == T
    assert list(host(toks)[:T]) == list(host(drafts))


def test_out_of_range_draft_reported(ctx):
    import torch
    rng = np.random.default_rng(12)
    T, V, seed = 6, 500, 3
    logits = (rng.standard_normal((T + 1, V)) * 3).astype(np.float32)
    y, margins = oracle.gumbel_sample(logits, seed, _positions(0, T + 1))
    assert margins.min() >= EPS
    drafts = y[:T].astype(np.int32)
    drafts[3] = V + 1
    n = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    toks = torch.full((T + 1,), -1, dtype=torch.int32, device="cuda")
    sv.spec_accept_gumbel(ctx, dev(logits), dev(drafts), T, V, seed, 0, n, toks)
    with pytest.raises(sv.SpecError):
        sv.spec_sync_status(ctx)
    assert int(host(n)[0]) == 3
    assert list(host(toks)[:4]) == [int(v) for v in y[:4]]


@pytest.mark.parametrize("rows,T,V", [(0, 0, 10), (258, 0, 10), (1, -1, 10), (1, 257, 10), (1, 1, 0)])
def test_bad_shapes_rejected(ctx, rows, T, V):
    import torch
    logits = torch.zeros(4096, dtype=torch.float32, device="cuda")
    out = torch.zeros(512, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    if rows != 1:
        with pytest.raises(sv.SpecError) as e:
            sv.spec_gumbel_sample(ctx, logits, rows, V, 1, 0, out)
    else:
        with pytest.raises(sv.SpecError) as e:
            sv.spec_accept_gumbel(ctx, logits, out, T, V, 1, 0, n, out)
    assert e.value.status == SPEC_ERR_SHAPE
