"""GPU parity of softmax, chain acceptance and greedy tree acceptance against
the fp64 oracle, through the C ABI.

Bars: probabilities within 1e-5 absolute; accepted lengths and token ids
bit-exact, except draws the oracle flags as near ties (|u - p/q| < 1e-4, or a
final draw within 1e-7 (relative) of a cumulative boundary), which are counted and
reported separately; tree results bit-exact.
"""
import json
import os

import numpy as np
import pytest
import scipy.stats

import oracle
import bit_qgemm_w4_gb300 as sv
from bit_qgemm_w4_gb300 import inputs
from tests.gpu_util import dev, host

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def ctx():
    from bit_qgemm_w4_gb300 import build
    build.build()
    c = sv.Context(0)
    yield c
    c.close()


def _gpu_accept(ctx, logits, q, drafts, u):
    import torch
    T = len(drafts)
    V = logits.shape[1]
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    toks = torch.full((T + 1,), -1, dtype=torch.int32, device="cuda")
    flags = torch.zeros(T + 1, dtype=torch.int32, device="cuda")
    qd = dev(q) if T > 0 else dev(np.zeros((1, V), np.float32))
    dd = dev(drafts) if T > 0 else dev(np.zeros(1, np.int32))
    sv.spec_accept(ctx, dev(logits), qd, dd, dev(u), T, V, n, toks, flags)
    sv.spec_sync_status(ctx)
    k = int(host(n)[0])
    return k, list(host(toks)[:k + 1]), host(flags)


def _check_case(ctx, a):
    n_o, toks_o, near_o = oracle.spec_accept(a.logits, a.q, a.drafts, a.u)
    n_g, toks_g, _ = _gpu_accept(ctx, a.logits, a.q, a.drafts, a.u)
    if near_o.any():
        return "near_tie"
    assert n_g == n_o and toks_g == list(toks_o), (n_g, toks_g, n_o, list(toks_o))
    return "exact"


@pytest.mark.parametrize("V", [1000, 151936])
def test_softmax_parity(ctx, V):
    import torch
    rng = np.random.default_rng(V)
    rows = 17 if V == 1000 else 33
    l = (rng.standard_normal((rows, V)) * (2.0 if V == 1000 else 3.0)).astype(np.float32)
    p = torch.empty((rows, V), dtype=torch.float32, device="cuda")
    sv.spec_softmax(ctx, dev(l), p, rows, V)
    torch.cuda.synchronize()
    err = np.max(np.abs(host(p) - oracle.softmax(l)))
    assert err <= 1e-5, err


def test_cat_sat_worked_example(ctx):
    g = json.load(open(os.path.join(GOLDEN, "cat_sat.json")))
    vocab = {w: i for i, w in enumerate(g["vocab"])}
    drafts = np.array([vocab[w] for w in g["drafts"]], dtype=np.int32)
    logits = np.array(g["logits"], dtype=np.float32)
    q = np.array(g["q"], dtype=np.float32)
    for u in g["uniform_sets"]:
        n, toks, _ = _gpu_accept(ctx, logits, q, drafts, np.array(u, dtype=np.float32))
        assert n == g["expected_n_accepted"]
        assert toks == [vocab[w] for w in g["expected_tokens"]]


def test_bonus_token(ctx):
    V, T = 64, 6
    rng = np.random.default_rng(2)
    drafts = rng.integers(0, V, size=T).astype(np.int32)
    logits = np.full((T + 1, V), -1e4, dtype=np.float32)
    logits[np.arange(T), drafts] = 0.0
    logits[T, 17] = 0.0
    q = np.full((T, V), 1.0 / V, dtype=np.float32)
    n, toks, _ = _gpu_accept(ctx, logits, q, drafts, inputs.uniforms(rng, T + 1))
    assert n == T and toks == list(drafts) + [17]


def test_no_drafts_and_single_token_vocab(ctx):
    rng = np.random.default_rng(3)
    l = (rng.standard_normal((1, 300)) * 2).astype(np.float32)
    u = np.array([0.37], dtype=np.float32)
    n, toks, _ = _gpu_accept(ctx, l, None, np.zeros(0, np.int32), u)
    n_o, t_o, _ = oracle.spec_accept(l, np.zeros((0, 300), np.float32), np.zeros(0, np.int32), u)
    assert n == 0 and toks == list(t_o)
    l1 = np.zeros((3, 1), dtype=np.float32)
    q1 = np.ones((2, 1), dtype=np.float32)
    n, toks, _ = _gpu_accept(ctx, l1, q1, np.zeros(2, np.int32), np.array([0.5, 0.9, 0.1], np.float32))
    assert n == 2 and toks == [0, 0, 0]


@pytest.mark.parametrize("seed", range(10))
def test_tiny_config_parity(ctx, seed):
    rng = np.random.default_rng(seed)
    a = inputs.accept_inputs(rng, 16, 1000, logit_std=2.0, noise_std=1.0)
    _check_case(ctx, a)


@pytest.mark.parametrize("target", [0.3, 0.6, 0.9])
def test_vocab_152k_sweep_parity(ctx, target):
    sigma = inputs.fit_noise_for_acceptance(target, 151936, 3.0, seed=int(target * 100))
    outcomes = []
    for seed in range(4):
        rng = np.random.default_rng(100 + seed + int(target * 1000))
        a = inputs.accept_inputs(rng, 32, 151936, logit_std=3.0, noise_std=sigma)
        outcomes.append(_check_case(ctx, a))
    assert outcomes.count("exact") >= 3, outcomes


def test_random_many_small(ctx):
    near = 0
    for seed in range(60):
        rng = np.random.default_rng(500 + seed)
        T = int(rng.integers(0, 9))
        V = int(rng.integers(1, 40))
        a = inputs.accept_inputs(rng, T, V, logit_std=1.5, noise_std=0.7)
        near += _check_case(ctx, a) == "near_tie"
    assert near <= 3


def test_chi_square_distribution_preserved(ctx):
    """1e6 trials on an 8-token vocabulary: the emitted first token follows p."""
    import torch
    V, T, n_trials = 8, 2, 1_000_000
    rng = np.random.default_rng(77)
    logits = (rng.standard_normal((T + 1, V)) * 1.5).astype(np.float32)
    q64 = np.exp(rng.standard_normal((T, V)) * 1.5)
    q = (q64 / q64.sum(axis=1, keepdims=True)).astype(np.float32)
    qc = np.cumsum(q.astype(np.float64), axis=1)
    draws = rng.random((n_trials, T))
    drafts = np.stack([np.minimum(np.searchsorted(qc[i], draws[:, i] * qc[i, -1], side="right"), V - 1)
                       for i in range(T)], axis=1).astype(np.int32)
    us = rng.random((n_trials, T + 1)).astype(np.float32)
    us = np.minimum(us, np.float32(np.nextafter(np.float32(1), np.float32(0))))
    d_l, d_q = dev(logits), dev(q)
    d_dr, d_u = dev(drafts), dev(us)
    n_out = torch.zeros(n_trials, dtype=torch.int32, device="cuda")
    t_out = torch.zeros((n_trials, T + 1), dtype=torch.int32, device="cuda")
    L = sv.lib()
    h = ctx.handle
    stream = torch.cuda.current_stream().cuda_stream
    for t in range(n_trials):
        rc = L.spec_accept(h, d_l.data_ptr(), d_q.data_ptr(), d_dr.data_ptr() + 4 * T * t,
                           d_u.data_ptr() + 4 * (T + 1) * t, T, V, n_out.data_ptr() + 4 * t,
                           t_out.data_ptr() + 4 * (T + 1) * t, None, stream)
        assert rc == 0
    sv.spec_sync_status(ctx)
    first = host(t_out)[:, 0]
    p = oracle.softmax(logits)
    obs = np.bincount(first, minlength=V)
    chi = ((obs - n_trials * p[0]) ** 2 / (n_trials * p[0])).sum()
    assert chi < scipy.stats.chi2.ppf(0.999, V - 1), chi
    acc = (host(n_out) >= 1).mean()
    assert abs(acc - np.minimum(p[0], q[0]).sum()) < 5 * np.sqrt(0.25 / n_trials)


# ----------------------------------------------------------------------------
# greedy tree
# ----------------------------------------------------------------------------

def _gpu_tree(ctx, logits, drafts, parent):
    import torch
    T = len(drafts)
    V = logits.shape[1]
    ln = torch.zeros(1, dtype=torch.int32, device="cuda")
    toks = torch.full((T + 1,), -1, dtype=torch.int32, device="cuda")
    nodes = torch.full((T,), -1, dtype=torch.int32, device="cuda")
    sv.spec_accept_tree(ctx, dev(logits), dev(drafts), dev(parent), T, V, ln, toks, nodes)
    sv.spec_sync_status(ctx)
    k = int(host(ln)[0])
    return k, list(host(toks)[:k + 1]), list(host(nodes)[:k])


@pytest.mark.parametrize("T", [1, 4, 8, 16, 32, 64])
def test_tree_config_parity(ctx, T):
    for seed in range(3):
        rng = np.random.default_rng(900 + T * 10 + seed)
        tin = inputs.tree_inputs(rng, T, 151936, logit_std=3.0, p_match=0.7)
        k, toks, nodes = _gpu_tree(ctx, tin.logits, tin.drafts, tin.parent)
        ko, to, no = oracle.spec_accept_tree(tin.logits, tin.drafts, tin.parent)
        assert (k, toks, nodes) == (ko, list(to), list(no))


def test_tree_random_shapes_and_ties(ctx):
    for seed in range(40):
        rng = np.random.default_rng(1300 + seed)
        T = int(rng.integers(1, 20))
        V = int(rng.integers(1, 6))
        parent = np.array([-1 if i == 0 or rng.random() < 0.3 else int(rng.integers(0, i))
                           for i in range(T)], dtype=np.int32)
        logits = rng.integers(0, 3, size=(T + 1, V)).astype(np.float32)   # many argmax ties
        drafts = rng.integers(0, V, size=T).astype(np.int32)
        k, toks, nodes = _gpu_tree(ctx, logits, drafts, parent)
        ko, to, no = oracle.spec_accept_tree(logits, drafts, parent)
        assert (k, toks, nodes) == (ko, list(to), list(no))


def test_fwht_parity(ctx):
    import torch
    rng = np.random.default_rng(11)
    for B in (32, 64, 128, 256, 512, 1024):
        T, K = 3, 2 * B if B > 32 else 96
        xb = inputs.activations(rng, T, K)
        s = inputs.hadamard_signs(rng, K)
        y = torch.empty((T, K), dtype=torch.bfloat16, device="cuda")
        from tests.gpu_util import bf16_dev
        sv.fwht_rotate(ctx, bf16_dev(xb), y, T, K, dev(s), B)
        torch.cuda.synchronize()
        ref = oracle.rht(oracle.bf16_bits_to_f64(xb), s, B)
        err = np.abs(host(y) - ref)
        assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 1e-6 * np.sqrt(np.mean(ref ** 2))), B


@pytest.mark.parametrize("aligned", [True, False])
def test_fwht_block32_in_place_any_sign_alignment(ctx, aligned):
    # block 32 (the split engine's rotation before each block-32 GEMM) at an
    # odd T, with 16-byte aligned and unaligned signs, out of place and in
    # place, against the oracle
    import torch
    from tests.gpu_util import bf16_dev
    rng = np.random.default_rng(12 + aligned)
    T, K = 33, 4096
    xb = inputs.activations(rng, T, K)
    s = inputs.hadamard_signs(rng, K)
    sbuf = torch.zeros(K + 16, dtype=torch.int8, device="cuda")
    off = 0 if aligned else 1
    sbuf[off:off + K] = torch.from_numpy(s).to("cuda")
    sig = sbuf[off:off + K]
    assert (sig.data_ptr() % 16 == 0) == aligned
    ref = oracle.rht(oracle.bf16_bits_to_f64(xb), s, 32)
    y = torch.empty((T, K), dtype=torch.bfloat16, device="cuda")
    sv.fwht_rotate(ctx, bf16_dev(xb), y, T, K, sig, 32)
    xin = bf16_dev(xb)
    sv.fwht_rotate(ctx, xin, xin, T, K, sig, 32)
    torch.cuda.synchronize()
    for out in (host(y), host(xin)):
        err = np.abs(out - ref)
        assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 1e-6 * np.sqrt(np.mean(ref ** 2)))
