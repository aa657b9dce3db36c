"""Pins for the oracle's shared-seed (Gumbel-max) sampling and acceptance
(CPU only).

Sources: the trymirai post feed (nitterts.pages.dev/trymirai), the post with
the "random number from 1 to 10" example: sample the speculator and the LLM
with the same seed through the Gumbel-max trick, so that matching
distributions give matching tokens (100% acceptance), where independent
draws agree only one time in ten.  The generator is Philox4x32-10 (Salmon,
Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3",
SC 2011), pinned by the known-answer vectors published with its reference
implementation (Random123).
"""
import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle

M32 = 0xFFFFFFFF


@pytest.mark.parametrize("ctr,key,want", [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((M32, M32, M32, M32), (M32, M32), (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
])
def test_philox_known_answers(ctr, key, want):
    got = oracle.philox4x32_10(np.array([ctr]), key)[0]
    assert [int(v) for v in got] == list(want)


def test_uniform_layout_and_range():
    # token v of position p is word v mod 4 at counter (v div 4, p low, p high, 0)
    seed, pos, V = (7 << 32) | 11, (3 << 32) | 5, 10
    u = oracle.gumbel_uniforms(seed, pos, V)
    for v in range(V):
        w = int(oracle.philox4x32_10(np.array([[v // 4, 5, 3, 0]]), (11, 7))[0][v % 4])
        assert u[v] == (2 * (w >> 9) + 1) / 2.0**24
    # odd multiples of 2^-24, strictly inside (0, 1)
    big = oracle.gumbel_uniforms(1, 0, 200003)
    k = big * 2.0**24
    assert np.all(k == np.round(k)) and np.all(k.astype(np.int64) % 2 == 1)
    assert big.min() > 0.0 and big.max() < 1.0
    assert scipy.stats.kstest(big, "uniform").pvalue > 1e-3


def test_position_and_seed_high_words_matter():
    V = 64
    base = oracle.gumbel_uniforms(5, 0, V)
    assert not np.array_equal(base, oracle.gumbel_uniforms(5, 1 << 32, V))
    assert not np.array_equal(base, oracle.gumbel_uniforms(5 + (1 << 32), 0, V))
    assert not np.array_equal(base, oracle.gumbel_uniforms(6, 0, V))


def test_gumbel_max_samples_the_softmax():
    # argmax(l + Gumbel noise) is distributed as softmax(l): a wrong sign, a
    # missing logarithm or a biased uniform changes the frequencies
    l = np.array([0.0, 1.0, -1.0, 2.0, 0.5, -3.0], dtype=np.float32)
    n = 20000
    toks, _ = oracle.gumbel_sample(np.tile(l, (n, 1)), 99, np.arange(n))
    obs = np.bincount(toks, minlength=l.size)
    exp = scipy.special.softmax(l.astype(np.float64)) * n
    assert scipy.stats.chisquare(obs, exp).pvalue > 1e-3


def test_matching_distributions_accept_every_draft():
    # "shared randomness means shared outcome when distributions match"
    rng = np.random.default_rng(3)
    T, V, seed, pos = 16, 1000, 1234, 77
    logits = (rng.standard_normal((T + 1, V)) * 3).astype(np.float32)
    drafts, _ = oracle.gumbel_sample(logits[:T], seed, pos + np.arange(T))
    n, toks, _ = oracle.spec_accept_gumbel(logits, drafts, seed, pos)
    bonus, _ = oracle.gumbel_sample(logits[T:], seed, [pos + T])
    assert n == T
    assert list(toks) == list(drafts) + [int(bonus[0])]


def test_random_number_from_one_to_ten():
    # uniform target and speculator over ten numbers: with the same seed
    # every draft is accepted; with independent draws one in ten is
    V, T, trials = 10, 1, 4000
    logits = np.zeros((T + 1, V), dtype=np.float32)
    shared = independent = 0
    for k in range(trials):
        pos = k * (T + 1)
        d_same, _ = oracle.gumbel_sample(logits[:T], 42, [pos])
        d_other, _ = oracle.gumbel_sample(logits[:T], 43, [pos])
        shared += oracle.spec_accept_gumbel(logits, d_same, 42, pos)[0]
        independent += oracle.spec_accept_gumbel(logits, d_other, 42, pos)[0]
    assert shared == trials
    rate = independent / trials
    assert abs(rate - 0.1) < 4.5 * np.sqrt(0.09 / trials)


def test_dominant_logit_reduces_to_the_greedy_chain():
    # a token 40 above the rest outweighs any noise (-log(-log u) lies in
    # [-2.9, 16.7] for u in [2^-24, 1 - 2^-24]), so the rule becomes the
    # greedy chain of the tree rule with parent i - 1
    rng = np.random.default_rng(8)
    T, V = 12, 500
    logits = rng.standard_normal((T + 1, V)).astype(np.float32)
    top = rng.integers(0, V, T + 1)
    logits[np.arange(T + 1), top] += 40.0
    for cut in [0, 3, T]:
        drafts = top[:T].copy()
        if cut < T:
            drafts[cut] = (drafts[cut] + 1) % V
        n, toks, _ = oracle.spec_accept_gumbel(logits, drafts, 9, 1000)
        m, toks_tree, _ = oracle.spec_accept_tree(logits, drafts, np.arange(T) - 1)
        assert n == m == cut
        assert list(toks) == list(toks_tree)


def test_first_mismatch_and_out_of_range_draft():
    rng = np.random.default_rng(5)
    T, V, seed = 5, 300, 2
    logits = (rng.standard_normal((T + 1, V)) * 2).astype(np.float32)
    y, _ = oracle.gumbel_sample(logits, seed, np.arange(T + 1))
    drafts = y[:T].copy()
    drafts[2] = V + 7                        # never matches
    n, toks, _ = oracle.spec_accept_gumbel(logits, drafts, seed, 0)
    assert n == 2 and list(toks) == [y[0], y[1], y[2]]
    n0, toks0, near0 = oracle.spec_accept_gumbel(logits[:1], np.zeros(0, np.int64), seed, 0)
    assert n0 == 0 and list(toks0) == [y[0]] and near0.shape == (1,)


def test_near_tie_flag_marks_small_margins():
    V, seed, pos = 50, 4, 9
    g = -np.log(-np.log(oracle.gumbel_uniforms(seed, pos, V)))
    l = np.zeros(V)
    l[3] = 30.0
    l[17] = 30.0 + g[3] - g[17] - 5e-5     # runner-up 5e-5 below token 3
    _, m = oracle.gumbel_sample(l[None, :].astype(np.float32), seed, [pos])
    _, _, near = oracle.spec_accept_gumbel(l[None, :].astype(np.float32), np.zeros(0, np.int64), seed, pos)
    assert m[0] < 1e-4 and near[0]
    l[17] = 0.0
    _, _, near = oracle.spec_accept_gumbel(l[None, :].astype(np.float32), np.zeros(0, np.int64), seed, pos)
    assert not near[0]
