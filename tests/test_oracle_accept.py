"""Pins for the oracle's softmax and acceptance rules (CPU only).

Sources: "Speculative Decoding Clearly Explained" (the cat-sat walkthrough,
bonus token, distribution preservation) and "Karpathy's Trick for Faster
Local LLMs Finally Has Proper Tooling", sections "Producing several tokens
from one model pass" (five drafts, four agree, advance five) and "Issue with
parallel draft generation" (a draft tree, its deepest confirmed path).
"""
import itertools
import json
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle
from bit_qgemm_w4_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_softmax_matches_scipy_and_sums_to_one():
    rng = np.random.default_rng(0)
    l = (rng.standard_normal((5, 1000)) * 3).astype(np.float32)
    p = oracle.softmax(l)
    np.testing.assert_allclose(p, scipy.special.softmax(l.astype(np.float64), axis=-1), rtol=1e-12)
    np.testing.assert_allclose(p.sum(axis=-1), 1.0, rtol=1e-13)


def test_cat_sat_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "cat_sat.json")))
    vocab = {w: i for i, w in enumerate(g["vocab"])}
    drafts = np.array([vocab[w] for w in g["drafts"]], dtype=np.int32)
    logits = np.array(g["logits"], dtype=np.float32)
    q = np.array(g["q"], dtype=np.float32)
    expect = [vocab[w] for w in g["expected_tokens"]]
    for u in g["uniform_sets"]:
        n, toks, _ = oracle.spec_accept(logits, q, drafts, np.array(u, dtype=np.float32))
        assert n == g["expected_n_accepted"]
        assert list(toks) == expect


def _one_hot_logits(rows, V):
    l = np.full((len(rows), V), -1e4, dtype=np.float32)
    for i, v in enumerate(rows):
        l[i, v] = 0.0
    return l


def test_bonus_token_when_all_accepted():
    V, T = 16, 5
    rng = np.random.default_rng(1)
    drafts = rng.integers(0, V, size=T).astype(np.int32)
    bonus = 11
    logits = _one_hot_logits(list(drafts) + [bonus], V)
    q = np.full((T, V), 1.0 / V, dtype=np.float32)
    for _ in range(5):
        u = inputs.uniforms(rng, T + 1)
        n, toks, _ = oracle.spec_accept(logits, q, drafts, u)
        assert n == T
        assert list(toks) == list(drafts) + [bonus]


def test_five_drafts_four_agree_advance_five():
    # Greedy target and drafter (one-hot distributions): drafts agree with the
    # target on the first four positions, so one pass yields five tokens,
    # the fifth being the target's own token.
    V = 10
    target = [3, 1, 4, 1, 5, 9]          # target's choice after each prefix
    drafts = np.array([3, 1, 4, 1, 2], dtype=np.int32)
    logits = _one_hot_logits(target, V)
    q = np.zeros((5, V), dtype=np.float32)
    q[np.arange(5), drafts] = 1.0
    n, toks, _ = oracle.spec_accept(logits, q, drafts, np.full(6, 0.5, dtype=np.float32))
    assert n == 4 and list(toks) == [3, 1, 4, 1, 5]
    # the same through the tree rule on a chain
    parent = np.array([-1, 0, 1, 2, 3], dtype=np.int32)
    ln, ttoks, nodes = oracle.spec_accept_tree(logits, drafts, parent)
    assert ln == 4 and list(ttoks) == [3, 1, 4, 1, 5] and list(nodes) == [0, 1, 2, 3]


def test_zero_draft_probability_always_accepts():
    V = 4
    logits = np.zeros((2, V), dtype=np.float32)
    q = np.array([[0.0, 0.5, 0.5, 0.0]], dtype=np.float32)
    n, toks, _ = oracle.spec_accept(logits, q, np.array([0], dtype=np.int32),
                                    np.array([0.999, 0.0], dtype=np.float32))
    assert n == 1 and toks[0] == 0 and toks[1] == 0


def test_strict_inequality_rejects_zero_ratio_at_zero_uniform():
    V = 4
    logits = np.array([[-1e4, 0, 0, 0], [0, 0, 0, 0]], dtype=np.float32)
    q = np.array([[0.25, 0.25, 0.25, 0.25]], dtype=np.float32)
    n, _, _ = oracle.spec_accept(logits, q, np.array([0], dtype=np.int32),
                                 np.array([0.0, 0.5], dtype=np.float32))
    assert n == 0


def test_inverse_cdf_picks_expected_token():
    # Bonus row with p = (0.1, 0.2, 0.3, 0.4): u = 0.05 -> 0, 0.25 -> 1, 0.55 -> 2, 0.95 -> 3.
    p = np.array([0.1, 0.2, 0.3, 0.4])
    logits = np.log(p).astype(np.float32)[None, :]
    q = np.zeros((0, 4), dtype=np.float32)
    for u, expect in [(0.05, 0), (0.25, 1), (0.55, 2), (0.95, 3)]:
        n, toks, _ = oracle.spec_accept(logits, q, np.zeros(0, dtype=np.int32),
                                        np.array([u], dtype=np.float32))
        assert n == 0 and list(toks) == [expect]


def test_near_tie_flags():
    V = 2
    # p = (0.5, 0.5); q(x0) = 0.625 -> ratio 0.8
    logits = np.zeros((2, V), dtype=np.float32)
    q = np.array([[0.625, 0.375]], dtype=np.float32)
    _, _, near = oracle.spec_accept(logits, q, np.array([0], dtype=np.int32),
                                    np.array([0.80001, 0.3], dtype=np.float32))
    assert near[0]
    _, _, near = oracle.spec_accept(logits, q, np.array([0], dtype=np.int32),
                                    np.array([0.9, 0.3], dtype=np.float32))
    assert not near[0]


def _chain_trials(p_rows, q_rows, n_trials, seed):
    """Run the oracle on n_trials fresh (drafts ~ q, uniforms) and return the
    emitted token at each position (-1 where the chain stopped before it)."""
    T = q_rows.shape[0]
    logits = np.log(p_rows).astype(np.float32)
    q = q_rows.astype(np.float32)
    rng = np.random.default_rng(seed)
    out = np.full((n_trials, T + 1), -1, dtype=np.int64)
    qc = np.cumsum(q.astype(np.float64), axis=1)
    draws = rng.random((n_trials, T))
    us = rng.random((n_trials, T + 1)).astype(np.float32)
    for t in range(n_trials):
        drafts = np.array([min(int(np.searchsorted(qc[i], draws[t, i] * qc[i, -1], side="right")),
                               q.shape[1] - 1) for i in range(T)], dtype=np.int32)
        n, toks, _ = oracle.spec_accept(logits, q, drafts, us[t])
        out[t, :n + 1] = toks
    return out


def test_distribution_preserved_chi_square():
    # Vocabulary of 8, two drafts: the emitted token at position 0, and at
    # position 1 given that position 0 was accepted, must follow p.
    V = 8
    rng = np.random.default_rng(7)
    p = scipy.special.softmax(rng.standard_normal((3, V)) * 1.5, axis=-1)
    q = scipy.special.softmax(rng.standard_normal((2, V)) * 1.5, axis=-1)
    # store p through float32 logits as the oracle reads them
    p = scipy.special.softmax(np.log(p).astype(np.float32).astype(np.float64), axis=-1)
    n_trials = 1_000_000
    out = _chain_trials(p, q, n_trials, seed=11)
    crit = scipy.stats.chi2.ppf(0.999, V - 1)   # 24.32
    obs0 = np.bincount(out[:, 0], minlength=V)
    chi0 = ((obs0 - n_trials * p[0]) ** 2 / (n_trials * p[0])).sum()
    assert chi0 < crit, chi0
    reached = out[:, 1] >= 0
    m = int(reached.sum())
    obs1 = np.bincount(out[reached, 1], minlength=V)
    chi1 = ((obs1 - m * p[1]) ** 2 / (m * p[1])).sum()
    assert chi1 < crit, chi1
    # acceptance rate at position 0 equals sum_v min(p, q) = 1 - TV(p, q)
    acc_rate = np.minimum(p[0], q[0]).sum()
    # position-0 acceptance <=> a second token exists
    k = m
    lo, hi = scipy.stats.binomtest(k, n_trials).proportion_ci(0.999)
    assert lo <= acc_rate <= hi, (acc_rate, lo, hi)


def test_residual_sign_matters():
    # If the resample used max(0, q - p) instead, the chi-square above would
    # fail; check directly that the residual picks the token where p > q.
    V = 3
    p = np.array([[0.1, 0.1, 0.8], [1 / 3, 1 / 3, 1 / 3]])
    q = np.array([[0.8, 0.1, 0.1]], dtype=np.float32)
    n, toks, _ = oracle.spec_accept(np.log(p).astype(np.float32), q,
                                    np.array([0], dtype=np.int32),
                                    np.array([0.99, 0.5], dtype=np.float32))
    assert n == 0 and toks[0] == 2


# ----------------------------------------------------------------------------
# tree
# ----------------------------------------------------------------------------

def _brute_tree(logits, drafts, parent):
    """Enumerate every root path and keep the longest whose tokens all match
    the argmax of the row that scores them."""
    T = len(drafts)
    amax = [int(np.argmax(logits[r])) for r in range(T + 1)]
    best_nodes = []
    for i in range(T):
        path = []
        n = i
        while n >= 0:
            path.append(n)
            n = int(parent[n])
        path.reverse()
        ok = all(drafts[nd] == amax[0 if parent[nd] < 0 else parent[nd] + 1] for nd in path)
        if ok and len(path) > len(best_nodes):
            best_nodes = path
    bonus = amax[best_nodes[-1] + 1] if best_nodes else amax[0]
    return len(best_nodes), [int(drafts[n]) for n in best_nodes] + [bonus], best_nodes


@pytest.mark.parametrize("seed", range(20))
def test_tree_matches_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    T = int(rng.integers(1, 9))
    V = 4
    parent = np.array([-1 if i == 0 or rng.random() < 0.3 else int(rng.integers(0, i))
                       for i in range(T)], dtype=np.int32)
    tin = inputs.tree_inputs(rng, T, V, p_match=0.8, parent=parent)
    n, toks, nodes = oracle.spec_accept_tree(tin.logits, tin.drafts, tin.parent)
    bn, btoks, bnodes = _brute_tree(tin.logits, tin.drafts, tin.parent)
    assert n == bn and list(toks) == btoks and list(nodes) == bnodes


def test_tree_chain_equals_greedy_chain():
    rng = np.random.default_rng(3)
    T, V = 8, 50
    tin = inputs.tree_inputs(rng, T, V, p_match=0.9)
    n, toks, nodes = oracle.spec_accept_tree(tin.logits, tin.drafts, tin.parent)
    amax = np.argmax(tin.logits, axis=1)
    k = 0
    while k < T and tin.drafts[k] == amax[k]:
        k += 1
    assert n == k and list(toks) == list(tin.drafts[:k]) + [int(amax[k])]
    assert list(nodes) == list(range(k))


def test_tree_no_node_accepted_takes_root_argmax():
    logits = _one_hot_logits([2, 0, 0], 4)
    n, toks, nodes = oracle.spec_accept_tree(logits, np.array([1, 1], dtype=np.int32),
                                             np.array([-1, -1], dtype=np.int32))
    assert n == 0 and list(toks) == [2] and len(nodes) == 0


def test_tree_equal_depth_tie_goes_to_smallest_node():
    # two branches of depth 2 whose tokens both match
    V = 5
    logits = _one_hot_logits([1, 2, 3, 2, 4], V)
    # nodes: 0 (root child, tok 1), 1 (child of 0, tok 2), 2 (root child, tok 1), 3 (child of 2, tok 2)
    drafts = np.array([1, 2, 1, 2], dtype=np.int32)
    parent = np.array([-1, 0, -1, 2], dtype=np.int32)
    n, toks, nodes = oracle.spec_accept_tree(logits, drafts, parent)
    assert n == 2 and list(nodes) == [0, 1] and list(toks) == [1, 2, 3]


def test_tree_argmax_tie_goes_to_smallest_token():
    logits = np.array([[1.0, 3.0, 3.0, 0.0], [0, 0, 0, 0]], dtype=np.float32)
    n, toks, _ = oracle.spec_accept_tree(logits, np.array([2], dtype=np.int32),
                                         np.array([-1], dtype=np.int32))
    assert n == 0 and list(toks) == [1]
    n, toks, _ = oracle.spec_accept_tree(logits, np.array([1], dtype=np.int32),
                                         np.array([-1], dtype=np.int32))
    assert n == 1 and list(toks) == [1, 0]


def test_tree_shapes():
    for T, want in [(1, [-1]), (4, [-1, 0, 1, 2])]:
        assert list(inputs.tree_parents(T)) == want
    p32 = inputs.tree_parents(32)
    assert list(np.nonzero(p32 < 0)[0]) == [0, 8, 16, 24]
    assert all(p32[i] == i - 1 for i in range(32) if i % 8)
