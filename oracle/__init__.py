"""fp64 CPU oracle for the speculative-decoding verify step.

TEST INFRASTRUCTURE ONLY.  Nothing on the library's product path imports,
calls or links this package; only the tests, the package entry's smoke check
and the benchmark's CPU-baseline/reference arm use it.  It shares no code with
the CUDA path (no kernels, headers, helpers or tables), and it reads the very
same host arrays the CUDA path receives, decoding the storage layouts itself.

Every function is a plain, slow, obviously-correct restatement of what the
sources define, in float64, with a library primitive (numpy matmul, cumsum,
argmax) standing in for a step where the definition is plain.  Sources:

* "Speculative Decoding Clearly Explained" (bittide.aicompass.dev post, the
  cat-sat walkthrough): accept left to right with probability min(1, p/q),
  stop at the first rejection, resample from the normalised positive part of
  p - q, bonus token when every draft is accepted.
* "Karpathy's Trick for Faster Local LLMs Finally Has Proper Tooling"
  (highsignal.app), section "How Uzu optimizes bytes and tokens per pass":
  4-bit asymmetric (Medium) and 8-bit symmetric (Large) integer weights with
  group-shared scales; block-diagonal random Hadamard transform with sign
  flips before the mixing, +/-1 entries and one overall scale.  Sections
  "Producing several tokens from one model pass" and "Issue with parallel
  draft generation": one target pass scores several positions or a whole
  draft tree; of the root paths the target confirms, the deepest is emitted.
* "Local LLM 4x Faster--Not Through Hardware, but Through Speculative
  Decoding" (wink.run): random Hadamard transform for outliers; a tree of
  drafts checked in one pass, its deepest confirmed path emitted.
* The trymirai post feed (nitterts.pages.dev/trymirai), the post on the
  "random number from 1 to 10" example: the speculator and the target both
  sample with the same seed through the Gumbel-max trick, so matching
  distributions give matching tokens.  The random numbers come from
  Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as
  easy as 1, 2, 3", SC 2011), a counter-based generator that the CUDA path
  implements separately from the same published definition.

Readings where the sources are silent:
dequantisation w = (code - zero) * scale with groups of g consecutive k
inside one output row; Sylvester (natural-order) Hadamard with 1/sqrt(B);
T+1 uniforms (u[0..T-1] for the accept tests, u[T] for the one final draw);
strict u < min(1, p/q); inverse-CDF sampling in ascending token order;
greedy tree rule (draft == argmax of the row that scores it), deepest node
wins, ties to the smallest node index, argmax ties to the smallest token id;
shared-seed rule: the noise of token v at draft position p is word v mod 4
of Philox4x32-10 at counter (v div 4, p low, p high, 0) under key (seed low,
seed high), made a uniform (2 floor(w / 2^9) + 1) / 2^24 and a Gumbel value
-log(-log u); the target's token at position p is argmax_v (logit + noise),
a draft is accepted while it equals that token, and the first position that
differs (or position T) emits the target's token.

Parity pins for every function live in tests/test_oracle_*.py.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "bf16_bits_to_f64", "unpack_w4_codes", "unpack_w4_zeros", "dequant_w4",
    "dequant_w8", "hadamard", "rht", "qgemm_w4a16", "qgemm_w8a16", "softmax",
    "spec_accept", "spec_accept_tree", "philox4x32_10", "gumbel_uniforms",
    "gumbel_sample", "spec_accept_gumbel",
]


# ----------------------------------------------------------------------------
# storage decoding
# ----------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly: a bf16 value is the
    top half of the float32 with the same bits."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def unpack_w4_codes(qcodes: np.ndarray, N: int, K: int) -> np.ndarray:
    """uint8 [N][K/2] -> int64 [N][K].  The row is read as little-endian
    32-bit words, one per eight consecutive k; nibble p of a word (counted
    from the least significant end) holds the word's element 2*(p % 4) + p // 4,
    so its four bytes carry (k0, k2), (k4, k6), (k1, k3), (k5, k7) as (low,
    high) nibbles."""
    q = np.asarray(qcodes, dtype=np.uint8).reshape(N, K // 8, 4).astype(np.int64)
    out = np.empty((N, K // 8, 8), dtype=np.int64)
    for p in range(8):
        byte, high = p // 2, p % 2
        nib = (q[:, :, byte] >> 4) if high else (q[:, :, byte] & 0xF)
        out[:, :, 2 * (p % 4) + p // 4] = nib
    return out.reshape(N, K)


def unpack_w4_zeros(zeros: np.ndarray, G: int, N: int) -> np.ndarray:
    """uint8 [G][N/2] -> int64 [G][N]; output row n's zero point sits in the
    low nibble of byte n//2 when n is even, the high nibble when odd."""
    z = np.asarray(zeros, dtype=np.uint8).reshape(G, N // 2).astype(np.int64)
    out = np.empty((G, N), dtype=np.int64)
    out[:, 0::2] = z & 0xF
    out[:, 1::2] = z >> 4
    return out


# ----------------------------------------------------------------------------
# dequantisation ("How Uzu optimizes bytes and tokens per pass")
# ----------------------------------------------------------------------------

def dequant_w4(qcodes, scales, zeros, group_size: int, N: int, K: int) -> np.ndarray:
    """4-bit asymmetric: w[n, k] = (code[n, k] - zero[g, n]) * scale[g, n]
    with g = k // group_size.  Scales fp16 [K/g][N], zeros uint4 [K/g][N/2]."""
    G = K // group_size
    codes = unpack_w4_codes(qcodes, N, K)
    z = unpack_w4_zeros(zeros, G, N)
    s = np.asarray(scales, dtype=np.float16).reshape(G, N).astype(np.float64)
    g_of_k = np.arange(K) // group_size
    # [N][K] views of the per-group parameters
    z_nk = z.T[:, g_of_k]
    s_nk = s.T[:, g_of_k]
    return (codes - z_nk).astype(np.float64) * s_nk


def dequant_w8(qcodes, scales, group_size: int, N: int, K: int) -> np.ndarray:
    """8-bit symmetric (no zero point): w[n, k] = code[n, k] * scale, with one
    scale per output channel (group_size == 0, scales [N]) or per group of
    group_size consecutive k (scales [K/g][N])."""
    c = np.asarray(qcodes, dtype=np.int8).reshape(N, K).astype(np.float64)
    s = np.asarray(scales, dtype=np.float16).astype(np.float64)
    if group_size == 0:
        return c * s.reshape(N, 1)
    g_of_k = np.arange(K) // group_size
    return c * s.reshape(K // group_size, N).T[:, g_of_k]


# ----------------------------------------------------------------------------
# random Hadamard transform ("How Uzu optimizes bytes and tokens per pass")
# ----------------------------------------------------------------------------

def hadamard(B: int) -> np.ndarray:
    """Sylvester Hadamard matrix H_B (entries +/-1): H_1 = [1],
    H_2m = [[H_m, H_m], [H_m, -H_m]]."""
    assert B >= 1 and (B & (B - 1)) == 0
    H = np.ones((1, 1), dtype=np.float64)
    while H.shape[0] < B:
        H = np.block([[H, H], [H, -H]])
    return H


def rht(x: np.ndarray, signs: np.ndarray, block: int) -> np.ndarray:
    """Block-diagonal random Hadamard rotation of the rows of x (float64
    [T][K]): each block of `block` consecutive columns becomes
    (1/sqrt(block)) * H_block @ (s * x_block), the random signs applied
    before the mixing."""
    x = np.asarray(x, dtype=np.float64)
    T, K = x.shape
    assert K % block == 0
    H = hadamard(block) / math.sqrt(block)
    s = np.asarray(signs, dtype=np.float64).reshape(K)
    out = np.empty_like(x)
    for b in range(K // block):
        cols = slice(b * block, (b + 1) * block)
        out[:, cols] = (x[:, cols] * s[cols]) @ H.T
    return out


# ----------------------------------------------------------------------------
# verify GEMMs
# ----------------------------------------------------------------------------

def _activations(x_bits, T, K, signs, block):
    x = bf16_bits_to_f64(x_bits).reshape(T, K)
    if block:
        x = rht(x, signs, block)
    return x


def qgemm_w4a16(qcodes, scales, zeros, group_size, x_bits, T, N, K,
                signs=None, block=0) -> np.ndarray:
    """y[t, n] = sum_k x[t, k] * w[n, k] in float64, w from dequant_w4; with
    a sign vector and block > 0 the activations are rotated first (the
    weights are taken as stored already rotated)."""
    W = dequant_w4(qcodes, scales, zeros, group_size, N, K)
    return _activations(x_bits, T, K, signs, block) @ W.T


def qgemm_w8a16(qcodes, scales, group_size, x_bits, T, N, K,
                signs=None, block=0) -> np.ndarray:
    """y[t, n] = sum_k x[t, k] * w[n, k] in float64, w from dequant_w8."""
    W = dequant_w8(qcodes, scales, group_size, N, K)
    return _activations(x_bits, T, K, signs, block) @ W.T


# ----------------------------------------------------------------------------
# softmax and the acceptance rule ("Speculative Decoding Clearly Explained")
# ----------------------------------------------------------------------------

def softmax(logits: np.ndarray) -> np.ndarray:
    """p[i, v] = exp(l[i, v] - max_w l[i, w]) / sum_w exp(l[i, w] - max_w l[i, w])."""
    l = np.asarray(logits, dtype=np.float64)
    l = l - l.max(axis=-1, keepdims=True)
    e = np.exp(l)
    return e / e.sum(axis=-1, keepdims=True)


def _inverse_cdf(weights: np.ndarray, u: float):
    """Smallest v with sum_{w<=v} weights[w] > u * sum(weights), plus the
    distance of that threshold to the nearest cumulative boundary (relative
    to the total) for the near-tie report."""
    c = np.cumsum(weights)
    Z = c[-1]
    target = u * Z
    v = int(np.searchsorted(c, target, side="right"))
    if v >= len(c):  # only through rounding: take the last token with mass
        v = int(np.nonzero(weights > 0)[0][-1])
    gap = float(np.min(np.abs(c - target))) / Z
    return v, gap


def spec_accept(logits, q, drafts, u, tie_eps: float = 1e-4, cdf_eps: float = 1e-7):
    """Chain acceptance of T drafts.

    Inputs: target logits [T+1][V] (row i scores draft i, row T follows the
    last draft), draft probabilities q [T][V], draft tokens [T], uniforms
    [T+1].  For i = 0..T-1: accept draft i iff u[i] < min(1, p_i(x_i) /
    q_i(x_i)) (q = 0 counts as ratio +inf); stop at the first rejection j and
    draw the replacement from normalize(max(0, p_j - q_j)) with u[T]; when
    every draft is accepted draw the bonus token from p_T with u[T].

    Returns (n_accepted, tokens[n_accepted+1], near_tie[T+1]): near_tie[i] for
    i < T marks |u[i] - p/q| < tie_eps at an evaluated position; near_tie[T]
    marks a final draw within cdf_eps (relative) of a cumulative boundary.
    """
    l = np.asarray(logits, dtype=np.float32).astype(np.float64)
    qq = np.asarray(q, dtype=np.float32).astype(np.float64)
    x = np.asarray(drafts, dtype=np.int64)
    uu = np.asarray(u, dtype=np.float32).astype(np.float64)
    T = x.shape[0]
    p = softmax(l)
    near = np.zeros(T + 1, dtype=bool)
    rejected = None
    for i in range(T):
        pi = p[i, x[i]]
        qi = qq[i, x[i]]
        r = math.inf if qi == 0.0 else pi / qi
        near[i] = abs(uu[i] - r) < tie_eps
        if uu[i] < min(1.0, r):
            continue
        rejected = i
        break
    if rejected is None:
        n_acc = T
        weights = p[T]
    else:
        n_acc = rejected
        weights = np.maximum(0.0, p[rejected] - qq[rejected])
        if not weights.sum() > 0.0:  # reachable only through rounding
            weights = p[rejected]
    tok, gap = _inverse_cdf(weights, uu[T])
    near[T] = gap < cdf_eps
    tokens = np.concatenate([x[:n_acc], [tok]]).astype(np.int64)
    return n_acc, tokens, near


def spec_accept_tree(logits, drafts, parent):
    """Greedy verification of a draft tree.

    logits [T+1][V]: row 0 is the target's distribution after the last
    committed token (it scores the root's children), row i+1 the one after
    node i.  parent[i] < i, -1 for a child of the root.  Node i is accepted
    iff its parent is accepted (the root always is) and drafts[i] equals the
    largest-logit token of the row that scores it (ties to the smallest id).
    The deepest accepted node wins (ties to the smallest node index); the
    output is the tokens on its root path plus the bonus token, the argmax of
    the row that follows it (row 0 if no node is accepted).

    Returns (path_len, tokens[path_len+1], nodes[path_len]).
    """
    l = np.asarray(logits, dtype=np.float32).astype(np.float64)
    x = np.asarray(drafts, dtype=np.int64)
    par = np.asarray(parent, dtype=np.int64)
    T = x.shape[0]
    amax = [int(np.argmax(l[r])) for r in range(T + 1)]
    accepted = [False] * T
    depth = [0] * T
    for i in range(T):
        if par[i] < 0:
            ok, row, d = True, 0, 1
        else:
            assert par[i] < i
            ok, row, d = accepted[par[i]], int(par[i]) + 1, depth[par[i]] + 1
        accepted[i] = ok and x[i] == amax[row]
        depth[i] = d
    best = -1
    for i in range(T):
        if accepted[i] and (best < 0 or depth[i] > depth[best]):
            best = i
    nodes = []
    n = best
    while n >= 0:
        nodes.append(n)
        n = int(par[n])
    nodes.reverse()
    bonus = amax[best + 1] if best >= 0 else amax[0]
    tokens = [int(x[n]) for n in nodes] + [bonus]
    return len(nodes), np.asarray(tokens, dtype=np.int64), np.asarray(nodes, dtype=np.int64)


# ----------------------------------------------------------------------------
# shared-seed sampling (trymirai post feed, the post on sampling the
# speculator and the LLM with the same seed via the Gumbel-max trick)
# ----------------------------------------------------------------------------

_PHILOX_MUL = (0xD2511F53, 0xCD9E8D57)     # round multipliers of Philox4x32
_PHILOX_WEYL = (0x9E3779B9, 0xBB67AE85)    # key increments between rounds
_U32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(counter, key) -> np.ndarray:
    """Philox4x32-10 (Salmon et al., SC 2011) over an array of counters.

    counter: integers [..., 4] (each < 2^32); key: (k0, k1).  One round takes
    the products M0 * x0 and M1 * x2 (64-bit, exact in uint64) and gives the
    next counter (hi(M1 x2) ^ x1 ^ k0, lo(M1 x2), hi(M0 x0) ^ x3 ^ k1,
    lo(M0 x0)); between rounds the key grows by the Weyl constants (mod 2^32).
    Returns uint32 [..., 4].
    """
    c = np.asarray(counter, dtype=np.uint64)
    x0, x1, x2, x3 = (c[..., i].copy() for i in range(4))
    k0, k1 = (int(key[0]) & 0xFFFFFFFF, int(key[1]) & 0xFFFFFFFF)
    m0, m1 = np.uint64(_PHILOX_MUL[0]), np.uint64(_PHILOX_MUL[1])
    for r in range(10):
        if r > 0:
            k0 = (k0 + _PHILOX_WEYL[0]) & 0xFFFFFFFF
            k1 = (k1 + _PHILOX_WEYL[1]) & 0xFFFFFFFF
        p0 = m0 * x0
        p1 = m1 * x2
        x0, x1, x2, x3 = ((p1 >> np.uint64(32)) ^ x1 ^ np.uint64(k0), p1 & _U32,
                          (p0 >> np.uint64(32)) ^ x3 ^ np.uint64(k1), p0 & _U32)
    return np.stack([x0, x1, x2, x3], axis=-1).astype(np.uint32)


def gumbel_uniforms(seed: int, position: int, V: int) -> np.ndarray:
    """The V uniforms of one draft position, in float64 (exact).

    Token v takes word v mod 4 of Philox4x32-10 at counter (v div 4,
    position mod 2^32, position div 2^32, 0) under key (seed mod 2^32,
    seed div 2^32); a word w gives u = (2 floor(w / 2^9) + 1) / 2^24, an odd
    multiple of 2^-24 strictly inside (0, 1).
    """
    seed = int(seed) % (1 << 64)
    position = int(position) % (1 << 64)
    nb = (V + 3) // 4
    ctr = np.zeros((nb, 4), dtype=np.uint64)
    ctr[:, 0] = np.arange(nb, dtype=np.uint64)
    ctr[:, 1] = position & 0xFFFFFFFF
    ctr[:, 2] = position >> 32
    w = philox4x32_10(ctr, (seed & 0xFFFFFFFF, seed >> 32)).reshape(-1)[:V]
    return (2.0 * (w.astype(np.float64) // 512.0) + 1.0) / float(1 << 24)


def gumbel_sample(logits, seed: int, positions):
    """One token per row by the Gumbel-max trick with shared noise.

    Row r's token is argmax_v (logits[r][v] + g_v), g_v = -log(-log u_v) with
    the uniforms of position positions[r] (smallest id among equal values).
    Because g is a standard Gumbel variable, the token is distributed as
    softmax(logits[r]).  Also returns each row's margin: its best value minus
    the best value of any other token (0 on an exact tie).
    """
    l = np.asarray(logits, dtype=np.float32).astype(np.float64)
    if l.ndim == 1:
        l = l[None, :]
    R, V = l.shape
    pos = [int(p) for p in np.atleast_1d(positions)]
    assert len(pos) == R
    tokens = np.zeros(R, dtype=np.int64)
    margins = np.zeros(R, dtype=np.float64)
    for r in range(R):
        z = l[r] + (-np.log(-np.log(gumbel_uniforms(seed, pos[r], V))))
        t = int(np.argmax(z))
        tokens[r] = t
        rest = np.delete(z, t)
        margins[r] = z[t] - rest.max() if rest.size else math.inf
    return tokens, margins


def spec_accept_gumbel(logits, drafts, seed: int, position: int, tie_eps: float = 1e-4):
    """Verification when the speculator sampled with the same seed.

    logits [T+1][V]: row i scores draft position i (row T follows the last
    draft).  The target's token at position i is the Gumbel-max sample of
    row i with the noise of position `position + i`.  Drafts are accepted
    left to right while they equal the target's token; the first position
    that differs, or position T when all T are accepted, emits the target's
    token.  A draft outside [0, V) never matches.

    Returns (n_accepted, tokens[n_accepted + 1], near_tie[T + 1]) where
    near_tie[i] marks a row whose margin is below tie_eps.
    """
    x = np.asarray(drafts, dtype=np.int64)
    T = x.shape[0]
    positions = [(int(position) + i) % (1 << 64) for i in range(T + 1)]
    y, margins = gumbel_sample(logits, seed, positions)
    n = T
    for i in range(T):
        if x[i] != y[i]:
            n = i
            break
    tokens = np.concatenate([x[:n], [y[n]]]).astype(np.int64)
    return n, tokens, margins < tie_eps
