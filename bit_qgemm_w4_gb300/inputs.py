"""Seeded synthetic inputs for the speculative-decoding verify step.

Both the CUDA path's tests/bench and the fp64 oracle's tests draw their inputs
from here.  This module only draws random numbers and stores them in the byte
layouts the library reads (packed int4 nibbles, fp16 scales, bf16 activation
bits); it performs none of the verify step's own arithmetic (no dequantisation,
no GEMM, no rotation, no acceptance rule).  The one place it evaluates a
softmax is to synthesise the *draft model's* distribution q, which is an input
of the verify step, not part of it.

Storage layouts (shared by the C ABI and the oracle):

* int4 codes    uint8  [N][K/2]   each little-endian 32-bit word w of a row holds
                                   k = 8w..8w+7, nibble p (from the least significant
                                   end) holding k = 8w + 2*(p % 4) + p // 4
* int4 scales   fp16   [K/g][N]   group-major (one row per quantisation group)
* int4 zeros    uint8  [K/g][N/2] uint4 zero points, two output rows per byte,
                                   low nibble = even n
* int8 codes    int8   [N][K]
* int8 scales   fp16   [N] (per output channel) or [K/g][N] (grouped)
* activations   bf16 bit patterns (uint16) [T][K], row-major
* signs         int8   [K], each +1 or -1
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


# ----------------------------------------------------------------------------
# dtype helpers (storage only)
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even) and
    return their 16-bit patterns as uint16."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 exactly."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def pack_w4_codes(codes: np.ndarray) -> np.ndarray:
    """Pack uint4 codes [..., K] (K % 8 == 0) into the int4 code layout: each
    group of eight consecutive k becomes one little-endian 32-bit word whose
    nibble p (from the least significant end) holds element 2*(p % 4) + p // 4,
    i.e. bytes (k0 | k2<<4), (k4 | k6<<4), (k1 | k3<<4), (k5 | k7<<4)."""
    c = np.asarray(codes, dtype=np.uint8)
    K = c.shape[-1]
    assert K % 8 == 0
    g = (c.reshape(c.shape[:-1] + (K // 8, 8)) & 0xF).astype(np.uint8)
    packed = np.stack([g[..., 0] | (g[..., 2] << 4), g[..., 4] | (g[..., 6] << 4),
                       g[..., 1] | (g[..., 3] << 4), g[..., 5] | (g[..., 7] << 4)], axis=-1)
    return packed.reshape(c.shape[:-1] + (K // 2,)).astype(np.uint8)


def pack_nibbles(vals: np.ndarray) -> np.ndarray:
    """Pack uint4 values along the last axis, two per byte, even index in
    the low nibble."""
    vals = np.asarray(vals, dtype=np.uint8)
    assert vals.shape[-1] % 2 == 0
    lo = vals[..., 0::2] & 0xF
    hi = vals[..., 1::2] & 0xF
    return (lo | (hi << 4)).astype(np.uint8)


# ----------------------------------------------------------------------------
# quantised weights
# ----------------------------------------------------------------------------

@dataclass
class W4Weights:
    N: int
    K: int
    group_size: int
    qcodes: np.ndarray   # uint8 [N][K/2]
    scales: np.ndarray   # float16 [K/g][N]
    zeros: np.ndarray    # uint8 [K/g][N/2]
    raw_codes: np.ndarray | None  # uint8 [N][K] (unpacked, for tests only)
    raw_zeros: np.ndarray  # uint8 [K/g][N] (unpacked, for tests only)

    @property
    def nbytes(self) -> int:
        return self.qcodes.nbytes + self.scales.nbytes + self.zeros.nbytes


@dataclass
class W8Weights:
    N: int
    K: int
    group_size: int      # 0 = one scale per output channel
    qcodes: np.ndarray   # int8 [N][K]
    scales: np.ndarray   # float16 [N] or [K/g][N]

    @property
    def nbytes(self) -> int:
        return self.qcodes.nbytes + self.scales.nbytes


def w4_weights(rng: np.random.Generator, N: int, K: int, group_size: int = 64,
               scale_lo: float = 0.005, scale_hi: float = 0.02,
               keep_raw: bool = True) -> W4Weights:
    """int4 asymmetric group-quantised weights: codes and zero points uniform
    on 0..15, fp16 scales uniform on [scale_lo, scale_hi].  With
    keep_raw=False the packed code bytes are drawn directly (a uniform byte is
    two independent uniform nibbles) and the unpacked codes are not kept."""
    assert K % group_size == 0 and K % 8 == 0 and N % 2 == 0
    G = K // group_size
    if keep_raw:
        codes = rng.integers(0, 16, size=(N, K), dtype=np.uint8)
        packed = pack_w4_codes(codes)
    else:
        codes = None
        packed = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    zeros = rng.integers(0, 16, size=(G, N), dtype=np.uint8)
    scales = rng.uniform(scale_lo, scale_hi, size=(G, N)).astype(np.float16)
    return W4Weights(N, K, group_size, packed, scales, pack_nibbles(zeros), codes, zeros)


def w8_weights(rng: np.random.Generator, N: int, K: int, group_size: int = 0,
               scale_lo: float = 0.002, scale_hi: float = 0.01) -> W8Weights:
    """int8 symmetric weights: codes uniform on -127..127, fp16 scales
    uniform on [scale_lo, scale_hi], per output channel when group_size == 0."""
    codes = rng.integers(-127, 128, size=(N, K), dtype=np.int16).astype(np.int8)
    if group_size == 0:
        scales = rng.uniform(scale_lo, scale_hi, size=(N,)).astype(np.float16)
    else:
        assert K % group_size == 0
        scales = rng.uniform(scale_lo, scale_hi,
                             size=(K // group_size, N)).astype(np.float16)
    return W8Weights(N, K, group_size, codes, scales)


def activations(rng: np.random.Generator, T: int, K: int, std: float = 1.0) -> np.ndarray:
    """bf16 activations ~ N(0, std^2), returned as uint16 bit patterns [T][K]."""
    return f32_to_bf16_bits(rng.standard_normal((T, K), dtype=np.float32) * np.float32(std))


def hadamard_signs(rng: np.random.Generator, K: int) -> np.ndarray:
    """Random +1/-1 sign vector (int8 [K])."""
    return (rng.integers(0, 2, size=K, dtype=np.int8) * 2 - 1).astype(np.int8)


# ----------------------------------------------------------------------------
# acceptance inputs
# ----------------------------------------------------------------------------

def _draft_softmax(z: np.ndarray) -> np.ndarray:
    # The draft model's output distribution (an input of the verify step).
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def uniforms(rng: np.random.Generator, n: int) -> np.ndarray:
    """float32 uniforms on [0, 1); values that round up to 1.0 are pulled
    back to the largest float32 below 1."""
    u = rng.random(n).astype(np.float32)
    return np.minimum(u, np.float32(np.nextafter(np.float32(1), np.float32(0))))


@dataclass
class AcceptInputs:
    T: int
    V: int
    logits: np.ndarray   # float32 [T+1][V]
    q: np.ndarray        # float32 [T][V]
    drafts: np.ndarray   # int32 [T]
    u: np.ndarray        # float32 [T+1]


def accept_inputs(rng: np.random.Generator, T: int, V: int, logit_std: float = 2.0,
                  alpha: float = 1.0, noise_std: float = 1.0) -> AcceptInputs:
    """Target logits ~ N(0, logit_std^2) [T+1][V]; draft probabilities
    q = softmax(alpha*logits[:T] + N(0, noise_std^2)); draft tokens sampled
    from q; T+1 uniforms."""
    logits = (rng.standard_normal((T + 1, V)) * logit_std).astype(np.float32)
    noise = rng.standard_normal((T, V)) * noise_std
    q64 = _draft_softmax(alpha * logits[:T].astype(np.float64) + noise)
    q = q64.astype(np.float32)
    drafts = np.empty(T, dtype=np.int32)
    for i in range(T):
        c = np.cumsum(q64[i])
        drafts[i] = min(int(np.searchsorted(c, rng.random() * c[-1], side="right")), V - 1)
    return AcceptInputs(T, V, logits, q, drafts, uniforms(rng, T + 1))


def mean_acceptance_for(logits: np.ndarray, alpha: float, noise_std: float,
                        rng: np.random.Generator) -> float:
    """Expected per-position acceptance sum_v min(p, q) of a draft built as
    q = softmax(alpha*l + noise), averaged over rows.  Used only to shape the
    synthetic draft distribution to a target acceptance level."""
    l64 = logits.astype(np.float64)
    p = _draft_softmax(l64)
    q = _draft_softmax(alpha * l64 + rng.standard_normal(l64.shape) * noise_std)
    return float(np.minimum(p, q).sum(axis=-1).mean())


def fit_noise_for_acceptance(target: float, V: int, logit_std: float, seed: int,
                             alpha: float = 1.0, rows: int = 8) -> float:
    """Bisection on the draft-noise std so that the mean acceptance of the
    synthetic draft distribution is close to `target`."""
    lo, hi = 0.0, 20.0
    base = np.random.default_rng(seed)
    logits = base.standard_normal((rows, V)) * logit_std
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        acc = mean_acceptance_for(logits, alpha, mid, np.random.default_rng(seed + 1))
        if acc > target:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


# ----------------------------------------------------------------------------
# tree inputs
# ----------------------------------------------------------------------------

def tree_parents(T: int) -> np.ndarray:
    """Draft tree of max(1, T // 8) chains of depth min(T, 8) that all hang
    off the root; parent[i] = -1 marks a child of the root.  T=32 gives four
    branches of depth eight."""
    depth = min(T, 8)
    branches = max(1, T // 8)
    assert branches * depth == T, "tree sizes are multiples of 8 or at most 8"
    parent = np.empty(T, dtype=np.int32)
    for b in range(branches):
        for d in range(depth):
            i = b * depth + d
            parent[i] = -1 if d == 0 else i - 1
    return parent


@dataclass
class TreeInputs:
    T: int
    V: int
    logits: np.ndarray   # float32 [T+1][V]; row 0 follows the root
    drafts: np.ndarray   # int32 [T]
    parent: np.ndarray   # int32 [T]


def tree_inputs(rng: np.random.Generator, T: int, V: int, logit_std: float = 3.0,
                p_match: float = 0.7, parent: np.ndarray | None = None) -> TreeInputs:
    """Logits ~ N(0, logit_std^2) [T+1][V]; node i's draft token equals the
    largest logit of the row that scores it (row 0 for children of the root,
    row parent+1 otherwise) with probability p_match, else a uniform token."""
    logits = (rng.standard_normal((T + 1, V)) * logit_std).astype(np.float32)
    if parent is None:
        parent = tree_parents(T)
    drafts = np.empty(T, dtype=np.int32)
    for i in range(T):
        row = 0 if parent[i] < 0 else int(parent[i]) + 1
        if rng.random() < p_match:
            drafts[i] = int(np.argmax(logits[row]))
        else:
            drafts[i] = int(rng.integers(0, V))
    return TreeInputs(T, V, logits, drafts, parent.astype(np.int32))


# ----------------------------------------------------------------------------
# model-shaped weight stacks
# ----------------------------------------------------------------------------

# (name, K, N) of the fused projections of one 9B-class decoder layer:
# q/k/v (4096 -> 4096+1024+1024) share one input, gate/up (4096 -> 2*12288)
# share one input; o and down read their own inputs.
LAYER_9B = (("qkv", 4096, 6144), ("o", 4096, 4096), ("gate_up", 4096, 24576),
            ("down", 12288, 4096))
LAYERS_9B = 36
VOCAB_9B = 151936

# The same for the 27B-class Large tier (hidden 5120).
LAYER_27B = (("qkv", 5120, 7168), ("o", 5120, 5120), ("gate_up", 5120, 34816),
             ("down", 17408, 5120))
LAYERS_27B = 64


# ----------------------------------------------------------------------------
# device-resident stacks (benchmark sizes; drawn on the GPU from a seeded
# torch generator, same value distributions as the numpy generators above)
# ----------------------------------------------------------------------------

def w4_weights_device(gen, N: int, K: int, device, group_size: int = 64,
                      scale_lo: float = 0.005, scale_hi: float = 0.02) -> dict:
    """int4 weights drawn on the device: packed code bytes and packed zero
    bytes uniform on 0..255 (two independent uniform nibbles each), fp16
    scales uniform on [scale_lo, scale_hi]."""
    import torch
    G = K // group_size
    qcodes = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=device, generator=gen)
    zeros = torch.randint(0, 256, (G, N // 2), dtype=torch.uint8, device=device, generator=gen)
    scales = (torch.rand((G, N), device=device, generator=gen) * (scale_hi - scale_lo)
              + scale_lo).to(torch.float16)
    return {"N": N, "K": K, "g": group_size, "qcodes": qcodes, "scales": scales, "zeros": zeros}


def w8_weights_device(gen, N: int, K: int, device, scale_lo: float = 0.002,
                      scale_hi: float = 0.01) -> dict:
    """int8 per-output-channel weights drawn on the device: codes uniform on
    -127..127, fp16 scales uniform on [scale_lo, scale_hi]."""
    import torch
    qcodes = torch.randint(-127, 128, (N, K), dtype=torch.int8, device=device, generator=gen)
    scales = (torch.rand((N,), device=device, generator=gen) * (scale_hi - scale_lo)
              + scale_lo).to(torch.float16)
    return {"N": N, "K": K, "g": 0, "qcodes": qcodes, "scales": scales}


def activations_device(gen, T: int, K: int, device):
    """bf16 activations ~ N(0, 1) drawn on the device."""
    import torch
    return torch.randn((T, K), device=device, generator=gen).to(torch.bfloat16)
