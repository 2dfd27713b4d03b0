"""Philox-4x32-10 and the draw layout of the speculative step (host side).

Test infrastructure: see the package docstring.

Philox-4x32-10 is restated from its published definition (Salmon, Moraes,
Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11, section on
the Philox S-box): a 4-word counter and a 2-word key; each of the 10 rounds
multiplies words 0 and 2 by two fixed odd 32-bit constants, keeps the high and
low halves of both products, XORs the high halves with the other two counter
words and the round key, and permutes; the key is bumped by two Weyl
increments (the golden ratio and sqrt(3)-1 in 32-bit fixed point) between
rounds.

Draw layout (how every random number of the method is keyed, so that the GPU
and this oracle draw identical uniforms):

    key     = (seed & 0xffffffff, seed >> 32)
    counter = (step, position, stream, row)
    u       = (word0 >> 8) * 2**-24            # in [0, 1), exact in fp32/fp64

``step`` counts speculative steps from 0 after prefill (autoregressive steps
for the plain-decoding baseline); ``position`` is the draft index i = 1..K,
K+1 for the bonus draw; ``row`` is the batch row.
"""
import numpy as np

# Multipliers and Weyl key increments of Philox-4x32 (SC'11 paper).
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
ROUNDS = 10

# Stream ids of the draw layout.
STREAM_DRAFT = 0      # inverse-CDF uniform for draft token d_i ~ q_i
STREAM_ACCEPT = 1     # r_i of the ratio test
STREAM_RESIDUAL = 2   # inverse-CDF uniform for the residual (p - q)+ draw
STREAM_BONUS = 3      # inverse-CDF uniform for the bonus draw from p_{K+1}
STREAM_AR = 4         # inverse-CDF uniform for plain autoregressive sampling

_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(counter, key):
    """Philox-4x32-10 block function.

    counter: array-like [..., 4] of uint32 words; key: array-like [..., 2].
    Returns a uint32 array [..., 4].  Vectorised over leading dimensions.
    """
    c = np.asarray(counter, dtype=np.uint64) & _MASK32
    k = np.asarray(key, dtype=np.uint64) & _MASK32
    c0, c1, c2, c3 = (c[..., j].copy() for j in range(4))
    k0 = np.broadcast_to(k[..., 0], c0.shape).copy()
    k1 = np.broadcast_to(k[..., 1], c0.shape).copy()
    m0 = np.uint64(PHILOX_M0)
    m1 = np.uint64(PHILOX_M1)
    for _ in range(ROUNDS):
        p0 = c0 * m0            # < 2**64: exact in uint64
        p1 = c2 * m1
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0), lo1, (hi0 ^ c3 ^ k1), lo0
        k0 = (k0 + np.uint64(PHILOX_W0)) & _MASK32
        k1 = (k1 + np.uint64(PHILOX_W1)) & _MASK32
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def to_uniform(word):
    """Top 24 bits of a uint32 word as a uniform in [0, 1) (exact in fp32)."""
    w = np.asarray(word, dtype=np.uint64)
    return (w >> np.uint64(8)).astype(np.float64) * (2.0 ** -24)


def uniform(seed, step, position, stream, row=0):
    """One uniform of the draw layout (scalars or broadcastable arrays)."""
    seed = int(seed)
    step, position, stream, row = np.broadcast_arrays(
        np.asarray(step, dtype=np.uint64), np.asarray(position, dtype=np.uint64),
        np.asarray(stream, dtype=np.uint64), np.asarray(row, dtype=np.uint64))
    ctr = np.stack([step, position, stream, row], axis=-1)
    key = np.array([seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF], dtype=np.uint64)
    out = to_uniform(philox4x32_10(ctr, key)[..., 0])
    return float(out) if out.ndim == 0 else out
