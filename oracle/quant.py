"""4-bit group-quantized weights: the format and its plain reference.

Test infrastructure: see the package docstring.

The pages' measurements run 4-bit models (the internals page's llama-bench
commands use Q4_K_M files, and its drafter advice pairs a Q4 target with a
Q8 drafter); streaming 4-bit weights cuts the bytes every verify pass reads
by ~3.8x.  The format here is this repository's own (not GGUF's):

* a weight matrix W [n][k] (row-major, the nn.Linear layout) is cut along k
  into groups of ``group`` consecutive elements per row;
* each group stores one scale s (bf16) and ``group`` signed 4-bit codes
  q in [-8, 7]; the weight it stands for is s * q;
* s = bf16(max |w| / 7) over the group (0 for an all-zero group), q =
  clamp(round_half_even(w / s), -8, 7);
* codes are packed two per byte along k: byte b of a row holds element 2b in
  its low nibble and element 2b + 1 in its high nibble (two's complement).

Speculative decoding with such a target is exact with respect to the
quantized target -- the distribution the method preserves is the one of the
model that verifies.
"""
import numpy as np
import torch


def bf16_round(x):
    """Round fp32/fp64 values to the nearest bf16 (round-half-even), as fp64."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.to(torch.float64).numpy()


def quantize_q4(w, group=64):
    """(codes int8 [n][k] in [-8, 7], scales fp64 [n][k/group] holding bf16 values)."""
    w = np.asarray(w, dtype=np.float64)
    n, k = w.shape
    if k % group:
        raise ValueError("k must be a multiple of the group size")
    g = w.reshape(n, k // group, group)
    scales = bf16_round(np.abs(g).max(axis=2) / 7.0)
    safe = np.where(scales > 0, scales, 1.0)
    q = np.rint(g / safe[..., None])                     # round half to even
    q = np.where(scales[..., None] > 0, np.clip(q, -8, 7), 0)
    return q.astype(np.int8).reshape(n, k), scales


def pack_q4(codes):
    """Two codes per byte along k: element 2b in the low nibble, 2b+1 in the high."""
    c = np.asarray(codes, dtype=np.int16)
    if c.shape[-1] % 2:
        raise ValueError("k must be even")
    nib = (c & 0xF).astype(np.uint8)
    return (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)


def unpack_q4(packed):
    """Inverse of pack_q4: int8 codes in [-8, 7]."""
    p = np.asarray(packed, dtype=np.uint8)
    lo = (p & 0xF).astype(np.int16)
    hi = (p >> 4).astype(np.int16)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int16)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    out = np.where(out >= 8, out - 16, out)
    return out.astype(np.int8)


def dequantize_q4(packed, scales, group=64):
    """W' = s * q in fp64, [n][k]."""
    q = unpack_q4(packed).astype(np.float64)
    n, k = q.shape
    s = np.repeat(np.asarray(scales, dtype=np.float64), group, axis=1)
    return (s * q).reshape(n, k)


def bytes_q4(n, k, group=64):
    """Bytes one pass streams for an [n][k] matrix: codes + bf16 scales."""
    return n * k // 2 + n * (k // group) * 2
