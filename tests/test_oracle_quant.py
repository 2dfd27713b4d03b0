"""Pins of the 4-bit group-quantized weight format (oracle/quant.py).

* Packing on a hand-worked row (nibble order and two's complement).
* Pack / unpack round trip over every code value.
* Values already on the grid (s * q with a bf16 s and max |q| = 7 in each
  group) come back exactly.
* Rounding error at most s / 2 per element for arbitrary weights; all-zero
  groups stay zero.
* Scales are bf16 values of max |w| / 7.
* Streamed bytes: codes + scales, ~3.8x fewer than bf16 at group 64.
* The benchmark's synthetic 4-bit matrices have the bf16 workloads' weight
  scale (std ~0.02), by closed form and by sample.
"""
import numpy as np
import pytest

from oracle import quant


def test_pack_hand_worked():
    # codes 1, -2 -> low nibble 0x1, high nibble 0xE -> 0xE1;
    # codes 7, -8 -> 0x7 | 0x8 << 4 -> 0x87
    assert quant.pack_q4(np.array([[1, -2, 7, -8]])).tolist() == [[0xE1, 0x87]]
    assert quant.unpack_q4(np.array([[0xE1, 0x87]], dtype=np.uint8)).tolist() == [[1, -2, 7, -8]]


def test_pack_roundtrip_all_codes():
    rng = np.random.default_rng(0)
    q = rng.integers(-8, 8, size=(5, 64)).astype(np.int8)
    q[0, :16] = np.arange(-8, 8)
    assert np.array_equal(quant.unpack_q4(quant.pack_q4(q)), q)


def test_grid_values_exact():
    rng = np.random.default_rng(1)
    n, k, group = 4, 128, 32
    s = quant.bf16_round(rng.uniform(0.01, 0.1, size=(n, k // group)))
    q = rng.integers(-7, 8, size=(n, k)).astype(np.int8)
    q[:, ::group] = 7                           # every group reaches |q| = 7
    w = np.repeat(s, group, axis=1) * q
    codes, scales = quant.quantize_q4(w, group)
    assert np.array_equal(scales, s)
    assert np.array_equal(codes, q)
    assert np.array_equal(quant.dequantize_q4(quant.pack_q4(codes), scales, group), w)


@pytest.mark.parametrize("group", [32, 64, 128])
def test_rounding_error_bound(group):
    rng = np.random.default_rng(2)
    w = rng.normal(0.0, 0.02, size=(16, 256))
    w[3, :group] = 0.0                           # an all-zero group
    codes, scales = quant.quantize_q4(w, group)
    assert np.array_equal(scales, quant.bf16_round(np.abs(w.reshape(16, -1, group)).max(axis=2) / 7.0))
    back = quant.dequantize_q4(quant.pack_q4(codes), scales, group)
    s = np.repeat(scales, group, axis=1)
    # the bf16 scale may sit just below max|w|/7: the largest code is then
    # clamped, which costs at most |w| - 7 s more
    bound = s / 2 + np.maximum(np.abs(w) - 7.5 * s, 0.0)
    assert (np.abs(w - back) <= bound + 1e-15).all()
    assert (back[3, :group] == 0).all() and (codes[3, :group] == 0).all()
    assert codes.min() >= -8 and codes.max() <= 7


def test_bytes():
    n, k = 4096, 4096
    assert quant.bytes_q4(n, k, 64) == n * k // 2 + n * 64 * 2
    assert (n * k * 2) / quant.bytes_q4(n, k, 64) == pytest.approx(3.765, abs=1e-3)


def test_synthetic_4bit_recipe_matches_bf16_weights():
    """The benchmark's synthetic 4-bit matrices (workloads.q4_matrix: uniform
    codes -8..7, scales 0.75-1.25 x 0.02/4.6 per group) dequantize to weights
    of standard deviation ~0.02, the bf16 workloads' N(0, 0.02^2): the closed
    form sqrt(E[c^2] E[s^2]) = sqrt(21.5 x 1.0208) x 0.02/4.6 = 0.0204, and
    the sample agrees to 2%."""
    import torch
    import workloads
    n, k = 256, 1024
    g = torch.Generator().manual_seed(3)
    buf = workloads.q4_matrix(n, k, g, "cpu")
    packed, scales = workloads.q4_parts(buf, n, k)
    w = quant.dequantize_q4(packed.numpy(), scales.numpy())
    closed = np.sqrt(21.5 * (1 + 0.25 / 12)) * 0.02 / 4.6
    assert abs(closed - 0.0204) < 1e-4
    assert abs(w.std() / closed - 1) < 0.02
