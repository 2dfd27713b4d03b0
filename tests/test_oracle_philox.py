"""Pins of the oracle's Philox-4x32-10 and its uniform mapping.

The known-answer vectors are those published with the Philox definition
(Salmon, Moraes, Dror, Shaw, SC'11, and the known-answer file distributed
with that paper's reference library): counter/key all zero, all ones, and the
hexadecimal digits of pi.  A wrong multiplier, a swapped high/low half, a
missing key bump or a wrong round count changes every output word.
"""
import numpy as np
import pytest
from scipy import stats

from oracle import philox

KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,want", KAT)
def test_known_answers(ctr, key, want):
    got = philox.philox4x32_10(np.array(ctr), np.array(key))
    assert tuple(int(x) for x in got) == want


def test_vectorised_matches_scalar():
    rng = np.random.default_rng(1)
    ctrs = rng.integers(0, 2**32, size=(64, 4), dtype=np.uint64)
    keys = rng.integers(0, 2**32, size=(64, 2), dtype=np.uint64)
    batch = philox.philox4x32_10(ctrs, keys)
    for i in range(64):
        assert np.array_equal(batch[i], philox.philox4x32_10(ctrs[i], keys[i]))


def test_uniform_mapping_exact():
    words = np.array([0, 255, 256, 0xFFFFFFFF, 0x80000000], dtype=np.uint64)
    u = philox.to_uniform(words)
    assert u[0] == 0.0 and u[1] == 0.0
    assert u[2] == 2.0 ** -24
    assert u[3] == 1.0 - 2.0 ** -24          # never reaches 1
    assert u[4] == 0.5
    # exactly representable in fp32
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)


def test_draw_layout_keys():
    # key = (seed lo, seed hi); counter = (step, position, stream, row); word 0.
    seed = (7 << 32) | 11
    w = philox.philox4x32_10(np.array([3, 2, philox.STREAM_ACCEPT, 5]), np.array([11, 7]))[0]
    assert philox.uniform(seed, 3, 2, philox.STREAM_ACCEPT, 5) == philox.to_uniform(w)


def test_uniformity_chi_square():
    n = 1_000_000
    u = philox.uniform(0, np.arange(n), 1, philox.STREAM_DRAFT, 0)
    counts = np.bincount((u * 100).astype(int), minlength=100)
    assert stats.chisquare(counts).pvalue > 1e-3
    # streams are not copies of one another
    v = philox.uniform(0, np.arange(n), 1, philox.STREAM_ACCEPT, 0)
    assert abs(np.corrcoef(u, v)[0, 1]) < 5e-3
