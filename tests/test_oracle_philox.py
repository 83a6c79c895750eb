"""Pins for oracle.philox: published known-answer vectors and uniformity."""
import os

import numpy as np

from oracle.philox import element_words, philox4x32_10

GOLD = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def test_known_answer_vectors():
    n = 0
    for line in open(GOLD):
        if line.startswith("#") or not line.strip():
            continue
        v = [int(t, 16) for t in line.split()]
        out = philox4x32_10(*[np.array([c], dtype=np.uint64) for c in v[:4]], v[4], v[5])
        assert [int(o[0]) for o in out] == v[6:]
        n += 1
    assert n == 3


def test_uniformity_and_bit_balance():
    w = element_words(1 << 21, 0, seed=0x1234_5678_9ABC, copy_id=0, offset=7)[::4]   # one word per group
    u = w.astype(np.float64) / 2.0 ** 32
    assert abs(u.mean() - 0.5) < 4 * np.sqrt(1 / 12 / u.size)
    hist = np.bincount((w >> 24).astype(np.int64), minlength=256)
    exp = u.size / 256
    chi2 = ((hist - exp) ** 2 / exp).sum()
    assert chi2 < 255 + 6 * np.sqrt(2 * 255)
    bits = ((w[:, None] >> np.arange(32, dtype=np.uint32)) & 1).mean(axis=0)
    assert np.all(np.abs(bits - 0.5) < 4 * 0.5 / np.sqrt(u.size))


def test_element_words_indexing():
    # element g reads word (g // 4) % 4 of counter g // 16; any window agrees
    full = element_words(64, 0, seed=5, copy_id=1, offset=3)
    part = element_words(10, 37, seed=5, copy_id=1, offset=3)
    np.testing.assert_array_equal(full[37:47], part)
    c = philox4x32_10(np.array([2]), np.array([1]), np.array([3]), np.array([0]), 5, 0)
    words = [int(x[0]) for x in c]
    np.testing.assert_array_equal(full[32:48], np.repeat(words, 4))
    # different copy ids / offsets / seeds give different streams
    assert not np.array_equal(full, element_words(64, 0, seed=5, copy_id=0, offset=3))
    assert not np.array_equal(full, element_words(64, 0, seed=5, copy_id=1, offset=4))
    assert not np.array_equal(full, element_words(64, 0, seed=6, copy_id=1, offset=3))
