"""Pins of the KV-commit oracle (CPU only): the lesson's exercise 4 built
by hand (sequence A accepts every draft, sequence B rejects at position 2,
each length right), with the KV lengths taken from the verify oracle; a
tree path by hand; in-place and scratch commits agree; refused overflows."""

import numpy as np

from oracle import kv as okv
from oracle import verify as ov


def _pattern(shape, base):
    """Distinct bytes per (layer, sequence, position, byte)."""
    L, B, S, E = shape
    v = np.zeros(shape, dtype=np.uint8)
    for l in range(L):
        for b in range(B):
            for s in range(S):
                v[l, b, s] = (base + 37 * l + 11 * b + 5 * s + np.arange(E)) % 251
    return v


def _two_sequences_kv_len():
    """Greedy verify of N = 3 drafts: A's drafts all equal the argmax, B's
    second draft does not -> out_kv_len [4, 2]."""
    vocab = 6
    z = np.zeros((2, 4, vocab), dtype=np.float32)
    arg = [[1, 2, 3, 4], [5, 0, 2, 1]]
    for b in range(2):
        for j in range(4):
            z[b, j, arg[b][j]] = 1.0
    drafts = np.array([[1, 2, 3], [5, 3, 2]], dtype=np.int32)   # B: position 2 rejected
    res = ov.verify(z, None, drafts, np.zeros(2, np.float32), 0, "f32")
    return res.kv_len


def test_exercise_4_two_sequences_by_hand():
    kv = _two_sequences_kv_len()
    assert kv.tolist() == [4, 2]
    L, B, S, E, W = 2, 2, 12, 16, 4
    cache = _pattern((L, B, S, E), 3)
    scratch = _pattern((L, B, W, E), 101)
    seq = np.array([5, 7])
    want = cache.copy()
    want[:, 0, 5:9] = scratch[:, 0, 0:4]
    want[:, 1, 7:9] = scratch[:, 1, 0:2]
    got, new_len, err = okv.commit(okv.SCRATCH, cache.copy(), seq, kv, scratch=scratch)
    assert err == 0 and new_len.tolist() == [9, 9]
    np.testing.assert_array_equal(got, want)
    # in place: the window already sits after each length; nothing moves
    placed = cache.copy()
    placed[:, 0, 5:9] = scratch[:, 0]
    placed[:, 1, 7:11] = scratch[:, 1]
    got2, len2, err2 = okv.commit(okv.INPLACE, placed.copy(), seq, kv)
    assert err2 == 0 and len2.tolist() == [9, 9]
    np.testing.assert_array_equal(got2, placed)
    assert okv.bytes_moved(okv.INPLACE, kv, E, L) == 0
    assert okv.bytes_moved(okv.SCRATCH, kv, E, L) == 2 * 6 * E * L


def test_tree_path_by_hand():
    L, B, S, E, W = 1, 1, 10, 16, 7
    cache = _pattern((L, B, S, E), 9)
    scratch = _pattern((L, B, W, E), 77)
    path = np.array([[2, 5, -1, -1]])
    kv = np.array([3])
    got, new_len, err = okv.commit(okv.SCRATCH, cache.copy(), [1], kv, scratch=scratch, path=path)
    want = cache.copy()
    want[0, 0, 1], want[0, 0, 2], want[0, 0, 3] = scratch[0, 0, 0], scratch[0, 0, 2], scratch[0, 0, 5]
    assert err == 0 and new_len.tolist() == [4]
    np.testing.assert_array_equal(got, want)
    placed = cache.copy()
    placed[0, 0, 1:8] = scratch[0, 0]
    got2, len2, _ = okv.commit(okv.INPLACE, placed.copy(), [1], kv, path=path)
    np.testing.assert_array_equal(got2[0, 0, 1:4], want[0, 0, 1:4])
    np.testing.assert_array_equal(got2[0, 0, 4:], placed[0, 0, 4:])   # past the length: untouched
    assert okv.bytes_moved(okv.INPLACE, kv, E, L, path=path) == 2 * 2 * E


def test_failed_and_overflowing_sequences_are_left_alone():
    L, B, S, E, W = 1, 3, 8, 16, 4
    cache = _pattern((L, B, S, E), 1)
    scratch = _pattern((L, B, W, E), 2)
    got, new_len, err = okv.commit(okv.SCRATCH, cache.copy(), [2, 6, 1], [-1, 3, 0], scratch=scratch)
    assert err == okv.ERR_KV and new_len.tolist() == [2, 6, 1]
    np.testing.assert_array_equal(got, cache)


def test_non_rising_path_is_refused():
    L, B, S, E, W = 1, 1, 10, 16, 7
    cache = _pattern((L, B, S, E), 4)
    scratch = _pattern((L, B, W, E), 5)
    got, new_len, err = okv.commit(okv.SCRATCH, cache.copy(), [1], [3], scratch=scratch,
                                   path=np.array([[4, 2]]))
    assert err == okv.ERR_KV and new_len.tolist() == [1]
    np.testing.assert_array_equal(got, cache)
