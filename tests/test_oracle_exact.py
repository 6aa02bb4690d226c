"""Exact pins of the oracle's walk (CPU only).

The oracle's ``walk``, ``accept``, ``residual`` and ``sample`` run here on
object arrays of ``fractions.Fraction``.  The uniform each draw consumes is
enumerated over the grid {0, 1/L, ..., (L-1)/L}; every threshold q/p and
every normalised residual / bonus CDF value in these fixtures is a multiple
of 1/L, and for such thresholds the grid gives each branch exactly its real
probability (#{k : k/L < x} = xL).  Summing over all draft tuples (weighted
by prod_j p_j(d_j)) and all uniform tuples therefore yields the exact law of
the walk's output, which must satisfy what the "Speculative Decoding and
EAGLE-3" lesson states ("Invariant: Leviathan rejection sampling";
"What determines the speedup"):

* every emitted token is distributed as the verifier's q at its slot, given
  the accepted prefix (the output law equals q, whatever p is);
* the acceptance probability at position j, given the walk reached j, is
  sum_t min(p_j(t), q_j(t));
* with that overlap alpha equal at every position, the expected number of
  tokens per verifier call is (1 - alpha^(N+1)) / (1 - alpha);
* the KV length to commit is accepted + 1.
"""

import itertools
from fractions import Fraction as Fr

import numpy as np
import pytest

from oracle import verify as ov


def fr_row(*nums, den=12):
    return np.array([Fr(n, den) for n in nums], dtype=object)


def enumerate_law(q_rows, p_rows, grid):
    """Exact joint law of (tokens, accepted, kv_len) of ``ov.walk``."""
    n = len(p_rows)
    vocab = len(q_rows[0])
    us = [Fr(k, grid) for k in range(grid)]
    law = {}
    for drafts in itertools.product(range(vocab), repeat=n):
        w_d = Fr(1)
        for j, d in enumerate(drafts):
            w_d *= p_rows[j][d]
        if w_d == 0:
            continue
        for utup in itertools.product(us, repeat=n + 1):
            def draw(j, kind, utup=utup):
                return utup[j - 1] if kind == 0 else utup[n]
            tokens, a, kv, _ = ov.walk(q_rows, p_rows, list(drafts), draw)
            key = (tuple(int(t) for t in tokens), a, kv)
            law[key] = law.get(key, Fr(0)) + w_d / grid ** (n + 1)
    return law


# Fixture A: V=4, N=2, grid 12.  q_1 has a zero entry (a draft there is
# always rejected); both positions have overlap sum min(p, q) = 2/3.
Q_A = [fr_row(4, 4, 4, 0), fr_row(1, 6, 2, 3), fr_row(1, 2, 3, 6)]
P_A = [fr_row(2, 3, 3, 4), fr_row(3, 3, 4, 2)]

# Fixture B: V=3, N=3, grid 6; overlaps 5/6, 2/3, 5/6 (not constant).
Q_B = [fr_row(3, 2, 1, den=6), fr_row(1, 1, 4, den=6), fr_row(2, 2, 2, den=6),
       fr_row(1, 4, 1, den=6)]
P_B = [fr_row(2, 2, 2, den=6), fr_row(2, 1, 3, den=6), fr_row(3, 2, 1, den=6)]


@pytest.fixture(scope="module")
def law_a():
    return enumerate_law(Q_A, P_A, 12)


@pytest.fixture(scope="module")
def law_b():
    return enumerate_law(Q_B, P_B, 6)


def _fixture_sanity(q_rows, p_rows, grid):
    for row in list(q_rows) + list(p_rows):
        assert sum(row) == 1
    for q, p in zip(q_rows, p_rows):
        for t in range(len(q)):
            if p[t] > 0:
                assert (min(1, q[t] / p[t]) * grid).denominator == 1
        r = ov.residual(q, p)
        for c in np.cumsum(r):
            assert (c * grid).denominator == 1
    for c in np.cumsum(q_rows[-1]):
        assert (c * grid).denominator == 1


def test_fixtures_are_on_the_grid():
    _fixture_sanity(Q_A, P_A, 12)
    _fixture_sanity(Q_B, P_B, 6)


def _check_law(law, q_rows, p_rows):
    n = len(p_rows)
    vocab = len(q_rows[0])
    assert sum(law.values()) == 1
    for (tokens, a, kv), _ in law.items():
        assert kv == a + 1
        assert len(tokens) == a + 1
    # Slot-by-slot: P(slot k = t, slots < k accepted, prefix) / P(prefix) = q_{k+1}(t).
    for k in range(n + 1):
        prefixes = {}
        for (tokens, a, _), pr in law.items():
            if a < k:
                continue  # slot k is not emitted or the prefix was not all accepted
            key = tokens[:k]
            prefixes.setdefault(key, {})
            t = tokens[k]
            prefixes[key][t] = prefixes[key].get(t, Fr(0)) + pr
        for key, dist in prefixes.items():
            total = sum(dist.values())
            for t in range(vocab):
                assert dist.get(t, Fr(0)) / total == q_rows[k][t], (k, key, t)
    # Acceptance at position j given the walk reached j.
    for j in range(1, n + 1):
        reach = sum(pr for (_, a, _), pr in law.items() if a >= j - 1)
        acc = sum(pr for (_, a, _), pr in law.items() if a >= j)
        alpha = sum(min(q, p) for q, p in zip(q_rows[j - 1], p_rows[j - 1]))
        assert acc / reach == alpha, j


def test_leviathan_invariant_fixture_a(law_a):
    _check_law(law_a, Q_A, P_A)


def test_leviathan_invariant_fixture_b(law_b):
    _check_law(law_b, Q_B, P_B)


def test_expected_tokens_closed_form(law_a):
    """E[accepted + 1] = (1 - alpha^(N+1)) / (1 - alpha) with alpha = 2/3, N = 2."""
    alpha = Fr(2, 3)
    for q, p in zip(Q_A, P_A):
        assert sum(min(a, b) for a, b in zip(q, p)) == alpha
    mean = sum(pr * (a + 1) for (_, a, _), pr in law_a.items())
    assert mean == (1 - alpha ** 3) / (1 - alpha)
    assert mean == Fr(19, 9)


def test_rejected_draft_never_reemitted(law_a):
    """A rejection at j needs q_j(d) < p_j(d), where (q - p)_+ is zero, so the
    correction never repeats the rejected draft.  Check on the walk itself."""
    us = [Fr(k, 12) for k in range(12)]
    for d1 in range(4):
        if P_A[0][d1] == 0:
            continue
        for u0, u1 in itertools.product(us, us):
            tokens, a, _, _ = ov.walk(Q_A, P_A, [d1, 0],
                                      lambda j, kind: u0 if kind == 0 else u1)
            if a == 0:
                assert tokens[0] != d1


def test_accept_rule_edges():
    # p(d) <= 0 is accepted whatever u is
    assert ov.accept(Fr(1, 2), Fr(0), Fr(999, 1000))
    assert ov.accept(0.0, 0.0, 0.99)
    # strict comparison u < min(1, q/p)
    assert not ov.accept(Fr(1, 4), Fr(1, 2), Fr(1, 2))
    assert ov.accept(Fr(1, 4), Fr(1, 2), Fr(1, 2) - Fr(1, 10 ** 9))
    # ratio above 1 always accepts
    assert ov.accept(0.9, 0.1, 1.0 - 2 ** -24)
    # q(d) = 0 always rejects
    assert not ov.accept(0.0, 0.3, 0.0)


def test_residual_edges():
    q = fr_row(6, 3, 3, 0)
    # (q - p)_+ normalised
    r = ov.residual(q, fr_row(3, 3, 3, 3))
    assert list(r) == [1, 0, 0, 0]
    # zero positive part: the residual falls back to q
    r = ov.residual(q, q.copy())
    assert list(r) == list(q)


def test_sample_inverse_cdf_edges():
    dist = fr_row(0, 3, 0, 9)
    assert ov.sample(dist, Fr(0))[0] == 1
    assert ov.sample(dist, Fr(3, 12) - Fr(1, 10 ** 6))[0] == 1
    assert ov.sample(dist, Fr(3, 12))[0] == 3      # C_1 = 3/12 is not > 3/12
    assert ov.sample(dist, Fr(11, 12))[0] == 3
    # rounding past the end falls back to the last index with mass
    assert ov.sample(np.array([0.5, 0.25, 0.0]), 0.9)[0] == 1
    t, margin = ov.sample(dist, Fr(1, 12))
    assert t == 1 and margin == Fr(1, 12)
