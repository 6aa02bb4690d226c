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
                # V <= 16: the first three levels of the grouped inverse CDF
                # have a single block, so only the last uniform matters
                return utup[j - 1] if kind == 0 else (Fr(0), Fr(0), Fr(0), utup[n])
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
                                      lambda j, kind: u0 if kind == 0 else (0, 0, 0, u1))
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
    # unnormalised masses: the comparison is against u times the total
    assert ov.sample(np.array([0.5, 0.25, 0.0]), 0.9)[0] == 1
    assert ov.sample(np.array([0.5, 0.25, 0.0]), 0.5)[0] == 0
    t, margin = ov.sample(dist, Fr(1, 12))
    assert t == 1 and margin == Fr(1, 12)
    # a zero-mass index is never chosen
    for k in range(12):
        assert ov.sample(fr_row(0, 4, 0, 0, 8, 0), Fr(k, 12))[0] in (1, 4)


def _grouped_fixture():
    """300 tokens: level 2 splits them into [0, 256) and [256, 300) with
    conditional masses 1/3, 2/3; level 3 blocks of 16 get 1/16 each in the
    first block and 1/4, 1/4, 1/2 in the second; level 4 tokens get
    multiples of 1/16 of their block (with zeros).  Every level's edges are
    then multiples of 1/3, 1/16 and 1/16."""
    dist = [Fr(0)] * 300
    tok_pattern = [0, 2, 1, 0, 3, 0, 0, 1, 2, 2, 0, 1, 0, 2, 1, 1]   # sums to 16
    tok_short = [4, 0, 2, 2, 0, 4, 1, 3, 0, 0, 0, 0]                 # 12 tokens, sums to 16
    for g in range(16):                      # block [0, 256): 16 blocks of 16
        for i in range(16):
            dist[16 * g + i] = Fr(1, 3) * Fr(1, 16) * Fr(tok_pattern[(i + g) % 16], 16)
    second = [Fr(1, 4), Fr(1, 4), Fr(1, 2)]  # blocks [256,272), [272,288), [288,300)
    for g in range(3):
        n = 16 if g < 2 else 12
        pat = tok_pattern if g < 2 else tok_short
        for i in range(n):
            dist[256 + 16 * g + i] = Fr(2, 3) * second[g] * Fr(pat[(i + g) % n] if g < 2 else pat[i], 16)
    return np.array(dist, dtype=object)


def test_grouped_sampler_is_exact_over_three_levels():
    dist = _grouped_fixture()
    assert sum(dist) == 1
    law = {}
    for u2 in range(3):
        for u3 in range(16):
            for u4 in range(16):
                t, _ = ov.sample_grouped(dist, (Fr(0), Fr(u2, 3), Fr(u3, 16), Fr(u4, 16)))
                law[t] = law.get(t, Fr(0)) + Fr(1, 3 * 16 * 16)
    for t in range(300):
        assert law.get(t, Fr(0)) == dist[t], t


def test_grouped_sampler_levels_and_scale_invariance():
    dist = _grouped_fixture()
    us = (Fr(1, 7), Fr(1, 2), Fr(5, 16), Fr(3, 16))
    t, margins = ov.sample_grouped(dist, us)
    t2, margins2 = ov.sample_grouped(dist * 5, us)        # unnormalised masses
    assert t == t2 and margins == margins2
    assert len(margins) == 4
    assert margins[0] == min(us[0], 1 - us[0])             # one block at level 1
    assert 256 <= t < 300                                  # u2 = 1/2 > 1/3 picks the 2nd block
