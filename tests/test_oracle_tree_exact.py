"""Exact pins of the tree walk itself, ``oracle.tree.walk`` (CPU only).

The pages ("Speculative Decoding and EAGLE-3" lesson, "Key terms" entry on
EAGLE-2's draft tree and exercise 3's [2, 2, 2] tree; "Invariant: Leviathan
rejection sampling") require that verifying a draft tree keeps the
verifier's law: whatever the drafter proposes, every emitted token is
distributed as the target's q at the node the walk has reached.  Here the
oracle's own ``walk`` (not a second statement of its sibling loop) is run
over every outcome of its random inputs, with exact rational weights:

* each uniform the walk asks for is a symbolic value known only to lie in
  an interval; the first comparison the interval does not decide splits it
  at the threshold and both halves are explored, so the weight of an
  outcome is the product of its intervals' lengths -- the exact probability
  for any rational thresholds, no grid needed;
* a Philox counter (depth, draw) stands for ONE uniform, used by every word
  and level of that counter, so two decisions that share a counter are
  correlated in this model -- the walk must give each decision its own;
* in SAMPLED mode a child's token is drawn from its parent's draft row the
  first time the walk reads it, weighted by p_parent(token).

The pin: for every accepted path prefix P (node ids), the token emitted in
slot |P| is distributed exactly as q at P's last node (the root for the
empty prefix), in SAMPLED and in TOPK mode.  Planted slips in ``walk``
(made by editing its source text here, on the CPU) must break it.
"""

import inspect
import itertools
import textwrap
from fractions import Fraction as F

import numpy as np
import pytest

from oracle import philox
from oracle import tree as ot


class _Split(Exception):
    def __init__(self, kind, key, at=None):
        super().__init__(kind, key, at)
        self.kind, self.key, self.at = kind, key, at


class SymU:
    """A uniform known to lie in [lo, hi).  ``u < x`` is answered when the
    interval decides it, otherwise the enumerator is asked to split at x."""

    def __init__(self, key, lo, hi):
        self.key, self.lo, self.hi = key, lo, hi

    def _below(self, x):
        x = F(x)
        if self.hi <= x:
            return True
        if self.lo >= x:
            return False
        raise _Split("u", self.key, x)

    def __lt__(self, x):
        return self._below(x)

    def __ge__(self, x):
        return not self._below(x)

    def __mul__(self, s):
        return _Scaled(self, F(s))

    __rmul__ = __mul__

    def __sub__(self, x):
        return F(0)  # only the bookkeeping margins subtract; they are not pinned here

    def __rsub__(self, x):
        return F(0)


class _Scaled:
    """u * s for s > 0, as ``sample`` forms it (compared against running sums)."""

    def __init__(self, u, s):
        self.u, self.s = u, s

    def __lt__(self, x):          # u s < x
        return self.u._below(F(x) / self.s)

    def __gt__(self, x):          # u s > x  <=>  not (u s < x) up to a null set
        return not self.u._below(F(x) / self.s)


class _LazyTokens:
    """Child tokens drawn from the parent's draft row on first read."""

    def __init__(self, assigned, m):
        self.assigned, self.m = assigned, m

    def __getitem__(self, i):
        if i not in self.assigned:
            raise _Split("tok", i)
        return self.assigned[i]

    def __len__(self):
        return self.m


def enumerate_walk(q_rows, p_rows, parents, mode, walk=None, tokens=None):
    """Exact law of (emitted tokens, path) of ``walk`` (default ``ot.walk``)
    over its uniforms and, in SAMPLED mode with ``tokens`` None, over the
    children's drafted tokens.  Returns {(emitted, path): Fraction}."""
    walk = walk or ot.walk
    m = len(parents)
    vocab = len(q_rows[0])
    law = {}
    stack = [({}, {})]  # (interval per counter, token per node index - 1)
    while stack:
        ivs, toks = stack.pop()

        def draw(j, kind, ivs=ivs):
            key = (j, kind)
            lo, hi = ivs.get(key, (F(0), F(1)))
            u = SymU(key, lo, hi)
            return (u, u, u, u) if kind == philox.SAMPLE_DRAW else u

        tok_seq = _LazyTokens(toks, m) if tokens is None else tokens
        try:
            emitted, path, a, kv, _ = walk(q_rows, p_rows, parents, tok_seq, mode, draw)
        except _Split as s:
            if s.kind == "u":
                lo, hi = ivs.get(s.key, (F(0), F(1)))
                for iv in ((lo, s.at), (s.at, hi)):
                    nxt = dict(ivs)
                    nxt[s.key] = iv
                    stack.append((nxt, toks))
            else:
                par = int(parents[s.key])
                for x in range(vocab):
                    if p_rows[par][x] > 0:
                        nxt = dict(toks)
                        nxt[s.key] = x
                        stack.append((ivs, nxt))
            continue
        assert kv == a + 1 and len(path) == a and len(emitted) == a + 1
        w = F(1)
        for lo, hi in ivs.values():
            w *= hi - lo
        if tokens is None:
            for i, x in toks.items():
                w *= p_rows[int(parents[i])][x]
        key = (tuple(int(t) for t in emitted), tuple(int(c) for c in path))
        law[key] = law.get(key, F(0)) + w
    return law


def slot_laws(law):
    """{path prefix: {token: P(slot |prefix| = token, path starts with prefix)}}."""
    out = {}
    for (emitted, path), w in law.items():
        for k in range(len(path) + 1):
            pre = path[:k]
            d = out.setdefault(pre, {})
            d[emitted[k]] = d.get(emitted[k], F(0)) + w
    return out


def check_slot_laws(law, q_rows):
    assert sum(law.values()) == 1
    vocab = len(q_rows[0])
    laws = slot_laws(law)
    assert () in laws
    for pre, dist in laws.items():
        node = pre[-1] if pre else 0
        total = sum(dist.values())
        for t in range(vocab):
            assert dist.get(t, F(0)) / total == q_rows[node][t], (pre, t, dist, q_rows[node])
    return laws


def fr(*nums):
    v = [F(n) for n in nums]
    s = sum(v)
    return np.array([x / s for x in v], dtype=object)


# A root with three children; child 1 has two children, child 4 one child;
# child 2 has one.  Distributions over V = 3 differ per node, with zeros.
# At the nodes with several children the residual changes after every
# rejection (root: (1/4, 3/4, 0) after one, (0, 1, 0) after two; node 1:
# (1/3, 2/3, 0), then (1/4, 3/4, 0)), so a walk that does not carry it from
# sibling to sibling is seen; at the root both the first and the second
# child's thresholds can lie strictly between 0 and 1 (1/5 for token 2,
# then 5/8 for token 0), so siblings that share a uniform are seen too.
PARENTS = [0, 0, 0, 1, 1, 4, 2]
Q_ROWS = [fr(5, 4, 1), fr(2, 3, 1), fr(2, 0, 3), fr(1, 1, 1), fr(5, 2, 1), fr(0, 1, 1), fr(4, 1, 1),
          fr(1, 2, 2)]
P_ROWS = [fr(4, 1, 5), fr(1, 1, 4), fr(1, 1, 0), None, fr(1, 3, 1), None, None, None]


@pytest.fixture(scope="module")
def sampled_law():
    return enumerate_walk(Q_ROWS, P_ROWS, PARENTS, ot.SAMPLED)


def test_sampled_tree_keeps_q_in_every_slot(sampled_law):
    laws = check_slot_laws(sampled_law, Q_ROWS)
    # the walk reaches depth 3 (root -> 1 -> 4 -> 6) with positive probability
    assert (1, 4, 6) in laws and (2,) in laws and (3,) in laws


# TOPK: fixed candidates, including a repeated sibling token and a token the
# verifier gives no mass at its node.
TOPK_TOKENS = [0, 2, 0, 1, 1, 2, 1]          # nodes 1..7
TOPK_Q = [fr(3, 1, 2), fr(1, 4, 1), fr(2, 0, 3), fr(1, 1, 1), fr(0, 2, 1), fr(0, 1, 1), fr(4, 1, 1),
          fr(1, 2, 2)]


def test_topk_tree_keeps_q_in_every_slot():
    law = enumerate_walk(TOPK_Q, None, PARENTS, ot.TOPK, tokens=TOPK_TOKENS)
    laws = check_slot_laws(law, TOPK_Q)
    assert (1, 4, 6) in laws


def test_two_level_binary_tree_both_modes():
    """The [2, 2] tree of exercise 3's shape, V = 4."""
    parents = list(ot.branching_tree((2, 2)))
    q = [fr(1, 2, 3, 4), fr(4, 1, 1, 2), fr(0, 3, 1, 1), fr(2, 2, 1, 1), fr(1, 0, 0, 1), fr(5, 1, 1, 1),
         fr(1, 1, 1, 3), ]
    p = [fr(2, 1, 1, 1), fr(1, 1, 3, 1), fr(1, 2, 0, 1), None, None, None, None]
    check_slot_laws(enumerate_walk(q, p, parents, ot.SAMPLED), q)
    check_slot_laws(enumerate_walk(q, None, parents, ot.TOPK, tokens=[3, 0, 1, 1, 2, 3]), q)


def test_one_child_per_node_matches_the_chain_law():
    """A line tree: slot k's law is q_k given the accepted prefix, and the
    acceptance at depth j given the walk reached it is sum min(p, q)."""
    parents = [0, 1]
    q = [fr(1, 2, 1), fr(3, 1, 1), fr(1, 1, 4)]
    p = [fr(2, 1, 1), fr(1, 1, 3), None]
    law = enumerate_walk(q, p, parents, ot.SAMPLED)
    check_slot_laws(law, q)
    for depth in (1, 2):
        reach = sum(w for (_, path), w in law.items() if len(path) >= depth - 1)
        acc = sum(w for (_, path), w in law.items() if len(path) >= depth)
        alpha = sum(min(a, b) for a, b in zip(q[depth - 1], p[depth - 1]))
        assert acc / reach == alpha


# ---------------------------------------------------------------- planted slips

def _mutated_walk(old, new):
    """``ot.walk`` with one source line edited (a planted mistake)."""
    src = textwrap.dedent(inspect.getsource(ot.walk))
    assert src.count(old) == 1, old
    ns = dict(vars(ot))
    exec(compile(src.replace(old, new), "<mutated walk>", "exec"), ns)
    return ns["walk"]


SLIPS = {
    # the residual is not carried to the next sibling: each rejection
    # restarts from the node's q
    "residual not carried": ("r = residual(r, p)", "r = residual(q_rows[node], p)"),
    # every sibling is tested with the same counter (draw 0), so their
    # uniforms are one and the same
    "siblings share a counter": ("u = draw_uniform(depth, accept_draw(i))",
                                 "u = draw_uniform(depth, accept_draw(0))"),
    # the i-th child's test takes draw i, so the second child asks for the
    # counter of the node's correction draw (four words where one is
    # expected: the walk fails outright)
    "draw i for child i": ("u = draw_uniform(depth, accept_draw(i))", "u = draw_uniform(depth, i)"),
    # a leaf's bonus drawn from the root's q
    "bonus from the root": ("t, margin = sample_grouped(q_rows[node], us)",
                            "t, margin = sample_grouped(q_rows[0], us)"),
}


@pytest.mark.parametrize("slip", sorted(SLIPS))
def test_planted_slips_break_the_pin(slip):
    walk = _mutated_walk(*SLIPS[slip])
    with pytest.raises((AssertionError, TypeError)):
        law = enumerate_walk(Q_ROWS, P_ROWS, PARENTS, ot.SAMPLED, walk=walk)
        check_slot_laws(law, Q_ROWS)


def test_planted_slip_in_topk_mode():
    walk = _mutated_walk(*SLIPS["residual not carried"])
    law = enumerate_walk(TOPK_Q, None, PARENTS, ot.TOPK, walk=walk, tokens=TOPK_TOKENS)
    with pytest.raises(AssertionError):
        check_slot_laws(law, TOPK_Q)


# ---------------------------------------------------------------- counters

@pytest.mark.parametrize("mode", [ot.SAMPLED, ot.TOPK])
def test_every_decision_takes_its_own_counter(mode):
    """On random trees and seeds, no Philox counter (depth, draw) is asked for
    twice within one walk, so every decision sees a fresh uniform."""
    rng = np.random.default_rng(3)
    vocab = 6
    for trial in range(200):
        m = int(rng.integers(1, 12))
        parents = [int(rng.integers(0, i + 1)) for i in range(m)]
        z = rng.normal(size=(m + 1, vocab))
        q = [np.exp(r) / np.exp(r).sum() for r in z]
        p = [np.exp(r + rng.normal(size=vocab)) for r in z]
        p = [x / x.sum() for x in p]
        toks = [int(rng.integers(0, vocab)) for _ in range(m)]
        seen = []
        base = ot.draws(trial, 0)

        def draw(j, kind):
            seen.append((j, kind))
            return base(j, kind)

        ot.walk(q, p if mode == ot.SAMPLED else None, parents, toks, mode, draw)
        assert len(seen) == len(set(seen)), seen


def test_the_counter_check_catches_a_shared_counter():
    walk = _mutated_walk(*SLIPS["siblings share a counter"])
    parents, vocab = [0, 0], 3
    q = [fr(1, 1, 1)] * 3
    toks = [0, 0]
    found = False
    for seed in range(50):
        seen = []
        base = ot.draws(seed, 0)

        def draw(j, kind):
            seen.append((j, kind))
            return base(j, kind)

        walk([np.array([float(x) for x in r]) for r in q], None, parents, toks, ot.TOPK, draw)
        found |= len(seen) != len(set(seen))
    assert found


def test_enumerator_reproduces_a_known_law():
    """The enumerator itself, on a one-node chain: accept with probability
    min(1, q(d)/p(d)) summed over d ~ p gives sum min(p, q), and the emitted
    token's law is q (the chain pin of the lesson's invariant)."""
    q, p = fr(1, 2, 3), fr(3, 2, 1)
    law = enumerate_walk([q, fr(1, 1, 1)], [p, None], [0], ot.SAMPLED)
    acc = sum(w for (_, path), w in law.items() if path)
    assert acc == sum(min(a, b) for a, b in zip(q, p)) == F(2, 3)
    first = {}
    for (emitted, _), w in law.items():
        first[emitted[0]] = first.get(emitted[0], F(0)) + w
    assert [first.get(t, F(0)) for t in range(3)] == list(q)
    assert list(itertools.accumulate(first[t] for t in range(3)))[-1] == 1
