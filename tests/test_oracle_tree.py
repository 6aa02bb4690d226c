"""Pins of the tree-verify oracle (CPU only).

* A tree with one child per node is the chain: same tokens, accepted
  lengths and KV lengths as ``oracle.verify`` on the same rows and seeds
  (sampled and greedy), which is itself pinned by the chain tests.
* Exact laws with fractions.Fraction: at a node whose children are
  independent draws from p (SAMPLED), or any fixed candidate list (TOPK),
  the law of the node's emitted token is exactly q -- recursive rejection
  sampling preserves the verifier's distribution.  A planted mistake in the
  residual breaks it.
* Monte Carlo over the whole walk of a two-level tree with Philox draws:
  the first emitted token follows q_root.
* Hand-checked greedy walks, topology helpers, error order.
"""

from fractions import Fraction as F
import itertools

import numpy as np
import pytest

from oracle import tree as ot
from oracle import verify as ov
from speculative_decoding_verification_73_gb300 import workloads


def _chain_tree(wl):
    """The chain workload as a tree: node i+1 under node i, draft row N unused."""
    b, n, v = wl.shape
    parents = np.tile(np.arange(n, dtype=np.int32), (b, 1))
    z, y = wl.raw()
    y_tree = np.concatenate([y, np.zeros_like(z[:, :1])], axis=1)
    return z, y_tree, parents


@pytest.mark.parametrize("gen_seed,dtype,vocab", [(11, "f32", 700), (12, "bf16", 1500), (13, "f32", 9000)])
def test_one_child_per_node_is_the_chain(gen_seed, dtype, vocab):
    wl = workloads.make_random(10, 5, vocab, dtype, gen_seed=gen_seed, verify_seed=gen_seed)
    z, y_tree, parents = _chain_tree(wl)
    temps = wl.temperature.numpy()
    for seed in (wl.seed, wl.seed + 101, 2 ** 63 + 7):
        chain = ov.verify(z, wl.raw()[1], wl.tokens.numpy(), temps, seed, dtype)
        tr = ot.verify_tree(z, y_tree, parents, wl.tokens.numpy(), temps, seed, dtype, ot.SAMPLED)
        np.testing.assert_array_equal(tr.tokens, chain.tokens)
        np.testing.assert_array_equal(tr.accept_len, chain.accept_len)
        np.testing.assert_array_equal(tr.kv_len, chain.kv_len)
        for b in range(10):
            a = int(chain.accept_len[b])
            np.testing.assert_array_equal(tr.path[b, :a], np.arange(1, a + 1))
            assert (tr.path[b, a:] == -1).all()


def _law_sampled(q, p, k):
    """Sum over k independent candidates x_i ~ p of the node's exact outcome."""
    vocab = len(q)
    law = np.array([F(0)] * vocab, dtype=object)
    for cands in itertools.product(range(vocab), repeat=k):
        w = F(1)
        for x in cands:
            w *= p[x]
        if w == 0:
            continue
        acc, final = ot.node_law(q, lambda i: p, list(cands))
        for i, x in enumerate(cands):
            law[x] += w * acc[i]
        law += w * final
    return law


def _fr(v):
    v = np.array([F(x) for x in v], dtype=object)
    return v / v.sum()


@pytest.mark.parametrize("q,p,k", [
    ((3, 1, 2), (1, 1, 1), 2),
    ((5, 1, 1, 3), (1, 4, 2, 1), 2),
    ((1, 6, 2, 1), (3, 1, 1, 5), 3),
    ((2, 0, 3, 1), (1, 2, 0, 4), 3),   # zeros on both sides
    ((1, 1, 1), (0, 0, 1), 2),          # p concentrated where q is small
])
def test_sampled_children_preserve_q_exactly(q, p, k):
    q, p = _fr(q), _fr(p)
    law = _law_sampled(q, p, k)
    assert list(law) == list(q)


@pytest.mark.parametrize("q,cands", [
    ((3, 1, 2, 4), [3, 0]),
    ((3, 1, 2, 4), [1, 2, 0]),
    ((1, 0, 5, 2), [1, 2]),        # a candidate the verifier gives no mass
    ((2, 3, 1), [0, 0, 2]),        # a repeated candidate
    ((1, 2, 3, 4, 5), [4, 3, 2, 1, 0]),
])
def test_fixed_candidates_preserve_q_exactly(q, cands):
    q = _fr(q)
    vocab = len(q)
    acc, final = ot.node_law(q, lambda i: ot.point_mass(vocab, cands[i], q), cands)
    law = final.copy()
    for i, x in enumerate(cands):
        law[x] += acc[i]
    assert list(law) == list(q)


def test_planted_residual_mistake_is_caught(monkeypatch):
    """Using (p - q)_+ as the residual (a sign slip) breaks the exact law."""
    q, p = _fr((3, 1, 2)), _fr((1, 1, 1))

    def wrong(r, pp):
        raw = np.maximum(pp - r, 0)
        s = raw.sum()
        return r.copy() if s == 0 else raw / s

    monkeypatch.setattr(ot, "residual", wrong)
    assert list(_law_sampled(q, p, 2)) != list(q)


def test_first_token_law_over_the_whole_walk():
    """Two-level tree, V = 5, children redrawn from p for each of 6000
    seeds: the first emitted token follows q_root (chi-square, 4 dof)."""
    rng = np.random.default_rng(5)
    vocab = 5
    parents = np.array([0, 0, 1, 1, 2], dtype=np.int32)
    z = rng.normal(size=(6, vocab))
    y = z + rng.normal(scale=0.8, size=(6, vocab))
    q = [ov.softmax(z[r], 1.0) for r in range(6)]
    p = [ov.softmax(y[r], 1.0) for r in range(6)]
    counts = np.zeros(vocab)
    trials = 6000
    for s in range(trials):
        toks = np.zeros(5, dtype=np.int64)
        for i, par in enumerate(parents):
            toks[i] = rng.choice(vocab, p=p[par])
        emitted, path, a, kv, _ = ot.walk(q, p, parents, toks, ot.SAMPLED, ot.draws(s, 0))
        counts[emitted[0]] += 1
    expect = trials * q[0]
    chi2 = float(((counts - expect) ** 2 / expect).sum())
    assert chi2 < 18.47, (chi2, counts, expect)  # 0.999 quantile, 4 dof


def test_greedy_walk_by_hand():
    # root argmax 2 -> child 2 (token 2); node 2's argmax 0 -> child 4
    # (token 0; child 3 has token 1); node 4 is a leaf with argmax 3.
    z = np.full((5, 4), -1.0)
    z[0, 2] = z[2, 0] = z[4, 3] = 1.0
    z[1, 1] = z[3, 1] = 1.0
    parents = [0, 0, 2, 2]
    tokens = [1, 2, 1, 0]
    emitted, path, a, kv = ot.greedy_walk(z, parents, tokens)
    assert path == [2, 4] and emitted == [2, 0, 3] and (a, kv) == (2, 3)
    # first matching child wins when two siblings carry the argmax
    emitted, path, _, _ = ot.greedy_walk(z, [0, 0, 0, 0], [2, 2, 1, 0])
    assert path == [1] and emitted == [2, 1]


def test_topology_helpers():
    par = ot.branching_tree((2, 2, 2))
    assert len(par) == 14
    kids = ot.children_of(par, 14)
    assert [len(k) for k in kids[:7]] == [2] * 7 and sum(1 for k in kids if not k) == 8
    np.testing.assert_array_equal(par, workloads.full_tree_parents((2, 2, 2)))
    assert ot.topology_is_valid(par, 14)
    assert not ot.topology_is_valid([0, 2], 2) and not ot.topology_is_valid([-1], 1)


def test_error_order():
    wl = workloads.make_tree(1, 40, "f32", gen_seed=3, widths=(2, 2), temps=(1.0,))
    z, y = wl.raw()
    par, tok = wl.parents.numpy().copy(), wl.tokens.numpy().copy()
    args = dict(seed=0, dtype="f32", mode=ot.SAMPLED)
    par[0, 3] = 5                       # node 4 under node 5: invalid
    tok[0, 0] = 40                      # out of range
    r = ot.verify_tree(z, y, par, tok, [float("nan")], **args)
    assert r.errors == ov.ERR_TEMP
    r = ot.verify_tree(z, y, par, tok, [1.0], **args)
    assert r.errors == ot.ERR_TREE and r.accept_len[0] == -1
    r = ot.verify_tree(z, y, wl.parents.numpy(), tok, [1.0], **args)
    assert r.errors == ov.ERR_TOKEN
    zz = z.copy()
    zz[0, 1, 3] = np.inf
    r = ot.verify_tree(zz, y, wl.parents.numpy(), wl.tokens.numpy(), [1.0], **args)
    assert r.errors == ov.ERR_LOGIT
    # a bad draft row of a leaf is never read
    yy = y.copy()
    yy[0, 6, 0] = np.nan
    r = ot.verify_tree(z, yy, wl.parents.numpy(), wl.tokens.numpy(), [1.0], **args)
    assert r.errors == 0


@pytest.mark.parametrize("shape", ["random", "star", "line"])
def test_255_node_trees_walk_validly(shape):
    """Trees of the largest size a context takes (255 draft nodes): the
    accepted path descends from the root along parent links, the emitted
    tokens are the path's tokens then one drawn token, and the lengths
    agree; greedy requests descend exactly while a child holds the argmax."""
    kw = {"random": {"m": 255}, "star": {"widths": (255,)}, "line": {"widths": (1,) * 255}}[shape]
    wl = workloads.make_tree(3, 1000, "f32", gen_seed=91, temps=(0.0, 0.7, 1.0), sigma=(0.0, 0.3),
                             verify_seed=4, **kw)
    res = ot.verify_tree(*wl.raw(), wl.parents.numpy(), wl.tokens.numpy(), wl.temperature.numpy(), 4,
                           wl.dtype, wl.mode)
    par, toks = wl.parents.numpy(), wl.tokens.numpy()
    z, _ = wl.raw()
    for b in range(3):
        assert res.request_errors[b] == 0
        a = int(res.accept_len[b])
        assert res.kv_len[b] == a + 1
        path = [int(x) for x in res.path[b][:a]]
        assert all(x == -1 for x in res.path[b][a:])
        node = 0
        for c in path:
            assert int(par[b, c - 1]) == node  # a child of the current node
            node = c
        emitted = [int(x) for x in res.tokens[b]]
        assert emitted[:a] == [int(toks[b, c - 1]) for c in path]
        assert 0 <= emitted[a] < 1000 and all(x == -1 for x in emitted[a + 1:])
        if float(wl.temperature[b]) == 0.0:
            # the walk stops at the first node none of whose children is the argmax
            rows = np.asarray(z[b], dtype=np.float64)
            kids = [i + 1 for i in range(par.shape[1]) if int(par[b, i]) == node]
            g = int(np.argmax(rows[node]))
            assert emitted[a] == g and all(int(toks[b, c - 1]) != g for c in kids)


LAZY_CASES = [
    dict(batch=12, vocab=3000, dtype="f32", gen_seed=401, widths=(2, 2, 2)),
    dict(batch=12, vocab=3000, dtype="bf16", gen_seed=402, widths=(3, 2)),
    dict(batch=10, vocab=2000, dtype="f32", gen_seed=403, m=20),
    dict(batch=10, vocab=2000, dtype="bf16", gen_seed=404, widths=(2, 2), mode=workloads.TREE_TOPK),
]


@pytest.mark.parametrize("case", range(len(LAZY_CASES)))
def test_lazy_reading_equals_the_eager_one_on_valid_rows(case):
    """Reading a node's rows only when the walk reaches it changes nothing
    on valid inputs (greedy, sampled and TOPK requests, fixed and random
    topologies, three seeds)."""
    wl = workloads.make_tree(**LAZY_CASES[case])
    z, y = wl.raw()
    for seed in (0, 7, 2 ** 64 - 1):
        args = (z, y, wl.parents.numpy(), wl.tokens.numpy(), wl.temperature.numpy(), seed, wl.dtype, wl.mode)
        e, l = ot.verify_tree(*args), ot.verify_tree(*args, lazy=True)
        assert e.errors == l.errors == 0
        for a, b in ((e.tokens, l.tokens), (e.path, l.path), (e.accept_len, l.accept_len), (e.kv_len, l.kv_len)):
            assert np.array_equal(a, b)


def test_lazy_reading_checks_only_the_rows_it_reads():
    """A NaN in the target row (or +inf in the draft row) of a node the walk
    never reaches fails the eager reading but not the lazy one, whose outputs
    stay those of the clean input; the same NaN in the root's row fails both."""
    wl = workloads.make_tree(16, 500, "f32", gen_seed=405, widths=(2, 2, 2), temps=(0.0, 1.0))
    z, y = wl.raw()
    par, tok, temp = wl.parents.numpy(), wl.tokens.numpy(), wl.temperature.numpy()
    clean = ot.verify_tree(z, y, par, tok, temp, 3, "f32", ot.SAMPLED)
    assert clean.errors == 0
    zz, yy = z.copy(), y.copy()
    kids = [ot.children_of([int(v) for v in par[b]], par.shape[1]) for b in range(par.shape[0])]
    planted = 0
    for b in range(par.shape[0]):
        seen = {0} | {int(n) for n in clean.path[b] if n >= 0}
        off = [n for n in range(1, par.shape[1] + 1) if n not in seen]
        zz[b, off[0], 7] = np.nan
        inner_off = [n for n in off if kids[b][n]]
        if inner_off and temp[b] > 0:
            yy[b, inner_off[0], 11] = np.inf
        planted += 1
    assert planted == par.shape[0]
    eager = ot.verify_tree(zz, yy, par, tok, temp, 3, "f32", ot.SAMPLED)
    lazy = ot.verify_tree(zz, yy, par, tok, temp, 3, "f32", ot.SAMPLED, lazy=True)
    assert eager.errors == ov.ERR_LOGIT and (eager.accept_len == -1).all()
    assert lazy.errors == 0
    for a, b in ((clean.tokens, lazy.tokens), (clean.path, lazy.path), (clean.accept_len, lazy.accept_len)):
        assert np.array_equal(a, b)
    zr = z.copy()
    zr[:, 0, 5] = np.nan
    both = [ot.verify_tree(zr, y, par, tok, temp, 3, "f32", ot.SAMPLED, lazy=lz) for lz in (False, True)]
    assert all(r.errors == ov.ERR_LOGIT and (r.accept_len == -1).all() for r in both)
