"""CPU oracle of draft-tree verification (test infrastructure only).

Source: the "Speculative Decoding and EAGLE-3" lesson (factory.pai-world.com,
phase 10 lesson 15): the "Key terms" entry on EAGLE-2 (the drafter proposes
a small candidate tree instead of one sequence, the verifier scores every
candidate in one forward pass under a tree mask, and the walk follows the
most probable path), the section "KV cache rollback" (tree attention with a
non-causal mask over the tree topology), exercise 3 (a [2, 2, 2] tree: eight
candidate paths, one verifier pass, the most probable accepted path is
kept), and "Invariant: Leviathan rejection sampling" for the per-node test.

Readings of points the pages leave open:

* Layout.  Node 0 is the root (the last verified token); draft nodes are
  1..M, node i's parent is ``parents[i-1]`` in [0, i-1] (topological
  order) and its token is ``tokens[i-1]``.  Target row r is the verifier's
  next-token distribution after node r (row 0: after the root); draft row r
  is the drafter's distribution from which node r's children were drawn.
* The walk starts at the root with depth 1.  At a node, its children are
  tried in increasing node index (the tree builder lists siblings most
  probable first, so the first accepted child is the most probable accepted
  branch).  Child c with token x is tested with the Leviathan rule against
  the node's current distribution r (initially q_node): accept iff
  p(x) <= 0 or u < min(1, r(x) / p(x)).  Accepting moves the walk to c at
  depth + 1.  Rejecting replaces r by the residual (r - p)_+ normalised
  (r itself if that is all zero) and the next sibling is tried.  When every
  child is rejected, one token is drawn from the final r; when the walk
  reaches a leaf, a bonus token is drawn from that leaf's q.  With one child
  per node this is exactly the chain of ``verify.walk``.
* Two drafting modes.  SAMPLED: the children are independent draws from
  the drafter's distribution p at the node (draft logits are read); the
  rule above then preserves q (recursive rejection sampling).  TOPK: the
  children are fixed candidates (for instance the drafter's top-k); each
  is then a draw from a point mass on its own token, so p = 1 at x and 0
  elsewhere: accept iff u < r(x), and the residual is r with x zeroed and
  renormalised.  Draft logits are not read.  This also preserves q.
* Uniforms: the test of the i-th child tried (0-based) at depth j uses
  Philox counter (b, j, draw, 0) with draw 0 for i = 0 and draw i + 1 for
  i >= 1; the token drawn at depth j (correction or bonus) uses draw 1 and
  the grouped inverse CDF of ``verify.sample_grouped``.  A one-child-per-
  node tree therefore consumes exactly the chain's draws.
* T = 0: the child whose token equals the argmax of the node's target row
  (lowest index on ties) is accepted, the first such child in index order;
  if none, or at a leaf, the argmax is emitted.  Draft logits are not read.
* Outputs: the tokens of the accepted path then the drawn token (-1
  padding), the accepted node indices (-1 padding), accepted = path
  length, KV length = accepted + 1.
* Errors, checked in this order: temperature, topology (a parent index
  outside [0, i-1]), tokens (outside [0, V)), logits (every target row, and
  in SAMPLED mode the draft rows of nodes that have children, must be
  valid rows as in ``verify.row_is_valid``).
* The lazy reading (``lazy=True``): the walk reads a node's rows only when
  it reaches the node, and the rows of nodes it never reaches do not enter
  the result (a node's children are tested against that node's rows
  alone), so only the rows it reads are checked: the same outputs on valid
  inputs, and a bad row off the walked path is not an error.

Floating point is float64; ``node_law`` drives the same accept and
residual code with exact ``fractions.Fraction`` arrays for the pins.
"""

import numpy as np

from . import philox
from .verify import (ERR_LOGIT, ERR_TEMP, ERR_TOKEN, Decision, argmax_lowest, logits_to_f64,
                     residual, row_is_valid, sample_grouped, softmax, temperature_is_valid)

SAMPLED = 0
TOPK = 1

ERR_TREE = 8


def accept_draw(i):
    """Philox draw index of the test of the i-th child tried at a node."""
    return philox.ACCEPT_DRAW if i == 0 else i + 1


def accept_threshold(r_x, p_x):
    """min(1, r(x) / p(x)), or 1 when the drafter gives x no mass (then the
    rule accepts whatever u is)."""
    if p_x <= 0:
        return 1
    return min(1, r_x / p_x)


def point_mass(vocab, x, like):
    """The drafter's law of a fixed candidate x: 1 at x, 0 elsewhere."""
    p = np.zeros(vocab, dtype=like.dtype) if like.dtype != object else np.array([0] * vocab, dtype=object)
    p[x] = 1
    return p


def children_of(parents, m):
    """Children of each node 0..m in increasing index order."""
    kids = [[] for _ in range(m + 1)]
    for i in range(m):
        kids[int(parents[i])].append(i + 1)
    return kids


def topology_is_valid(parents, m):
    return all(0 <= int(parents[i]) <= i for i in range(m))


def node_law(q, p_for, cand_tokens):
    """Exact law of one node's outcome, for pins: returns (accept, final)
    where accept[i] is the probability that the i-th candidate is the one
    accepted and final is the distribution the token is drawn from when all
    are rejected, weighted by the probability of that event.  ``p_for(i)``
    is the drafter's law of candidate i.  Uses the walk's own rules."""
    r = q
    stay = 1
    accept = []
    for i, x in enumerate(cand_tokens):
        p = p_for(i)
        a = accept_threshold(r[x], p[x])
        accept.append(stay * a)
        stay = stay * (1 - a)
        r = residual(r, p)
    return accept, r * stay


def walk(q_rows, p_rows, parents, tokens, mode, draw_uniform):
    """The sampled tree walk of one request.  q_rows[r] / p_rows[r]: target
    / drafter distributions at node r (p_rows unused in TOPK mode);
    draw_uniform(j, draw) as in ``verify.walk``.

    Returns (emitted tokens, path node indices, accepted, kv_len, decisions).
    """
    m = len(tokens)
    kids = children_of(parents, m)
    node, depth = 0, 1
    path, emitted, decisions = [], [], []
    while True:
        if not kids[node]:
            us = draw_uniform(depth, philox.SAMPLE_DRAW)
            t, margin = sample_grouped(q_rows[node], us)
            decisions.append(Decision("bonus", depth, us, margin=margin, taken=t))
            break
        r = q_rows[node]
        moved = False
        for i, c in enumerate(kids[node]):
            x = int(tokens[c - 1])
            p = p_rows[node] if mode == SAMPLED else point_mass(len(r), x, r)
            u = draw_uniform(depth, accept_draw(i))
            thr = accept_threshold(r[x], p[x])
            ok = p[x] <= 0 or u < thr
            decisions.append(Decision("accept", depth, u, threshold=None if p[x] <= 0 else thr, taken=ok))
            if ok:
                path.append(c)
                emitted.append(x)
                node, depth, moved = c, depth + 1, True
                break
            r = residual(r, p)
        if not moved:
            us = draw_uniform(depth, philox.SAMPLE_DRAW)
            t, margin = sample_grouped(r, us)
            decisions.append(Decision("residual", depth, us, margin=margin, taken=t))
            break
    emitted.append(t)
    return emitted, path, len(path), len(path) + 1, decisions


def greedy_walk(z_rows, parents, tokens):
    """Temperature-0 tree walk: descend into the first child whose token is
    the argmax of the node's target row; emit the argmax where none is."""
    m = len(tokens)
    kids = children_of(parents, m)
    node = 0
    path, emitted = [], []
    while True:
        g = argmax_lowest(z_rows[node])
        nxt = next((c for c in kids[node] if int(tokens[c - 1]) == g), None)
        emitted.append(g)
        if nxt is None:
            break
        path.append(nxt)
        node = nxt
    return emitted, path, len(path), len(path) + 1


def draws(seed, b):
    def draw(j, kind):
        if kind == philox.SAMPLE_DRAW:
            return philox.uniforms4(seed, b, j, kind)
        return philox.uniform(seed, b, j, kind)
    return draw


class _BadRow(Exception):
    """A row the lazy walk read is not a valid row."""


class _RowsOnUse:
    """Rows widened, checked and transformed when the walk first reads them
    (the lazy reading)."""

    def __init__(self, raw, dtype, make):
        self.raw, self.dtype, self.make, self.cache = raw, dtype, make, {}

    def __getitem__(self, r):
        if r not in self.cache:
            x = logits_to_f64(self.raw[r], self.dtype)
            if not row_is_valid(x):
                raise _BadRow
            self.cache[r] = self.make(x)
        return self.cache[r]


def verify_request(z_raw, y_raw, parents, tokens, temperature, seed, b, dtype, mode, lazy=False):
    """One request: z_raw [M+1, V], y_raw [M+1, V] (None in TOPK mode or at
    T = 0), parents [M], tokens [M]; ``lazy`` selects the lazy reading.

    Returns (err_bit, emitted, path, accepted, kv_len, decisions).
    """
    z_raw = np.asarray(z_raw)
    m = z_raw.shape[0] - 1
    vocab = z_raw.shape[1]
    t = float(np.float32(temperature))
    if not temperature_is_valid(t):
        return ERR_TEMP, None, None, None, None, []
    parents = [int(x) for x in np.asarray(parents).reshape(-1)[:m]]
    if not topology_is_valid(parents, m):
        return ERR_TREE, None, None, None, None, []
    tokens = [int(x) for x in np.asarray(tokens).reshape(-1)[:m]]
    if any(x < 0 or x >= vocab for x in tokens):
        return ERR_TOKEN, None, None, None, None, []
    if lazy:
        try:
            if t == 0.0:
                emitted, path, a, kv = greedy_walk(_RowsOnUse(z_raw, dtype, lambda x: x), parents, tokens)
                return 0, emitted, path, a, kv, []
            q_rows = _RowsOnUse(z_raw, dtype, lambda x: softmax(x, t))
            p_rows = _RowsOnUse(y_raw, dtype, lambda x: softmax(x, t)) if mode == SAMPLED else None
            emitted, path, a, kv, dec = walk(q_rows, p_rows, parents, tokens, mode, draws(seed, b))
            return 0, emitted, path, a, kv, dec
        except _BadRow:
            return ERR_LOGIT, None, None, None, None, []
    z = logits_to_f64(z_raw, dtype)
    if not all(row_is_valid(z[r]) for r in range(m + 1)):
        return ERR_LOGIT, None, None, None, None, []
    if t == 0.0:
        emitted, path, a, kv = greedy_walk(z, parents, tokens)
        return 0, emitted, path, a, kv, []
    kids = children_of(parents, m)
    q_rows = [softmax(z[r], t) for r in range(m + 1)]
    p_rows = None
    if mode == SAMPLED:
        y = logits_to_f64(y_raw, dtype)
        inner = [r for r in range(m + 1) if kids[r]]
        if not all(row_is_valid(y[r]) for r in inner):
            return ERR_LOGIT, None, None, None, None, []
        p_rows = [softmax(y[r], t) if kids[r] else None for r in range(m + 1)]
    emitted, path, a, kv, dec = walk(q_rows, p_rows, parents, tokens, mode, draws(seed, b))
    return 0, emitted, path, a, kv, dec


class TreeResult:
    """Outputs of one batched tree verify, laid out like the library's."""

    def __init__(self, batch, m):
        self.tokens = np.full((batch, m + 1), -1, dtype=np.int32)
        self.path = np.full((batch, m), -1, dtype=np.int32)
        self.accept_len = np.zeros(batch, dtype=np.int32)
        self.kv_len = np.zeros(batch, dtype=np.int32)
        self.errors = 0
        self.request_errors = np.zeros(batch, dtype=np.int32)
        self.decisions = [[] for _ in range(batch)]


def verify_tree(target, draft, parents, tokens, temperature, seed, dtype, mode, lazy=False):
    """Batched tree verify: target [B, M+1, V], draft [B, M+1, V] (None when
    unused), parents [B, M], tokens [B, M], temperature [B], 64-bit seed;
    ``lazy`` selects the lazy reading (rows checked only where the walk
    reads them).  Failed requests get tokens and path -1, accept_len -1,
    kv_len 0."""
    target = np.asarray(target)
    batch, m1, _ = target.shape
    m = m1 - 1
    res = TreeResult(batch, m)
    parents = np.asarray(parents).reshape(batch, m)
    tokens = np.asarray(tokens).reshape(batch, m)
    temperature = np.asarray(temperature, dtype=np.float32).reshape(batch)
    for b in range(batch):
        y_b = None if draft is None else np.asarray(draft[b])
        err, emitted, path, a, kv, dec = verify_request(
            target[b], y_b, parents[b], tokens[b], temperature[b], seed, b, dtype, mode, lazy)
        if err:
            res.errors |= err
            res.request_errors[b] = err
            res.accept_len[b] = -1
            continue
        res.tokens[b, :len(emitted)] = emitted
        res.path[b, :len(path)] = path
        res.accept_len[b] = a
        res.kv_len[b] = kv
        res.decisions[b] = dec
    return res


def branching_tree(widths):
    """Parents of a full tree in breadth-first order: ``widths[d]`` children
    under every node of depth d (the pages' [2, 2, 2] tree is
    ``branching_tree((2, 2, 2))``: 14 draft nodes, 8 leaves)."""
    parents, level = [], [0]
    nxt_id = 1
    for w in widths:
        new = []
        for node in level:
            for _ in range(w):
                parents.append(node)
                new.append(nxt_id)
                nxt_id += 1
        level = new
    return np.array(parents, dtype=np.int32)
