"""Plain CPU oracle of the batched draft-verify step (test infrastructure only).

Source: the "Speculative Decoding and EAGLE-3" lesson
(factory.pai-world.com, phase 10 lesson 15), sections

* "Invariant: Leviathan rejection sampling" -- the draft p, the verifier
  q, accept d ~ p with probability min(1, q(d)/p(d)), otherwise sample the
  residual (q - p)_+ / ||(q - p)_+||_1; one verifier pass over
  prefix + d_1..d_N returns q_1..q_{N+1}; walk left to right, stop at the
  first rejection with a residual sample, and add a bonus token from
  q_{N+1} when every draft is accepted;
* "Build it", step 1 (rejection rule: a draft with p(d) <= 0 is accepted,
  otherwise accept iff u < min(1, q/p)), step 2 (residual: fall back to q
  when the positive part sums to zero), step 3 (the full speculative step)
  and step 4 (KV rollback bookkeeping);
* "KV cache rollback" -- on a rejection at position j the logical length
  stops right after the correction token.

Temperature and the greedy path come from the method statement this
library implements: rows are softmaxed at the request's temperature T, and
T = 0 is argmax matching.

Readings of points the pages leave open:

* both the target and the draft rows use the request's T;
* a valid T is 0 (greedy) or a finite float32 >= 2^-126; anything else
  (negative, NaN, inf, subnormal) is a per-request temperature error;
* the uniform u is the Philox draw in ``oracle.philox``;
* a correction or bonus token is drawn by a grouped inverse CDF: the
  vocabulary is split into blocks of 2^13 consecutive tokens, each block
  into blocks of 2^8, then 2^4, then single tokens; at each of these four
  levels one sub-block is chosen by inverse CDF over the sub-blocks' masses
  (smallest index whose running sum exceeds u times the total; the last
  one with mass if rounding leaves none), each level with its own uniform.
  This draws exactly from the normalised residual (or q), and each
  decision compares u against at most max(V / 2^13, 32) bucket edges;
* greedy ties go to the lowest vocabulary index; draft logits are not read
  at T = 0; a draft is accepted iff it equals the row's argmax, and the
  emitted token after the first mismatch (or after N matches) is the
  argmax of the next target row;
* the KV length to commit from this window is accepted + 1 (the verified
  input token plus the accepted drafts), the same on rejection and on full
  acceptance;
* a logit row holding NaN or +inf, or whose maximum is -inf, is a
  per-request logit error; -inf entries are allowed and mean probability 0.

Floating point is float64 throughout.  ``residual`` and ``sample`` are
written with numpy operations that also run on object arrays of
``fractions.Fraction``, so the exact-enumeration tests drive this very code.
"""

import math

import numpy as np

from . import philox

# Per-request error bits, checked in this order (the first failing check
# is the one reported for the request).
ERR_TEMP = 1
ERR_TOKEN = 2
ERR_LOGIT = 4

FLT_MIN_NORMAL = 2.0 ** -126


# --------------------------------------------------------------------------
# Input widening
# --------------------------------------------------------------------------

def logits_to_f64(raw, dtype):
    """Widen stored logits to float64 exactly.

    ``dtype`` is "f32" (``raw`` holds float32 values) or "bf16" (``raw``
    holds the 16-bit patterns as uint16: a bfloat16 is the top half of an
    IEEE binary32, so shifting the pattern left by 16 gives that float32).
    """
    if dtype == "f32":
        return np.asarray(raw, dtype=np.float32).astype(np.float64)
    if dtype == "bf16":
        bits = np.asarray(raw, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        with np.errstate(invalid="ignore"):  # NaN patterns stay NaN
            return bits.view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def row_is_valid(x):
    """A row is usable iff it has no NaN, no +inf and a finite maximum."""
    if np.any(np.isnan(x)) or np.any(x == np.inf):
        return False
    return bool(np.max(x) > -np.inf)


def temperature_is_valid(t):
    t = float(t)
    return t == 0.0 or (math.isfinite(t) and t >= FLT_MIN_NORMAL)


# --------------------------------------------------------------------------
# One row: temperature softmax
# --------------------------------------------------------------------------

def softmax(x, temperature):
    """softmax(x / T) in float64: subtract the row maximum, exponentiate,
    divide by the sum.  -inf entries get probability 0."""
    s = np.asarray(x, dtype=np.float64) / float(temperature)
    m = np.max(s)
    e = np.exp(s - m)
    return e / np.sum(e)


def log_partition(x, temperature):
    """logZ = log sum_t exp(x_t / T), float64 (for row-statistic parity)."""
    s = np.asarray(x, dtype=np.float64) / float(temperature)
    m = np.max(s)
    return float(m + np.log(np.sum(np.exp(s - m))))


# --------------------------------------------------------------------------
# The three page-level operations
# --------------------------------------------------------------------------

def accept(q_prob, p_prob, u):
    """Rejection rule: a draft the drafter gives no mass is accepted;
    otherwise accept iff u < min(1, q(d) / p(d))."""
    if p_prob <= 0:
        return True
    return u < min(1, q_prob / p_prob)


def residual(q, p):
    """(q - p)_+ normalised to sum 1; q itself if the positive part is 0."""
    raw = np.maximum(q - p, 0)
    s = np.sum(raw)
    if s == 0:
        return q.copy()
    return raw / s


def sample(masses, u):
    """Inverse CDF over a short list of masses.

    Returns ``(c, margin)``: c is the smallest index whose running sum C_c
    exceeds u times the total (the last index with mass > 0 if none does,
    which only rounding can cause), and margin = min(|u - C_{c-1}/M|,
    |u - C_c/M|) is how far u sits from the edges of c's bucket in units of
    the total M (C_{-1} = 0).
    """
    c_sum = np.cumsum(masses)
    total = c_sum[-1]
    above = np.nonzero(c_sum > u * total)[0]
    if len(above):
        c = int(above[0])
    else:
        c = int(np.nonzero(masses > 0)[0][-1])
    lo = c_sum[c - 1] if c > 0 else 0
    margin = min(abs(u - lo / total), abs(u - c_sum[c] / total))
    return c, margin


# Token groups of the grouped inverse CDF: level 1 splits the vocabulary
# into blocks of 2^13 consecutive tokens, level 2 a block into blocks of
# 2^8, level 3 into blocks of 2^4, level 4 into single tokens.
LEVEL_SHIFTS = (13, 8, 4, 0)


def sample_grouped(dist, us):
    """Draw a token from ``dist`` (any non-negative masses) with four
    uniforms, one per level: at each level the current block is split into
    consecutive sub-blocks (sizes 2^13, 2^8, 2^4, 1) and one is chosen by
    ``sample`` over their masses.  The chance of token t is the product of
    its blocks' conditional masses, which telescopes to dist[t] / sum(dist),
    so this is an exact draw from the normalised ``dist``.

    Returns ``(t, margins)`` with the margin of each level's choice.
    """
    lo, hi = 0, len(dist)
    margins = []
    for level, shift in enumerate(LEVEL_SHIFTS):
        size = 1 << shift
        starts = list(range(lo, hi, size))
        masses = np.array([np.sum(dist[s:min(s + size, hi)]) for s in starts], dtype=dist.dtype)
        c, margin = sample(masses, us[level])
        margins.append(margin)
        lo = starts[c]
        hi = min(lo + size, hi)
    return lo, margins


# --------------------------------------------------------------------------
# One request
# --------------------------------------------------------------------------

class Decision:
    """One random decision of the walk, for near-threshold bookkeeping.

    kind is "accept" (threshold = min(1, q/p), or None when p(d) <= 0),
    "residual" or "bonus" (margin = for each level of the grouped inverse
    CDF, the distance of that level's uniform to its bucket edges).
    """

    __slots__ = ("kind", "j", "u", "threshold", "margin", "taken")

    def __init__(self, kind, j, u, threshold=None, margin=None, taken=None):
        self.kind, self.j, self.u = kind, j, u
        self.threshold, self.margin, self.taken = threshold, margin, taken

    def distance(self, level=None):
        """How close the uniform(s) came to flipping this decision (at one
        level of a sampling decision, or the closest level)."""
        if self.kind == "accept":
            if self.threshold is None:
                return math.inf
            return abs(self.u - self.threshold)
        if level is not None:
            return self.margin[level]
        return min(self.margin)

    def __repr__(self):
        return (f"Decision({self.kind}, j={self.j}, u={self.u!r}, "
                f"thr={self.threshold!r}, margin={self.margin!r}, taken={self.taken!r})")


def walk(q_rows, p_rows, drafts, draw_uniform):
    """The sampled chain for one request.

    q_rows: N+1 verifier distributions q_1..q_{N+1}; p_rows: N draft
    distributions p_1..p_N; drafts: d_1..d_N; draw_uniform(j, draw) gives,
    for 1-based position j, the uniform of draw 0 (accept) or the four
    uniforms of draw 1 (correction / bonus, one per level of
    ``sample_grouped``).

    Returns (tokens, accepted, kv_len, decisions): tokens are the accepted
    drafts followed by one correction or bonus token.
    """
    n = len(drafts)
    tokens, decisions = [], []
    for j in range(1, n + 1):
        d = int(drafts[j - 1])
        q_d, p_d = q_rows[j - 1][d], p_rows[j - 1][d]
        u = draw_uniform(j, philox.ACCEPT_DRAW)
        ok = accept(q_d, p_d, u)
        thr = None if p_d <= 0 else min(1, q_d / p_d)
        decisions.append(Decision("accept", j, u, threshold=thr, taken=ok))
        if ok:
            tokens.append(d)
            continue
        r = residual(q_rows[j - 1], p_rows[j - 1])
        u2 = draw_uniform(j, philox.SAMPLE_DRAW)
        t, margin = sample_grouped(r, u2)
        decisions.append(Decision("residual", j, u2, margin=margin, taken=t))
        tokens.append(t)
        accepted = j - 1
        return tokens, accepted, accepted + 1, decisions
    u2 = draw_uniform(n + 1, philox.SAMPLE_DRAW)
    t, margin = sample_grouped(q_rows[n], u2)
    decisions.append(Decision("bonus", n + 1, u2, margin=margin, taken=t))
    tokens.append(t)
    return tokens, n, n + 1, decisions


def philox_draws(seed, b):
    """The uniform provider of request b for ``walk``."""
    def draw(j, kind):
        if kind == philox.ACCEPT_DRAW:
            return philox.uniform(seed, b, j, kind)
        return philox.uniforms4(seed, b, j, kind)
    return draw


def argmax_lowest(x):
    """Index of the maximum, lowest index among equal maxima."""
    return int(np.argmax(x))  # numpy returns the first occurrence


def greedy_walk(z_rows, drafts):
    """Temperature-0 chain: accept d_j iff d_j = argmax z_j; the token after
    the accepted prefix is the argmax of the next target row."""
    n = len(drafts)
    tokens = []
    for j in range(1, n + 1):
        g = argmax_lowest(z_rows[j - 1])
        tokens.append(g)
        if int(drafts[j - 1]) != g:
            return tokens, j - 1, j
    tokens.append(argmax_lowest(z_rows[n]))
    return tokens, n, n + 1


def verify_request(z_raw, y_raw, drafts, temperature, seed, b, dtype):
    """One request.  z_raw: [N+1, V], y_raw: [N, V] or None, drafts: [N].

    Returns (err_bit, tokens, accepted, kv_len, decisions); err_bit is 0 or
    one of ERR_*.
    """
    z_raw = np.asarray(z_raw)
    n = z_raw.shape[0] - 1
    vocab = z_raw.shape[1]
    t = float(np.float32(temperature))
    if not temperature_is_valid(t):
        return ERR_TEMP, None, None, None, []
    drafts = [int(x) for x in np.asarray(drafts).reshape(-1)[:n]]
    if any(d < 0 or d >= vocab for d in drafts):
        return ERR_TOKEN, None, None, None, []
    z = logits_to_f64(z_raw, dtype)
    if not all(row_is_valid(z[j]) for j in range(n + 1)):
        return ERR_LOGIT, None, None, None, []
    if t == 0.0:
        tokens, a, kv = greedy_walk(z, drafts)
        return 0, tokens, a, kv, []
    y = logits_to_f64(y_raw, dtype) if n > 0 else np.zeros((0, vocab))
    if not all(row_is_valid(y[j]) for j in range(n)):
        return ERR_LOGIT, None, None, None, []
    q_rows = [softmax(z[j], t) for j in range(n + 1)]
    p_rows = [softmax(y[j], t) for j in range(n)]
    tokens, a, kv, decisions = walk(
        q_rows, p_rows, drafts, philox_draws(seed, b))
    return 0, tokens, a, kv, decisions


def verify_request_lazy(z_raw, y_raw, drafts, temperature, seed, b, dtype):
    """The lazy reading of one request: the same walk, but a row is only
    read (and so only checked) when the walk reaches it -- target and draft
    row j-1 for the test at position j, target row N for the bonus.  Rows
    past the point where the walk stops are never looked at, so a bad row
    there is not an error.  Otherwise identical to ``verify_request``."""
    z_raw = np.asarray(z_raw)
    n = z_raw.shape[0] - 1
    vocab = z_raw.shape[1]
    t = float(np.float32(temperature))
    if not temperature_is_valid(t):
        return ERR_TEMP, None, None, None, []
    drafts = [int(x) for x in np.asarray(drafts).reshape(-1)[:n]]
    if any(d < 0 or d >= vocab for d in drafts):
        return ERR_TOKEN, None, None, None, []
    z = logits_to_f64(z_raw, dtype)
    y = logits_to_f64(y_raw, dtype) if (n > 0 and t != 0.0) else None

    class _Bad(Exception):
        pass

    def target(j):
        if not row_is_valid(z[j]):
            raise _Bad
        return z[j]

    def draft(j):
        if not row_is_valid(y[j]):
            raise _Bad
        return y[j]

    try:
        if t == 0.0:
            tokens = []
            for j in range(1, n + 1):
                g = argmax_lowest(target(j - 1))
                tokens.append(g)
                if drafts[j - 1] != g:
                    return 0, tokens, j - 1, j, []
            tokens.append(argmax_lowest(target(n)))
            return 0, tokens, n, n + 1, []
        q_rows = _LazyRows(lambda j: softmax(target(j), t))
        p_rows = _LazyRows(lambda j: softmax(draft(j), t))
        tokens, a, kv, decisions = walk(q_rows, p_rows, drafts, philox_draws(seed, b))
        return 0, tokens, a, kv, decisions
    except _Bad:
        return ERR_LOGIT, None, None, None, []


class _LazyRows:
    """Rows computed on first use (for the lazy reading)."""

    def __init__(self, make):
        self.make, self.cache = make, {}

    def __getitem__(self, j):
        if j not in self.cache:
            self.cache[j] = self.make(j)
        return self.cache[j]


# --------------------------------------------------------------------------
# The batch
# --------------------------------------------------------------------------

class Result:
    """Outputs of one batched verify call, laid out like the library's."""

    def __init__(self, batch, n):
        self.tokens = np.full((batch, n + 1), -1, dtype=np.int32)
        self.accept_len = np.zeros(batch, dtype=np.int32)
        self.kv_len = np.zeros(batch, dtype=np.int32)
        self.errors = 0
        self.request_errors = np.zeros(batch, dtype=np.int32)
        self.decisions = [[] for _ in range(batch)]


def verify(target, draft, drafts, temperature, seed, dtype, lazy=False):
    """Batched verify: target [B, N+1, V], draft [B, N, V] (may be None when
    every T is 0), drafts [B, N] int, temperature [B] float32, 64-bit seed;
    ``lazy`` selects ``verify_request_lazy`` (rows checked only when read).

    A request that fails a check gets tokens -1, accept_len -1, kv_len 0,
    and its error bit is OR-ed into ``errors``.
    """
    target = np.asarray(target)
    batch, n1, _ = target.shape
    n = n1 - 1
    res = Result(batch, n)
    drafts = np.asarray(drafts).reshape(batch, n)
    temperature = np.asarray(temperature, dtype=np.float32).reshape(batch)
    for b in range(batch):
        y_b = None if draft is None or n == 0 else np.asarray(draft[b])
        one = verify_request_lazy if lazy else verify_request
        err, tokens, a, kv, dec = one(target[b], y_b, drafts[b], temperature[b], seed, b, dtype)
        if err:
            res.errors |= err
            res.request_errors[b] = err
            res.accept_len[b] = -1
            res.kv_len[b] = 0
            continue
        res.tokens[b, :len(tokens)] = tokens
        res.accept_len[b] = a
        res.kv_len[b] = kv
        res.decisions[b] = dec
    return res


def acceptance_probabilities(target, draft, drafts, temperature, dtype):
    """min(1, q_j(d_j) / p_j(d_j)) for every (b, j) of sampled requests
    (NaN for greedy requests), plus logZ of every row (NaN for rows a greedy
    request does not normalise).  Used for the 1e-5 relative parity of the
    row statistics."""
    target = np.asarray(target)
    batch, n1, _ = target.shape
    n = n1 - 1
    probs = np.full((batch, n), np.nan)
    logz_t = np.full((batch, n + 1), np.nan)
    logz_d = np.full((batch, n), np.nan)
    vocab = target.shape[2]
    for b in range(batch):
        t = float(np.float32(temperature[b]))
        if t == 0.0 or not temperature_is_valid(t):
            continue
        if any(int(x) < 0 or int(x) >= vocab for x in np.asarray(drafts[b]).reshape(-1)[:n]):
            continue
        z = logits_to_f64(target[b], dtype)
        y = logits_to_f64(draft[b], dtype) if n > 0 else None
        if not all(row_is_valid(r) for r in z) or (n > 0 and not all(row_is_valid(r) for r in y)):
            continue
        for j in range(n + 1):
            logz_t[b, j] = log_partition(z[j], t)
        for j in range(n):
            logz_d[b, j] = log_partition(y[j], t)
            d = int(drafts[b][j])
            q = softmax(z[j], t)[d]
            p = softmax(y[j], t)[d]
            probs[b, j] = 1.0 if p <= 0 else min(1.0, q / p)
    return probs, logz_t, logz_d
