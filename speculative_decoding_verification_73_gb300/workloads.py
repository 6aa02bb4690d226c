"""Seeded synthetic inputs for the batched draft-verify step.

This module is the one piece that the CUDA library's tests and the CPU
oracle both consume.  It holds none of the verify method's arithmetic: it
builds logit rows, picks temperatures, and draws draft tokens from the
drafter's own law (by the Gumbel-max trick, argmax_t(y_t / T + G_t) with
G_t standard Gumbel, which is a draw from softmax(y / T) without forming
it; or by the inverse CDF of a probability vector this module itself
constructed).  It never normalises a logit row, never evaluates an
acceptance test and never samples a residual.

Logit recipe ("Speculative Decoding and EAGLE-3" lesson, "Build it" step 6:
the draft is the target perturbed by noise of a chosen amplitude): a target
row is Zipf-shaped, z_t = -s ln(rank_t) + N(0, 0.3) with the ranks a fresh
random permutation of 1..V per row; its draft row is z + N(0, sigma).  Rows
are built in float32/float64 and cast to the storage dtype last, so both
sides see the same quantised values.

The five named workloads follow the method statement's five configurations:

  tiny-f32         B=1,   N=4, V=1024,   fp32, sigma 0.5, T 1
  single-bf16      B=1,   N=5, V=128256, bf16, sigma tuned so that the mean
                   sum_t min(p, q) over rows is about 0.8; T 1 (or 0)
  batch64-bf16     B=64,  N=7, V=128256, bf16, sigma_b ~ U[0.2, 1.5],
                   T_b uniform over {0, 0.7, 1.0}
  mixture-bf16     B=16,  N=3, V=163840, bf16, half of the 64 target rows
                   peaked (top-1 mass 0.95 on a Zipf-0.8 base), half flat
                   Zipf-0.8; sigma 0.4, T 1
  alpha09-f32      B=256, N=8, V=32000,  fp32, drafts built with per-position
                   overlap sum_t min(p, q) = 0.9 exactly in real arithmetic;
                   T 1; draft tokens redrawn for every verify seed
"""

import dataclasses
import math

import numpy as np
import torch

DTYPES = {"bf16": torch.bfloat16, "f32": torch.float32}

# Draft noise for the single-request V=128256 workload, chosen by bisection
# on the oracle's mean overlap sum_t min(p, q) (target 0.8).  The script
# that finds it is tests/golden/make_single_bf16_sigma.py; a CPU test checks
# that the value still gives 0.80 +- 0.01.
SINGLE_BF16_SIGMA = 0.47816771268844604


@dataclasses.dataclass
class Workload:
    """One batch of verify inputs on the host (torch CPU tensors)."""

    name: str
    dtype: str                  # "bf16" | "f32"
    target: torch.Tensor        # [B, N+1, V]
    draft: torch.Tensor         # [B, N, V]
    tokens: torch.Tensor        # [B, N] int32
    temperature: torch.Tensor   # [B] float32
    seed: int                   # verify seed

    @property
    def shape(self):
        b, n1, v = self.target.shape
        return b, n1 - 1, v

    def raw(self):
        """(target, draft) as numpy arrays in the oracle's input form:
        uint16 bit patterns for bf16, float32 values for fp32."""
        if self.dtype == "bf16":
            return (self.target.view(torch.int16).numpy().view(np.uint16),
                    self.draft.view(torch.int16).numpy().view(np.uint16))
        return self.target.numpy(), self.draft.numpy()

    def bytes_read(self):
        """Logit bytes one full verify pass reads: every target row, plus the
        draft rows of requests with T > 0."""
        b, n, v = self.shape
        esize = self.target.element_size()
        sampled = int((self.temperature > 0).sum())
        return (b * (n + 1) + sampled * n) * v * esize


# --------------------------------------------------------------------------
# Building blocks
# --------------------------------------------------------------------------

def _gen(seed):
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def _neg_log_rank(gen, rows, vocab):
    """-ln(rank_t) per row, with ranks a fresh random permutation of 1..V."""
    out = torch.empty(rows, vocab, dtype=torch.float64)
    base = -torch.log(torch.arange(1, vocab + 1, dtype=torch.float64))
    for r in range(rows):
        perm = torch.randperm(vocab, generator=gen)
        out[r, perm] = base
    return out


def _gumbel_argmax(gen, logits_f64, temperature):
    """One draw from softmax(logits / T) per row via argmax(logits/T + G),
    G standard Gumbel; argmax of the logits when T == 0 (first index on
    ties)."""
    rows = logits_f64.shape[0]
    out = np.zeros(rows, dtype=np.int32)
    for r in range(rows):
        x = logits_f64[r]
        if temperature == 0:
            out[r] = int(np.argmax(x))
            continue
        u = torch.rand(x.shape[0], generator=gen, dtype=torch.float64).numpy()
        u = np.clip(u, 1e-300, 1.0 - 1e-16)
        g = -np.log(-np.log(u))
        out[r] = int(np.argmax(x / temperature + g))
    return out


def _widen(t):
    """Stored logits as float64 (exact)."""
    return t.to(torch.float64).numpy()


def _zipf_rows(gen, rows, vocab, s, noise):
    z = s * _neg_log_rank(gen, rows, vocab)
    if noise:
        z += noise * torch.randn(rows, vocab, generator=gen, dtype=torch.float64)
    return z


def make_zipf(batch, n, vocab, dtype, *, gen_seed, verify_seed=0, s=1.1,
              target_noise=0.3, sigma=0.5, temperatures=1.0, name="zipf"):
    """Zipf-shaped target rows, draft = target + N(0, sigma_b), tokens drawn
    from the drafter at each request's temperature.

    ``sigma`` and ``temperatures`` are a scalar or one value per request.
    """
    gen = _gen(gen_seed)
    sig = np.broadcast_to(np.asarray(sigma, dtype=np.float64), (batch,))
    temps = np.broadcast_to(np.asarray(temperatures, dtype=np.float32), (batch,)).copy()
    tdt = DTYPES[dtype]
    target = torch.empty(batch, n + 1, vocab, dtype=tdt)
    draft = torch.empty(batch, n, vocab, dtype=tdt)
    tokens = np.zeros((batch, n), dtype=np.int32)
    for b in range(batch):
        z = _zipf_rows(gen, n + 1, vocab, s, target_noise)
        target[b] = z.to(tdt)
        if n == 0:
            continue
        y = z[:n] + float(sig[b]) * torch.randn(n, vocab, generator=gen, dtype=torch.float64)
        draft[b] = y.to(tdt)
        tokens[b] = _gumbel_argmax(gen, _widen(draft[b]), float(temps[b]))
    return Workload(name, dtype, target, draft, torch.from_numpy(tokens),
                    torch.from_numpy(temps), int(verify_seed))


def make_random(batch, n, vocab, dtype, *, gen_seed, verify_seed=0, temps=(0.0, 0.7, 1.0),
                sigma=(0.2, 1.5), s=1.1):
    """A small mixed batch for parity tests: per-request sigma ~ U[sigma],
    per-request T uniform over ``temps``."""
    gen = _gen(gen_seed + 7919)
    lo, hi = sigma
    sig = (lo + (hi - lo) * torch.rand(batch, generator=gen, dtype=torch.float64)).numpy()
    pick = torch.randint(0, len(temps), (batch,), generator=gen).numpy()
    tv = np.asarray(temps, dtype=np.float32)[pick]
    return make_zipf(batch, n, vocab, dtype, gen_seed=gen_seed, verify_seed=verify_seed,
                     s=s, sigma=sig, temperatures=tv, name=f"random-{dtype}-B{batch}-N{n}-V{vocab}")


# --------------------------------------------------------------------------
# The five named workloads
# --------------------------------------------------------------------------

def tiny_f32():
    """B=1, N=4, V=1024, fp32, sigma 0.5, T 1, verify seed 0."""
    return make_zipf(1, 4, 1024, "f32", gen_seed=1001, verify_seed=0, sigma=0.5,
                     temperatures=1.0, name="tiny-f32")


def single_bf16(temperature=1.0, sigma=None):
    """B=1, N=5, V=128256, bf16, sigma tuned for mean overlap ~0.8."""
    sig = SINGLE_BF16_SIGMA if sigma is None else sigma
    return make_zipf(1, 5, 128256, "bf16", gen_seed=1002, verify_seed=0, sigma=sig,
                     temperatures=temperature, name=f"single-bf16-T{temperature:g}")


def batch64_bf16(verify_seed=0, gen_seed=1003):
    """B=64, N=7, V=128256, bf16; sigma_b ~ U[0.2, 1.5]; T_b from {0, 0.7, 1}."""
    gen = _gen(gen_seed + 104729)
    sig = (0.2 + 1.3 * torch.rand(64, generator=gen, dtype=torch.float64)).numpy()
    pick = torch.randint(0, 3, (64,), generator=gen).numpy()
    temps = np.array([0.0, 0.7, 1.0], dtype=np.float32)[pick]
    return make_zipf(64, 7, 128256, "bf16", gen_seed=gen_seed, verify_seed=verify_seed,
                     sigma=sig, temperatures=temps, name="batch64-bf16")


def low_accept_bf16(verify_seed=0, sigma=3.0):
    """B=64, N=7, V=128256, bf16, every request at T 1 with draft noise
    sigma 3 (the drafter far from the target: most requests reject their
    first draft) -- the regime where reading rows only up to the first
    rejection pays."""
    return make_zipf(64, 7, 128256, "bf16", gen_seed=4242, verify_seed=verify_seed, sigma=sigma,
                     temperatures=1.0, name="lowaccept64-bf16")


def mixture_bf16(verify_seed=0):
    """B=16, N=3, V=163840, bf16: half of the 64 target rows peaked (top-1
    mass 0.95 over a Zipf-0.8 base), half flat Zipf-0.8; sigma 0.4; T 1."""
    batch, n, vocab = 16, 3, 163840
    gen = _gen(1004)
    rows = batch * (n + 1)
    peaked = torch.zeros(rows, dtype=torch.bool)
    peaked[torch.randperm(rows, generator=gen)[: rows // 2]] = True
    tdt = torch.bfloat16
    target = torch.empty(batch, n + 1, vocab, dtype=tdt)
    draft = torch.empty(batch, n, vocab, dtype=tdt)
    tokens = np.zeros((batch, n), dtype=np.int32)
    for b in range(batch):
        nlr = _neg_log_rank(gen, n + 1, vocab)          # -ln(rank)
        z = 0.8 * nlr                                    # flat Zipf-0.8 logits
        for j in range(n + 1):
            if not peaked[b * (n + 1) + j]:
                continue
            # Probability vector: rank 1 gets 0.95, the rest share 0.05 in
            # Zipf-0.8 proportions; the logits are its logarithm.
            w = torch.exp(z[j])                          # rank^-0.8
            top = int(torch.argmax(nlr[j]))
            rest = w.clone()
            rest[top] = 0.0
            q = 0.05 * rest / rest.sum()
            q[top] = 0.95
            z[j] = torch.log(q)
        target[b] = z.to(tdt)
        y = z[:n] + 0.4 * torch.randn(n, vocab, generator=gen, dtype=torch.float64)
        draft[b] = y.to(tdt)
        tokens[b] = _gumbel_argmax(gen, _widen(draft[b]), 1.0)
    temps = np.ones(batch, dtype=np.float32)
    return Workload("mixture-bf16", "bf16", target, draft, torch.from_numpy(tokens),
                    torch.from_numpy(temps), int(verify_seed))


class Alpha09:
    """B=256, N=8, V=32000, fp32 rows with sum_t min(p_j, q_j) = 0.9.

    Per row the target law q is built directly as a probability vector
    (Zipf-1.1 weights times log-normal(0, 0.3) noise, divided by their sum);
    a random set S with q(S) >= 0.2 is chosen by walking a random token order;
    the draft law is p = q (1 - 0.1/q(S)) on S and q (1 + 0.1/(1 - q(S)))
    off S, so the total-variation distance is 0.1.  Logits are ln q and ln p
    stored as float32.  ``tokens(s)`` redraws every d_{b,j} ~ p_{b,j} for
    verify seed s by the inverse CDF of this module's own p.
    """

    batch, n, vocab = 256, 8, 32000
    alpha = 0.9

    def __init__(self, gen_seed=1005):
        gen = _gen(gen_seed)
        b, n, v = self.batch, self.n, self.vocab
        self.q = np.zeros((b, n + 1, v))
        self.p = np.zeros((b, n, v))
        base = torch.arange(1, v + 1, dtype=torch.float64) ** -1.1
        for i in range(b):
            for j in range(n + 1):
                w = torch.empty(v, dtype=torch.float64)
                w[torch.randperm(v, generator=gen)] = base
                w *= torch.exp(0.3 * torch.randn(v, generator=gen, dtype=torch.float64))
                q = (w / w.sum()).numpy()
                self.q[i, j] = q
                if j == n:
                    continue
                order = torch.randperm(v, generator=gen).numpy()
                k = int(np.searchsorted(np.cumsum(q[order]), 0.2)) + 1
                in_s = np.zeros(v, dtype=bool)
                in_s[order[:k]] = True
                qs = q[in_s].sum()
                p = np.where(in_s, q * (1.0 - 0.1 / qs), q * (1.0 + 0.1 / (1.0 - qs)))
                self.p[i, j] = p
        self.target = torch.from_numpy(np.log(self.q).astype(np.float32))
        self.draft = torch.from_numpy(np.log(self.p).astype(np.float32))
        self._cdf = np.cumsum(self.p, axis=2)
        self.temperature = torch.ones(b, dtype=torch.float32)

    def tokens(self, verify_seed):
        gen = _gen(50000 + int(verify_seed))
        u = torch.rand(self.batch, self.n, generator=gen, dtype=torch.float64).numpy()
        out = np.zeros((self.batch, self.n), dtype=np.int32)
        for i in range(self.batch):
            for j in range(self.n):
                c = self._cdf[i, j]
                t = int(np.searchsorted(c, u[i, j] * c[-1], side="right"))
                out[i, j] = min(t, self.vocab - 1)
        return torch.from_numpy(out)

    def workload(self, verify_seed):
        return Workload("alpha09-f32", "f32", self.target, self.draft,
                        self.tokens(verify_seed), self.temperature, int(verify_seed))


NAMED = {
    "tiny-f32": tiny_f32,
    "single-bf16": single_bf16,
    "batch64-bf16": batch64_bf16,
    "mixture-bf16": mixture_bf16,
}


# --------------------------------------------------------------------------
# Draft trees
# --------------------------------------------------------------------------

TREE_SAMPLED = 0   # children are independent draws from the parent's draft row
TREE_TOPK = 1      # children are the parent's top draft tokens, most probable first


@dataclasses.dataclass
class TreeWorkload:
    """One batch of tree-verify inputs on the host (torch CPU tensors).
    Node 0 is the root, nodes 1..M the drafts; row r of both logit tensors
    belongs to node r."""

    name: str
    dtype: str
    mode: int                   # TREE_SAMPLED | TREE_TOPK
    target: torch.Tensor        # [B, M+1, V]
    draft: torch.Tensor         # [B, M+1, V]
    parents: torch.Tensor       # [B, M] int32, parent of node i+1 in [0, i]
    tokens: torch.Tensor        # [B, M] int32
    temperature: torch.Tensor   # [B] float32
    seed: int

    @property
    def shape(self):
        b, m1, v = self.target.shape
        return b, m1 - 1, v

    def raw(self):
        if self.dtype == "bf16":
            return (self.target.view(torch.int16).numpy().view(np.uint16),
                    self.draft.view(torch.int16).numpy().view(np.uint16))
        return self.target.numpy(), self.draft.numpy()

    def inner_rows(self):
        """Number of nodes with children, per request."""
        b, m, _ = self.shape
        out = np.zeros(b, dtype=np.int64)
        par = self.parents.numpy()
        for i in range(b):
            out[i] = len(set(int(x) for x in par[i]))
        return out

    def bytes_read(self):
        """Logit bytes of one tree verify: every target row, plus (SAMPLED
        mode, T > 0) the draft rows of nodes with children."""
        b, m, v = self.shape
        esize = self.target.element_size()
        rows = b * (m + 1)
        if self.mode == TREE_SAMPLED:
            inner = self.inner_rows()
            rows += int(sum(inner[i] for i in range(b) if float(self.temperature[i]) > 0))
        return rows * v * esize


def full_tree_parents(widths):
    """Parents (breadth-first ids) of the tree with widths[d] children under
    every node of depth d: (2, 2, 2) gives 14 draft nodes and 8 leaves."""
    parents, level, nxt = [], [0], 1
    for w in widths:
        new = []
        for node in level:
            for _ in range(w):
                parents.append(node)
                new.append(nxt)
                nxt += 1
        level = new
    return np.array(parents, dtype=np.int32)


def random_tree_parents(gen, m, max_children=4):
    """A random topology with m draft nodes: node i+1 hangs under a uniformly
    chosen earlier node that still has fewer than max_children children."""
    parents, kids = [], [0] * (m + 1)
    for i in range(m):
        while True:
            p = int(torch.randint(0, i + 1, (1,), generator=gen))
            if kids[p] < max_children:
                break
        kids[p] += 1
        parents.append(p)
    return np.array(parents, dtype=np.int32)


def make_tree(batch, vocab, dtype, *, gen_seed, widths=None, m=None, mode=TREE_SAMPLED,
              verify_seed=0, temps=(0.0, 0.7, 1.0), sigma=(0.2, 1.5), s=1.1,
              target_noise=0.3, name=None):
    """Tree workload: a full tree of ``widths`` for every request, or (with
    ``m``) a random topology of m draft nodes per request.  Target rows are
    Zipf-shaped; draft row r = target row r + N(0, sigma_b).  Children of a
    node take tokens from the node's draft row at the request's temperature:
    independent Gumbel-max draws (SAMPLED) or its largest logits in
    decreasing order (TOPK, and every request with T = 0)."""
    gen = _gen(gen_seed + 4409)
    lo, hi = sigma
    sig = (lo + (hi - lo) * torch.rand(batch, generator=gen, dtype=torch.float64)).numpy()
    pick = torch.randint(0, len(temps), (batch,), generator=gen).numpy()
    tv = np.asarray(temps, dtype=np.float32)[pick]
    if widths is not None:
        par = np.tile(full_tree_parents(widths), (batch, 1))
    else:
        par = np.stack([random_tree_parents(gen, m) for _ in range(batch)])
    mm = par.shape[1]
    tdt = DTYPES[dtype]
    target = torch.empty(batch, mm + 1, vocab, dtype=tdt)
    draft = torch.empty(batch, mm + 1, vocab, dtype=tdt)
    tokens = np.zeros((batch, mm), dtype=np.int32)
    for b in range(batch):
        z = _zipf_rows(gen, mm + 1, vocab, s, target_noise)
        target[b] = z.to(tdt)
        y = z + float(sig[b]) * torch.randn(mm + 1, vocab, generator=gen, dtype=torch.float64)
        draft[b] = y.to(tdt)
        yw = _widen(draft[b])
        for node in range(mm + 1):
            kids = [i for i in range(mm) if par[b, i] == node]
            if not kids:
                continue
            if mode == TREE_TOPK or tv[b] == 0:
                order = np.argsort(-yw[node], kind="stable")
                for k, i in enumerate(kids):
                    tokens[b, i] = int(order[k])
            else:
                rows = np.repeat(yw[node:node + 1], len(kids), axis=0)
                tokens[b, kids] = _gumbel_argmax(gen, rows, float(tv[b]))
    label = name or f"tree-{'topk' if mode == TREE_TOPK else 'sampled'}-{dtype}-B{batch}-M{mm}-V{vocab}"
    return TreeWorkload(label, dtype, mode, target, draft, torch.from_numpy(par),
                        torch.from_numpy(tokens), torch.from_numpy(tv), int(verify_seed))


# --------------------------------------------------------------------------
# FC-norm inputs
# --------------------------------------------------------------------------

@dataclasses.dataclass
class FcNormWorkload:
    """Hidden states of three target layers and the FC weights (CPU tensors).
    The later layers' states are larger, as the EAGLE 3.1 page describes
    (residual accumulation): standard deviations 1, 4 and 16, means 0, 0.5
    and 2."""

    name: str
    h: list                     # 3 x [T, d] bf16
    weight: torch.Tensor        # [d_out, 3d] bf16
    gamma: torch.Tensor         # [3, d] float32
    beta: torch.Tensor          # [3, d] float32
    bias: torch.Tensor          # [d_out] float32


def make_fcnorm(T, d, d_out, *, gen_seed, name=None):
    gen = _gen(gen_seed + 313)
    h = []
    for scale, mean in ((1.0, 0.0), (4.0, 0.5), (16.0, 2.0)):
        x = mean + scale * torch.randn(T, d, generator=gen, dtype=torch.float64)
        h.append(x.to(torch.bfloat16))
    w = torch.randn(d_out, 3 * d, generator=gen, dtype=torch.float64) / math.sqrt(3 * d)
    gamma = 1.0 + 0.1 * torch.randn(3, d, generator=gen, dtype=torch.float64)
    beta = 0.1 * torch.randn(3, d, generator=gen, dtype=torch.float64)
    bias = 0.1 * torch.randn(d_out, generator=gen, dtype=torch.float64)
    return FcNormWorkload(name or f"fcnorm-T{T}-d{d}-o{d_out}", h, w.to(torch.bfloat16),
                          gamma.to(torch.float32), beta.to(torch.float32), bias.to(torch.float32))
