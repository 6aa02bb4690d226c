"""GPU parity of tree verification through the C ABI against the tree
oracle, and bit-for-bit agreement with spec_verify on one-child-per-node
trees.  Every input is a seeded synthetic tree from ``workloads``."""

import numpy as np
import pytest
import torch

from speculative_decoding_verification_73_gb300 import binding, build, workloads

from parity import compare_tree, run_tree_oracle

pytestmark = pytest.mark.gpu

TORCH_DT = {"bf16": torch.bfloat16, "f32": torch.float32}


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return binding.load()


def run_tree(wl, seed=None, ctx=None, lazy=False):
    B, M, V = wl.shape
    own = ctx is None
    if own:
        ctx = binding.SpecVerify(max(B, 1), max(M, 1), V, TORCH_DT[wl.dtype])
    draft = wl.draft.cuda() if wl.mode == binding.SV_TREE_SAMPLED else None
    toks, path, acc, kv = ctx.tree(wl.target.cuda(), draft, wl.parents.cuda(), wl.tokens.cuda(),
                                   wl.temperature.cuda(), wl.seed if seed is None else seed, wl.mode,
                                   lazy=lazy)
    code, bits = ctx.get_error()
    out = (toks.cpu().numpy().copy(), path.cpu().numpy().copy(), acc.cpu().numpy().copy(),
           kv.cpu().numpy().copy(), code, bits)
    if own:
        ctx.close()
    return out


def check_tree(wl, seed=None, label=""):
    res = run_tree_oracle(wl, seed)
    toks, path, acc, kv, code, bits = run_tree(wl, seed)
    assert bits == res.errors, (bits, res.errors)
    return res, compare_tree(res, toks, path, acc, kv, wl.temperature.numpy(), label or wl.name)


def test_one_child_per_node_is_spec_verify_bit_for_bit():
    for wl in (workloads.make_random(16, 6, 5000, "bf16", gen_seed=61, verify_seed=3),
               workloads.make_random(9, 4, 3001, "f32", gen_seed=62, verify_seed=4)):
        B, N, V = wl.shape
        ctx = binding.SpecVerify(B, N, V, TORCH_DT[wl.dtype])
        z, y = wl.target.cuda(), wl.draft.cuda()
        d, t = wl.tokens.cuda(), wl.temperature.cuda()
        par = torch.arange(N, dtype=torch.int32).repeat(B, 1).cuda()
        y_tree = torch.cat([y, torch.zeros_like(z[:, :1])], dim=1)
        for seed in (0, 1, 77):
            ct, ca, ck = (x.cpu().clone() for x in ctx(z, y, d, t, seed))
            tt, tp, ta, tk = (x.cpu().clone() for x in ctx.tree(z, y_tree, par, d, t, seed))
            assert torch.equal(tt, ct) and torch.equal(ta, ca) and torch.equal(tk, ck)
            for b in range(B):
                a = int(ca[b])
                assert tp[b, :a].tolist() == list(range(1, a + 1)) and (tp[b, a:] == -1).all()
        ctx.close()


CASES = {
    "222-sampled-bf16": lambda: workloads.make_tree(24, 32000, "bf16", gen_seed=71, widths=(2, 2, 2),
                                                    verify_seed=5),
    "222-topk-bf16": lambda: workloads.make_tree(24, 32000, "bf16", gen_seed=72, widths=(2, 2, 2),
                                                 mode=workloads.TREE_TOPK, verify_seed=6),
    "random-sampled-f32-ragged": lambda: workloads.make_tree(12, 3001, "f32", gen_seed=73, m=40,
                                                             verify_seed=7),
    "random-topk-f32-ragged": lambda: workloads.make_tree(12, 3001, "f32", gen_seed=74, m=40,
                                                          mode=workloads.TREE_TOPK, verify_seed=8),
    "wide-sampled-bf16": lambda: workloads.make_tree(8, 50000, "bf16", gen_seed=75, widths=(4, 3),
                                                     verify_seed=9),
    "root-only": lambda: workloads.make_tree(5, 4096, "f32", gen_seed=76, widths=(), verify_seed=1),
    # seven spans per fp32 row: partials merged past the first four
    "many-spans-sampled-f32": lambda: workloads.make_tree(4, 100000, "f32", gen_seed=79, widths=(3, 2),
                                                          verify_seed=12),
    # 21 level-1 blocks of bf16: three per CTA, so the rows are not staged and
    # each block is picked on its own
    "three-blocks-per-cta-bf16": lambda: workloads.make_tree(6, 170000, "bf16", gen_seed=86,
                                                             widths=(2, 2, 2), temps=(0.7, 1.0),
                                                             verify_seed=13),
    # 135 level-1 blocks: the draw's masses and candidates go through the
    # workspace instead of distributed shared memory
    "huge-vocabulary-bf16": lambda: workloads.make_tree(2, 1100000, "bf16", gen_seed=87, widths=(2, 2),
                                                        temps=(0.7, 1.0), verify_seed=14),
}


@pytest.mark.parametrize("name", list(CASES))
def test_tree_parity(name):
    wl = CASES[name]()
    logged = []
    for seed in (wl.seed, wl.seed + 1000, 2 ** 64 - 3):
        res, lg = check_tree(wl, seed, f"{name} seed {seed}")
        logged += lg
        assert res.errors == 0
    B, M, _ = wl.shape
    assert len(logged) == 0 or len(logged) < 1e-5 * 3 * B * max(M, 1)


def test_tree_222_full_vocabulary():
    """The pages' [2, 2, 2] tree over V = 128256 bf16 logits, 32 requests."""
    wl = workloads.make_tree(32, 128256, "bf16", gen_seed=77, widths=(2, 2, 2), verify_seed=11)
    for seed in (11, 12):
        check_tree(wl, seed, "222-full")


def test_tree_errors_are_flagged_per_request():
    wl = workloads.make_tree(6, 2048, "f32", gen_seed=78, widths=(2, 2), temps=(1.0,), verify_seed=2)
    wl.temperature[0] = float("nan")
    wl.parents[1, 3] = 5            # node 4 under node 5
    wl.tokens[2, 0] = 2048          # out of range
    wl.target[3, 2, 7] = float("inf")
    wl.parents[4, 0] = -1
    res, _ = check_tree(wl, label="errors")
    toks, path, acc, kv, code, bits = run_tree(wl)
    assert code == binding.SV_EBADTEMP and bits == 1 | 2 | 4 | 8
    for b, bit in ((0, 1), (1, 8), (2, 2), (3, 4), (4, 8)):
        assert res.request_errors[b] == bit
        assert acc[b] == -1 and kv[b] == 0 and (toks[b] == -1).all() and (path[b] == -1).all()
    assert acc[5] >= 0


MAX_CASES = {
    # 255 draft nodes per tree: the largest M a context accepts
    "random-255-sampled-f32": lambda: workloads.make_tree(3, 3001, "f32", gen_seed=81, m=binding.SV_MAX_N,
                                                          verify_seed=21),
    "random-255-topk-bf16": lambda: workloads.make_tree(3, 4099, "bf16", gen_seed=82, m=binding.SV_MAX_N,
                                                        mode=workloads.TREE_TOPK, verify_seed=22),
    "star-255-sampled-bf16": lambda: workloads.make_tree(3, 4099, "bf16", gen_seed=83, widths=(255,),
                                                         verify_seed=23),
    "star-255-topk-f32": lambda: workloads.make_tree(3, 3001, "f32", gen_seed=84, widths=(255,),
                                                     mode=workloads.TREE_TOPK, verify_seed=24),
    "line-255-sampled-f32": lambda: workloads.make_tree(3, 3001, "f32", gen_seed=85, widths=(1,) * 255,
                                                        sigma=(0.0, 0.05), verify_seed=25),
}


@pytest.mark.parametrize("name", list(MAX_CASES))
def test_tree_max_size(name):
    wl = MAX_CASES[name]()
    assert wl.shape[1] == binding.SV_MAX_N
    for seed in (wl.seed, wl.seed + 7):
        res, _ = check_tree(wl, seed, f"{name} seed {seed}")
        assert res.errors == 0


def _repeat_first_sibling(wl):
    """Give the second child of every node the token of its first child."""
    B, M, _ = wl.shape
    par = wl.parents.numpy()
    for b in range(B):
        kids = {}
        for i in range(M):
            kids.setdefault(int(par[b, i]), []).append(i)
        for ks in kids.values():
            if len(ks) > 1:
                wl.tokens[b, ks[1]] = wl.tokens[b, ks[0]]
    return wl


@pytest.mark.parametrize("mode", [workloads.TREE_SAMPLED, workloads.TREE_TOPK])
def test_repeated_sibling_tokens(mode):
    """A token tried twice at one node: in TOPK mode the residual has already
    removed it, so the second try is always rejected and the removed mass is
    counted once; in SAMPLED mode the second try faces the residual."""
    wl = _repeat_first_sibling(workloads.make_tree(16, 32000, "bf16", gen_seed=86, widths=(3, 2, 2),
                                                   mode=mode, verify_seed=26))
    for seed in (26, 27, 28):
        res, _ = check_tree(wl, seed, f"repeat mode {mode} seed {seed}")
        assert res.errors == 0


# ------------------------------------------------------------------ lazy walk

LAZY_NAMES = [n for n in CASES if n != "huge-vocabulary-bf16"]


@pytest.mark.parametrize("name", LAZY_NAMES + ["222-full"] + list(MAX_CASES))
def test_lazy_tree_is_the_eager_tree_bit_for_bit(name):
    """spec_verify_tree_lazy reduces each row the walk reaches with the same
    span reduction as the eager row statistics and merges the same partials
    in the same order: identical outputs on valid inputs (three seeds, one
    context, eager and lazy calls interleaved), up to 255-node trees (the
    line tree's walks visit up to 256 nodes each)."""
    wl = (workloads.make_tree(32, 128256, "bf16", gen_seed=77, widths=(2, 2, 2), verify_seed=11)
          if name == "222-full" else MAX_CASES[name]() if name in MAX_CASES else CASES[name]())
    B, M, V = wl.shape
    ctx = binding.SpecVerify(max(B, 1), max(M, 1), V, TORCH_DT[wl.dtype])
    for seed in (wl.seed, wl.seed + 1000, 2 ** 64 - 3):
        eager = run_tree(wl, seed, ctx)
        lazy = run_tree(wl, seed, ctx, lazy=True)
        for a, b in zip(eager[:4], lazy[:4]):
            assert np.array_equal(a, b), name
        assert eager[4:] == lazy[4:] == (0, 0)
    ctx.close()


def test_lazy_tree_reads_only_the_walked_rows():
    """Bad rows off every request's walked path (a NaN target row of a node
    the walk never reaches, a +inf draft row of an unvisited inner node) are
    not errors for the lazy walk: its outputs are those of the clean input,
    and equal the oracle's lazy reading; the same inputs fail the eager walk.
    A NaN in the root's row fails both."""
    from oracle import tree as ot
    wl = workloads.make_tree(16, 5000, "bf16", gen_seed=405, widths=(2, 2, 2), temps=(0.0, 1.0), verify_seed=3)
    clean = run_tree(wl, 3)
    assert clean[4:] == (0, 0)
    B, M, V = wl.shape
    par = wl.parents.numpy()
    kids = [ot.children_of([int(v) for v in par[b]], M) for b in range(B)]
    for b in range(B):
        seen = {0} | {int(n) for n in clean[1][b] if n >= 0}
        off = [n for n in range(1, M + 1) if n not in seen]
        wl.target[b, off[0], 7] = float("nan")
        inner_off = [n for n in off if kids[b][n]]
        if inner_off and float(wl.temperature[b]) > 0:
            wl.draft[b, inner_off[0], 11] = float("inf")
    lazy = run_tree(wl, 3, lazy=True)
    assert lazy[4:] == (0, 0)
    for a, b in zip(clean[:4], lazy[:4]):
        assert np.array_equal(a, b)
    z, y = wl.raw()
    res = ot.verify_tree(z, y, par, wl.tokens.numpy(), wl.temperature.numpy(), 3, wl.dtype, wl.mode, lazy=True)
    assert res.errors == 0
    compare_tree(res, *lazy[:4], wl.temperature.numpy(), "lazy-off-path")
    eager = run_tree(wl, 3)
    assert eager[5] == binding.SV_ERRBIT_LOGIT and (eager[2] == -1).all()
    wl.target[:, 0, 5] = float("nan")
    for lz in (False, True):
        out = run_tree(wl, 3, lazy=lz)
        assert out[5] == binding.SV_ERRBIT_LOGIT and (out[2] == -1).all() and (out[0] == -1).all()


def test_lazy_tree_takes_rows_of_at_most_32_spans():
    """Rows of more than 32 spans of 64 KB are refused before anything is
    enqueued (SV_EINVAL); the eager walk takes them."""
    wl = CASES["huge-vocabulary-bf16"]()
    with pytest.raises(binding.SpecVerifyError):
        run_tree(wl, lazy=True)


def test_lazy_tree_errors_are_flagged_per_request():
    """The eager error workload through the lazy walk: temperature, topology
    and token errors as in spec_verify_tree (checked before the walk); the
    +inf logit sits in node 2's row, an error only if that request's walk
    reaches node 2 -- exactly the oracle's lazy reading."""
    from oracle import tree as ot
    wl = workloads.make_tree(6, 2048, "f32", gen_seed=78, widths=(2, 2), temps=(1.0,), verify_seed=2)
    wl.temperature[0] = float("nan")
    wl.parents[1, 3] = 5            # node 4 under node 5
    wl.tokens[2, 0] = 2048          # out of range
    wl.target[3, 2, 7] = float("inf")
    wl.parents[4, 0] = -1
    toks, path, acc, kv, code, bits = run_tree(wl, lazy=True)
    z, y = wl.raw()
    res = ot.verify_tree(z, y, wl.parents.numpy(), wl.tokens.numpy(), wl.temperature.numpy(), wl.seed,
                         wl.dtype, wl.mode, lazy=True)
    assert bits == res.errors
    for b, bit in ((0, 1), (1, 8), (2, 2), (4, 8)):
        assert res.request_errors[b] == bit
        assert acc[b] == -1 and kv[b] == 0 and (toks[b] == -1).all() and (path[b] == -1).all()
    compare_tree(res, toks, path, acc, kv, wl.temperature.numpy(), "lazy-errors")
