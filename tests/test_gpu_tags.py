"""The chain's tagged row statistics across calls on one context.

The sampler takes a partial once it carries the call's sequence number, so
whatever earlier calls left in the workspace must never pass for this
call's: calls of other shapes, tree and lazy calls (which write their own
partials) and the counter's wrap past 2^32 - 1 all have to give exactly the
results of a fresh context on the same inputs.
"""

import time

import pytest
import torch

from speculative_decoding_verification_73_gb300 import binding, build, workloads

pytestmark = pytest.mark.gpu

MAX_B, MAX_N, MAX_V = 24, 14, 32000


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return binding.load()


def _inputs(wl):
    B, N, V = wl.shape
    return (wl.target.cuda(), wl.draft.cuda() if N > 0 else None, wl.tokens.cuda(),
            wl.temperature.cuda())


def _host(outs):
    return [x.cpu().clone() for x in outs]


def _fresh(wl, seed):
    B, N, V = wl.shape
    ctx = binding.SpecVerify(B, max(N, 1), V, torch.bfloat16)
    out = _host(ctx(*_inputs(wl), seed))
    err = ctx.get_error()
    ctx.close()
    return out, err


CHAINS = {
    "a": lambda: workloads.make_random(16, 6, 5000, "bf16", gen_seed=301, verify_seed=1),
    "b": lambda: workloads.make_random(24, 14, 32000, "bf16", gen_seed=302, verify_seed=2),
    "c": lambda: workloads.make_random(9, 3, 3001, "bf16", gen_seed=303, verify_seed=3),
    "d": lambda: workloads.make_random(20, 7, 24576, "bf16", gen_seed=304, verify_seed=4),
}


def test_chain_calls_between_other_shapes_tree_and_lazy_calls():
    chains = {k: f() for k, f in CHAINS.items()}
    tree = workloads.make_tree(12, 5000, "bf16", gen_seed=305, widths=(2, 2, 2), verify_seed=5)
    want = {(k, s): _fresh(wl, s) for k, wl in chains.items() for s in (11, 12)}
    ctx = binding.SpecVerify(MAX_B, MAX_N, MAX_V, torch.bfloat16)
    order = ["a", "tree", "b", "lazy-c", "c", "a", "d", "tree", "b", "lazy-d", "d", "c"]
    for i, step in enumerate(order):
        seed = 11 + (i % 2)
        if step == "tree":
            draft = tree.draft.cuda()
            ctx.tree(tree.target.cuda(), draft, tree.parents.cuda(), tree.tokens.cuda(),
                     tree.temperature.cuda(), seed, tree.mode)
            torch.cuda.synchronize()
            continue
        if step.startswith("lazy-"):
            ctx.lazy(*_inputs(chains[step[5:]]), seed)
            torch.cuda.synchronize()
            continue
        got = _host(ctx(*_inputs(chains[step]), seed))
        err = ctx.get_error()
        ref, ref_err = want[(step, seed)]
        for a, b in zip(got, ref):
            assert torch.equal(a, b), (i, step)
        assert err == ref_err == (0, 0), (i, step)
    ctx.close()


def test_call_counter_wrap():
    first = workloads.make_random(16, 6, 5000, "bf16", gen_seed=311, verify_seed=1)
    other = workloads.make_random(24, 14, 32000, "bf16", gen_seed=312, verify_seed=2)
    again = workloads.make_random(16, 6, 5000, "bf16", gen_seed=313, verify_seed=3)
    ctx = binding.SpecVerify(MAX_B, MAX_N, MAX_V, torch.bfloat16)
    # tags of call 1 left in the slots of `first`'s shape ...
    ctx(*_inputs(first), 7)
    torch.cuda.synchronize()
    # ... then calls 2^32 - 1, (wrap: every tag cleared) 1, 2, 3
    ctx.debug_seek_calls(0xFFFFFFFE)
    for i, wl in enumerate((other, again, first, again)):
        got = _host(ctx(*_inputs(wl), 20 + i))
        ref, ref_err = _fresh(wl, 20 + i)
        for a, b in zip(got, ref):
            assert torch.equal(a, b), i
        assert ctx.get_error() == ref_err == (0, 0)
    ctx.close()


def test_chain_waits_run_out_without_row_statistics():
    """No row statistics ever come: the sampler's bounded polls run out, every
    request with a valid temperature fails with the wait bit, and the context
    gives a fresh context's results on the next normal call."""
    wl = workloads.make_random(6, 3, 5000, "bf16", gen_seed=321, temps=(0.0, 1.0), verify_seed=1)
    wl.temperature[5] = -1.0  # an input error still wins over the wait
    ctx = binding.SpecVerify(MAX_B, MAX_N, MAX_V, torch.bfloat16)
    ctx.debug_skip_row_stats(True)
    t0 = time.time()
    toks, acc, kv = _host(ctx(*_inputs(wl), 5))
    elapsed = time.time() - t0
    code, bits = ctx.get_error()
    assert code == binding.SV_EBADTEMP and bits == binding.SV_ERRBIT_WAIT | binding.SV_ERRBIT_TEMP
    assert (acc == -1).all() and (kv == 0).all() and (toks == -1).all()
    assert elapsed < 60
    ctx.debug_skip_row_stats(False)
    wl.temperature[5] = 1.0
    got = _host(ctx(*_inputs(wl), 5))
    ref, ref_err = _fresh(wl, 5)
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    assert ctx.get_error() == ref_err == (0, 0)
    ctx.close()


def test_tree_waits_run_out_without_row_statistics():
    """The same for the tree walk: the cluster fails each request together."""
    tree = workloads.make_tree(5, 5000, "bf16", gen_seed=322, widths=(2, 2), temps=(0.0, 1.0), verify_seed=2)
    ctx = binding.SpecVerify(MAX_B, MAX_N, MAX_V, torch.bfloat16)
    args = (tree.target.cuda(), tree.draft.cuda(), tree.parents.cuda(), tree.tokens.cuda(),
            tree.temperature.cuda(), 9, tree.mode)
    ctx.debug_skip_row_stats(True)
    toks, path, acc, kv = _host(ctx.tree(*args))
    code, bits = ctx.get_error()
    assert code == binding.SV_ETIMEOUT and bits == binding.SV_ERRBIT_WAIT
    assert (acc == -1).all() and (kv == 0).all() and (toks == -1).all() and (path == -1).all()
    ctx.debug_skip_row_stats(False)
    got = _host(ctx.tree(*args))
    assert ctx.get_error() == (0, 0)
    fresh = binding.SpecVerify(MAX_B, MAX_N, MAX_V, torch.bfloat16)
    ref = _host(fresh.tree(*args))
    fresh.close()
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    ctx.close()


@pytest.mark.parametrize("cta", [0, 1, 4])
def test_one_sampler_cta_gives_up_while_the_others_finish(cta):
    """One sampler CTA of every request acts as if its wait for the row
    statistics ran out, while the request's other CTAs finish their blocks
    and count in (V = 70000 bf16: five CTAs per request).  Every sampled
    request fails as a whole with the wait bit (greedy requests too when
    the CTA is 0, the one that walks them); the next normal calls on the
    same context give a fresh context's results, so nothing the CTAs share
    outlives the call."""
    wl = workloads.make_random(12, 5, 70000, "bf16", gen_seed=323, temps=(0.0, 1.0), verify_seed=3)
    sampled = (wl.temperature > 0).numpy()
    assert sampled.any() and (~sampled).any()
    ctx = binding.SpecVerify(12, 5, 70000, torch.bfloat16)
    ctx.debug_late_cta(cta)
    toks, acc, kv = _host(ctx(*_inputs(wl), 7))
    code, bits = ctx.get_error()
    assert code == binding.SV_ETIMEOUT and bits == binding.SV_ERRBIT_WAIT
    failed = sampled if cta > 0 else sampled | ~sampled
    assert (acc[failed] == -1).all() and (kv[failed] == 0).all() and (toks[failed] == -1).all()
    ref, ref_err = _fresh(wl, 7)
    assert ref_err == (0, 0)
    for a, b in zip((toks, acc, kv), ref):
        assert torch.equal(a[~failed], b[~failed])
    ctx.debug_late_cta(-1)
    for seed in (7, 8):
        got = _host(ctx(*_inputs(wl), seed))
        ref, ref_err = _fresh(wl, seed)
        for a, b in zip(got, ref):
            assert torch.equal(a, b), seed
        assert ctx.get_error() == ref_err == (0, 0)
    ctx.close()


@pytest.mark.parametrize("cta", [1, 4])
def test_sampler_cta_gives_up_on_a_request_with_a_bad_logit(cta):
    """One sampler CTA of every request acts as if its wait ran out, on a
    batch where two sampled requests also carry a NaN / +inf logit: that
    CTA stops at the wait, its peers at the logit check.  Each failed
    request's CTAs still all count in, so the next normal calls on the same
    context (clean inputs) give a fresh context's results and no error."""
    wl = workloads.make_random(12, 5, 70000, "bf16", gen_seed=324, temps=(0.0, 1.0), verify_seed=3)
    sampled = (wl.temperature > 0).numpy()
    bad = [int(b) for b in sampled.nonzero()[0][:2]]
    assert len(bad) == 2 and (~sampled).any()
    target = wl.target.clone()
    target[bad[0], 1, 12345] = float("nan")
    target[bad[1], 0, 69999] = float("inf")
    ctx = binding.SpecVerify(12, 5, 70000, torch.bfloat16)
    ctx.debug_late_cta(cta)
    toks, acc, kv = _host(ctx(target.cuda(), wl.draft.cuda(), wl.tokens.cuda(), wl.temperature.cuda(), 7))
    code, bits = ctx.get_error()
    assert bits & binding.SV_ERRBIT_WAIT and bits & binding.SV_ERRBIT_LOGIT, (code, bits)
    assert (acc[sampled] == -1).all() and (kv[sampled] == 0).all() and (toks[sampled] == -1).all()
    ctx.debug_late_cta(-1)
    for seed in (7, 8):
        got = _host(ctx(*_inputs(wl), seed))
        ref, ref_err = _fresh(wl, seed)
        for a, b in zip(got, ref):
            assert torch.equal(a, b), seed
        assert ctx.get_error() == ref_err == (0, 0)
    ctx.close()
