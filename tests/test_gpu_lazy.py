"""spec_verify_lazy on the GPU: bit for bit spec_verify's results on valid
inputs (which are pinned to the oracle elsewhere), the lazy oracle's errors
when a bad row lies past the stop, and parity with the oracle directly."""

import numpy as np
import pytest
import torch

from oracle import verify as ov
from speculative_decoding_verification_73_gb300 import binding, build, workloads

from parity import compare, run_oracle

pytestmark = pytest.mark.gpu
TORCH_DT = {"bf16": torch.bfloat16, "f32": torch.float32}


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return binding.load()


def _both(wl, seeds):
    B, N, V = wl.shape
    ctx = binding.SpecVerify(B, N, V, TORCH_DT[wl.dtype])
    z = wl.target.cuda()
    y = wl.draft.cuda() if N > 0 else None
    d, t = wl.tokens.cuda(), wl.temperature.cuda()
    out = []
    for s in seeds:
        e = [x.cpu().clone() for x in ctx(z, y, d, t, s)]
        ee = ctx.get_error()
        l = [x.cpu().clone() for x in ctx.lazy(z, y, d, t, s)]
        le = ctx.get_error()
        out.append((e, ee, l, le))
    ctx.close()
    return out


LAZY_CASES = {
    "tiny-f32": workloads.tiny_f32,
    "random-bf16": lambda: workloads.make_random(24, 7, 40960, "bf16", gen_seed=91, verify_seed=1),
    "random-f32-ragged": lambda: workloads.make_random(12, 5, 3001, "f32", gen_seed=92, verify_seed=2),
    "mixture-bf16": workloads.mixture_bf16,
    "batch64-bf16": workloads.batch64_bf16,
    "lowaccept64-bf16": workloads.low_accept_bf16,
    "no-drafts": lambda: workloads.make_random(6, 0, 5000, "f32", gen_seed=93),
    # 34 spans and 135 level-1 blocks per row: partials, token logits and the
    # draw's masses go through the workspace instead of distributed shared memory
    "huge-vocabulary-bf16": lambda: workloads.make_random(3, 3, 1100000, "bf16", gen_seed=96, verify_seed=5,
                                                          temps=(0.7, 1.0)),
}


@pytest.mark.parametrize("name", list(LAZY_CASES))
def test_lazy_is_spec_verify_bit_for_bit(name):
    wl = LAZY_CASES[name]()
    for e, ee, l, le in _both(wl, (0, 1, 2 ** 63 + 5)):
        for a, b in zip(e, l):
            assert torch.equal(a, b), name
        assert ee == le == (0, 0)


def test_lazy_matches_the_oracle():
    wl = workloads.make_random(32, 6, 20000, "bf16", gen_seed=94, verify_seed=4)
    B, N, V = wl.shape
    ctx = binding.SpecVerify(B, N, V, torch.bfloat16)
    for seed in (4, 5):
        toks, acc, kv = ctx.lazy(wl.target.cuda(), wl.draft.cuda(), wl.tokens.cuda(),
                                 wl.temperature.cuda(), seed)
        res = run_oracle(wl, seed)
        compare(res, toks.cpu().numpy(), acc.cpu().numpy(), kv.cpu().numpy(), wl.temperature.numpy(), N,
                f"lazy seed {seed}")
    ctx.close()


def test_bad_rows_past_the_stop_are_not_errors():
    wl = workloads.make_random(8, 5, 3000, "f32", gen_seed=95, verify_seed=3,
                               temps=(0.0, 1.0))
    wl.target[:, 5, 17] = float("nan")          # the bonus row: read only after 5 matches
    wl.draft[:, 4, 3] = float("inf")            # draft row 4: read only at position 5
    z, y = wl.raw()
    lazy = ov.verify(z, y, wl.tokens.numpy(), wl.temperature.numpy(), wl.seed, "f32", lazy=True)
    B, N, V = wl.shape
    ctx = binding.SpecVerify(B, N, V, torch.float32)
    toks, acc, kv = ctx.lazy(wl.target.cuda(), wl.draft.cuda(), wl.tokens.cuda(), wl.temperature.cuda(),
                             wl.seed)
    code, bits = ctx.get_error()
    assert bits == lazy.errors
    compare(lazy, toks.cpu().numpy(), acc.cpu().numpy(), kv.cpu().numpy(), wl.temperature.numpy(), N,
            "lazy-errors")
    assert (lazy.request_errors == 0).any()
    ctx.close()
