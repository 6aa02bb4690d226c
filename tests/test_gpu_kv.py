"""GPU KV commit through the C ABI against the KV-commit oracle, byte for
byte, driven by real out_kv_len / out_path from the verify kernels."""

import numpy as np
import pytest
import torch

from oracle import kv as okv
from speculative_decoding_verification_73_gb300 import binding, build, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return binding.load()


def _bytes(shape, seed):
    g = torch.Generator()
    g.manual_seed(seed)
    return torch.randint(0, 256, shape, generator=g, dtype=torch.uint8)


def _commit_both(ctx, mode, cache, scratch, seq, kv, path=None):
    want, want_len, want_err = okv.commit(mode, cache.numpy().copy(), seq.numpy(), kv.numpy(),
                                          scratch=None if scratch is None else scratch.numpy(),
                                          path=None if path is None else path.numpy())
    d_cache, d_seq = cache.cuda(), seq.cuda()
    binding.spec_verify_kv_commit(ctx.ctx, mode, d_cache, d_seq, kv.cuda(),
                                  scratch=None if scratch is None else scratch.cuda(),
                                  path=None if path is None else path.cuda())
    code, bits = ctx.get_error()
    np.testing.assert_array_equal(d_cache.cpu().numpy(), want)
    np.testing.assert_array_equal(d_seq.cpu().numpy(), want_len)
    assert bits == want_err, (bits, want_err)
    return want_err


def test_chain_commit_from_spec_verify():
    wl = workloads.make_random(16, 6, 2000, "f32", gen_seed=81, verify_seed=1)
    B, N, V = wl.shape
    ctx = binding.SpecVerify(B, N, V, torch.float32)
    _, _, kv = ctx(wl.target.cuda(), wl.draft.cuda(), wl.tokens.cuda(), wl.temperature.cuda(), 5)
    kv = kv.cpu().clone()
    L, S, E, W = 3, 40, 64, N + 1
    cache = _bytes((L, B, S, E), 1)
    scratch = _bytes((L, B, W, E), 2)
    seq = torch.randint(0, S - W, (B,), generator=torch.Generator().manual_seed(3), dtype=torch.int32)
    assert _commit_both(ctx, binding.SV_KV_SCRATCH, cache, scratch, seq, kv) == 0
    # in place: the window already sits after each length
    placed = cache.clone()
    for b in range(B):
        placed[:, b, int(seq[b]):int(seq[b]) + W] = scratch[:, b]
    assert _commit_both(ctx, binding.SV_KV_INPLACE, placed, None, seq, kv) == 0
    ctx.close()


def test_tree_commit_from_spec_verify_tree():
    wl = workloads.make_tree(12, 3000, "f32", gen_seed=82, m=20, verify_seed=2)
    B, M, V = wl.shape
    ctx = binding.SpecVerify(B, M, V, torch.float32)
    _, path, _, kv = ctx.tree(wl.target.cuda(), wl.draft.cuda(), wl.parents.cuda(), wl.tokens.cuda(),
                              wl.temperature.cuda(), 9)
    path, kv = path.cpu().clone(), kv.cpu().clone()
    assert (kv > 1).any()
    L, S, E, W = 2, 48, 32, M + 1
    cache = _bytes((L, B, S, E), 4)
    scratch = _bytes((L, B, W, E), 5)
    seq = torch.randint(0, S - W, (B,), generator=torch.Generator().manual_seed(6), dtype=torch.int32)
    assert _commit_both(ctx, binding.SV_KV_SCRATCH, cache, scratch, seq, kv, path) == 0
    placed = cache.clone()
    for b in range(B):
        placed[:, b, int(seq[b]):int(seq[b]) + W] = scratch[:, b]
    assert _commit_both(ctx, binding.SV_KV_INPLACE, placed, None, seq, kv, path) == 0
    ctx.close()


def test_refused_commits_leave_the_sequence_alone():
    ctx = binding.SpecVerify(4, 4, 64, torch.float32)
    L, B, S, E, W = 2, 4, 10, 48, 5
    cache = _bytes((L, B, S, E), 7)
    scratch = _bytes((L, B, W, E), 8)
    seq = torch.tensor([8, 2, 1, 3], dtype=torch.int32)
    kv = torch.tensor([3, 0, 3, -1], dtype=torch.int32)          # seq 0 overflows S
    path = torch.tensor([[1, 2, -1], [1, -1, -1], [3, 2, -1], [1, 2, 3]], dtype=torch.int32)  # seq 2 falls
    err = _commit_both(ctx, binding.SV_KV_SCRATCH, cache, scratch, seq, kv, path)
    assert err == okv.ERR_KV
    ctx.close()


def test_full_size_commit_32_layers():
    """32 layers x 64 sequences x 4 KB entries (8 KV heads x 128 dims x K,V
    in bf16), an 8-position window, KV lengths of the 64-request verify."""
    wl = workloads.batch64_bf16()
    B, N, V = wl.shape
    ctx = binding.SpecVerify(B, N, V, torch.bfloat16)
    _, _, kv = ctx(wl.target.cuda(), wl.draft.cuda(), wl.tokens.cuda(), wl.temperature.cuda(), 0)
    kv = kv.cpu().clone()
    L, S, E, W = 32, 24, 4096, N + 1
    cache = _bytes((L, B, S, E), 9)
    scratch = _bytes((L, B, W, E), 10)
    seq = torch.randint(0, S - W, (B,), generator=torch.Generator().manual_seed(11), dtype=torch.int32)
    assert _commit_both(ctx, binding.SV_KV_SCRATCH, cache, scratch, seq, kv) == 0
    ctx.close()


def _commit_chain(ctx, mode, cache, scratch_list, seq, kv_list, path_list=None):
    """Several commits back to back on one context (no host sync between
    them), against the oracle applied in the same order."""
    want, want_len = cache.numpy().copy(), seq.numpy().copy()
    d_cache, d_seq = cache.cuda(), seq.cuda()
    for i, kv in enumerate(kv_list):
        scratch = None if scratch_list is None else scratch_list[i]
        path = None if path_list is None else path_list[i]
        want, want_len, _ = okv.commit(mode, want, want_len, kv.numpy(),
                                       scratch=None if scratch is None else scratch.numpy(),
                                       path=None if path is None else path.numpy())
        binding.spec_verify_kv_commit(ctx.ctx, mode, d_cache, d_seq, kv.cuda(),
                                      scratch=None if scratch is None else scratch.cuda(),
                                      path=None if path is None else path.cuda())
    code, bits = ctx.get_error()
    assert bits == 0, bits
    np.testing.assert_array_equal(d_seq.cpu().numpy(), want_len)
    np.testing.assert_array_equal(d_cache.cpu().numpy(), want)


@pytest.mark.parametrize("E", [48, 8192], ids=["one-slice", "two-slices"])
def test_back_to_back_commits_advance_each_length_once(E):
    """Four commits issued back to back (no host sync): each one's lengths
    move exactly once, after every layer's copy has read them; entries of
    one column slice and of two 4 KB slices."""
    ctx = binding.SpecVerify(8, 4, 64, torch.float32)
    L, B, S, W = 3, 5, 40, 5
    cache = _bytes((L, B, S, E), 21)
    g = torch.Generator().manual_seed(22)
    scratch = [_bytes((L, B, W, E), 23 + i) for i in range(4)]
    kv = [torch.randint(0, W + 1, (B,), generator=g, dtype=torch.int32) for _ in range(4)]
    seq = torch.randint(0, 8, (B,), generator=g, dtype=torch.int32)
    _commit_chain(ctx, binding.SV_KV_SCRATCH, cache, scratch, seq, kv)
    ctx.close()


def test_back_to_back_in_place_commits_between_verify_calls():
    """In-place commits driven by tree paths, with verify calls on the same
    context in between (the calls share the context's sequence numbers)."""
    B, M, V = 4, 6, 96
    ctx = binding.SpecVerify(B, M, V, torch.float32)
    L, S, E = 2, 48, 32
    cache = _bytes((L, B, S, E), 31)
    seq = torch.tensor([0, 5, 9, 2], dtype=torch.int32)
    g = torch.Generator().manual_seed(32)
    want, want_len = cache.numpy().copy(), seq.numpy().copy()
    d_cache, d_seq = cache.cuda(), seq.cuda()
    z = torch.randn(B, M + 1, V, generator=g).cuda()
    tok = torch.randint(0, V, (B, M), generator=g, dtype=torch.int32).cuda()
    temp = torch.ones(B).cuda()
    for i in range(3):
        ctx(z, z[:, :M].contiguous(), tok, temp, i)  # a chain verify in between
        path = torch.tensor([[1, 3, -1, -1, -1, -1], [2, -1, -1, -1, -1, -1],
                             [1, 2, 4, -1, -1, -1], [-1] * 6], dtype=torch.int32)
        kv = torch.tensor([3, 2, 4, 1], dtype=torch.int32)
        want, want_len, err = okv.commit(binding.SV_KV_INPLACE, want, want_len, kv.numpy(), path=path.numpy())
        assert err == 0
        binding.spec_verify_kv_commit(ctx.ctx, binding.SV_KV_INPLACE, d_cache, d_seq, kv.cuda(), path=path.cuda())
    code, bits = ctx.get_error()
    assert bits == 0, bits
    np.testing.assert_array_equal(d_seq.cpu().numpy(), want_len)
    np.testing.assert_array_equal(d_cache.cpu().numpy(), want)
    ctx.close()
