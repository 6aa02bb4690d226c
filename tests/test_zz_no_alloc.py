"""spec_verify_noalloc (no context, working memory in the library's static
device array) against spec_verify on the same inputs.

The file name sorts last, so in a full run these tests come after every
other test of the session; each one also passes alone in a fresh process,
where its first call is the one that looks up the array's address.
"""

import ctypes

import pytest
import torch

from speculative_decoding_verification_73_gb300 import binding, build, workloads

TORCH_DT = {"bf16": torch.bfloat16, "f32": torch.float32}


@pytest.fixture(scope="module")
def lib():
    try:
        build.build()
    except RuntimeError as e:
        pytest.skip(str(e))
    return binding.load()


def test_oversized_problem_is_refused_before_any_device_work(lib):
    """Size checks answer on the host: no pointer is read, nothing enqueued."""
    fake = ctypes.c_void_p(256)
    args = (fake, fake, fake, fake, ctypes.c_uint64(0), fake, fake, fake, None)
    # 4096 requests x 15 rows x 4 spans x 16 B of partials alone is ~3.9 MB > 1 MiB
    code = lib.spec_verify_noalloc(4096, 7, 128256, binding.SV_BF16, *args)
    assert code == binding.SV_ESCRATCH
    assert "SV_NOALLOC_SCRATCH_BYTES" in binding.strerror(code)
    # one request with 15 drafts over the largest vocabulary does not fit either
    assert lib.spec_verify_noalloc(1, 15, 1 << 26, binding.SV_F32, *args) == binding.SV_ESCRATCH
    # ordinary argument errors keep their code; B == 0 is a no-op
    assert lib.spec_verify_noalloc(1, 4, 100, 2, *args) == binding.SV_EINVAL
    assert lib.spec_verify_noalloc(1, 256, 100, 0, *args) == binding.SV_EINVAL
    assert lib.spec_verify_noalloc(1, 4, 0, 0, *args) == binding.SV_EINVAL
    assert lib.spec_verify_noalloc(1, 4, 100, 0, None, None, None, None, ctypes.c_uint64(0),
                                   None, None, None, None) == binding.SV_EINVAL
    assert lib.spec_verify_noalloc(0, 4, 100, 0, None, None, None, None, ctypes.c_uint64(0),
                                   None, None, None, None) == binding.SV_OK


def _device_inputs(wl):
    B, N, V = wl.shape
    z = wl.target.cuda()
    y = wl.draft.cuda() if N > 0 else None
    return z, y, wl.tokens.cuda(), wl.temperature.cuda()


def _outputs(B, N):
    # sentinel-filled so that a slot the kernels fail to write shows up
    return (torch.full((B, N + 1), -7, dtype=torch.int32, device="cuda"),
            torch.full((B,), -7, dtype=torch.int32, device="cuda"),
            torch.full((B,), -7, dtype=torch.int32, device="cuda"))


def _host(outs):
    return tuple(o.cpu().clone() for o in outs)


def _run_noalloc(wl, seeds, stream=None):
    B, N, V = wl.shape
    z, y, d, t = _device_inputs(wl)
    res = []
    for seed in seeds:
        outs = _outputs(B, N)
        if stream is not None:
            stream.wait_stream(torch.cuda.current_stream())
        binding.spec_verify_noalloc(z, y, d, t, seed, *outs, stream=stream)
        if stream is not None:
            stream.synchronize()
        torch.cuda.synchronize()
        res.append(_host(outs))
    return res


def _run_context(wl, seeds):
    B, N, V = wl.shape
    z, y, d, t = _device_inputs(wl)
    sv = binding.SpecVerify(B, N, V, TORCH_DT[wl.dtype])
    res = []
    try:
        for seed in seeds:
            outs = _outputs(B, N)
            binding.spec_verify(sv.ctx, z, y, d, t, seed, *outs)
            torch.cuda.synchronize()
            res.append(_host(outs))
    finally:
        sv.close()
    return res


def _assert_same(got, want, label):
    for (gt, ga, gk), (wt, wa, wk) in zip(got, want):
        assert torch.equal(ga, wa), f"{label}: accept lengths differ"
        assert torch.equal(gk, wk), f"{label}: KV lengths differ"
        assert torch.equal(gt, wt), f"{label}: tokens differ"
        assert int((ga == -7).sum()) == 0 and int((gt == -7).sum()) == 0, label


WORKLOADS = {
    "tiny-f32": workloads.tiny_f32,
    # ragged V (not a multiple of 8 elements): the scalar path; mixed temperatures
    "random-f32-ragged": lambda: workloads.make_random(12, 5, 3001, "f32", gen_seed=77,
                                                       verify_seed=5),
    "random-bf16": lambda: workloads.make_random(24, 3, 40960, "bf16", gen_seed=78,
                                                 verify_seed=9),
    "batch64-bf16": workloads.batch64_bf16,
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(WORKLOADS))
def test_two_calls_in_a_row_match_spec_verify(lib, name):
    """Integer outputs: identical, call after call, to the context entry point
    (the second call runs on the scratch the first one left behind)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wl = WORKLOADS[name]()
    seeds = (wl.seed, wl.seed + 1)
    got = _run_noalloc(wl, seeds)
    want = _run_context(wl, seeds)
    _assert_same(got, want, name)


@pytest.mark.gpu
def test_side_stream_and_bad_request(lib):
    """On a non-default stream; a request with a bad temperature is marked in
    its own outputs only, and the next call starts clean."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wl = workloads.make_random(8, 4, 2048, "bf16", gen_seed=79, verify_seed=3)
    bad = workloads.Workload(wl.name + "-bad", wl.dtype, wl.target, wl.draft, wl.tokens,
                             wl.temperature.clone(), wl.seed)
    bad.temperature[2] = -1.0
    stream = torch.cuda.Stream()
    got_bad = _run_noalloc(bad, (bad.seed,), stream=stream)
    got = _run_noalloc(wl, (wl.seed, wl.seed + 1), stream=stream)
    want_bad = _run_context(bad, (bad.seed,))
    want = _run_context(wl, (wl.seed, wl.seed + 1))
    _assert_same(got_bad, want_bad, "bad")
    t, a, k = got_bad[0]
    assert int(a[2]) == -1 and int(k[2]) == 0 and bool((t[2] == -1).all())
    _assert_same(got, want, "after-bad")
    assert bool((got[0][1] >= 0).all())
