"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Every test here needs a CUDA device; all inputs are seeded synthetic
workloads from ``workloads`` and every expected value comes from
``oracle``.
"""

import numpy as np
import pytest
import torch

from oracle import philox as oph
from oracle import verify as ov
from speculative_decoding_verification_73_gb300 import binding, build, workloads

from parity import (check_quota, compare, max_prob_rel, max_rel, near_threshold_count, prob_close,
                    rel_close, run_oracle)

pytestmark = pytest.mark.gpu

TORCH_DT = {"bf16": torch.bfloat16, "f32": torch.float32}


@pytest.fixture(scope="session", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return binding.load()


def run_gpu(wl, seed=None, ctx=None):
    B, N, V = wl.shape
    own = ctx is None
    if own:
        ctx = binding.SpecVerify(max(B, 1), N, V, TORCH_DT[wl.dtype])
    z = wl.target.cuda()
    y = wl.draft.cuda() if N > 0 else None
    d = wl.tokens.cuda()
    t = wl.temperature.cuda()
    toks, acc, kv = ctx(z, y, d, t, wl.seed if seed is None else seed)
    code, bits = ctx.get_error()
    stats = ctx.debug_stats(B, N) if B > 0 else (None, None)
    out = (toks.cpu().numpy().copy(), acc.cpu().numpy().copy(), kv.cpu().numpy().copy(), code, bits,
           [s.cpu().numpy() if s is not None else None for s in stats])
    if own:
        ctx.close()
    return out


def check(wl, seed=None, label="", stats=True):
    res = run_oracle(wl, seed)
    toks, acc, kv, code, bits, (acc_prob, logz) = run_gpu(wl, seed)
    B, N, V = wl.shape
    assert bits == res.errors, (bits, res.errors)
    logged = compare(res, toks, acc, kv, wl.temperature.numpy(), N, label or wl.name)
    if stats and B > 0:
        z, y = wl.raw()
        probs, lz_t, lz_d = ov.acceptance_probabilities(z, y, wl.tokens.numpy(),
                                                        wl.temperature.numpy(), wl.dtype)
        ok_req = res.request_errors == 0
        if N > 0:
            assert prob_close(acc_prob[ok_req], probs[ok_req]), max_prob_rel(acc_prob[ok_req], probs[ok_req])
        ref_lz = np.concatenate([lz_t, lz_d], axis=1)
        assert rel_close(logz[ok_req], ref_lz[ok_req]), max_rel(logz[ok_req], ref_lz[ok_req])
    return res, logged


# ------------------------------------------------------------------ Philox

def test_philox_matches_oracle_on_a_million_counters():
    n = 1 << 20
    rng = np.random.default_rng(0)
    for seed in (0, 0x0123456789ABCDEF, 2 ** 64 - 1):
        ctr = rng.integers(0, 2 ** 32, size=(n, 3), dtype=np.uint64)
        ctr[: n // 2, 1] = rng.integers(1, 300, size=n // 2)   # the walk's (b, j, draw) range
        ctr[: n // 2, 2] = rng.integers(0, 2, size=n // 2)
        got = binding.spec_verify_debug_philox(seed, torch.from_numpy(ctr.astype(np.int64)).cuda())
        k0, k1 = oph.split_seed(seed)
        want = oph.philox4x32_10(ctr[:, 0], ctr[:, 1], ctr[:, 2], 0, k0, k1)
        got = got.cpu().numpy().astype(np.uint64)
        for w in range(4):
            assert np.array_equal(got[:, w], want[w]), (seed, w)


# ------------------------------------------------------------------ the five workloads

def test_tiny_f32():
    res, _ = check(workloads.tiny_f32())
    assert res.errors == 0


@pytest.mark.parametrize("temperature", [1.0, 0.0])
def test_single_bf16(temperature):
    wl = workloads.single_bf16(temperature)
    res, _ = check(wl)
    for seed in range(1, 6):
        check(wl, seed=seed, stats=False)


def test_batch64_bf16_full_size():
    wl = workloads.batch64_bf16()
    near = 0
    for seed in range(4):
        res, _ = check(wl, seed=seed, stats=(seed == 0))
        near += near_threshold_count(res)
    print("in-window decisions (oracle):", near)


def test_mixture_bf16_full_size():
    check(workloads.mixture_bf16())


@pytest.fixture(scope="module")
def alpha09():
    return workloads.Alpha09()


def test_alpha09_parity_on_sampled_seeds(alpha09):
    for seed in (0, 1, 2, 517, 999):
        check(alpha09.workload(seed), stats=(seed == 0))


def test_alpha09_mean_tokens_per_call_1000_seeds(alpha09):
    """(1 - 0.9^9) / (1 - 0.9) = 6.12579511 tokens per verifier call; 256 x
    1000 samples, var(a+1) = 9.129 -> standard error 0.00597; allow 4 sigma."""
    B, N, V = alpha09.batch, alpha09.n, alpha09.vocab
    ctx = binding.SpecVerify(B, N, V, torch.float32)
    z, y = alpha09.target.cuda(), alpha09.draft.cuda()
    t = alpha09.temperature.cuda()
    total = 0
    for seed in range(1000):
        d = alpha09.tokens(seed).cuda()
        _, acc, _ = ctx(z, y, d, t, seed)
        total += int(acc.sum().item()) + B
    assert ctx.get_error()[0] == 0
    ctx.close()
    mean = total / (B * 1000)
    closed = (1 - 0.9 ** 9) / (1 - 0.9)
    print("mean tokens per call", mean, "closed form", closed)
    assert abs(mean - closed) < 4 * 0.00597


def test_mismatch_rate_over_many_seeds():
    """100 verify seeds of a 64-request sampled batch (V = 32000, bf16):
    44,800 draft positions and 6,400 correction / bonus draws compared with
    the oracle; every mismatch must be near-threshold and there must be
    fewer than 1e-5 of the positions, i.e. none."""
    wl = workloads.make_random(64, 7, 32000, "bf16", gen_seed=4242, temps=(0.7, 1.0))
    B, N, V = wl.shape
    ctx = binding.SpecVerify(B, N, V, torch.bfloat16)
    z, y = wl.target.cuda(), wl.draft.cuda()
    d, t = wl.tokens.cuda(), wl.temperature.cuda()
    logged, near = [], 0
    for seed in range(100):
        toks, acc, kv = ctx(z, y, d, t, seed)
        res = run_oracle(wl, seed)
        near += near_threshold_count(res)
        logged += compare(res, toks.cpu().numpy(), acc.cpu().numpy(), kv.cpu().numpy(),
                          wl.temperature.numpy(), N, f"seed {seed}", quota=False)
    ctx.close()
    print(f"mismatches {len(logged)} over {B * N * 100} positions; in-window oracle decisions {near}")
    check_quota(len(logged), B * N * 100)


# ------------------------------------------------------------------ shapes and edges

SHAPES = [
    # B, N, V, dtype     (row spans: 32768 bf16 / 16384 f32 elements; sampler blocks 8192)
    (1, 0, 1, "f32"),
    (3, 1, 3, "bf16"),          # scalar path (6 bytes per row)
    (5, 3, 8191, "bf16"),       # scalar path, one chunk minus one
    (4, 2, 8192, "f32"),        # exactly one row chunk
    (7, 4, 20000, "bf16"),      # two row chunks, ragged tail
    (6, 5, 4097, "f32"),        # scalar path, ragged
    (9, 8, 40000, "f32"),       # several chunks
    (33, 2, 24577, "bf16"),     # scalar path, several chunks
    (2, 0, 50000, "bf16"),      # bonus only
    (17, 6, 65536, "bf16"),
    (4, 3, 150000, "f32"),      # ten spans per row: partials merged past the first four
    (3, 2, 150001, "f32"),      # the same on the scalar path
]


@pytest.mark.parametrize("B,N,V,dtype", SHAPES)
def test_shapes_mixed_temperatures(B, N, V, dtype):
    wl = workloads.make_random(B, N, V, dtype, gen_seed=B * 1000 + N * 10 + V % 97, verify_seed=V)
    check(wl)


@pytest.mark.parametrize("B,N,V,dtype", [(3, 2, 300000, "bf16"), (2, 3, 270000, "f32")])
def test_more_than_32_level1_blocks(B, N, V, dtype):
    """37 (bf16) and 33 (fp32) level-1 blocks of 8192 tokens: the last
    sampler CTA picks level 1 over more than 32 masses (the tiled pass of the
    warp pick) and fetches the chosen block's candidate by index; sampled
    requests only, three verify seeds each."""
    wl = workloads.make_random(B, N, V, dtype, gen_seed=V % 1000 + B, verify_seed=V, temps=(0.7, 1.0))
    for seed in range(3):
        check(wl, seed=seed, stats=(seed == 0))


def test_max_drafts():
    wl = workloads.make_random(3, 255, 96, "f32", gen_seed=5, temps=(0.0, 1.0, 2.0), sigma=(0.0, 0.05))
    check(wl)


def test_max_drafts_bf16_two_spans():
    # every walk thread holds a row pair, each row two spans
    wl = workloads.make_random(2, 255, 40000, "bf16", gen_seed=6, temps=(0.0, 1.0), sigma=(0.0, 0.05))
    check(wl)


def test_batch_of_zero_is_a_noop():
    ctx = binding.SpecVerify(4, 3, 100, torch.float32)
    z = torch.zeros(0, 4, 100, device="cuda")
    binding.spec_verify(ctx.ctx, z, torch.zeros(0, 3, 100, device="cuda"),
                        torch.zeros(0, 3, dtype=torch.int32, device="cuda"),
                        torch.zeros(0, device="cuda"), 0, ctx.out_tokens[:0], ctx.out_accept[:0],
                        ctx.out_kv[:0])
    assert ctx.get_error() == (0, 0)
    ctx.close()


def test_size_checks_on_device_context():
    ctx = binding.SpecVerify(2, 3, 100, torch.float32)
    out_t = torch.empty(64, dtype=torch.int32, device="cuda")
    out_a = torch.empty(8, dtype=torch.int32, device="cuda")
    out_k = torch.empty(8, dtype=torch.int32, device="cuda")
    z = torch.zeros(3, 4, 100, device="cuda")          # B = 3 > max_B
    with pytest.raises(binding.SpecVerifyError):
        binding.spec_verify(ctx.ctx, z, torch.zeros(3, 3, 100, device="cuda"),
                            torch.zeros(3, 3, dtype=torch.int32, device="cuda"),
                            torch.ones(3, device="cuda"), 0, out_t[:12], out_a[:3], out_k[:3])
    z = torch.zeros(1, 5, 101, device="cuda")          # N = 4 > max_N and V > max_V
    with pytest.raises(binding.SpecVerifyError):
        binding.spec_verify(ctx.ctx, z, torch.zeros(1, 4, 101, device="cuda"),
                            torch.zeros(1, 4, dtype=torch.int32, device="cuda"),
                            torch.ones(1, device="cuda"), 0, out_t[:5], out_a[:1], out_k[:1])
    assert ctx.get_error() == (0, 0)
    ctx.close()


def test_greedy_ties_lowest_index():
    B, N, V = 6, 4, 3000
    g = torch.Generator().manual_seed(3)
    z = torch.randint(-3, 2, (B, N + 1, V), generator=g).to(torch.bfloat16)  # many ties at 1
    d = torch.zeros(B, N, dtype=torch.int32)
    for b in range(B):
        for j in range(N):
            am = int(np.argmax(z[b, j].float().numpy()))
            d[b, j] = am if (b + j) % 3 else (am + 1) % V
    wl = workloads.Workload("ties", "bf16", z, z[:, :N].contiguous(), d, torch.zeros(B), 0)
    check(wl)


def test_masked_vocabulary_entries():
    wl = workloads.make_random(8, 4, 10000, "bf16", gen_seed=77)
    wl.target[:, :, 5000:6000] = float("-inf")
    wl.draft[:, :, 5500:7000] = float("-inf")
    wl.draft[0, 0, int(wl.tokens[0, 0])] = float("-inf")   # p(d) = 0 -> accepted
    res, _ = check(wl)
    if wl.temperature[0] > 0:
        assert res.accept_len[0] >= 1


def test_kv_rollback_two_sequences():
    """Sequence A accepts every draft, sequence B is rejected at position 2."""
    n, v = 4, 8
    z = torch.zeros(2, n + 1, v)
    y = torch.zeros(2, n, v)
    d = torch.tensor([[1, 2, 3, 4], [5, 6, 7, 0]], dtype=torch.int32)
    for j in range(n):
        z[0, j, d[0, j]] = 2.0
    z[1, 0, d[1, 0]] = 2.0
    z[1, 1, d[1, 1]] = float("-inf")
    for seed in range(5):
        wl = workloads.Workload("rollback", "f32", z, y, d, torch.ones(2), seed)
        toks, acc, kv, code, _, _ = run_gpu(wl)
        assert code == 0
        assert acc.tolist() == [n, 1] and kv.tolist() == [n + 1, 2]
        assert toks[1, 1] != d[1, 1] and (toks[1, 2:] == -1).all()
        check(wl, stats=False)


def test_input_errors_are_flagged_per_request():
    wl = workloads.make_random(8, 3, 5000, "bf16", gen_seed=11, temps=(0.7, 1.0))
    wl.temperature[0] = -1.0
    wl.temperature[1] = float("nan")
    wl.temperature[2] = 1e-40
    wl.tokens[3, 1] = 5000
    wl.tokens[4, 0] = -3
    wl.target[5, 2, 17] = float("nan")
    wl.draft[6, 1, :] = float("-inf")
    wl.target[7, 0, 99] = float("inf")
    res = run_oracle(wl)
    assert res.request_errors.tolist() == [1, 1, 1, 2, 2, 4, 4, 4]
    toks, acc, kv, code, bits, _ = run_gpu(wl)
    assert code == binding.SV_EBADTEMP and bits == 7
    assert (acc == -1).all() and (kv == 0).all() and (toks == -1).all()
    # a greedy request never reads its draft rows: a NaN there is not an error
    wl2 = workloads.make_random(2, 3, 5000, "bf16", gen_seed=12, temps=(0.0,))
    wl2.draft[0, 1, 3] = float("nan")
    check(wl2)
    # errors clear after a read, and other requests are unaffected
    wl3 = workloads.make_random(4, 3, 5000, "f32", gen_seed=13, temps=(0.0, 1.0))
    wl3.tokens[2, 2] = 10 ** 6
    res3, _ = check(wl3)
    assert res3.errors == ov.ERR_TOKEN


def test_repeat_calls_are_deterministic():
    wl = workloads.make_random(16, 5, 30000, "bf16", gen_seed=21)
    a = run_gpu(wl)
    b = run_gpu(wl)
    for x, y in zip(a[:3], b[:3]):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("slot", [0, 1, 2])
def test_slot_law_matches_q(slot):
    """The Leviathan invariant on the GPU path itself, slot by slot: given
    that the first ``slot`` drafts were accepted, the token emitted in that
    slot (the next accepted draft, or the correction / bonus) is distributed
    as q_{slot+1} (chi-square over 16 tokens at 99.9 %).  Each call verifies
    256 copies of one request whose drafts are redrawn from p; the Philox
    counters differ by request index and by seed."""
    v, n, batch, calls = 16, 3, 256, 48
    g = torch.Generator().manual_seed(8)
    z = torch.randn(1, n + 1, v, generator=g) * 1.5
    y = z[:, :n] + torch.randn(1, n, v, generator=g)
    q = [ov.softmax(z[0, j].double().numpy(), 1.0) for j in range(n + 1)]
    p = [ov.softmax(y[0, j].double().numpy(), 1.0) for j in range(n)]
    rng = np.random.default_rng(1 + slot)
    ctx = binding.SpecVerify(batch, n, v, torch.float32)
    zc = z.expand(batch, n + 1, v).contiguous().cuda()
    yc = y.expand(batch, n, v).contiguous().cuda()
    t = torch.ones(batch, device="cuda")
    counts = np.zeros(v)
    for s in range(calls):
        d = np.stack([rng.choice(v, size=batch, p=p[j]) for j in range(n)], axis=1)
        toks, acc, _ = ctx(zc, yc, torch.from_numpy(d.astype(np.int32)).cuda(), t, 1000 * slot + s)
        toks, acc = toks.cpu().numpy(), acc.cpu().numpy()
        reached = acc >= slot
        np.add.at(counts, toks[reached, slot], 1)
    assert ctx.get_error()[0] == 0
    ctx.close()
    total = counts.sum()
    assert total > 2000, total
    exp = total * q[slot]
    chi2 = float(np.sum((counts - exp) ** 2 / exp))
    print(f"slot {slot}: {int(total)} samples, chi2 {chi2:.1f}")
    assert chi2 < 37.7   # 15 degrees of freedom, 99.9%
