"""Pins of the oracle's float64 row math, greedy path, validation and batch
driver (CPU only)."""

import math

import numpy as np
import pytest
import torch

from oracle import philox
from oracle import verify as ov


# ---------------------------------------------------------------- widening

def test_bf16_widening_bit_patterns():
    # bfloat16 = sign, 8 exponent bits, 7 fraction bits (the top half of an
    # IEEE binary32): values below follow from that definition.
    cases = {
        0x3F80: 1.0, 0xC000: -2.0, 0x4049: 3.140625, 0x0000: 0.0,
        0x8000: -0.0, 0x7F80: math.inf, 0xFF80: -math.inf,
        0x0001: 2.0 ** -133, 0x7F7F: (2 - 2 ** -7) * 2.0 ** 127,
        0x3C00: 2.0 ** -7,
    }
    bits = np.array(list(cases), dtype=np.uint16)
    got = ov.logits_to_f64(bits, "bf16")
    for g, want in zip(got, cases.values()):
        assert g == want
    assert math.isnan(ov.logits_to_f64(np.array([0x7FC0], np.uint16), "bf16")[0])
    # agrees with torch's own bf16 -> float64 conversion on random patterns
    rnd = np.random.default_rng(0).integers(0, 2 ** 16, 4096).astype(np.uint16)
    t = torch.from_numpy(rnd.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    o = ov.logits_to_f64(rnd, "bf16")
    same = (t == o) | (np.isnan(t) & np.isnan(o))
    assert same.all()


# ---------------------------------------------------------------- softmax

def test_softmax_uniform_row():
    for v in (1, 7, 1024):
        x = np.full(v, 3.25)
        q = ov.softmax(x, 0.7)
        assert np.allclose(q, 1.0 / v, rtol=1e-15, atol=0)
        assert ov.log_partition(x, 0.7) == pytest.approx(3.25 / 0.7 + math.log(v), rel=1e-15)


def test_softmax_spike_closed_form():
    v, a, t = 1000, 5.0, 0.5
    x = np.zeros(v)
    x[17] = a
    q = ov.softmax(x, t)
    e = math.exp(a / t)
    assert q[17] == pytest.approx(e / (e + v - 1), rel=1e-14)
    assert q[0] == pytest.approx(1 / (e + v - 1), rel=1e-14)


def test_softmax_temperature_and_shift_invariance():
    rng = np.random.default_rng(3)
    x = rng.normal(size=513) * 4
    q1 = ov.softmax(x, 0.25)
    q2 = ov.softmax(x / 0.25 + 100.0, 1.0)
    assert np.allclose(q1, q2, rtol=1e-12, atol=1e-300)
    assert abs(np.sum(q1) - 1) < 1e-14


def test_softmax_matches_library():
    rng = np.random.default_rng(4)
    for t in (0.05, 0.7, 1.0, 3.0):
        x = rng.normal(size=2000) * 3
        want = torch.softmax(torch.from_numpy(x) / t, dim=0).numpy()
        assert np.allclose(ov.softmax(x, t), want, rtol=1e-12, atol=1e-300)
        lz = torch.logsumexp(torch.from_numpy(x) / t, dim=0).item()
        assert ov.log_partition(x, t) == pytest.approx(lz, rel=1e-13)


def test_softmax_neg_inf_and_large():
    x = np.array([-np.inf, 1e4, 1e4 - 1.0, -np.inf])
    q = ov.softmax(x, 1.0)
    assert q[0] == 0 and q[3] == 0
    assert q[1] == pytest.approx(1 / (1 + math.exp(-1)), rel=1e-14)


# ---------------------------------------------------------------- greedy

def _brute_argmax(row):
    return sorted(range(len(row)), key=lambda t: (-row[t], t))[0]


def test_greedy_chain_brute_force_with_ties():
    rng = np.random.default_rng(5)
    for trial in range(200):
        n, v = int(rng.integers(0, 5)), int(rng.integers(1, 9))
        z = rng.integers(-2, 3, size=(n + 1, v)).astype(np.float64)  # many ties
        g = [_brute_argmax(z[j]) for j in range(n + 1)]
        d = [g[j] if rng.random() < 0.7 else int(rng.integers(0, v)) for j in range(n)]
        tokens, a, kv = ov.greedy_walk(z, d)
        want_a = next((j for j in range(n) if d[j] != g[j]), n)
        assert a == want_a and kv == want_a + 1
        assert tokens == g[: want_a + 1]


# ---------------------------------------------------------------- validation

def _one(z, y, d, t, dtype="f32"):
    res = ov.verify(np.asarray(z, np.float32)[None], None if y is None else np.asarray(y, np.float32)[None],
                    np.asarray(d, np.int32)[None], np.array([t], np.float32), 0, dtype)
    return res


def test_validation_errors_and_order():
    z = np.zeros((3, 4), np.float32)
    y = np.zeros((2, 4), np.float32)
    for bad_t in (-1.0, float("nan"), float("inf"), 1e-40):
        r = _one(z, y, [0, 1], bad_t)
        assert r.errors == ov.ERR_TEMP and r.accept_len[0] == -1 and r.kv_len[0] == 0
        assert (r.tokens == -1).all()
    assert _one(z, y, [0, 4], 1.0).errors == ov.ERR_TOKEN
    assert _one(z, y, [-1, 0], 0.0).errors == ov.ERR_TOKEN
    zn = z.copy()
    zn[1, 2] = np.nan
    assert _one(zn, y, [0, 1], 1.0).errors == ov.ERR_LOGIT
    assert _one(zn, y, [0, 1], 0.0).errors == ov.ERR_LOGIT
    zi = z.copy()
    zi[2, 0] = np.inf
    assert _one(zi, y, [0, 1], 1.0).errors == ov.ERR_LOGIT
    yi = y.copy()
    yi[:] = -np.inf
    assert _one(z, yi, [0, 1], 1.0).errors == ov.ERR_LOGIT
    # a greedy request never reads its draft rows
    assert _one(z, yi, [0, 0], 0.0).errors == 0
    # the temperature check comes first, then tokens, then logits
    assert _one(zn, y, [0, 9], -1.0).errors == ov.ERR_TEMP
    assert _one(zn, y, [0, 9], 1.0).errors == ov.ERR_TOKEN


def test_neg_inf_draft_mass_is_accepted_and_q_zero_rejected():
    z = np.zeros((3, 4), np.float32)
    y = np.zeros((2, 4), np.float32)
    y[0, 2] = -np.inf          # p_1(2) = 0 -> accepted by the rule's guard
    z[1, 3] = -np.inf          # q_2(3) = 0 -> rejected whatever u is
    for seed in range(20):
        r = ov.verify(z[None], y[None], np.array([[2, 3]], np.int32), np.array([1.0], np.float32),
                      seed, "f32")
        assert r.accept_len[0] == 1 and r.kv_len[0] == 2
        assert r.tokens[0, 0] == 2 and r.tokens[0, 1] != 3 and r.tokens[0, 2] == -1


def test_no_drafts_samples_bonus_from_q1():
    rng = np.random.default_rng(9)
    z = rng.normal(size=(1, 1, 6)).astype(np.float32)
    q = ov.softmax(z[0, 0].astype(np.float64), 1.0)
    counts = np.zeros(6)
    for seed in range(3000):
        r = ov.verify(z, None, np.zeros((1, 0), np.int32), np.ones(1, np.float32), seed, "f32")
        assert r.accept_len[0] == 0 and r.kv_len[0] == 1
        counts[r.tokens[0, 0]] += 1
    chi2 = np.sum((counts - 3000 * q) ** 2 / (3000 * q))
    assert chi2 < 20.5  # 5 degrees of freedom, 99.9%


def test_batched_kv_rollback_exercise():
    """Two sequences (lesson exercise 4): A accepts every draft, B is
    rejected at position 2; each gets its own KV length."""
    n, v = 4, 8
    z = np.zeros((2, n + 1, v), np.float32)
    y = np.zeros((2, n, v), np.float32)
    d = np.array([[1, 2, 3, 4], [5, 6, 7, 0]], np.int32)
    # A: q(d) >= p(d) everywhere -> ratio >= 1 -> always accepted
    for j in range(n):
        z[0, j, d[0, j]] = 2.0
    # B: position 1 accepted (ratio >= 1), position 2 has q(d) = 0
    z[1, 0, d[1, 0]] = 2.0
    z[1, 1, d[1, 1]] = -np.inf
    for seed in range(10):
        r = ov.verify(z, y, d, np.ones(2, np.float32), seed, "f32")
        assert r.accept_len.tolist() == [n, 1]
        assert r.kv_len.tolist() == [n + 1, 2]
        assert r.tokens[0, :n].tolist() == d[0].tolist()
        assert r.tokens[1, 0] == d[1, 0] and r.tokens[1, 1] != d[1, 1]
        assert (r.tokens[1, 2:] == -1).all()


# ---------------------------------------------------------------- statistics

def test_leviathan_chi_square_like_lesson_step5():
    """The lesson's check (step 5): 50,000 speculative steps against 50,000
    direct draws from q; also against q itself."""
    v, n = 12, 3
    rng = np.random.default_rng(11)
    z = rng.normal(size=(n + 1, v)) * 1.2
    y = z[:n] + rng.normal(size=(n, v)) * 0.9
    q_rows = [ov.softmax(z[j], 1.0) for j in range(n + 1)]
    p_rows = [ov.softmax(y[j], 1.0) for j in range(n)]
    steps = 50_000
    first = np.zeros(v)
    cdfs = [np.cumsum(p) for p in p_rows]
    ud = rng.random((steps, n))
    for s in range(steps):
        drafts = [min(int(np.searchsorted(cdfs[j], ud[s, j], side="right")), v - 1) for j in range(n)]
        tokens, _, _, _ = ov.walk(q_rows, p_rows, drafts, ov.philox_draws(777, s))
        first[tokens[0]] += 1
    direct = np.bincount(np.searchsorted(np.cumsum(q_rows[0]), rng.random(steps), side="right"),
                         minlength=v)[:v]
    exp = steps * q_rows[0]
    chi2_q = float(np.sum((first - exp) ** 2 / exp))
    tot = first + direct
    e1, e2 = tot / 2, tot / 2
    mask = tot > 0
    chi2_two = float(np.sum((first[mask] - e1[mask]) ** 2 / e1[mask] + (direct[mask] - e2[mask]) ** 2 / e2[mask]))
    # 11 degrees of freedom: 95% critical value 19.68
    assert chi2_q < 19.68
    assert chi2_two < 19.68


def test_alpha09_mean_tokens_per_call():
    """alpha09 rows: overlap 0.9 at each of N=8 positions, so E[a+1] =
    (1 - 0.9^9) / 0.1 = 6.12579511.  100 seeds x 256 requests; var(a+1) =
    9.129 gives a standard error of 0.0189; allow 4 sigma."""
    from speculative_decoding_verification_73_gb300 import workloads
    wl = workloads.Alpha09()
    q_rows = [[ov.softmax(ov.logits_to_f64(wl.target[b, j].numpy(), "f32"), 1.0) for j in range(9)]
              for b in range(256)]
    p_rows = [[ov.softmax(ov.logits_to_f64(wl.draft[b, j].numpy(), "f32"), 1.0) for j in range(8)]
              for b in range(256)]
    for b in range(0, 256, 37):
        for j in range(8):
            ov_alpha = float(np.sum(np.minimum(q_rows[b][j], p_rows[b][j])))
            assert abs(ov_alpha - 0.9) < 1e-5
    total, count = 0, 0
    for seed in range(100):
        d = wl.tokens(seed).numpy()
        for b in range(256):
            _, a, _, _ = ov.walk(q_rows[b], p_rows[b], d[b], ov.philox_draws(seed, b))
            total += a + 1
            count += 1
    closed = (1 - 0.9 ** 9) / (1 - 0.9)
    assert closed == pytest.approx(6.12579511, abs=1e-8)
    assert abs(total / count - closed) < 4 * 0.0189


def test_single_bf16_sigma_gives_overlap_08():
    """The stored draft noise of the single-request V=128256 workload gives a
    mean overlap sum_t min(p, q) of 0.80 +- 0.01 under the oracle."""
    import json
    import os
    from speculative_decoding_verification_73_gb300 import workloads
    path = os.path.join(os.path.dirname(__file__), "golden", "single_bf16_sigma.json")
    stored = json.load(open(path))
    assert stored["sigma"] == workloads.SINGLE_BF16_SIGMA
    wl = workloads.single_bf16(1.0)
    z, y = wl.raw()
    zf, yf = ov.logits_to_f64(z[0], "bf16"), ov.logits_to_f64(y[0], "bf16")
    al = [float(np.sum(np.minimum(ov.softmax(zf[j], 1.0), ov.softmax(yf[j], 1.0)))) for j in range(5)]
    assert abs(np.mean(al) - 0.8) < 0.01


def test_grouped_sampler_chi_square_across_level1_blocks():
    """float64: draws with Philox uniforms over V = 20000 (three level-1
    blocks, ragged tail) follow the normalised masses."""
    rng = np.random.default_rng(21)
    v = 20000
    w = rng.random(v) ** 8                      # skewed masses, many tiny
    w[5000:5100] = 0.0
    bins = np.minimum(np.arange(v) // 400, 49)  # 50 bins of ~400 tokens
    p_bin = np.bincount(bins, weights=w, minlength=50) / w.sum()
    counts = np.zeros(50)
    n = 20000
    for s in range(n):
        t, _ = ov.sample_grouped(w, philox.uniforms4(99, s, 1, 1))
        assert w[t] > 0
        counts[bins[t]] += 1
    chi2 = float(np.sum((counts - n * p_bin) ** 2 / (n * p_bin)))
    assert chi2 < 85.4   # 49 degrees of freedom, 99.9%
