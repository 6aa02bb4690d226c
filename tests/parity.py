"""GPU-vs-oracle comparison under the method's tolerances (test helper).

* greedy requests: tokens, accept length and KV length bit-exact;
* sampled requests: bit-exact, except where the oracle's decision at the
  point of divergence had its uniform within WINDOW (1e-5) of its threshold
  (|u - min(1, q/p)| for an accept test; for a correction / bonus draw, the
  distance of that level's uniform to the edges of the chosen sub-block at
  the first level of the grouped inverse CDF where the two tokens' blocks
  differ); every such mismatch is logged, and mismatches must stay below
  1e-5 of the verified positions;
* error requests: identical error bits and the -1 / 0 markers.
"""

import math

import numpy as np

from oracle.verify import LEVEL_SHIFTS

WINDOW = 1e-5


def oracle_inputs(wl):
    z, y = wl.raw()
    return z, y, wl.tokens.numpy(), wl.temperature.numpy()


def run_oracle(wl, seed=None):
    from oracle import verify as ov
    z, y, d, t = oracle_inputs(wl)
    return ov.verify(z, y, d, t, wl.seed if seed is None else seed, wl.dtype)


def near_threshold_count(res):
    return sum(1 for decs in res.decisions for dec in decs if dec.distance() < WINDOW)


def compare(res, tokens, accept, kv, temperature, n, label="", quota=True):
    """Check GPU outputs (numpy) against an oracle Result.  Returns the list
    of logged in-window mismatches; with quota=False the caller checks the
    mismatch count against its own total of positions."""
    tokens = np.asarray(tokens).reshape(res.tokens.shape)
    accept = np.asarray(accept).reshape(-1)
    kv = np.asarray(kv).reshape(-1)
    temperature = np.asarray(temperature).reshape(-1)
    logged = []
    for b in range(res.tokens.shape[0]):
        same = (np.array_equal(tokens[b], res.tokens[b]) and accept[b] == res.accept_len[b]
                and kv[b] == res.kv_len[b])
        if same:
            continue
        where = f"{label} request {b}: gpu a={accept[b]} kv={kv[b]} tok={tokens[b].tolist()} " \
                f"oracle a={res.accept_len[b]} kv={res.kv_len[b]} tok={res.tokens[b].tolist()}"
        assert res.request_errors[b] == 0, "error request differs: " + where
        assert float(temperature[b]) != 0.0, "greedy request differs: " + where
        assert kv[b] == accept[b] + 1, where
        decs = res.decisions[b]
        if accept[b] != res.accept_len[b]:
            j = min(int(accept[b]), int(res.accept_len[b])) + 1
            dec = [x for x in decs if x.kind == "accept" and x.j == j]
            assert dec, "no oracle decision at the divergence: " + where
            dist = dec[0].distance()
        else:
            dec = [x for x in decs if x.kind in ("residual", "bonus")]
            assert dec, "no oracle decision at the divergence: " + where
            # the accepted prefix must agree exactly
            a = int(accept[b])
            assert np.array_equal(tokens[b, :a], res.tokens[b, :a]), where
            t_gpu, t_ref = int(tokens[b, a]), int(res.tokens[b, a])
            level = next(lv for lv, sh in enumerate(LEVEL_SHIFTS) if (t_gpu >> sh) != (t_ref >> sh))
            dist = dec[0].distance(level)
        assert dist < WINDOW, f"mismatch outside the 1e-5 window (distance {dist:.3g}): " + where
        logged.append((label, b, dec[0].kind, dec[0].j, dist))
        print("near-threshold mismatch:", where, f"distance={dist:.3g}")
    if quota:
        check_quota(len(logged), tokens.shape[0] * max(n, 1))
    return logged


def check_quota(mismatches, positions):
    """Mismatches must stay below 1e-5 of the verified draft positions."""
    assert mismatches == 0 or mismatches < 1e-5 * positions, \
        f"{mismatches} mismatches over {positions} positions"


def rel_close(gpu, ref, rtol=WINDOW):
    """Row log-normalisers: |gpu - ref| <= rtol * max(|ref|, 1) elementwise,
    NaN where ref is NaN.  A logZ has magnitude near the row's largest
    scaled logit, so this is a relative bound wherever |logZ| >= 1."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    nan = np.isnan(ref)
    if not np.array_equal(nan, np.isnan(gpu)):
        return False
    d = np.abs(gpu[~nan] - ref[~nan])
    return bool(np.all(d <= rtol * np.maximum(np.abs(ref[~nan]), 1.0)))


def max_rel(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    m = ~np.isnan(ref)
    if not m.any():
        return 0.0
    return float(np.max(np.abs(gpu[m] - ref[m]) / np.maximum(np.abs(ref[m]), 1.0)))


# Smallest normal float32.  An acceptance probability below it is a float32
# subnormal on the GPU (or flushes to zero), whose spacing is no longer
# relative to the value; such a threshold is also below the 2^-24 step of
# the uniforms, so it decides like 0 for every uniform but u = 0.
FLT_MIN_NORMAL = 2.0 ** -126


def prob_close(gpu, ref, rtol=WINDOW):
    """Acceptance probabilities min(1, q(d)/p(d)): |gpu - ref| <= rtol * |ref|
    elementwise (relative, as the method statement fixes), NaN where ref is
    NaN; an absolute FLT_MIN_NORMAL is allowed on top only for references
    below FLT_MIN_NORMAL (exact zeros must come back as zeros)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    nan = np.isnan(ref)
    if not np.array_equal(nan, np.isnan(gpu)):
        return False
    g, r = gpu[~nan], ref[~nan]
    floor = np.where(np.abs(r) < FLT_MIN_NORMAL, FLT_MIN_NORMAL, 0.0)
    return bool(np.all(np.abs(g - r) <= rtol * np.abs(r) + floor))


def max_prob_rel(gpu, ref):
    """Largest relative error of acceptance probabilities with a normal
    float32 reference (for the assertion message)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    m = ~np.isnan(ref) & (np.abs(ref) >= FLT_MIN_NORMAL)
    if not m.any():
        return 0.0
    return float(np.max(np.abs(gpu[m] - ref[m]) / np.abs(ref[m])))


def run_tree_oracle(wl, seed=None):
    from oracle import tree as ot
    z, y = wl.raw()
    return ot.verify_tree(z, y, wl.parents.numpy(), wl.tokens.numpy(), wl.temperature.numpy(),
                          wl.seed if seed is None else seed, wl.dtype, wl.mode)


def compare_tree(res, tokens, path, accept, kv, temperature, label=""):
    """Tree outputs against an oracle TreeResult, with the same rules as
    ``compare``: greedy and error requests exact; a sampled request may
    differ only where the oracle's decision at the depth where the two walks
    part had its uniform within WINDOW of its threshold (any child test at
    that depth when the paths part there, else the drawn token's level)."""
    tokens = np.asarray(tokens).reshape(res.tokens.shape)
    path = np.asarray(path).reshape(res.path.shape)
    accept = np.asarray(accept).reshape(-1)
    kv = np.asarray(kv).reshape(-1)
    temperature = np.asarray(temperature).reshape(-1)
    logged = []
    for b in range(res.tokens.shape[0]):
        same = (np.array_equal(tokens[b], res.tokens[b]) and np.array_equal(path[b], res.path[b])
                and accept[b] == res.accept_len[b] and kv[b] == res.kv_len[b])
        if same:
            continue
        where = f"{label} request {b}: gpu a={accept[b]} path={path[b].tolist()} tok={tokens[b].tolist()} " \
                f"oracle a={res.accept_len[b]} path={res.path[b].tolist()} tok={res.tokens[b].tolist()}"
        assert res.request_errors[b] == 0, "error request differs: " + where
        assert float(temperature[b]) != 0.0, "greedy request differs: " + where
        assert kv[b] == accept[b] + 1, where
        a_g, a_o = int(accept[b]), int(res.accept_len[b])
        common = 0
        while common < min(a_g, a_o) and path[b, common] == res.path[b, common]:
            common += 1
        decs = res.decisions[b]
        depth = common + 1
        if common < a_g or common < a_o:
            cand = [x for x in decs if x.kind == "accept" and x.j == depth]
            assert cand, "no oracle decision at the divergence: " + where
            dist = min(x.distance() for x in cand)
            kind = "accept"
        else:
            cand = [x for x in decs if x.kind in ("residual", "bonus") and x.j == depth]
            assert cand, "no oracle decision at the divergence: " + where
            t_gpu, t_ref = int(tokens[b, a_g]), int(res.tokens[b, a_o])
            level = next(lv for lv, sh in enumerate(LEVEL_SHIFTS) if (t_gpu >> sh) != (t_ref >> sh))
            accept_cands = [x for x in decs if x.kind == "accept" and x.j == depth]
            dist = min([cand[0].distance(level)] + [x.distance() for x in accept_cands])
            kind = cand[0].kind
        assert dist < WINDOW, f"mismatch outside the 1e-5 window (distance {dist:.3g}): " + where
        logged.append((label, b, kind, depth, dist))
        print("near-threshold mismatch:", where, f"distance={dist:.3g}")
    return logged
