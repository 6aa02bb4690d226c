"""Pins of the FC-norm oracle (CPU only): normalisations worked by hand and
by their invariants, and the FC reduced to special weights."""

import numpy as np
import pytest

from oracle import fcnorm as ofc


def test_layernorm_by_hand():
    h = np.array([[1.0, 2.0, 3.0, 6.0]])            # mean 3, population var 3.5
    x = ofc.normalise(h, ofc.LAYER, gamma=np.ones(4), beta=np.zeros(4), eps=0.0)
    np.testing.assert_allclose(x, (h - 3.0) / np.sqrt(3.5), rtol=1e-15)
    x2 = ofc.normalise(h, ofc.LAYER, gamma=np.full(4, 2.0), beta=np.full(4, 0.5), eps=0.0)
    np.testing.assert_allclose(x2, 2.0 * (h - 3.0) / np.sqrt(3.5) + 0.5, rtol=1e-15)


def test_rmsnorm_by_hand():
    h = np.array([[3.0, -4.0]])                      # mean square 12.5
    x = ofc.normalise(h, ofc.RMS, gamma=np.array([1.0, 2.0]), eps=0.0)
    np.testing.assert_allclose(x, [[3.0 / np.sqrt(12.5), -8.0 / np.sqrt(12.5)]], rtol=1e-15)


def test_invariants():
    rng = np.random.default_rng(3)
    h = rng.normal(size=(5, 16)) * 7.0 + 2.0
    g, b = rng.normal(size=16), rng.normal(size=16)
    ln = ofc.normalise(h, ofc.LAYER, g, b, eps=0.0)
    # a positive scale and a shift of the whole row leave LayerNorm unchanged
    np.testing.assert_allclose(ofc.normalise(3.0 * h + 5.0, ofc.LAYER, g, b, eps=0.0), ln, rtol=1e-12)
    # without gamma/beta every row has mean 0 and variance 1
    raw = ofc.normalise(h, ofc.LAYER, np.ones(16), np.zeros(16), eps=0.0)
    np.testing.assert_allclose(raw.mean(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose((raw ** 2).mean(axis=1), 1.0, rtol=1e-12)
    # RMSNorm: invariant to a positive scale; equals LayerNorm on zero-mean rows with beta 0
    rms = ofc.normalise(h, ofc.RMS, g, eps=0.0)
    np.testing.assert_allclose(ofc.normalise(0.25 * h, ofc.RMS, g, eps=0.0), rms, rtol=1e-12)
    hz = h - h.mean(axis=1, keepdims=True)
    np.testing.assert_allclose(ofc.normalise(hz, ofc.RMS, g, eps=0.0),
                               ofc.normalise(hz, ofc.LAYER, g, np.zeros(16), eps=0.0), rtol=1e-12)


@pytest.mark.parametrize("kind", [ofc.NONE, ofc.LAYER, ofc.RMS])
def test_fc_with_selector_weights_returns_a_segment(kind):
    rng = np.random.default_rng(4)
    T, d = 6, 8
    hs = [rng.normal(size=(T, d)) * (1 + 3 * s) for s in range(3)]
    gamma, beta = rng.normal(size=(3, d)), rng.normal(size=(3, d))
    for s in range(3):
        w = np.zeros((d, 3 * d))
        w[:, s * d:(s + 1) * d] = np.eye(d)
        y = ofc.fc_norm(*hs, w, kind, gamma, beta if kind == ofc.LAYER else None, eps=1e-5)
        want = ofc.normalise(hs[s], kind, gamma[s], beta[s] if kind == ofc.LAYER else None, eps=1e-5)
        np.testing.assert_allclose(y, want, rtol=1e-14, atol=1e-14)


def test_bias_and_linearity():
    rng = np.random.default_rng(5)
    T, d, do = 4, 8, 5
    hs = [rng.normal(size=(T, d)) for _ in range(3)]
    g = rng.normal(size=(3, d))
    w1, w2 = rng.normal(size=(do, 3 * d)), rng.normal(size=(do, 3 * d))
    bias = rng.normal(size=do)
    y1 = ofc.fc_norm(*hs, w1, ofc.RMS, g)
    y2 = ofc.fc_norm(*hs, w2, ofc.RMS, g)
    np.testing.assert_allclose(ofc.fc_norm(*hs, w1 + w2, ofc.RMS, g, bias=bias), y1 + y2 + bias,
                               rtol=1e-12, atol=1e-12)
    # the error-scale bound dominates |y| (triangle inequality)
    assert (ofc.abs_bound(*hs, w1, ofc.RMS, g) >= np.abs(y1) - 1e-12).all()
