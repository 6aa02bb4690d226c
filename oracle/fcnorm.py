"""CPU oracle of the drafter's input fusion with FC normalisation (test
infrastructure only).

Source: the EAGLE-3 / EAGLE 3.1 page ("FC normalisation: the key change of
EAGLE 3.1"): EAGLE-3 concatenates three target hidden states (early, middle,
late layer) and projects them with one FC layer to the draft head's input
width, fused = FC([h_early; h_mid; h_late]); EAGLE 3.1 normalises each of
the three before the FC, fused = FC([LayerNorm(h_early); LayerNorm(h_mid);
LayerNorm(h_late)]), because the late layers' vectors are larger (residual
accumulation) and would otherwise dominate the projection.  The news page on
EAGLE 3.1 ("EAGLE 3.1 changed something small and low-level") speaks of
RMSNorm on each target hidden state instead.

Readings of points the pages leave open:

* norm: NONE (EAGLE-3), LAYER (LayerNorm: subtract the mean, divide by
  sqrt(population variance + eps), scale by gamma, add beta) or RMS
  (divide by sqrt(mean square + eps), scale by gamma); each of the three
  segments has its own gamma (and beta); eps is an input.
* FC: out = concat . W^T + bias with W [d_out, 3 d] and an optional bias.
* Float64 throughout; inputs are read as the stored bf16 / fp32 values.
"""

import numpy as np

NONE = 0
LAYER = 1
RMS = 2


def normalise(h, kind, gamma=None, beta=None, eps=1e-5):
    """One segment [T, d] -> normalised [T, d] (float64)."""
    h = np.asarray(h, dtype=np.float64)
    if kind == NONE:
        return h.copy()
    if kind == LAYER:
        mu = h.mean(axis=1, keepdims=True)
        var = ((h - mu) ** 2).mean(axis=1, keepdims=True)
        x = (h - mu) / np.sqrt(var + eps)
        x = x * np.asarray(gamma, dtype=np.float64)[None, :]
        if beta is not None:
            x = x + np.asarray(beta, dtype=np.float64)[None, :]
        return x
    if kind == RMS:
        ms = (h ** 2).mean(axis=1, keepdims=True)
        return h / np.sqrt(ms + eps) * np.asarray(gamma, dtype=np.float64)[None, :]
    raise ValueError(f"unknown norm {kind}")


def fused_input(h_early, h_mid, h_late, kind, gamma=None, beta=None, eps=1e-5):
    """The concatenation [norm(h_early); norm(h_mid); norm(h_late)] [T, 3 d]."""
    segs = []
    for s, h in enumerate((h_early, h_mid, h_late)):
        g = None if gamma is None else np.asarray(gamma)[s]
        b = None if beta is None else np.asarray(beta)[s]
        segs.append(normalise(h, kind, g, b, eps))
    return np.concatenate(segs, axis=1)


def fc_norm(h_early, h_mid, h_late, weight, kind, gamma=None, beta=None, bias=None, eps=1e-5):
    """fused = FC([norm(h_early); norm(h_mid); norm(h_late)]): [T, d_out]."""
    x = fused_input(h_early, h_mid, h_late, kind, gamma, beta, eps)
    y = x @ np.asarray(weight, dtype=np.float64).T
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float64)[None, :]
    return y


def abs_bound(h_early, h_mid, h_late, weight, kind, gamma=None, beta=None, eps=1e-5):
    """sum_k |x_k| |w_k| per output: the scale of the rounding error of a
    product whose inputs are rounded (for tolerances)."""
    x = np.abs(fused_input(h_early, h_mid, h_late, kind, gamma, beta, eps))
    return x @ np.abs(np.asarray(weight, dtype=np.float64)).T
