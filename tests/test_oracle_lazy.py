"""Pins of the lazy reading (CPU only): on valid inputs it is the eager
oracle exactly; a bad row is an error only if the walk reaches it."""

import numpy as np

from oracle import verify as ov
from speculative_decoding_verification_73_gb300 import workloads


def test_lazy_equals_eager_on_valid_rows():
    for gs, dt, v in ((21, "f32", 800), (22, "bf16", 3000)):
        wl = workloads.make_random(12, 5, v, dt, gen_seed=gs, verify_seed=gs)
        z, y = wl.raw()
        for seed in (0, 5, 2 ** 40 + 1):
            e = ov.verify(z, y, wl.tokens.numpy(), wl.temperature.numpy(), seed, dt)
            l = ov.verify(z, y, wl.tokens.numpy(), wl.temperature.numpy(), seed, dt, lazy=True)
            np.testing.assert_array_equal(e.tokens, l.tokens)
            np.testing.assert_array_equal(e.accept_len, l.accept_len)
            np.testing.assert_array_equal(e.kv_len, l.kv_len)
            assert e.errors == l.errors == 0


def test_bad_rows_past_the_stop_are_not_read():
    # greedy, N = 3: request 0 matches at position 1, mismatches at 2 -> reads
    # target rows 0 and 1 only; a NaN in row 3 is an error only eagerly.
    vocab = 5
    z = np.zeros((2, 4, vocab), dtype=np.float32)
    for j, g in enumerate((1, 2, 3, 4)):
        z[:, j, g] = 1.0
    drafts = np.array([[1, 0, 3], [1, 2, 3]], dtype=np.int32)
    z[:, 3, 0] = np.nan
    t = np.zeros(2, np.float32)
    eager = ov.verify(z, None, drafts, t, 0, "f32")
    lazy = ov.verify(z, None, drafts, t, 0, "f32", lazy=True)
    assert eager.request_errors.tolist() == [ov.ERR_LOGIT, ov.ERR_LOGIT]
    # request 0 stops at position 2 (rows 0, 1 read); request 1 matches all
    # three and needs row 3 for the bonus -> error
    assert lazy.request_errors.tolist() == [0, ov.ERR_LOGIT]
    assert lazy.tokens[0].tolist() == [1, 2, -1, -1] and lazy.accept_len[0] == 1
