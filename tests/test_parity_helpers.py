"""The parity bound itself: a whole-call normwise error can hide a few wrong tokens, the
per-token bound the GPU tests also apply cannot."""
import numpy as np

from ref import normwise_err, out_err, token_err


def test_one_wrong_token_among_many_is_caught():
    rng = np.random.default_rng(0)
    ref = rng.standard_normal((64, 256))
    got = ref.copy()
    got[17] *= 1.05                      # one token 5 % off, the other 63 exact
    assert normwise_err(got, ref) < 1e-2  # the whole-call error stays under 1e-2 ...
    assert token_err(got, ref) > 4e-2     # ... the per-token error does not
    assert out_err(got, ref) == token_err(got, ref)


def test_token_err_exact_and_scale_free():
    rng = np.random.default_rng(1)
    ref = rng.standard_normal((8, 32))
    assert token_err(ref, ref) == 0.0
    got = ref * (1 + 1e-3)
    assert abs(token_err(got, ref) - 1e-3) < 1e-12
    assert abs(token_err(1e6 * got, 1e6 * ref) - 1e-3) < 1e-12
    assert token_err(np.zeros((0, 4)), np.zeros((0, 4))) == 0.0
