"""Pins for the oracle's error feedback (THC section 5), CPU only.

The page sends x = grad + e (the previous error added to the current
gradient) and afterwards updates e to account for the quantization error,
e = x - x_hat.  Fixed by: e = 0 sends the gradient itself; a lossless round
(x_hat = x) leaves no error; and the telescoping identity of error feedback
-- over T rounds the values sent add up to the gradients plus the first error
minus the last, sum_t x_hat_t = sum_t grad_t + e_0 - e_T -- which holds exactly
on integer-valued inputs (every fp32 operation exact) and within rounding on
random ones.
"""
import numpy as np

import oracle


def test_zero_error_sends_the_gradient():
    g = np.random.default_rng([171, 0]).standard_normal(1000).astype(np.float32)
    np.testing.assert_array_equal(oracle.ef_apply(g, np.zeros_like(g)), g)


def test_lossless_round_leaves_no_error():
    x = np.random.default_rng([171, 1]).standard_normal(1000).astype(np.float32)
    assert not np.any(oracle.ef_update(x, x))


def _rounds(T, n, rng, integer):
    e = np.zeros(n, np.float32)
    e0 = e.copy()
    sent = np.zeros(n, np.float64)
    grads = np.zeros(n, np.float64)
    for _ in range(T):
        if integer:
            g = rng.integers(-50, 51, n).astype(np.float32)
        else:
            g = rng.standard_normal(n).astype(np.float32)
        x = oracle.ef_apply(g, e)
        # a quantizer: round to a coarse grid (any lossy map will do)
        q = (np.round(x / 8.0) * 8.0).astype(np.float32)
        e = oracle.ef_update(x, q)
        sent += q
        grads += g
    return sent, grads, e0, e


def test_telescoping_exact_on_integers():
    sent, grads, e0, eT = _rounds(20, 4096, np.random.default_rng([171, 2]), integer=True)
    np.testing.assert_array_equal(sent, grads + e0 - eT)
    assert np.all(np.abs(eT) <= 4.0)  # the carried error stays within half a grid step


def test_telescoping_within_rounding():
    sent, grads, e0, eT = _rounds(20, 4096, np.random.default_rng([171, 3]), integer=False)
    # each round adds at most two fp32 roundings of values below ~16 in magnitude
    assert np.max(np.abs(sent - (grads + e0 - eT))) <= 20 * 2 * 16 * 2.0 ** -24
