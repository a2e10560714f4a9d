"""The oracle pins catch plausible mistakes: each case plants one mistake in
the oracle (on the CPU, through monkeypatch) and checks that at least one pin
of tests/test_oracle_pins.py then fails."""
import numpy as np
import pytest

import oracle.linear_logp as OL
import test_oracle_pins as pins

PINS = [
    pins.test_single_class_vocab,
    pins.test_two_class_softplus,
    pins.test_uniform_logits_give_minus_log_v,
    pins.test_probability_bounds,
    pins.test_bruteforce_logsumexp_without_shift,
    lambda: pins.test_finite_differences(0),
    pins.test_finite_differences_logits,
    pins.test_gradient_rows_sum_to_zero,
    pins.test_invalid_targets_give_zero_rows,
    pins.test_zero_upstream_gives_positive_zeros,
    pins.test_empty_input,
    pins.test_masked_tail_logits,
    pins.test_temperature_two_class_softplus,
    pins.test_temperature_limits,
    lambda: pins.test_temperature_finite_differences(0.7),
]


def _some_pin_fails():
    for pin in PINS:
        try:
            pin()
        except Exception:  # an assertion, or a shape / index error
            return True
    return False


def test_unmodified_oracle_passes_every_pin():
    assert not _some_pin_fails()


_orig_logits = OL.linear_logits
_orig_grad = OL.grad_logits
_orig_lse = OL.logsumexp_rows
_orig_logp = OL.logp_from_logits


def _drop_bias(h, W, b=None):
    return h @ W.T


def _bias_twice(h, W, b=None):
    z = _orig_logits(h, W, b)
    return z if b is None else z + b[None, :]


def _grad_sign(z, y, gl, lse=None):
    return -_orig_grad(z, y, gl, lse)


def _grad_no_onehot(z, y, gl, lse=None):
    N, V = z.shape
    lse = _orig_lse(z) if lse is None else lse
    g = -np.asarray(gl, np.float64)[:, None] * np.exp(z - lse[:, None])
    return g + 0.0


def _grad_p_unnormalised(z, y, gl, lse=None):
    # softmax without subtracting lse (exp(z) instead of exp(z - lse))
    return _orig_grad(z, y, gl, np.zeros(z.shape[0]))


def _lse_max_only(z):
    return z.max(axis=1)


def _lse_no_log(z):
    M = z.max(axis=1)
    return M + np.exp(z - M[:, None]).sum(axis=1)


def _logp_off_by_one(z, y):
    y1 = np.minimum(np.asarray(y) + 1, z.shape[1] - 1)
    return _orig_logp(z, y1)


def _logp_sign(z, y):
    logp, lse = _orig_logp(z, y)
    return -logp, lse


def _logits_transposed_weight(h, W, b=None):
    # uses W's leading columns as if it were [D, V] (a transposed operand)
    D = h.shape[1]
    Wt = W.reshape(-1)[: D * W.shape[0]].reshape(W.shape[0], D)[::-1]
    z = h @ Wt.T
    return z if b is None else z + b[None, :]


_orig_tempered = OL._tempered
_orig_tgrad = OL._tempered_grad


def _temper_multiplies(z, temperature):
    _orig_tempered(z, temperature)  # keeps the argument check
    return z * temperature


def _tgrad_no_inverse(zT, y, gl, temperature, lse=None):
    return _orig_grad(zT, y, gl, lse)  # the 1 / T factor dropped


def _tgrad_squared(zT, y, gl, temperature, lse=None):
    return _orig_grad(zT, y, gl, lse) / temperature ** 2 + 0.0


MUTATIONS = {
    "temperature_multiplies": ("_tempered", _temper_multiplies),
    "temperature_grad_no_inverse": ("_tempered_grad", _tgrad_no_inverse),
    "temperature_grad_squared": ("_tempered_grad", _tgrad_squared),
    "drop_bias": ("linear_logits", _drop_bias),
    "bias_twice": ("linear_logits", _bias_twice),
    "transposed_weight": ("linear_logits", _logits_transposed_weight),
    "grad_sign": ("grad_logits", _grad_sign),
    "grad_without_onehot": ("grad_logits", _grad_no_onehot),
    "softmax_unnormalised": ("grad_logits", _grad_p_unnormalised),
    "lse_max_only": ("logsumexp_rows", _lse_max_only),
    "lse_missing_log": ("logsumexp_rows", _lse_no_log),
    "target_off_by_one": ("logp_from_logits", _logp_off_by_one),
    "logp_sign": ("logp_from_logits", _logp_sign),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(monkeypatch, name):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(OL, attr, fn)
    assert _some_pin_fails(), f"no pin caught the planted mistake {name!r}"
