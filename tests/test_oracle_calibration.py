"""Pins of the oracle's Sequential Temperature Scaling ([GN] "Calibração
posterior": per-position temperatures found left to right by a 1-D grid
search minimising the ECE of the cumulative survival)."""
import numpy as np
import pytest

from oracle import calibration as C

GRID = np.exp(np.linspace(np.log(0.25), np.log(4.0), 64))


def test_ece_by_hand():
    # two bins of [0, 1]: predictions 0.2, 0.4 (bin 0) and 0.6, 0.9 (bin 1), outcomes 0, 1, 1, 1
    pred = [0.2, 0.4, 0.6, 0.9]
    y = [0, 1, 1, 1]
    # bin 0: |0.6 - 1| = 0.4; bin 1: |1.5 - 2| = 0.5; total 0.9 / 4
    assert C.ece(pred, y, 2) == pytest.approx(0.225, abs=1e-15)
    # a prediction of exactly 1.0 falls in the last bin
    assert C.ece([1.0, 1.0], [1, 0], 4) == pytest.approx(0.5, abs=1e-15)
    assert C.ece([0.3] * 10, [1] * 3 + [0] * 7, 10) == pytest.approx(0.0, abs=1e-12)


def test_unit_temperature_is_identity_and_order_is_kept():
    rng = np.random.default_rng(0)
    c = rng.uniform(0.01, 0.99, size=1000)
    assert np.allclose(C.calibrate(c, 1.0), c, rtol=0, atol=1e-12)
    for T in (0.3, 2.5):
        out = C.calibrate(c, T)
        assert np.array_equal(np.argsort(c, kind="stable"), np.argsort(out, kind="stable"))


def _synthetic(seed, N, gamma, true_scale):
    """Outcomes drawn from survivals of sigmoid(logit(c) * true_scale): the raw
    confidences c have temperature 1 / true_scale relative to the truth."""
    rng = np.random.default_rng(seed)
    z = rng.normal(1.0, 1.5, size=(N, gamma))
    c = 1.0 / (1.0 + np.exp(-z))
    p_true = 1.0 / (1.0 + np.exp(-z * true_scale))
    u = rng.uniform(size=(N, gamma))
    passed = u < p_true
    A = np.where(passed.all(axis=1), gamma, np.argmin(passed, axis=1))
    return c, A


@pytest.mark.parametrize("scale,expect", [(0.5, 2.0), (2.0, 0.5), (1.0, 1.0)])
def test_fit_recovers_known_temperature(scale, expect):
    c, A = _synthetic(1, 60000, 3, scale)
    T, curves = C.sts_fit(c, A, GRID, 15)
    # the first position's temperature is identified directly; later ones within sampling noise
    assert abs(np.log(T[0] / expect)) < 0.12
    assert np.all(np.abs(np.log(T / expect)) < 0.35)
    assert curves[0].min() < 0.01


def test_fit_beats_raw_confidences():
    c, A = _synthetic(2, 40000, 4, 0.6)  # over-confident raw scores
    T, _ = C.sts_fit(c, A, GRID, 15)
    a_raw = np.cumprod(c, axis=1)
    a_cal = np.cumprod(C.sts_apply(c, T), axis=1)
    for j in range(1, 5):
        y = A >= j
        assert C.ece(a_cal[:, j - 1], y, 15) < C.ece(a_raw[:, j - 1], y, 15)
