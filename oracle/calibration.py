"""Sequential Temperature Scaling of the confidence head -- oracle.

Test infrastructure: imported only by the tests, the smoke entry point and the
benchmark's CPU legs; never by the library.

What the pages define ([GN] "Calibração posterior — Sequential Temperature
Scaling (STS)" and "O papel do confidence head"): the scheduler needs absolute
survival probabilities, the raw confidences are over-confident, each c_i is a
conditional probability so the survival of a prefix is the product of the
c_i, and on a held-out set a left-to-right 1-D grid search minimises the
expected calibration error (ECE) position by position, preserving the order
of the tokens; after STS the mean ECE falls to about 1%.

Readings where the pages are silent (each listed in the design notes):
  * One temperature per position k: c'_k = sigmoid(logit(c_k) / T_k), with c
    clipped to [1e-6, 1 - 1e-6] before the logit. This is monotone in c, so
    within a position the order of the candidates is kept.
  * The held-out set is N blocks with confidences c [N, gamma] and the number
    of leading drafted tokens that passed verification, A [N] (every position
    verified). The outcome of prefix j is y_j = [A >= j]; its prediction is
    the calibrated survival a'_j = prod_{i <= j} c'_i.
  * ECE with B equal-width bins of the prediction on [0, 1] (bin
    min(floor(a' B), B - 1)): sum over bins of |sum of a' - sum of y| / N.
  * Left to right: T_j is the first grid temperature that minimises ECE_j
    given T_1..T_{j-1}; the grid is an input (the benchmark uses 64
    log-spaced values from 1/4 to 4).

Pins (tests/test_oracle_calibration.py): ECE of hand-made sets against their
value by hand; T = 1 is the identity; order within a position is kept; data
drawn from known over-confidence (logits scaled by 2 or 1/2) is recovered
(T near 2 or 1/2); data drawn from the survivals themselves gives T near 1 and
an ECE near the sampling floor.
"""

import numpy as np

CLIP = 1e-6


def calibrate(c, T):
    """c' = sigmoid(logit(clip(c)) / T), float64, elementwise; T broadcasts."""
    c = np.clip(np.asarray(c, dtype=np.float64), CLIP, 1.0 - CLIP)
    z = np.log(c) - np.log1p(-c)
    return 1.0 / (1.0 + np.exp(-z / np.asarray(T, dtype=np.float64)))


def ece(pred, y, n_bins):
    """Expected calibration error: sum_b |sum_{i in b} pred_i - sum_{i in b} y_i| / N."""
    pred = np.asarray(pred, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    b = np.minimum((pred * n_bins).astype(np.int64), n_bins - 1)
    sp = np.bincount(b, weights=pred, minlength=n_bins)
    sy = np.bincount(b, weights=y, minlength=n_bins)
    return float(np.abs(sp - sy).sum() / pred.shape[0])


def sts_fit(conf, accepted, grid, n_bins):
    """Left-to-right grid search. Returns (T [gamma], ece_curves [gamma, len(grid)])."""
    conf = np.asarray(conf, dtype=np.float64)
    accepted = np.asarray(accepted)
    N, gamma = conf.shape
    grid = np.asarray(grid, dtype=np.float64)
    a = np.ones(N)
    T = np.zeros(gamma)
    curves = np.zeros((gamma, grid.shape[0]))
    for j in range(1, gamma + 1):
        y = (accepted >= j).astype(np.float64)
        for t, Tg in enumerate(grid):
            curves[j - 1, t] = ece(a * calibrate(conf[:, j - 1], Tg), y, n_bins)
        best = int(np.argmin(curves[j - 1]))  # first minimum
        T[j - 1] = grid[best]
        a = a * calibrate(conf[:, j - 1], T[j - 1])
    return T, curves


def sts_apply(conf, T):
    """Calibrated confidences c'[:, k] = sigmoid(logit(c[:, k]) / T_k)."""
    return calibrate(conf, np.asarray(T, dtype=np.float64)[None, :])
