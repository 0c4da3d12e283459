"""Confidence-scheduled verification length (hardware-aware prefix scheduler) -- oracle.

What the pages define ([GN] §"Verificação com agendamento por confiança";
[AI] "Verificar solo lo que importa"; [JD] the scheduler sections):
  * c_{r,k} in (0,1) is the probability that draft token k of request r passes
    verification given all earlier tokens were accepted; the cumulative prefix
    survival is a_{r,j} = prod_{i<=j} c_{r,i}, non-increasing in j ([GN]
    "Calibração posterior" and "Hardware-Aware Prefix Scheduler").
  * The scheduler maximises Theta = tau * SPS(B), SPS(B) being a steps-per-
    second cost table profiled once at engine start, by sorting all R x gamma
    candidates by a in descending order and admitting them greedily with an
    O(1) table lookup each; monotone a makes the result prefix-closed.
  * Early stop: admission halts at the first candidate that lowers Theta, so
    each decision depends only on the prefix processed so far (non-anticipation).
  * Production variant ([GN] §"Aplicação prática do scheduler"; [AI] the
    asynchronous-scheduler paragraph; [JD] the causal-barrier paragraph): the
    cut length K is chosen by an unconstrained (no early stop) search on the
    confidences of two steps earlier; the current candidates are ranked by
    their latest cumulative confidence and the top K are admitted.

Readings where the pages are silent (each listed in the design notes):
  * a is formed in float32, left to right: a_j = fl32(a_{j-1} * c_j), a_0 = 1.
    Confidences are clamped to [0, 1]; a non-finite confidence is an error.
  * Sort ties go to the smaller flat index r*gamma + (j-1) (keeps prefix
    closure when a product repeats).
  * tau counts the +1 corrected/bonus token of every request: before any
    admission tau = R and the batch holds B = R tokens (each request verifies
    its anchor). After i admissions B_i = R + i and
    tau_i = R + S_i * 2**-40, S_i the sum of the admitted a's each rounded to
    fixed point floor(a * 2**40 + 1/2) (exact and order-free);
    Theta_i = tau_i * SPS[B_i - 1] in float64, table entry i <-> B = i + 1.
  * B beyond the table is infeasible: it stops admission. If R exceeds the
    table, nothing is admitted (K = 0, Theta reported as 0).
  * Only a strict decrease stops admission; ties are admitted.
  * LAGGED: K = smallest argmax_i Theta_i over i = 0..min(R*gamma, n_table-R)
    on the lagged confidences; then the top K of the current order.
  * ALL: every position is verified (the offline evaluation setting, [GN]
    §"Resultados principais": scheduler off, fixed block).

Pins (tests/test_oracle_schedule.py): prefix closure and monotone a; brute
force over all prefix-closed length vectors equals the greedy choice when
Theta is unimodal; a constant table admits up to the table bound; a table
falling faster than R/(R+1) per token admits nothing; LAGGED equals CAUSAL
when the lagged confidences equal the current ones and Theta is unimodal.
"""

import math

import numpy as np

CAUSAL, LAGGED, ALL = 0, 1, 2
FIXED_SHIFT = 40


class NonFiniteInput(ValueError):
    pass


def survival(conf):
    """a_{r,j} = fl32(a_{r,j-1} * clamp(c_{r,j})), a_{r,0} = 1 (float32)."""
    c = np.asarray(conf, dtype=np.float32)
    if not np.all(np.isfinite(c)):
        raise NonFiniteInput("confidence is not finite")
    c = np.clip(c, np.float32(0.0), np.float32(1.0))
    R, gamma = c.shape
    a = np.zeros((R, gamma), dtype=np.float32)
    for r in range(R):
        acc = np.float32(1.0)
        for j in range(gamma):
            acc = np.float32(acc * c[r, j])
            a[r, j] = acc
    return a


def fixed_point(a):
    """floor(a * 2**40 + 1/2) for a float32 a in [0, 1] (exact in float64)."""
    return int(math.floor(float(a) * 2.0 ** FIXED_SHIFT + 0.5))


def descending_order(a):
    """Flat candidate indices r*gamma + (j-1), a descending, ties by index."""
    flat = np.asarray(a, dtype=np.float32).reshape(-1)
    return sorted(range(flat.size), key=lambda i: (-float(flat[i]), i))


def theta(R, S, sps_entry):
    """Theta = (R + S * 2**-40) * SPS, in this exact operation order."""
    tau = float(R) + float(S) * 2.0 ** -FIXED_SHIFT
    return tau, tau * float(sps_entry)


def _lengths(order, K, R, gamma):
    L = np.zeros(R, dtype=np.int64)
    for i in order[:K]:
        L[i // gamma] += 1
    return L


def schedule(conf, sps, mode=CAUSAL, conf_lagged=None):
    """Returns dict(L [R], K, tau, theta, a [R, gamma] float32).

    conf [R, gamma] current confidences; sps [n_table] float32 steps/s with
    entry i = SPS(B = i + 1); conf_lagged [R, gamma] for mode LAGGED.
    """
    sps = np.asarray(sps, dtype=np.float32)
    if not np.all(np.isfinite(sps)):
        raise NonFiniteInput("cost table is not finite")
    a = survival(conf)
    R, gamma = a.shape
    n = R * gamma
    n_table = sps.shape[0]
    flat = a.reshape(-1)
    f = [fixed_point(x) for x in flat]

    if mode == ALL:
        K = n
        S = sum(f)
        tau, th = theta(R, S, sps[R + K - 1]) if 0 < R + K <= n_table else (theta(R, S, 0.0)[0], 0.0)
        return dict(L=np.full(R, gamma, dtype=np.int64), K=K, tau=tau, theta=th, a=a)

    if R == 0 or R > n_table:
        return dict(L=np.zeros(R, dtype=np.int64), K=0, tau=float(R), theta=0.0, a=a)

    order = descending_order(a)

    if mode == CAUSAL:
        S, K = 0, 0
        tau, th = theta(R, 0, sps[R - 1])
        for i in range(n):
            B = R + i + 1
            if B > n_table:
                break
            S_next = S + f[order[i]]
            tau_next, th_next = theta(R, S_next, sps[B - 1])
            if th_next < th:  # the first admission that lowers Theta stops it
                break
            S, K, tau, th = S_next, K + 1, tau_next, th_next
        return dict(L=_lengths(order, K, R, gamma), K=K, tau=tau, theta=th, a=a)

    if mode == LAGGED:
        a_lag = survival(conf_lagged)
        f_lag = [fixed_point(x) for x in a_lag.reshape(-1)]
        order_lag = descending_order(a_lag)
        i_max = min(n, n_table - R)
        best_i, best_th, S = 0, None, 0
        for i in range(i_max + 1):
            if i > 0:
                S += f_lag[order_lag[i - 1]]
            _, th_i = theta(R, S, sps[R + i - 1])
            if best_th is None or th_i > best_th:  # smallest argmax
                best_i, best_th = i, th_i
        K = best_i
        S_now = sum(f[i] for i in order[:K])
        tau, th = theta(R, S_now, sps[R + K - 1])
        return dict(L=_lengths(order, K, R, gamma), K=K, tau=tau, theta=th, a=a)

    raise ValueError(f"unknown scheduler mode {mode}")
