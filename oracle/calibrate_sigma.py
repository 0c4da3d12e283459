"""Choose the target-noise scale of the DeepSeek-scale synthetic workload.

The pages report accepted lengths per round of 5.1-5.6 on math/code and
3.1-3.6 on chat at a 7-token window with the scheduler off and temperature 1
([JD] the section on fixed-length verification; [GN] §"Resultados
principais"). The synthetic target logits are base + N(0, sigma^2); this
script bisects sigma so that the mean accepted length (accepted draft tokens
+ 1) reaches a target at gamma = 7, using only the oracle: 5.0 for the
DeepSeek-scale workload, 5.5 and 3.3 for the structured and chat halves of the
mixed-domain workload.

The per-request expectation given the drafted tokens is used instead of one
sampled outcome (Rao-Blackwellised: E[tau | x] = 1 + sum_k prod_{i<=k}
min(1, p_i / q_i)), which removes the accept/reject noise.

Usage: python -m oracle.calibrate_sigma [target_tau] [n_requests]  (prints sigma)
"""
import sys

import numpy as np

import workloads as W
from oracle.draft import decode, draft_request
from oracle.verify import verify_request


def mean_tau(sigma, n_req, gamma=7):
    cfg = W.with_(W.CONFIGS["ds"], gamma=gamma, target_sd=(sigma,), mode=W.ALL)
    base, tgt = W.logits_rows_np(cfg, range(n_req))
    W1, W2 = W.weights_np(cfg)
    W1f, W2f = decode(W1).astype(np.float64), decode(W2).astype(np.float64)
    anchors = W.anchors(cfg)
    taus = []
    for i in range(n_req):
        b, t = decode(base[i]), decode(tgt[i])
        d = draft_request(b, int(anchors[i]), W1f, W2f, cfg.T, 0, i)
        v = verify_request(t, b, int(anchors[i]), W1f, W2f, d["tokens"], gamma, cfg.T, 0, i)
        acc = np.minimum(1.0, v["p"] / v["q"])
        taus.append(1.0 + np.sum(np.cumprod(acc)))
    return float(np.mean(taus))


def main():
    target = float(sys.argv[1]) if len(sys.argv) > 1 else 5.0
    n_req = int(sys.argv[2]) if len(sys.argv) > 2 else 32
    lo, hi = 0.05, 2.0
    for _ in range(9):
        mid = 0.5 * (lo + hi)
        tau = mean_tau(mid, n_req)
        print(f"sigma={mid:.4f} tau={tau:.3f}", flush=True)
        if tau > target:
            lo = mid
        else:
            hi = mid
    print(f"SIGMA {0.5 * (lo + hi):.3f}")


if __name__ == "__main__":
    main()
