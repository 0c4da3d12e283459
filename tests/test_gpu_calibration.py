"""GPU parity of Sequential Temperature Scaling against the oracle: the device
picks, position by position, a grid temperature that is optimal for the
oracle's own ECE curve (ties within 1e-12 may go either way), its ECE curve
matches the oracle's, and the calibrated confidences match."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import calibration as C

pytestmark = pytest.mark.gpu

GRID = np.exp(np.linspace(np.log(0.25), np.log(4.0), 64)).astype(np.float32)


def _synthetic(seed, N, gamma, scale):
    rng = np.random.default_rng(seed)
    z = rng.normal(1.0, 1.5, size=(N, gamma))
    c = (1.0 / (1.0 + np.exp(-z))).astype(np.float32)
    p_true = 1.0 / (1.0 + np.exp(-z * scale))
    passed = rng.uniform(size=(N, gamma)) < p_true
    A = np.where(passed.all(axis=1), gamma, np.argmin(passed, axis=1)).astype(np.int32)
    return c, A


@pytest.mark.parametrize("N,gamma,scale,n_bins", [(50000, 5, 0.5, 15), (20000, 16, 1.3, 10), (777, 3, 2.0, 64)])
def test_sts_fit_matches_oracle(N, gamma, scale, n_bins):
    from speculative_decoding_draft_seq_gb300 import dspark
    c, A = _synthetic(N + gamma, N, gamma, scale)
    T_ref, curves = C.sts_fit(c, A, GRID.astype(np.float64), n_bins)
    dev = torch.device("cuda")
    T = torch.zeros(gamma, dtype=torch.float32, device=dev)
    ece = torch.zeros((gamma, GRID.size), dtype=torch.float32, device=dev)
    st = dspark.sts_fit(torch.from_numpy(c).to(dev), torch.from_numpy(A).to(dev), torch.from_numpy(GRID).to(dev),
                        n_bins, T, ece)
    assert st == dspark.OK
    T = T.cpu().numpy()
    ece = ece.cpu().numpy()
    # the same choices as the oracle (a different choice only between equal ECE values)
    a = np.ones(N)
    for j in range(gamma):
        y = A >= j + 1
        ref_curve = np.array([C.ece(a * C.calibrate(c[:, j], g), y, n_bins) for g in GRID.astype(np.float64)])
        ti = int(np.where(GRID == T[j])[0][0])
        assert ref_curve[ti] <= ref_curve.min() + 1e-12, (j, T[j], T_ref[j])
        np.testing.assert_allclose(ece[j], ref_curve, rtol=1e-5, atol=1e-7)
        a = a * C.calibrate(c[:, j], float(T[j]))


def test_sts_apply_matches_oracle():
    from speculative_decoding_draft_seq_gb300 import dspark
    rng = np.random.default_rng(3)
    R, gamma = 128, 16
    c = rng.uniform(0.0, 1.0, size=(R, gamma)).astype(np.float32)
    c[0, 0], c[1, 1] = 0.0, 1.0  # clipped ends
    T = np.exp(rng.uniform(np.log(0.3), np.log(3.0), size=gamma)).astype(np.float32)
    dev = torch.device("cuda")
    out = torch.empty((R, gamma), dtype=torch.float32, device=dev)
    dspark.sts_apply(torch.from_numpy(c).to(dev), torch.from_numpy(T).to(dev), out)
    ref = C.sts_apply(c, T.astype(np.float64)).astype(np.float32)
    np.testing.assert_allclose(out.cpu().numpy(), ref, rtol=2e-7, atol=0)
