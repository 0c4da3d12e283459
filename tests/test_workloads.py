"""The seeded input generators: deterministic, identical on the numpy and torch
paths, and shaped as the workloads describe (host-side, no GPU)."""
import numpy as np
import pytest

import workloads as W


def test_numpy_and_torch_cpu_generators_are_bit_identical():
    torch = pytest.importorskip("torch")
    cfg = W.with_(W.CONFIGS["small"], R=3)
    b, t = W.logits_rows_np(cfg, range(3))
    bd, td = W.logits_device(cfg, "cpu")
    assert np.array_equal(bd.view(torch.int16).numpy().view(np.uint16), b)
    assert np.array_equal(td.view(torch.int16).numpy().view(np.uint16), t)
    w1, w2 = W.weights_np(cfg)
    w1d, w2d = W.weights_device(cfg, "cpu")
    assert np.array_equal(w1d.view(torch.int16).numpy().view(np.uint16), w1)
    assert np.array_equal(w2d.view(torch.int16).numpy().view(np.uint16), w2)


def test_rows_of_a_request_do_not_depend_on_which_requests_are_generated():
    cfg = W.with_(W.CONFIGS["small"], R=6)
    b_all, t_all = W.logits_rows_np(cfg, range(6))
    b4, t4 = W.logits_rows_np(cfg, [4])
    assert np.array_equal(b_all[4], b4[0]) and np.array_equal(t_all[4], t4[0])


def test_shapes_and_value_distributions():
    cfg = W.CONFIGS["tiny"]
    b, t = W.logits_rows_np(cfg, range(cfg.R))
    assert b.shape == (4, 4, 64) and t.shape == (4, 5, 64) and b.dtype == np.float32
    assert abs(b.std() - 1.5) < 0.15
    assert abs((t[:, :4] - b).std() - 0.5) < 0.06
    c = W.confidences(cfg)
    assert c.shape == (4, 4) and c.min() >= 0.5 and c.max() <= 1.0
    s = W.sps_table(cfg)
    assert s.shape == (16,) and s[0] == 1.0 and s[-1] == np.float32(1 - 15 / 32)


def test_stress_table_is_step_shaped_with_dip():
    cfg = W.CONFIGS["stress"]
    s = W.sps_table(cfg)
    assert s.shape == (16384,)
    assert s[0] == s[63] and s[64] < s[63]          # plateaus of 64 tokens
    assert s[8192] < 0.85 * s[8191]                  # dip past 8192


def test_norm_table_is_symmetric_gaussian_quantiles():
    q = W.norm_table()
    assert q.shape == (65536,)
    np.testing.assert_array_equal(q[:32768], -q[::-1][:32768])
    assert abs(float(np.std(q.astype(np.float64))) - 1.0) < 2e-3


def test_host_built_inputs_equal_the_device_generator():
    """device_inputs_from_host (numpy + one copy per tensor, used by smoke())
    gives the same tensors as the torch generator, here both on the CPU."""
    torch = pytest.importorskip("torch")
    for cfg in (W.with_(W.CONFIGS["small"], R=3, V=640, rank=64, gated=True), W.CONFIGS["tiny"]):
        a = W.device_inputs(cfg, "cpu")
        b = W.device_inputs_from_host(cfg, "cpu")
        assert a.keys() == b.keys()
        for k, v in a.items():
            if isinstance(v, torch.Tensor):
                assert v.dtype == b[k].dtype and v.shape == b[k].shape, k
                assert torch.equal(v.view(torch.int16) if v.dtype == torch.bfloat16 else v,
                                   b[k].view(torch.int16) if v.dtype == torch.bfloat16 else b[k]), k
            else:
                assert v == b[k], k
