"""dspark_schedule_static: the scheduler entry point for callers that cannot
allocate device memory (an engine that owns every byte of the device, with no
allocator reachable from its decode step). It keeps its scratch in a fixed
array inside the library instead of a caller workspace; its results must equal
those of dspark_schedule bit for bit, call after call.

Named to be collected last, so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads as W

pytestmark = pytest.mark.gpu


def _inputs(cfg, dev):
    h = W.host_inputs(cfg)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    return t(h["conf"]), t(h["conf_lag"]), t(h["sps"]), cfg.mode


def _outputs(R, dev):
    return (torch.full((R,), -7, dtype=torch.int32, device=dev),
            torch.full((1,), -7, dtype=torch.int32, device=dev),
            torch.full((2,), -7.0, dtype=torch.float64, device=dev))


def _with_workspace(cfg, dev):
    from speculative_decoding_draft_seq_gb300 import dspark
    conf, lag, sps, mode = _inputs(cfg, dev)
    L, K, tt = _outputs(cfg.R, dev)
    ws = dspark.new_workspace(cfg.R, cfg.gamma, 1, 1, dspark.FP32, sps.numel(), dev)
    dspark.schedule(conf, lag, sps, mode, L, K, tt, ws)
    assert dspark.device_status(ws) == dspark.OK
    return L.cpu().numpy(), K.cpu().numpy(), tt.cpu().numpy()


def _static(cfg, dev, conf_override=None):
    from speculative_decoding_draft_seq_gb300 import dspark
    conf, lag, sps, mode = _inputs(cfg, dev)
    if conf_override is not None:
        conf = conf_override
    L, K, tt = _outputs(cfg.R, dev)
    st = torch.full((1,), 99, dtype=torch.int32, device=dev)
    rc = dspark.schedule_static(conf, lag, sps, mode, L, K, tt, device_status=st)
    assert rc == dspark.OK, dspark.status_string(rc)
    torch.cuda.synchronize()
    return L.cpu().numpy(), K.cpu().numpy(), tt.cpu().numpy(), int(st.item())


CASES = [W.CONFIGS["stress"],                       # R * gamma = 16384, the scratch maximum, LAGGED (radix form)
         W.CONFIGS["ds"],                           # CAUSAL
         W.with_(W.CONFIGS["ds"], mode=W.LAGGED),   # LAGGED on the small form: its lagged Theta by position
                                                    # shares bytes with the radix form's keys
         W.with_(W.CONFIGS["mixed"], mode=W.ALL),   # ALL
         W.CONFIGS["mixed"]]                        # CAUSAL again, after a smaller problem


def test_static_scheduler_matches_workspace_scheduler_call_after_call():
    dev = torch.device("cuda")
    for repeat in range(2):               # two calls in a row for each problem
        for cfg in CASES:
            ref = _with_workspace(cfg, dev)
            got = _static(cfg, dev)
            assert got[3] == 0, f"device status {got[3]}"
            np.testing.assert_array_equal(got[0], ref[0])
            np.testing.assert_array_equal(got[1], ref[1])
            np.testing.assert_array_equal(got[2], ref[2])   # tau, Theta: exact float64


def test_static_scheduler_reports_device_status_per_call():
    from speculative_decoding_draft_seq_gb300 import dspark
    dev = torch.device("cuda")
    cfg = W.CONFIGS["ds"]
    conf, _, _, _ = _inputs(cfg, dev)
    bad = conf.clone()
    bad[5, 3] = float("nan")
    assert _static(cfg, dev, conf_override=bad)[3] == dspark.ERR_NONFINITE
    assert _static(cfg, dev)[3] == dspark.OK        # the next call starts clean


def test_static_scheduler_rejects_sizes_beyond_its_scratch():
    from speculative_decoding_draft_seq_gb300 import dspark
    dev = torch.device("cuda")
    cfg = W.with_(W.CONFIGS["stress"], R=1025, mode=W.CAUSAL)
    conf, _, sps, _ = _inputs(cfg, dev)
    L, K, tt = _outputs(cfg.R, dev)
    rc = dspark.schedule_static(conf, None, sps, W.CAUSAL, L, K, tt)
    assert rc == dspark.ERR_TOO_LARGE
    torch.cuda.synchronize()
    assert int(K.item()) == -7    # nothing was launched
