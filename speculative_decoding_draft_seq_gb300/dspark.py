"""Python binding of the DSpark C-ABI library (libdspark.so).

Argument marshalling only: every step of the round runs in the library's CUDA
kernels. Tensors are torch CUDA tensors (device memory and streams are
PyTorch's); the binding passes their data pointers and the current stream's
handle to the C entry points declared in include/dspark.h. If the library is
missing the import fails: there is no fallback implementation.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdspark.so")

OK, ERR_INVALID_ARG, ERR_NONFINITE, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_RANGE, ERR_TOO_LARGE = range(8)
FP32, BF16 = 0, 1
CAUSAL, LAGGED, ALL = 0, 1, 2


class DSparkError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    i32, u64, f32, vp, sz = ctypes.c_int32, ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
    lib.dspark_workspace_bytes.restype = sz
    lib.dspark_workspace_bytes.argtypes = [i32] * 6
    lib.dspark_workspace_init.restype = i32
    lib.dspark_workspace_init.argtypes = [vp, sz, vp]
    lib.dspark_draft_sequential.restype = i32
    lib.dspark_draft_sequential.argtypes = [i32] * 5 + [vp] * 4 + [f32, u64] + [vp] * 3 + [vp, sz, vp]
    lib.dspark_schedule.restype = i32
    lib.dspark_schedule.argtypes = [i32, i32, vp, vp, vp, i32, i32, vp, vp, vp, vp, sz, vp]
    lib.dspark_schedule_static.restype = i32
    lib.dspark_schedule_static.argtypes = [i32, i32, vp, vp, vp, i32, i32, vp, vp, vp, vp, vp]
    lib.dspark_verify.restype = i32
    lib.dspark_verify.argtypes = [i32] * 5 + [vp] * 9 + [f32, u64] + [vp] * 3 + [vp, sz, vp]
    lib.dspark_round.restype = i32
    lib.dspark_round.argtypes = ([i32] * 5 + [vp] * 5 + [vp, vp, vp, i32, i32, f32, u64] +
                                 [vp] * 9 + [vp, sz, vp])
    lib.dspark_draft_sequential_gated.restype = i32
    lib.dspark_draft_sequential_gated.argtypes = [i32] * 5 + [vp] * 5 + [f32, u64] + [vp] * 3 + [vp, sz, vp]
    lib.dspark_verify_gated.restype = i32
    lib.dspark_verify_gated.argtypes = [i32] * 5 + [vp] * 10 + [f32, u64] + [vp] * 3 + [vp, sz, vp]
    lib.dspark_round_gated.restype = i32
    lib.dspark_round_gated.argtypes = ([i32] * 5 + [vp] * 6 + [vp, vp, vp, i32, i32, f32, u64] +
                                       [vp] * 9 + [vp, sz, vp])
    lib.dspark_lm_head.restype = i32
    lib.dspark_lm_head.argtypes = [i32, i32, i32, vp, vp, vp, vp, sz, vp]
    lib.dspark_copy_scheduled_rows.restype = i32
    lib.dspark_copy_scheduled_rows.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp]
    lib.dspark_wait_selftest.restype = i32
    lib.dspark_wait_selftest.argtypes = [i32, vp, sz, vp]
    lib.dspark_acceptance_labels.restype = i32
    lib.dspark_acceptance_labels.argtypes = [i32] * 5 + [vp] * 7 + [f32, vp, vp, sz, vp]
    lib.dspark_sts_scratch_bytes.restype = sz
    lib.dspark_sts_scratch_bytes.argtypes = [i32] * 4
    lib.dspark_sts_fit.restype = i32
    lib.dspark_sts_fit.argtypes = [i32, i32, vp, vp, i32, vp, i32, vp, vp, vp, sz, vp]
    lib.dspark_sts_status.restype = i32
    lib.dspark_sts_status.argtypes = [vp, vp]
    lib.dspark_sts_apply.restype = i32
    lib.dspark_sts_apply.argtypes = [i32, i32, vp, vp, vp, vp]
    lib.dspark_device_status.restype = i32
    lib.dspark_device_status.argtypes = [vp, vp]
    lib.dspark_status_string.restype = ctypes.c_char_p
    lib.dspark_status_string.argtypes = [i32]
    lib.dspark_last_launch_count.restype = i32
    lib.dspark_last_launch_count.argtypes = []
    return lib


lib = _load()


def status_string(status):
    return lib.dspark_status_string(int(status)).decode()


def last_launch_count():
    return int(lib.dspark_last_launch_count())


_I32, _F32, _F64, _U8 = torch.int32, torch.float32, torch.float64, torch.uint8


def _ptr(t, dtype=None, host=False):
    """Data pointer of a dense tensor for the C ABI, which takes row-major arrays without strides:
    a non-contiguous view, a tensor on the wrong side of the host/device split or (where the entry
    point fixes it) the wrong element type is refused here rather than read or written wrongly."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous (the C ABI takes dense row-major arrays)")
    if t.is_cuda == host:
        raise ValueError("expected a host tensor" if host else "expected a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return FP32
    raise TypeError(f"logits/weights must be bfloat16 or float32, got {t.dtype}")


def _check(status, where):
    if status != OK:
        raise DSparkError(status, where)


def workspace_bytes(R, gamma, V, rank, dtype, n_table):
    return int(lib.dspark_workspace_bytes(R, gamma, V, rank, dtype, n_table))


def new_workspace(R, gamma, V, rank, dtype, n_table, device="cuda", stream=None):
    """Allocates (with PyTorch) and clears a workspace for these sizes."""
    n = workspace_bytes(R, gamma, V, rank, dtype, n_table)
    ws = torch.empty(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + n]
    _check(lib.dspark_workspace_init(_ptr(ws, _U8), n, _stream(stream)), "dspark_workspace_init")
    return ws


def draft_sequential(base, anchor, W1, W2, temperature, seed, tokens, q_tok, q_stats, ws, stream=None):
    R, gamma, V = base.shape
    rank = W1.shape[1]
    _check(lib.dspark_draft_sequential(R, gamma, V, rank, _dtype_code(base), _ptr(base), _ptr(anchor, _I32),
                                       _ptr(W1), _ptr(W2), float(temperature), int(seed), _ptr(tokens, _I32),
                                       _ptr(q_tok, _F32), _ptr(q_stats, _F32), _ptr(ws, _U8), ws.numel(),
                                       _stream(stream)), "dspark_draft_sequential")


def draft_sequential_gated(base, anchor, W1, gate, W2, temperature, seed, tokens, q_tok, q_stats, ws,
                           stream=None):
    """Drafting with the recurrent (gated) head; `gate` [V, rank] like W1."""
    R, gamma, V = base.shape
    rank = W1.shape[1]
    _check(lib.dspark_draft_sequential_gated(R, gamma, V, rank, _dtype_code(base), _ptr(base), _ptr(anchor, _I32),
                                             _ptr(W1), _ptr(gate), _ptr(W2), float(temperature), int(seed),
                                             _ptr(tokens, _I32), _ptr(q_tok, _F32), _ptr(q_stats, _F32),
                                             _ptr(ws, _U8), ws.numel(), _stream(stream)),
           "dspark_draft_sequential_gated")


def lm_head(hidden, lm_head_w, logits, ws, stream=None):
    """Base logits bf16(hidden . lm_head): hidden [..., d], lm_head [d, V],
    logits [..., V] (bf16 tensors; the leading dimensions are flattened)."""
    d, V = lm_head_w.shape
    M = hidden.numel() // d
    _check(lib.dspark_lm_head(M, d, V, _ptr(hidden), _ptr(lm_head_w), _ptr(logits), _ptr(ws, _U8), ws.numel(),
                              _stream(stream)), "dspark_lm_head")


def schedule(conf, conf_lagged, sps, mode, sched_len, K, tau_theta, ws, stream=None):
    R, gamma = conf.shape
    _check(lib.dspark_schedule(R, gamma, _ptr(conf, _F32), _ptr(conf_lagged, _F32), _ptr(sps, _F32), sps.numel(),
                               int(mode), _ptr(sched_len, _I32), _ptr(K, _I32), _ptr(tau_theta, _F64),
                               _ptr(ws, _U8), ws.numel(), _stream(stream)), "dspark_schedule")


def schedule_static(conf, conf_lagged, sps, mode, sched_len, K, tau_theta, device_status=None,
                    stream=None):
    """dspark_schedule_static: the scheduler without a workspace (fixed library
    scratch, R * gamma <= 16384). Returns the C status code without raising."""
    R, gamma = conf.shape
    return int(lib.dspark_schedule_static(R, gamma, _ptr(conf, _F32), _ptr(conf_lagged, _F32), _ptr(sps, _F32),
                                          sps.numel(), int(mode), _ptr(sched_len, _I32), _ptr(K, _I32),
                                          _ptr(tau_theta, _F64), _ptr(device_status), _stream(stream)))


def verify(target, base, anchor, W1, W2, tokens, q_tok, q_stats, sched_len, temperature, seed,
           out_tokens, accepted_len, p_tok, ws, stream=None):
    R, gamma, V = base.shape
    rank = W1.shape[1]
    _check(lib.dspark_verify(R, gamma, V, rank, _dtype_code(base), _ptr(target), _ptr(base), _ptr(anchor, _I32),
                             _ptr(W1), _ptr(W2), _ptr(tokens, _I32), _ptr(q_tok, _F32), _ptr(q_stats, _F32),
                             _ptr(sched_len, _I32), float(temperature), int(seed), _ptr(out_tokens, _I32),
                             _ptr(accepted_len, _I32), _ptr(p_tok, _F32), _ptr(ws, _U8), ws.numel(),
                             _stream(stream)), "dspark_verify")


def verify_gated(target, base, anchor, W1, gate, W2, tokens, q_tok, q_stats, sched_len, temperature, seed,
                 out_tokens, accepted_len, p_tok, ws, stream=None):
    R, gamma, V = base.shape
    rank = W1.shape[1]
    _check(lib.dspark_verify_gated(R, gamma, V, rank, _dtype_code(base), _ptr(target), _ptr(base),
                                   _ptr(anchor, _I32), _ptr(W1), _ptr(gate), _ptr(W2), _ptr(tokens, _I32),
                                   _ptr(q_tok, _F32), _ptr(q_stats, _F32), _ptr(sched_len, _I32),
                                   float(temperature), int(seed), _ptr(out_tokens, _I32), _ptr(accepted_len, _I32),
                                   _ptr(p_tok, _F32), _ptr(ws, _U8), ws.numel(), _stream(stream)),
           "dspark_verify_gated")


def acceptance_labels(target, base, anchor, W1, W2, tokens, q_stats, temperature, labels, ws, stream=None):
    """dspark_acceptance_labels: labels [R, gamma] float32 = 1 - TV(P_{k-1}, Q_k) per position."""
    R, gamma, V = base.shape
    rank = W1.shape[1]
    _check(lib.dspark_acceptance_labels(R, gamma, V, rank, _dtype_code(base), _ptr(target), _ptr(base),
                                        _ptr(anchor, _I32), _ptr(W1), _ptr(W2), _ptr(tokens, _I32),
                                        _ptr(q_stats, _F32), float(temperature), _ptr(labels, _F32), _ptr(ws, _U8),
                                        ws.numel(), _stream(stream)), "dspark_acceptance_labels")


def sts_fit(conf, accepted, grid, n_bins, temperature, ece=None, stream=None):
    """dspark_sts_fit with a scratch it allocates (PyTorch); returns the device status."""
    N, gamma = conf.shape
    n = int(lib.dspark_sts_scratch_bytes(N, gamma, grid.numel(), n_bins))
    if n == 0:
        raise DSparkError(ERR_INVALID_ARG, "dspark_sts_scratch_bytes")
    raw = torch.empty(n + 256, dtype=torch.uint8, device=conf.device)
    off = (-raw.data_ptr()) % 256
    scratch = raw[off:off + n]
    _check(lib.dspark_sts_fit(N, gamma, _ptr(conf, _F32), _ptr(accepted, _I32), grid.numel(), _ptr(grid, _F32),
                              n_bins, _ptr(temperature, _F32), _ptr(ece, _F32), _ptr(scratch, _U8), n,
                              _stream(stream)), "dspark_sts_fit")
    return int(lib.dspark_sts_status(_ptr(scratch, _U8), _stream(stream)))


def sts_apply(conf, temperature, conf_out, stream=None):
    R, gamma = conf.shape
    _check(lib.dspark_sts_apply(R, gamma, _ptr(conf, _F32), _ptr(temperature, _F32), _ptr(conf_out, _F32),
                                _stream(stream)), "dspark_sts_apply")


def round_(base, target, anchor, W1, W2, conf, conf_lagged, sps, mode, temperature, seed, out, ws,
           stream=None):
    """One whole round; `out` is a RoundOutputs holding the output tensors."""
    R, gamma, V = base.shape
    rank = W1.shape[1]
    _check(lib.dspark_round(R, gamma, V, rank, _dtype_code(base), _ptr(base), _ptr(target), _ptr(anchor, _I32),
                            _ptr(W1), _ptr(W2), _ptr(conf, _F32), _ptr(conf_lagged, _F32), _ptr(sps, _F32),
                            sps.numel(), int(mode), float(temperature), int(seed), _ptr(out.tokens, _I32),
                            _ptr(out.q_tok, _F32), _ptr(out.q_stats, _F32), _ptr(out.sched_len, _I32),
                            _ptr(out.K, _I32), _ptr(out.tau_theta, _F64), _ptr(out.out_tokens, _I32),
                            _ptr(out.accepted_len, _I32), _ptr(out.p_tok, _F32), _ptr(ws, _U8), ws.numel(),
                            _stream(stream)), "dspark_round")


def round_gated(base, target, anchor, W1, gate, W2, conf, conf_lagged, sps, mode, temperature, seed, out, ws,
                stream=None):
    """One whole round with the recurrent (gated) head."""
    R, gamma, V = base.shape
    rank = W1.shape[1]
    _check(lib.dspark_round_gated(R, gamma, V, rank, _dtype_code(base), _ptr(base), _ptr(target),
                                  _ptr(anchor, _I32), _ptr(W1), _ptr(gate), _ptr(W2), _ptr(conf, _F32),
                                  _ptr(conf_lagged, _F32), _ptr(sps, _F32), sps.numel(), int(mode),
                                  float(temperature), int(seed), _ptr(out.tokens, _I32), _ptr(out.q_tok, _F32),
                                  _ptr(out.q_stats, _F32), _ptr(out.sched_len, _I32), _ptr(out.K, _I32),
                                  _ptr(out.tau_theta, _F64), _ptr(out.out_tokens, _I32),
                                  _ptr(out.accepted_len, _I32), _ptr(out.p_tok, _F32), _ptr(ws, _U8), ws.numel(),
                                  _stream(stream)), "dspark_round_gated")


def copy_scheduled_rows(host_target, device_target, host_sched_len, stream=None):
    """Host-to-device copy of target rows 0..L_r of every request (host_target pinned)."""
    R, g1, V = host_target.shape
    _check(lib.dspark_copy_scheduled_rows(R, g1 - 1, V, _dtype_code(host_target),
                                          _ptr(host_target, host=True), _ptr(device_target),
                                          _ptr(host_sched_len, _I32, host=True), _stream(stream)),
           "dspark_copy_scheduled_rows")


def wait_selftest(which, ws, stream=None):
    """A bounded device wait (0: grid barrier, 1: mbarrier, 2: counter poll) on a condition nothing meets; it
    gives up and records ERR_TIMEOUT in the workspace's status word."""
    _check(lib.dspark_wait_selftest(int(which), _ptr(ws, _U8), ws.numel(), _stream(stream)), "dspark_wait_selftest")


def device_status(ws, stream=None):
    return int(lib.dspark_device_status(_ptr(ws, _U8), _stream(stream)))


class RoundOutputs:
    """Device output tensors of one round for R requests and block length gamma."""

    def __init__(self, R, gamma, device="cuda"):
        i32, f32 = torch.int32, torch.float32
        self.tokens = torch.zeros((R, gamma), dtype=i32, device=device)
        self.q_tok = torch.zeros((R, gamma), dtype=f32, device=device)
        self.q_stats = torch.zeros((R, gamma, 2), dtype=f32, device=device)
        self.sched_len = torch.zeros((R,), dtype=i32, device=device)
        self.K = torch.zeros((1,), dtype=i32, device=device)
        self.tau_theta = torch.zeros((2,), dtype=torch.float64, device=device)
        self.out_tokens = torch.zeros((R, gamma + 1), dtype=i32, device=device)
        self.accepted_len = torch.zeros((R,), dtype=i32, device=device)
        self.p_tok = torch.zeros((R, gamma), dtype=f32, device=device)

    def host(self):
        return {k: v.cpu().numpy() for k, v in vars(self).items()}
