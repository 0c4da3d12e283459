"""The C-ABI library builds for sm_103a, loads, and exports every entry point
that include/dspark.h declares (no compute calls: this runs without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dspark.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(dspark_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_draft_seq_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("dspark_draft_sequential", "dspark_schedule", "dspark_verify", "dspark_round",
              "dspark_acceptance_labels", "dspark_workspace_bytes", "dspark_device_status",
              "dspark_status_string", "dspark_draft_sequential_gated", "dspark_verify_gated",
              "dspark_round_gated"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} not exported"


def test_host_only_calls(lib):
    lib.dspark_workspace_bytes.restype = ctypes.c_size_t
    n = lib.dspark_workspace_bytes(128, 16, 129280, 256, 1, 2176)
    assert n > 0 and n % 256 == 0
    assert lib.dspark_workspace_bytes(0, 16, 100, 8, 1, 10) == 0
    lib.dspark_status_string.restype = ctypes.c_char_p
    assert lib.dspark_status_string(0) == b"ok"
    # argument errors are returned before anything touches the GPU
    lib.dspark_schedule.restype = ctypes.c_int32
    assert lib.dspark_schedule(0, 4, None, None, None, 0, 0, None, None, None, None, 0, None) == 1
    lib.dspark_acceptance_labels.restype = ctypes.c_int32
    assert lib.dspark_acceptance_labels(0, 4, 100, 64, 1, *([None] * 7), ctypes.c_float(1.0), None, None,
                                        ctypes.c_size_t(0), None) == 1
    # the gated entry points refuse a missing gate table on the host
    f = ctypes.c_float(1.0)
    lib.dspark_draft_sequential_gated.restype = ctypes.c_int32
    assert lib.dspark_draft_sequential_gated(4, 4, 128, 64, 1, *([None] * 5), f, ctypes.c_uint64(0),
                                             None, None, None, None, ctypes.c_size_t(0), None) == 1
    lib.dspark_verify_gated.restype = ctypes.c_int32
    assert lib.dspark_verify_gated(4, 4, 128, 64, 1, *([None] * 10), f, ctypes.c_uint64(0),
                                   None, None, None, None, ctypes.c_size_t(0), None) == 1
    lib.dspark_round_gated.restype = ctypes.c_int32
    assert lib.dspark_round_gated(4, 4, 128, 64, 1, *([None] * 9), ctypes.c_int32(0), ctypes.c_int32(0), f,
                                  ctypes.c_uint64(0), *([None] * 10), ctypes.c_size_t(0), None) == 1


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "dspark_copy", os.path.join(ROOT, "speculative_decoding_draft_seq_gb300", "dspark.py"))
    mod = importlib.util.module_from_spec(spec)
    monkeypatch.setattr(os.path, "exists", lambda p: False if p.endswith("libdspark.so") else os.path.isfile(p))
    with pytest.raises(ImportError):
        spec.loader.exec_module(mod)


def test_binding_refuses_tensors_the_abi_cannot_describe():
    """The C ABI takes dense arrays without strides: the binding refuses views
    that are not contiguous, tensors on the wrong side of the host/device split
    and, where an entry point fixes it, the wrong element type."""
    torch = pytest.importorskip("torch")
    from speculative_decoding_draft_seq_gb300 import dspark
    assert dspark._ptr(None) is None
    x = torch.zeros((4, 6), dtype=torch.int32)
    assert dspark._ptr(x, torch.int32, host=True).value == x.data_ptr()
    with pytest.raises(ValueError, match="contiguous"):
        dspark._ptr(x.t(), host=True)
    with pytest.raises(ValueError, match="CUDA"):
        dspark._ptr(x)  # device arguments must be CUDA tensors
    with pytest.raises(TypeError):
        dspark._ptr(x.float(), torch.int32, host=True)
