"""Host-side checks of the C ABI that need no GPU.

The library must load, export every entry point include/armt.h declares, and
reject bad arguments with a status code before touching a device.
"""
import ctypes
import dataclasses
import os
import re

import pytest

from recurrent_memory_transformer_gb300 import armt as B
from recurrent_memory_transformer_gb300 import build as build_mod
from recurrent_memory_transformer_gb300 import inputs as I

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "armt.h")).read()
    return sorted(set(re.findall(r"ARMT_API\s+[\w\s\*]+?\b(armt_\w+)\s*\(", src)))


def test_header_declares_expected_entry_points():
    names = declared_functions()
    for n in ("armt_create", "armt_forward", "armt_forward_sequential", "armt_destroy",
              "armt_status_string", "armt_forward_host", "armt_grouped_gemm_bf16"):
        assert n in names
    assert set(names) == set(B.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(8):
        s = lib.armt_status_string(code)
        assert s and s != b"unknown status"
    assert lib.armt_status_string(99) == b"unknown status"


def _weights_struct(cfg):
    import numpy as np
    w = B.armt_weights()
    keep = [np.zeros(4, np.float32)]
    for k in B._WKEYS:
        setattr(w, k, keep[0].ctypes.data)
    w.on_device = 0
    return w, keep


def test_create_rejects_null_and_bad_configs_before_any_device_work(lib):
    h = ctypes.c_void_p()
    assert lib.armt_create(None, None, None, ctypes.byref(h)) == 1  # ARMT_ERR_ARG
    cases = [
        (dict(n_layers=0), 1),
        (dict(n_kv_heads=3), 2),                        # Hq % Hkv
        (dict(ffn_dim=100), 2),                         # F % 128
        (dict(head_dim=48), 3),                         # unsupported head_dim
        (dict(n_mem=40), 3),                            # n_mem > 32
        (dict(dpfp_nu=40), 2),                          # nu >= 2k
    ]
    for over, want in cases:
        cfg = dataclasses.replace(I.TINY, **over)
        c = B.make_config(cfg)
        w, keep = _weights_struct(cfg)
        st = lib.armt_create(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(h))
        assert st == want, (over, st, lib.armt_last_error())
        assert lib.armt_last_error()
    # bf16 models need tensor-core-friendly widths
    cfg = dataclasses.replace(I.TINY, dtype="bf16", head_dim=64, n_q_heads=1, n_kv_heads=1)
    c = B.make_config(cfg)
    w, keep = _weights_struct(cfg)
    assert lib.armt_create(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(h)) == 2
    # a NULL weight pointer
    c = B.make_config(I.TINY)
    w, keep = _weights_struct(I.TINY)
    w.wq = None
    assert lib.armt_create(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(h)) == 1


def test_forward_and_gemm_reject_null_arguments(lib):
    assert lib.armt_forward(None, None, 1, None, None, None, 0, None) == 1
    assert lib.armt_forward_sequential(None, None, 1, None, None, None, 0, None) == 1
    assert lib.armt_forward_host(None, None, 1, None, None, None, 0, 0, None) == 1
    assert lib.armt_forward_batch(None, None, 1, 1, None, None, None, 0, 0, None) == 1
    assert lib.armt_grouped_gemm_bf16(None, None, None, 1, 1, 256, 64, None) == 1
    i64 = ctypes.c_int64()
    assert lib.armt_launch_count(None, 1, 0, ctypes.byref(i64)) == 1
    assert lib.armt_state_sizes(None, ctypes.byref(i64), ctypes.byref(i64)) == 1
    assert lib.armt_memory_bytes(None, ctypes.byref(i64), None, None) == 1
    assert lib.armt_destroy(None) == 0


def test_valid_config_reports_missing_device_without_gpu(lib):
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except ImportError:
        pass
    c = B.make_config(I.TINY)
    w, keep = _weights_struct(I.TINY)
    h = ctypes.c_void_p()
    assert lib.armt_create(ctypes.byref(c), ctypes.byref(w), None, ctypes.byref(h)) == 7


def test_binding_argument_counts_match_the_header(lib):
    # every entry point the header declares takes as many arguments as the
    # ctypes binding passes (a mismatch would only surface on a GPU)
    src = open(os.path.join(ROOT, "include", "armt.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    for m in re.finditer(r"ARMT_API\s+[\w\s\*]+?\b(armt_\w+)\s*\(([^)]*)\)", src):
        name, params = m.group(1), m.group(2).strip()
        n = 0 if params in ("", "void") else len(params.split(","))
        argtypes = getattr(lib, name).argtypes
        if argtypes is None:
            assert n == 0, name
        else:
            assert len(argtypes) == n, (name, len(argtypes), n)
