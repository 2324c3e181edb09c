"""The C-ABI library builds, loads and exports every symbol include/sf.h
declares; host-only size queries behave (no GPU needed, no compute calls)."""

import ctypes
import os
import re

import pytest

from greedy_speculative_decoding_gb300 import _lib as L
from greedy_speculative_decoding_gb300 import build as B
from greedy_speculative_decoding_gb300.engine import model_cfg, weight_order
from synth import QWEN05B, QWEN05B_SHARED, QWEN7B, TINY_DRAFT, TINY_TARGET, weight_names

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "sf.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.load()


def _declared():
    with open(HEADER) as f:
        src = f.read()
    return sorted(set(re.findall(r"^SF_API\s+[\w\s\*]+?\b(sf_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_binding_exports():
    assert set(_declared()) == set(L.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_weight_order_matches_inputs():
    for s in (TINY_TARGET, TINY_DRAFT, QWEN7B):
        assert weight_order(s) == weight_names(s)


def test_weight_count_and_sizes(lib):
    c = model_cfg(TINY_TARGET)
    assert lib.sf_weight_count(ctypes.byref(c)) == 1 + 2 * 12 + 1
    c7 = model_cfg(QWEN7B)
    assert lib.sf_weight_count(ctypes.byref(c7)) == 1 + 28 * 12 + 1 + 1
    # KV cache: layers x 2 x batch x kv heads x slots x head_dim x 2 bytes
    assert lib.sf_kv_bytes(ctypes.byref(c7), 1, 4096) == 28 * 2 * 4 * 4096 * 128 * 2
    d = model_cfg(QWEN05B_SHARED)
    ws = lib.sf_workspace_bytes(ctypes.byref(c7), ctypes.byref(d), 1, 8, 4096)
    assert 0 < ws < 512 * 2**20
    # invalid shapes are refused (0 bytes)
    bad = model_cfg(TINY_TARGET.with_(head_dim=96))
    assert lib.sf_workspace_bytes(ctypes.byref(bad), None, 1, 4, 256) == 0
    assert lib.sf_workspace_bytes(ctypes.byref(c), None, 1, 4, 100) == 0


def test_status_strings(lib):
    for s in range(8):
        assert lib.sf_status_str(s)
    assert lib.sf_status_str(L.SF_OK) == b"ok"


def test_create_rejects_bad_arguments_without_gpu_work(lib):
    c = model_cfg(TINY_TARGET)
    h = ctypes.c_void_p()
    # null weights
    st = lib.sf_create(ctypes.byref(c), None, None, None, 1, 4, 256, None, None, None, None, ctypes.byref(h))
    assert st == L.SF_ERR_ARG and h.value is None
    # too many rows per forward
    arr = (ctypes.c_void_p * lib.sf_weight_count(ctypes.byref(c)))()
    st = lib.sf_create(ctypes.byref(c), arr, None, None, 8, 15, 256, 256, None, 256, None, ctypes.byref(h))
    assert st == L.SF_ERR_UNSUPPORTED
    assert b"exceeds" in lib.sf_last_error()
    # more sequences than the acceptance kernel's one-warp-per-sequence block holds
    st = lib.sf_create(ctypes.byref(c), arr, None, None, 33, 1, 256, 256, None, 256, None, ctypes.byref(h))
    assert st == L.SF_ERR_ARG and h.value is None
