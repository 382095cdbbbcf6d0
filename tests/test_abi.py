"""The C-ABI library builds, loads and exports what include/pa.h declares.

Host-only: argument checks that return before any CUDA call are exercised;
nothing here launches a kernel.
"""
import ctypes
import os
import re

import pytest

import paged_kv_cache_186_gb300 as pa
from paged_kv_cache_186_gb300 import build as pabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


@pytest.fixture(scope="module")
def L():
    pabuild.build()
    return pa.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(pa.EXPORTED)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_abi_version_and_status_strings(L):
    assert L.pa_abi_version() == 1
    for code in range(8):
        assert L.pa_status_string(code)
    assert L.pa_status_string(99) == b"unknown status"


def test_wait_timeout_hook_checks_its_bound(L):
    # host-only: arming and disarming touch no device
    assert L.pa_debug_inject_wait_timeout(0, 0) == 2            # PA_ERR_SHAPE
    assert L.pa_debug_inject_wait_timeout(0, 3_000_000_000) == 2
    assert L.pa_debug_inject_wait_timeout(-1, 0) == 0           # disarmed


def _cache(**kw):
    c = dict(num_blocks=8, block_size=16, num_kv_heads=2, head_dim=64, dtype=pa.PA_KV_BF16,
             k_cache=0x1000, v_cache=0x2000, k_scale=None, v_scale=None)
    c.update(kw)
    return pa.KVCache(**c)


@pytest.mark.parametrize("kw, want", [
    (dict(k_cache=None), 1),
    (dict(num_blocks=0), 2),
    (dict(dtype=7), 3),
    (dict(dtype=pa.PA_KV_FP8_E4M3, head_dim=128), 3),        # FP8 without scales
    (dict(k_scale=0x3000, v_scale=0x4000), 3),                  # scales on a bf16 cache
    (dict(block_size=8), 4),
    (dict(head_dim=96), 4),
    (dict(dtype=pa.PA_KV_FP8_E4M3, head_dim=64, k_scale=0x3000, v_scale=0x4000), 4),
    (dict(k_cache=0x1004), 7),
])
def test_cache_descriptor_is_validated_before_launch(L, kw, want):
    c = _cache(**kw)
    rc = L.pa_store_kv(ctypes.c_void_p(0x10), ctypes.c_void_p(0x20), None, None,
                       ctypes.c_void_p(0x30), 4, ctypes.byref(c), None)
    assert rc == want
    rc = L.pa_decode(ctypes.c_void_p(0x10), ctypes.byref(c), ctypes.c_void_p(0x20), 4,
                     ctypes.c_void_p(0x30), 0, 2, 4, 0.125, ctypes.c_void_p(0x40), None, 0, None)
    assert rc == want


def test_decode_argument_checks(L):
    c = _cache()
    P = ctypes.c_void_p
    call = lambda q=P(0x10), bt=P(0x20), mb=4, cl=P(0x30), B=2, H=4, scale=0.125, out=P(0x40): \
        L.pa_decode(q, ctypes.byref(c), bt, mb, cl, 0, B, H, scale, out, None, 0, None)
    assert call(B=0) == 0            # empty batch: nothing to do, no launch
    assert call(B=-1) == 2
    assert call(H=3) == 2            # not a multiple of num_kv_heads
    assert call(H=18) == 4           # 9 query heads per kv head
    assert call(mb=0) == 2
    assert call(q=None) == 1
    assert call(bt=None) == 1
    assert call(cl=None) == 1
    assert call(out=None) == 1
    assert call(scale=float("nan")) == 2
    assert call(q=P(0x18)) == 7      # misaligned q


def test_store_kv_argument_checks(L):
    c = _cache()
    P = ctypes.c_void_p
    assert L.pa_store_kv(P(0x10), P(0x20), None, None, P(0x30), 0, ctypes.byref(c), None) == 0
    assert L.pa_store_kv(P(0x10), P(0x20), None, None, P(0x30), -1, ctypes.byref(c), None) == 2
    assert L.pa_store_kv(None, P(0x20), None, None, P(0x30), 3, ctypes.byref(c), None) == 1
    assert L.pa_store_kv(P(0x10), P(0x20), None, None, None, 3, ctypes.byref(c), None) == 1
    # scales given for a bf16 cache
    assert L.pa_store_kv(P(0x10), P(0x20), ctypes.cast(P(0x40), ctypes.POINTER(ctypes.c_float)),
                         None, P(0x30), 3, ctypes.byref(c), None) == 3
    assert L.pa_store_kv(P(0x18), P(0x20), None, None, P(0x30), 3, ctypes.byref(c), None) == 7


def test_workspace_size_is_zero_for_invalid_arguments(L):
    c = _cache(num_blocks=0)
    assert L.pa_decode_workspace_size(ctypes.byref(c), 4, 8, 4, 0) == 0
    c = _cache()
    assert L.pa_decode_workspace_size(ctypes.byref(c), 0, 8, 4, 0) == 0


def test_binding_refuses_to_run_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(pa, "_lib", None)
    monkeypatch.setattr(pa, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        pa.lib()
