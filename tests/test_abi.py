"""The C ABI without a GPU: liboscar.so builds, loads, exports every symbol that
include/oscar.h declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

from bit_kv_cache_oscar_gb300 import binding as ob
from bit_kv_cache_oscar_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_symbols():
    text = open(os.path.join(ROOT, "include", "oscar.h")).read()
    return sorted(set(re.findall(r"OSCAR_API\s+[\w\s\*]*?\b(oscar_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ctypes.CDLL(build.LIB)


def test_every_declared_symbol_is_exported(lib):
    syms = header_symbols()
    assert len(syms) >= 13
    for s in syms:
        assert hasattr(lib, s), s


def test_binding_covers_the_header():
    assert sorted(ob.EXPORTS) == header_symbols()


def test_sizes_and_split_suggestion(lib):
    L = ob.Layout(8, 4, 64)
    assert ob.oscar_partials_ml_floats(L, 2, 7) == 2 * 32 * 8
    assert ob.oscar_partials_acc_floats(L, 2, 7) == 2 * 32 * 8 * 128
    s = ob.oscar_suggest_splits(L, 1, 99680, 152)
    assert 1 <= s <= 1024
    assert ob.oscar_suggest_splits(L, 1, 100, 152) >= 1
    # the documented rule: A resident clusters, W = 2 window clusters at batch 1 and 1 above it;
    # one wave while batch * (1 + W) <= A, else about four waves
    A = s + 2
    for b in (2, 4, 8, 16, 20, 32, 64):
        want = A // b - 1 if 2 * b <= A else 4 * A // b - 1
        assert ob.oscar_suggest_splits(L, b, 99680, 152) == max(1, want), b
    assert ob.oscar_version() == "0.1.0"


@pytest.mark.parametrize("field,value,msg", [
    ("head_dim", 64, "head_dim"), ("gqa", 3, "gqa"), ("page_size", 48, "page_size"),
    ("group", 16, "group"), ("sink", 40, "sink"), ("n_kv_heads", 0, "n_kv_heads"),
])
def test_layout_validation_on_host(lib, field, value, msg):
    lay = ob.LayoutC(128, 8, 4, 64, 128, 64, 256)
    setattr(lay, field, value)
    L = ob.lib()
    rc = L.oscar_quantize_rotated(ctypes.byref(lay), None, 1, 0.96, None, None, None, None)
    assert rc in (1, 2)
    assert msg in L.oscar_last_error_string().decode()


def test_codebook_validation_on_host(lib):
    """A non-uniform codebook must be four finite, strictly increasing levels per tensor."""
    L = ob.lib()
    for bad in ((0.5, 0.4, 2.0, 3.0), (0.0, 1.0, float("nan"), 3.0), (1.0, 1.0, 2.0, 3.0)):
        lay = ob.LayoutC(128, 8, 4, 64, 128, 64, 256)
        lay.levels_k = (ctypes.c_float * 4)(*bad)
        lay.levels_v = (ctypes.c_float * 4)(0.5, 1.2, 1.8, 2.5)
        rc = L.oscar_quantize_rotated(ctypes.byref(lay), None, 1, 0.96, None, None, None, None)
        assert rc in (1, 2)
        assert "codebook" in L.oscar_last_error_string().decode()


def test_null_and_range_checks_on_host(lib):
    L = ob.lib()
    lay = ob.LayoutC(128, 8, 4, 64, 128, 64, 256)
    assert L.oscar_quantize_rotated(ctypes.byref(lay), None, 1, 0.96, None, None, None, None) == 1
    assert L.oscar_quantize_rotated(None, None, 1, 0.96, None, None, None, None) == 1
    part = ob.PartialsC(None, None, None, 0)
    assert L.oscar_merge(ctypes.byref(lay), ctypes.byref(part), None, 1, None, None, None, None) == 1
    assert "partials" in L.oscar_last_error_string().decode()
    # zero-sized work is a no-op that needs no device
    assert L.oscar_quantize_rotated(ctypes.byref(lay), None, 0, 0.96, None, None, None, None) == 0
