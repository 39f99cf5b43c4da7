"""Host-side checks of the C ABI: the library loads, exports every function
include/h2o.h declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

from kv_cache_eviction_03_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^H2O_API\s+[\w\s\*]+?\b(h2o_\w+)\s*\(", text, flags=re.M)
    return names


def test_header_declares_the_abi():
    names = declared_functions()
    for required in ("h2o_cache_create", "h2o_prefill", "h2o_decode_step", "h2o_cache_destroy"):
        assert required in names
    assert set(names) == set(B.SIGNATURES), "binding and header disagree"


def test_library_exports_every_declared_symbol():
    lib = B.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name


@pytest.mark.parametrize("args", [
    (0, 4, 64, 4, 4, 0),       # batch
    (1, 0, 64, 4, 4, 0),       # heads
    (1, 4, 96, 4, 4, 0),       # head_dim
    (1, 4, 64, -1, 4, 0),      # heavy
    (1, 4, 64, 4, 0, 0),       # recent
    (1, 4, 64, 4, 4, 7),       # dtype
    (1, 4, 64, 60000, 6000, 0),  # slots
    (300, 300, 64, 4, 4, 0),   # pairs
])
def test_create_rejects_bad_arguments(args):
    lib = B.lib()
    out = ctypes.c_void_p(1234)
    assert lib.h2o_cache_create(*args, ctypes.byref(out)) == -1
    assert out.value is None
    assert lib.h2o_last_error().decode().startswith("h2o_cache_create")


def test_null_cache_is_rejected_everywhere():
    lib = B.lib()
    assert lib.h2o_prefill(None, None, None, None, 4, 1.0, None, None) == -1
    assert lib.h2o_prefill_ex(None, None, None, None, 4, 1.0, None, None, None, None) == -1
    assert lib.h2o_decode_step(None, None, None, None, 1.0, None, None, None) == -1
    assert lib.h2o_cache_reset(None, None) == -1
    assert lib.h2o_cache_export_state(None, None, 0, None) == -1
    assert lib.h2o_cache_import_state(None, None, 0, None) == -1
    assert lib.h2o_cache_check(None, None) == -1
    assert lib.h2o_cache_set_decode_shape(None, 2, 0) == -1
    assert lib.h2o_cache_info(None, None) == -1
    assert lib.h2o_cache_set_position_rolling(None, 10000.0) == -1
    assert lib.h2o_cache_set_rolling_digits(None, 4, 4) == -1
    assert lib.h2o_cache_rolling_digits(None, None) == -1
    assert lib.h2o_cache_state_bytes(None) == 0
    lib.h2o_cache_destroy(None)  # NULL-safe
    with pytest.raises(B.H2OError) as ei:
        B._check(lib.h2o_cache_reset(None, None))
    assert ei.value.code == -1 and "NULL" in str(ei.value)


def test_state_layout_arithmetic():
    lay = B.state_layout(2, 3, 64, 5, 4, B.H2O_F16)
    P, C = 6, 9
    assert lay["K"] == (64, P * C * 64 * 2)
    assert lay["total"] == 64 + 2 * P * C * 64 * 2 + P * C * 8 + P * 4 * 4 + P * 16


def test_selftest_rejects_bad_poll_counts():
    lib = B.lib()
    gave_up = (ctypes.c_int * 2)()
    ns = ctypes.c_ulonglong(0)
    for polls in (0, 1_000_001):
        assert lib.h2o_selftest_wait_timeout(polls, gave_up, ctypes.byref(ns)) == -1
        assert lib.h2o_last_error().decode().startswith("h2o_selftest_wait_timeout")
    assert lib.h2o_selftest_wait_timeout(10, None, ctypes.byref(ns)) == -1



def test_static_pattern_and_alloc_hook_reject_bad_arguments():
    lib = B.lib()
    assert lib.h2o_cache_set_static_pattern(None, 0, 1, 0) == -1
    assert lib.h2o_last_error().decode().startswith("h2o_cache_set_static_pattern")
    assert lib.h2o_debug_fail_alloc(-2) == -1
    assert lib.h2o_debug_fail_alloc(-1) == 0  # disarm: always accepted


def test_alloc_hook_fails_the_chosen_allocation_on_the_host():
    """Host-side fault injection: with the hook armed at 0 the very next
    device allocation fails.  Without a GPU, create fails first on the
    missing device, so this runs the hook path only where a device exists;
    the hook itself is a host counter and is disarmed after the test."""
    lib = B.lib()
    out = ctypes.c_void_p(1234)
    try:
        assert lib.h2o_debug_fail_alloc(0) == 0
        code = lib.h2o_cache_create(1, 2, 64, 4, 4, 0, ctypes.byref(out))
        assert code in (-2, -3)  # ENOMEM from the hook, or ECUDA without a device
        assert out.value is None
    finally:
        lib.h2o_debug_fail_alloc(-1)
