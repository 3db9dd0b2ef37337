"""CPU checks of the C ABI boundary: liblmoe.so loads without a GPU and exports every
function include/lmoe.h declares; status strings are defined; nothing is computed."""
import ctypes

import pytest

import nvfp4_latentmoe_fwd_02_b300 as lm


def test_library_exports_every_declared_function():
    lib = lm.lib()
    names = lm.header_functions()
    assert len(names) >= 15
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings():
    for st in range(7):
        s = lm.lmoe_status_string(st)
        assert isinstance(s, str) and s
    assert lm.lmoe_status_string(lm.LMOE_ETIMEOUT) != lm.lmoe_status_string(lm.LMOE_OK)


def test_null_context_calls_fail_without_touching_a_device():
    lib = lm.lib()
    assert lib.lmoe_workspace_size(None, 8) == 0
    assert lib.lmoe_forward_kernel_count(None, 8) == 0
    assert lib.lmoe_set_debug(None, 1) == lm.LMOE_EINVAL
    assert lib.lmoe_check(None, None) == lm.LMOE_EINVAL
    out = ctypes.c_void_p()
    assert lib.lmoe_create(256, 64, 16, 4, 128, None, None, ctypes.byref(out)) == lm.LMOE_EINVAL
    assert lib.lmoe_quantize_nvfp4(None, 0, 4, 24, -1.0, None, None, None, None) == lm.LMOE_EINVAL
    lib.lmoe_destroy(None)
