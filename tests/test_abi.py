"""CPU checks of the C-ABI library: it builds for sm_103a, loads, exports every
function include/moe.h declares, and rejects bad arguments on the host before
touching a GPU. No compute call is made here."""
import ctypes
import os
import re

import pytest

import quantized_moe_expert_sort_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_symbol():
    L = moe.lib()
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n


def test_status_strings():
    L = moe.lib()
    for s in range(7):
        assert L.moe_status_string(s).decode()
    assert L.moe_status_string(99).decode() == "unknown status"


def test_host_side_argument_checks():
    L = moe.lib()
    # NULL context / out-pointer
    assert L.moe_create(None, 256, 128, 8, 2, 16, 0) == 1
    assert L.moe_forward(None, None, None, None, 1, None, None, None, None, 1, 4.0, 25.0, 0, None, None) == 1
    assert L.moe_sort(None, None, 1, 8, None, None) == 1
    assert L.moe_get_workspace(None, None) == 1
    assert L.moe_destroy(None) == 0
    # bad sizes are rejected before any CUDA call
    h = ctypes.c_void_p()
    assert L.moe_create(ctypes.byref(h), 200, 128, 8, 2, 16, 0) == 2     # hidden % 128
    assert L.moe_create(ctypes.byref(h), 256, 128, 0, 2, 16, 0) == 1     # no experts
    assert L.moe_create(ctypes.byref(h), 256, 128, 5000, 2, 16, 0) == 2  # too many experts
    assert L.moe_quantize_mxfp4(None, 4, 33, None, None, None) == 1
    assert L.moe_quantize_activations(None, 4, 48, 1, None, None, None) == 1
    assert L.moe_quantize_activations(None, 4, 64, 9, None, None, None) == 2
    assert "multiple" in L.moe_last_error_message().decode() or L.moe_last_error_message()


def test_no_gpu_means_a_clean_error():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    st = moe.lib().moe_create(ctypes.byref(h), 256, 128, 8, 2, 16, 0)
    assert st in (1, 3)  # device out of range / CUDA error, never a crash
    with pytest.raises(moe.MoEError):
        moe.MoE(256, 128, 8, 2, 16)


def test_fault_injection_hook_on_the_host():
    L = moe.lib()
    assert L.moe_debug_inject(99, 0) == 1           # unknown injection
    assert L.moe_debug_inject(moe.INJECT_ALLOC_FAIL, 3) == 0
    assert L.moe_debug_inject(moe.INJECT_ALLOC_FAIL, -1) == 0  # disarm
    assert L.moe_selftest_wait(None, 1000, 0, None) == 1      # NULL context
