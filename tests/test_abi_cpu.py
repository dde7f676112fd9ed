"""Host-side checks of the C ABI that need no GPU: the library builds, loads and
exports every entry point include/moe_ep.h declares; argument errors are found
on the host before any CUDA call."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("no CUDA toolkit")
    from combine_layout_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def _declared():
    text = open(os.path.join(ROOT, "include", "moe_ep.h")).read()
    return sorted(set(re.findall(r"^\s*MOE_EP_API\s+(?:int|const char\*)\s+(moe_ep_\w+)\s*\(",
                                 text, re.M)))


def test_header_declares_the_path():
    names = _declared()
    for n in ("moe_ep_create_group", "moe_ep_route", "moe_ep_dispatch", "moe_ep_combine",
              "moe_ep_get_num_recv_tokens"):
        assert n in names
    # every declaration carries a comment citing its passage or stating its contract
    text = open(os.path.join(ROOT, "include", "moe_ep.h")).read()
    assert "核心功能函数" in text and "高吞吐模式" in text and "低延迟模式" in text


def test_library_exports_every_declared_symbol(lib):
    for n in _declared():
        assert hasattr(lib, n), n


def test_binding_names_match_header(lib):
    import combine_layout_gb300.moe_ep as ep
    assert ep.declared_symbols() == _declared()
    for n in _declared():
        if n != "moe_ep_status_string":
            assert callable(getattr(ep, n)), n


def test_host_argument_checks_without_gpu(lib):
    f = lib.moe_ep_create_group
    f.argtypes = [ctypes.POINTER(ctypes.c_void_p)] + [ctypes.c_int] * 5
    out = ctypes.c_void_p()
    INVALID = 1
    assert f(None, 1, 256, 64, 4096, 7168) == INVALID
    assert f(ctypes.byref(out), 7, 256, 64, 4096, 7168) == INVALID      # bad mode
    assert f(ctypes.byref(out), 1, 250, 64, 4096, 7168) == INVALID      # E % R
    assert f(ctypes.byref(out), 1, 1024, 64, 4096, 7168) == INVALID     # E too large
    assert f(ctypes.byref(out), 1, 256, 64, 0, 7168) == INVALID         # no tokens
    assert f(ctypes.byref(out), 1, 256, 64, 4096, 7164) == INVALID      # H % 8
    assert out.value is None
    for name in ("moe_ep_destroy_group", "moe_ep_destroy_handle", "moe_ep_clear_device_errors"):
        g = getattr(lib, name)
        g.argtypes = [ctypes.c_void_p]
        assert g(None) == INVALID
    for name in ("moe_ep_set_row_align", "moe_ep_set_x_before_route"):
        g = getattr(lib, name)
        g.argtypes = [ctypes.c_void_p, ctypes.c_int]
        assert g(None, 1) == INVALID
    # the signal primitives and the staged calls reject a null group / handle
    # on the host, before any CUDA call
    sa = lib.moe_ep_signal_add
    sa.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_void_p]
    assert sa(None, None, 1, None) == INVALID
    ws = lib.moe_ep_wait_signal
    ws.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_int64, ctypes.c_void_p]
    assert ws(None, None, 1, 1000, None) == INVALID
    cp = lib.moe_ep_complete
    cp.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    assert cp(None, None) == INVALID
    s = lib.moe_ep_status_string
    s.restype = ctypes.c_char_p
    assert s(0) == b"ok" and s(2).startswith(b"more tokens")
    assert b"bounded wait" in s(5) and s(6) == b"unknown status"
