"""The C-ABI library builds, loads and exports every function include/sv.h
declares; host-side argument checks answer without touching a GPU."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sv_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from draft_block_verification_gb300 import _build
    return C.CDLL(_build.build())


def test_header_declares_the_four_verify_calls():
    names = declared_functions()
    for n in ("sv_verify_greedy", "sv_verify_sample", "sv_verify_tree", "sv_packed_step",
              "sv_create", "sv_destroy", "sv_sync_status", "sv_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    lib.sv_status_string.restype = C.c_char_p
    for code in range(7):
        s = lib.sv_status_string(code)
        assert s and s != b"unknown status"
    assert lib.sv_status_string(99) == b"unknown status"


def test_null_handle_is_rejected_on_the_host(lib):
    vp = C.c_void_p
    lib.sv_verify_greedy.restype = C.c_int
    rc = lib.sv_verify_greedy(vp(0), vp(0), 1, C.c_int64(8), 1, 1, 8, vp(0), vp(0), vp(0),
                              vp(0), vp(0))
    assert rc == 1  # SV_ERR_INVALID_ARG
    lib.sv_create.restype = C.c_int
    assert lib.sv_create(vp(0)) == 1
    assert lib.sv_destroy(vp(0)) == 0


def test_binding_exports_the_c_names():
    import draft_block_verification_gb300 as dbv
    for n in ("sv_verify_greedy", "sv_verify_sample", "sv_verify_tree", "sv_packed_step"):
        assert callable(getattr(dbv, n))


def test_static_greedy_rejects_bad_arguments_on_the_host(lib):
    vp = C.c_void_p
    lib.sv_verify_greedy_static.restype = C.c_int
    # a missing status word, or a negative batch, is refused before any CUDA call
    rc = lib.sv_verify_greedy_static(vp(0), 1, C.c_int64(8), 1, 1, 8, vp(0), vp(0), vp(0),
                                     vp(0), vp(0), vp(0))
    assert rc == 1  # SV_ERR_INVALID_ARG
    rc = lib.sv_verify_greedy_static(vp(16), 1, C.c_int64(8), -1, 1, 8, vp(16), vp(0), vp(16),
                                     vp(16), vp(16), vp(0))
    assert rc == 1


def test_fault_injection_hook_answers_without_a_gpu(lib, monkeypatch):
    """SV_FAULT_INJECT makes the listed call return the given status before it
    touches the GPU: sv_create reports an injected SV_ERR_OOM (3) instead of
    whatever the device would have answered; malformed or unlisted entries
    inject nothing."""
    vp = C.c_void_p
    lib.sv_create.restype = C.c_int
    h = vp(0)
    monkeypatch.setenv("SV_FAULT_INJECT", "sv_verify_tree:2,sv_create:3")
    assert lib.sv_create(C.byref(h)) == 3 and not h.value
    monkeypatch.setenv("SV_FAULT_INJECT", "sv_create:5")
    assert lib.sv_create(C.byref(h)) == 5
    # a NULL out-pointer is still an argument error, checked first
    assert lib.sv_create(vp(0)) == 1
    monkeypatch.setenv("SV_FAULT_INJECT", "sv_create:9,sv_create,sv_creat:3,sv_create:2x")
    rc = lib.sv_create(C.byref(h))
    assert rc not in (2, 3, 9)  # nothing injected: the device's own answer
    if rc == 0:
        lib.sv_destroy(h)
