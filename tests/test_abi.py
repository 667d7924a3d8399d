"""The C-ABI library without a GPU: it loads, exports every function that
include/pa.h declares, and its host-side argument checks return the
documented statuses before anything touches a device."""
import ctypes
import os
import re

import pytest

from paged_kv_decode_18_gb300 import binding as B
from paged_kv_decode_18_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return B.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert _declared_functions() == sorted(B.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert B.pa_status_string(0) == "PA_OK"
    for st in (B.PA_ERR_ARG, B.PA_ERR_UNSUPPORTED, B.PA_ERR_WORKSPACE, B.PA_ERR_CUDA,
               B.PA_ERR_DEVICE):
        assert B.pa_status_string(st).startswith("PA_ERR_")
    assert "sm_103a" in B.pa_version()


def _shape(**kw):
    base = dict(num_seqs=4, num_q_heads=16, num_kv_heads=8, head_dim=128, block_size=16,
                max_blocks_per_seq=24, num_blocks=128)
    base.update(kw)
    return B.make_shape(**base)


def _decode(lib, sh, num_splits=0, null_q=False):
    p = ctypes.c_void_p(0x1000)  # never dereferenced: every case fails host checks first
    q = None if null_q else p
    return lib.pa_decode(q, p, p, p, p, 0.1, p, None, ctypes.byref(sh), num_splits, None, 0,
                         None)


def test_decode_host_checks(lib):
    assert lib.pa_decode(None, None, None, None, None, 0.1, None, None, None, 0, None, 0,
                         None) == B.PA_ERR_ARG
    assert _decode(lib, _shape(head_dim=64)) == B.PA_ERR_UNSUPPORTED
    assert _decode(lib, _shape(block_size=32)) == B.PA_ERR_UNSUPPORTED
    assert _decode(lib, _shape(num_kv_heads=4)) == B.PA_ERR_UNSUPPORTED  # group 4 not built
    assert _decode(lib, _shape(num_q_heads=12, num_kv_heads=8)) == B.PA_ERR_ARG
    assert _decode(lib, _shape(), num_splits=-1) == B.PA_ERR_ARG
    assert _decode(lib, _shape(), num_splits=5000) == B.PA_ERR_ARG
    assert _decode(lib, _shape(num_seqs=-1)) == B.PA_ERR_ARG
    assert _decode(lib, _shape(), null_q=True) == B.PA_ERR_ARG
    assert _decode(lib, _shape(num_seqs=0)) == B.PA_OK  # empty batch: nothing to do


def test_cache_write_host_checks(lib):
    p = ctypes.c_void_p(0x1000)
    sh = _shape()
    f = lib.pa_reshape_and_cache
    assert f(p, p, p, -1, p, p, ctypes.byref(sh), None) == B.PA_ERR_ARG
    assert f(p, p, p, 0, p, p, ctypes.byref(sh), None) == B.PA_OK
    assert f(None, p, p, 3, p, p, ctypes.byref(sh), None) == B.PA_ERR_ARG
    assert f(ctypes.c_void_p(0x1001), p, p, 3, p, p, ctypes.byref(sh), None) == B.PA_ERR_ARG
    sh2 = _shape(head_dim=96)
    assert f(p, p, p, 3, p, p, ctypes.byref(sh2), None) == B.PA_ERR_UNSUPPORTED


def test_splitk_reduce_host_checks(lib):
    p = ctypes.c_void_p(0x1000)
    f = lib.pa_splitk_reduce
    assert f(p, p, 4, 16, 0, 128, p, None, None) == B.PA_ERR_ARG
    assert f(p, p, 4, 16, 8, 126, p, None, None) == B.PA_ERR_UNSUPPORTED
    assert f(p, p, 4, 16, 8, 2048, p, None, None) == B.PA_ERR_UNSUPPORTED
    assert f(p, p, 0, 16, 8, 128, p, None, None) == B.PA_OK
    assert f(None, p, 4, 16, 8, 128, p, None, None) == B.PA_ERR_ARG


def test_varlen_host_checks(lib):
    p = ctypes.c_void_p(0x1000)
    sh = _shape(head_dim=64)
    f = lib.pa_decode_varlen
    assert f(p, p, p, p, p, p, 8, 2, 1, 0.1, p, None, ctypes.byref(sh), None, 0,
             None) == B.PA_ERR_UNSUPPORTED
    sh = _shape()
    assert f(p, p, p, p, p, p, -1, 2, 1, 0.1, p, None, ctypes.byref(sh), None, 0,
             None) == B.PA_ERR_ARG


def test_workspace_size_of_bad_shape_is_zero(lib):
    assert B.pa_decode_workspace_size(_shape(head_dim=64), 0) == 0
    assert B.pa_decode_workspace_size(_shape(), 1) == 0
