"""The C-ABI library builds, loads without a GPU and exports every entry point
the header declares; argument checks that need no GPU return their codes."""
import ctypes as C
import os
import re

import pytest

import paged_kv_prep_gb300 as pkv
from paged_kv_prep_gb300 import build as pbuild

HEADER = os.path.join(pbuild.INCLUDE, "pkv.h")


@pytest.fixture(scope="module")
def L():
    pbuild.build()
    return pkv.lib()


def header_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^int\s+(pkv_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_binding_exports():
    assert header_functions() == sorted(pkv.EXPORTS)


def test_every_declared_symbol_is_exported(L):
    for name in header_functions():
        assert hasattr(L, name), name
    assert L.pkv_version() == 100


def test_argument_checks_without_gpu(L):
    h = C.c_void_p()
    spec = (pkv._lib.GroupSpec * 1)(pkv._lib.GroupSpec(16, 4, 100))
    assert L.pkv_state_create(None, 4, 64, 1, spec, 0, None) == pkv.ERR_INVALID_ARG
    assert L.pkv_state_create(C.byref(h), 0, 64, 1, spec, 0, None) == pkv.ERR_INVALID_ARG
    assert L.pkv_state_create(C.byref(h), 4, 64, 0, spec, 0, None) == pkv.ERR_INVALID_ARG
    assert L.pkv_state_create(C.byref(h), 4, 64, 9, spec, 0, None) == pkv.ERR_INVALID_ARG
    bad = (pkv._lib.GroupSpec * 1)(pkv._lib.GroupSpec(0, 4, 100))
    assert L.pkv_state_create(C.byref(h), 4, 64, 1, bad, 0, None) == pkv.ERR_INVALID_ARG
    assert L.pkv_state_destroy(None) == pkv.ERR_INVALID_ARG
    assert L.pkv_prepare_batch(None, None, None, 0, 0, None, None, None) == pkv.ERR_INVALID_ARG
    assert L.pkv_get_error(None, None) == pkv.ERR_INVALID_ARG
    # KV store: alignment of line and strides is checked before any CUDA call
    p = C.c_void_p(4096)
    assert L.pkv_kv_cache_write(p, p, 24, 32, p, p, 10, 24, p, 4, None, None) == pkv.ERR_ALIGN
    assert L.pkv_kv_cache_write(p, p, 40, 32, p, p, 10, 32, p, 4, None, None) == pkv.ERR_ALIGN
    assert L.pkv_kv_cache_write(p, p, 16, 32, p, p, 10, 32, p, 4, None, None) == \
        pkv.ERR_INVALID_ARG   # stride shorter than a line
    assert L.pkv_kv_cache_write(p, p, 32, 32, p, p, 10, 32, None, 4, None, None) == \
        pkv.ERR_INVALID_ARG
    assert L.pkv_kv_cache_write(p, p, 32, 32, p, p, 10, 32, p, 0, None, None) == pkv.OK
    assert L.pkv_kv_cache_write_layers(-1, None, None, 32, 32, None, None, 10, 32, p, 4,
                                       None, None) == pkv.ERR_INVALID_ARG

