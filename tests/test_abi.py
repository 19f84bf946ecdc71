"""The C-ABI library builds, loads and exports every entry point include/kvs.h declares (no GPU)."""
import os
import re

import pytest

from conftest import ROOT


def _declared():
    with open(os.path.join(ROOT, "include", "kvs.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvs_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def libkvs():
    from sparse_kv_cache_decode_gb300 import build as B
    B.build()
    import sparse_kv_cache_decode_gb300 as K
    return K.lib()


def test_every_declared_symbol_is_exported(libkvs):
    names = _declared()
    assert len(names) >= 17
    for n in names:
        assert hasattr(libkvs, n), n


def test_binding_covers_every_declared_symbol(libkvs):
    import sparse_kv_cache_decode_gb300 as K
    assert sorted(K._SIGS) == _declared()


def test_workspace_sizing_and_validation(libkvs):
    import ctypes
    import sparse_kv_cache_decode_gb300 as K
    import workload as W
    cfg = K.make_config(W.LLAMA8B_32K)
    n = libkvs.kvs_workspace_bytes(ctypes.byref(cfg))
    # slot pools dominate: 32 layers x 64 units x 192 slots x 16 rows x 256 B x (K and V)
    assert n > 32 * 64 * 192 * 16 * 256 * 2
    bad = K.make_config(W.LLAMA8B_32K.with_(cap_blocks=100))       # cache smaller than the budget
    assert libkvs.kvs_workspace_bytes(ctypes.byref(bad)) == 0
    bad2 = K.make_config(W.TINY.with_(n_q_head=7))                  # H_q not a multiple of H_kv
    assert libkvs.kvs_workspace_bytes(ctypes.byref(bad2)) == 0
    h = ctypes.c_void_p()
    assert libkvs.kvs_create(ctypes.byref(cfg), None, 0, ctypes.byref(h)) == 1   # KVS_ERR_INVALID_ARG


def test_version(libkvs):
    import sparse_kv_cache_decode_gb300 as K
    assert "sm_103a" in K.version()
