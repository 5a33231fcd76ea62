"""The C-ABI library loads and exports every symbol include/kvs.h declares;
host-side argument checks return the documented status without touching a
GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from shared_paged_kv_gb300 import kvs as K
    return K.load()


def declared_symbols():
    with open(os.path.join(ROOT, "include", "kvs.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(kvs_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    syms = declared_symbols()
    assert len(syms) >= 13
    for s in syms:
        assert hasattr(lib, s), s
    from shared_paged_kv_gb300 import kvs as K
    assert sorted(K.EXPORTED) == syms


def test_host_argument_errors(lib):
    from shared_paged_kv_gb300 import kvs as K
    P = ctypes.c_void_p
    out = P()
    # null descriptor
    assert lib.kvs_pool_create(None, None, None, None, None, None, None, ctypes.byref(out)) == K.KVS_ERR_INVALID_ARG
    # unsupported head_dim is rejected before any CUDA call
    d = K.PoolDesc(1, 2, 96, 16, K.KVS_DTYPE_BF16, 8, 0, 4)
    arr = (P * 1)(16)
    assert lib.kvs_pool_create(ctypes.byref(d), arr, arr, None, None, None, None, ctypes.byref(out)) == K.KVS_ERR_UNSUPPORTED
    assert b"head_dim" in lib.kvs_last_error_string()
    d = K.PoolDesc(1, 2, 64, 32, K.KVS_DTYPE_BF16, 8, 0, 4)
    assert lib.kvs_pool_create(ctypes.byref(d), arr, arr, None, None, None, None, ctypes.byref(out)) == K.KVS_ERR_UNSUPPORTED
    d = K.PoolDesc(1, 2, 128, 256, K.KVS_DTYPE_Q4G64, 8, 0, 4)
    assert lib.kvs_pool_create(ctypes.byref(d), arr, arr, None, None, None, None, ctypes.byref(out)) == K.KVS_ERR_INVALID_ARG
    d = K.PoolDesc(1, 2, 64, 16, 7, 8, 0, 4)
    assert lib.kvs_pool_create(ctypes.byref(d), arr, arr, None, None, None, None, ctypes.byref(out)) == K.KVS_ERR_INVALID_ARG
    d = K.PoolDesc(1, 64, 128, 16, K.KVS_DTYPE_BF16, 1 << 22, 0, 4)
    assert lib.kvs_pool_create(ctypes.byref(d), arr, arr, None, None, None, None, ctypes.byref(out)) == K.KVS_ERR_CAPACITY
    assert lib.kvs_pool_destroy(None) == K.KVS_ERR_INVALID_ARG
    # every compute entry point rejects a null pool on the host
    assert lib.kvs_decode_attn(None, 0, None, 8, None, 1, None, 1, None, None, None, 1.0, 1.0, None, None, 0, None) == K.KVS_ERR_INVALID_ARG
    assert lib.kvs_decode_attn_q4(None, 0, None, 8, None, 1, None, 1, None, 1.0, None, None, 0, None) == K.KVS_ERR_INVALID_ARG
    assert lib.kvs_fingerprint_dedup(None, None, None, 1, None, None, None, None, None, 1, None, None, None, None, None,
                                     0, None, 0, None) == K.KVS_ERR_INVALID_ARG
    assert lib.kvs_rope_rerotate(None, 0, None, 1, 16, 1e4, None, None, 1, None) == K.KVS_ERR_INVALID_ARG
    assert lib.kvs_quantize_q4(None, 0, None, None, None, 1, None) == K.KVS_ERR_INVALID_ARG
    sz = ctypes.c_size_t()
    assert lib.kvs_workspace_size(None, 0, 1, 1, 1, ctypes.byref(sz)) == K.KVS_ERR_INVALID_ARG
    # selection: bad row width, and the empty call is a no-op
    assert lib.kvs_select_critical(None, None, None, 1, 8, 12, 0.1, None, None, None, 0, None) == K.KVS_ERR_INVALID_ARG
    off = (ctypes.c_int64 * 1)(0)
    assert lib.kvs_select_critical(None, None, off, 0, 8, 16, 0.1, None, off, None, 0, None) == K.KVS_OK
    assert lib.kvs_launch_count() == 0
