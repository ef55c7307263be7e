"""The C-ABI library builds, loads and exports what include/nvfp4_indexer.h
declares; host-side argument checks (no GPU needed, no kernel launched)."""
import ctypes

import pytest

import __graft_entry__
import sparse_attention_block_nvfp4_gb300 as idx


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return idx.load_library()


def test_exports_every_declared_symbol(lib):
    names = idx.declared_symbols()
    assert set(names) >= {"indexer_plan", "indexer_plan_destroy", "indexer_decode", "indexer_prefill",
                          "nvfp4_insert", "indexer_get_status", "indexer_last_error", "indexer_version"}
    for n in names:
        assert hasattr(lib, n), f"{n} declared in the header but not exported"


def test_version(lib):
    assert b"sm_103a" in lib.indexer_version()


P = ctypes.c_void_p
FAKE = ctypes.c_void_p(0x100000)   # never dereferenced: every call below fails its host checks


def test_plan_rejects_unsupported_config(lib):
    h = ctypes.c_void_p()
    assert lib.indexer_plan(ctypes.byref(h), 3, 8, 1, 64, 0, 0) == idx.IDX_EUNSUPPORTED
    assert b"num_heads" in lib.indexer_last_error()
    assert lib.indexer_plan(ctypes.byref(h), 4, 8, 9, 64, 0, 0) == idx.IDX_EUNSUPPORTED
    assert b"max_query_len" in lib.indexer_last_error()
    assert lib.indexer_plan(ctypes.byref(h), 4, -1, 1, 64, 0, 0) == idx.IDX_EINVAL
    assert lib.indexer_plan(None, 4, 8, 1, 64, 0, 0) == idx.IDX_EINVAL
    assert h.value is None


def test_decode_rejects_bad_arguments(lib):
    assert lib.indexer_decode(None, FAKE, FAKE, 1, FAKE, 1, FAKE, 1, 1, FAKE, None, 0, None) == idx.IDX_EINVAL
    assert b"plan is NULL" in lib.indexer_last_error()


def test_prefill_rejects_bad_arguments(lib):
    assert lib.indexer_prefill(None, FAKE, FAKE, 1, 1, 1, FAKE, 1, FAKE, 1, FAKE, FAKE, None, 0, None) \
        == idx.IDX_EINVAL


def test_insert_argument_checks(lib):
    assert lib.nvfp4_insert(FAKE, FAKE, -1, FAKE, 1, None, None) == idx.IDX_EINVAL
    assert lib.nvfp4_insert(None, None, 0, None, 0, None, None) == idx.IDX_OK      # n = 0: no-op
    assert lib.nvfp4_insert(None, FAKE, 4, FAKE, 1, None, None) == idx.IDX_EINVAL
    assert b"NULL" in lib.indexer_last_error()
    misaligned = ctypes.c_void_p(0x100008)
    assert lib.nvfp4_insert(misaligned, FAKE, 4, FAKE, 1, None, None) == idx.IDX_EINVAL
    assert b"aligned" in lib.indexer_last_error()
    assert lib.nvfp4_insert(FAKE, FAKE, 4, FAKE, 0, None, None) == idx.IDX_EINVAL


def test_status_rejects_null_plan(lib):
    bits = ctypes.c_int32(0)
    assert lib.indexer_get_status(None, None, ctypes.byref(bits)) == idx.IDX_EINVAL


def test_insert_norm_rope_argument_checks(lib):
    f = lib.nvfp4_insert_norm_rope
    # k, positions, slots, n, weight, eps, cos_sin, max_pos, rotary_dim, is_neox, pages, num_blocks, status, stream
    assert f(FAKE, FAKE, FAKE, -1, FAKE, 1e-6, FAKE, 16, 128, 1, FAKE, 1, None, None) == idx.IDX_EINVAL
    assert f(FAKE, FAKE, FAKE, 4, FAKE, 1e-6, FAKE, 16, 96, 1, FAKE, 1, None, None) == idx.IDX_EUNSUPPORTED
    assert b"NeoX" in lib.indexer_last_error()
    assert f(FAKE, FAKE, FAKE, 4, FAKE, 1e-6, FAKE, 16, 7, 0, FAKE, 1, None, None) == idx.IDX_EINVAL
    assert f(FAKE, FAKE, FAKE, 4, FAKE, 1e-6, FAKE, 16, 130, 0, FAKE, 1, None, None) == idx.IDX_EINVAL
    assert f(FAKE, FAKE, FAKE, 4, FAKE, -1.0, FAKE, 16, 128, 1, FAKE, 1, None, None) == idx.IDX_EINVAL
    assert f(FAKE, FAKE, FAKE, 4, FAKE, float("nan"), FAKE, 16, 128, 1, FAKE, 1, None, None) == idx.IDX_EINVAL
    assert b"eps" in lib.indexer_last_error()
    assert f(None, None, None, 0, None, 1e-6, None, 0, 0, 1, None, 0, None, None) == idx.IDX_OK   # n = 0
    # a rotation needs positions and a table
    assert f(FAKE, None, FAKE, 4, FAKE, 1e-6, FAKE, 16, 64, 1, FAKE, 1, None, None) == idx.IDX_EINVAL
    assert f(FAKE, FAKE, FAKE, 4, FAKE, 1e-6, None, 16, 64, 1, FAKE, 1, None, None) == idx.IDX_EINVAL
    # the table's vector loads: 16-byte alignment for NeoX and rotary_dim % 8 == 0, 4 otherwise
    odd = ctypes.c_void_p(0x100004)
    assert f(FAKE, FAKE, FAKE, 4, FAKE, 1e-6, odd, 16, 64, 1, FAKE, 1, None, None) == idx.IDX_EINVAL
    assert b"aligned" in lib.indexer_last_error()
    assert f(FAKE, FAKE, FAKE, 4, FAKE, 1e-6, odd, 16, 64, 0, FAKE, 1, None, None) == idx.IDX_EINVAL
    misaligned = ctypes.c_void_p(0x100008)
    assert f(misaligned, FAKE, FAKE, 4, FAKE, 1e-6, FAKE, 16, 128, 1, FAKE, 1, None, None) == idx.IDX_EINVAL
    assert f(FAKE, FAKE, FAKE, 4, FAKE, 1e-6, FAKE, 16, 128, 1, FAKE, 0, None, None) == idx.IDX_EINVAL
