"""The C-ABI library loads, exports every symbol include/ddtree.h declares, and
rejects bad arguments on the host before touching a GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

from speculative_decoding_tree_05_gb300 import ddtree

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ddtree.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"DDT_API\s+[\w\s\*]*?\b(ddtree_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_tree_05_gb300 import build
    build.build()
    return ddtree.lib()


def test_header_declares_the_api():
    assert declared_symbols() == sorted(ddtree.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert ddtree.status_string(0) == "ok"
    for code in ddtree.ERRORS:
        assert ddtree.status_string(code) != "unknown status"
    assert ddtree.status_string(12345) == "unknown status"


def dims(**kw):
    d = dict(batch=1, nodes=9, heads=16, pool_slots=4096, slot_stride=256, max_prefix_len=256)
    d.update(kw)
    return ddtree.make_dims(d["batch"], d["nodes"], d["heads"], d["pool_slots"], d["slot_stride"],
                            d["max_prefix_len"])


def call_verify(lib, d, ptr=0x10000, ws=1 << 30, q=None):
    p = ctypes.c_void_p(ptr)
    qp = p if q is None else ctypes.c_void_p(q)
    return lib.ddtree_verify_attn(qp, p, p, p, p, p, 0.1, p, p, None if d is None else ctypes.byref(d), p, ws,
                                  None)


def test_null_dims(lib):
    assert call_verify(lib, None) == -1


@pytest.mark.parametrize("bad", [dict(nodes=0), dict(nodes=129), dict(heads=0), dict(heads=1025),
                                 dict(batch=-1), dict(pool_slots=0), dict(max_prefix_len=-1),
                                 dict(slot_stride=100, max_prefix_len=256), dict(pool_slots=1 << 32)])
def test_bad_dims(lib, bad):
    assert call_verify(lib, dims(**bad)) == -2


def test_empty_batch_is_ok(lib):
    assert call_verify(lib, dims(batch=0), ptr=0) == 0


def test_null_pointer(lib):
    assert call_verify(lib, dims(), q=0) == -1


def test_misaligned_pointer(lib):
    assert call_verify(lib, dims(), q=0x10008) == -4


def test_compact_host_checks(lib):
    p = ctypes.c_void_p(0x10000)
    d = dims()
    assert lib.ddtree_kv_compact(p, p, p, p, p, p, None, p, None) == -1
    assert lib.ddtree_kv_compact(None, p, p, p, p, p, ctypes.byref(d), p, None) == -1
    assert lib.ddtree_kv_compact(ctypes.c_void_p(0x10004), p, p, p, p, p, ctypes.byref(d), p, None) == -4


def test_read_status_null(lib):
    assert lib.ddtree_read_device_status(None, None, None) == -1


def test_workspace_bytes_bad_dims(lib):
    assert ddtree.workspace_bytes(dims(nodes=0)) == 0


def test_ragged_host_checks(lib):
    p = ctypes.c_void_p(0x10000)
    d = dims(batch=2)

    def ragged(tree_len, dd=d):
        return lib.ddtree_verify_attn_ragged(p, p, p, p, p, p, tree_len, 0.1, p, p, ctypes.byref(dd), p, 1 << 30,
                                             None)
    assert ragged(None) == -1                       # tree_len is required when B > 0
    assert ragged(ctypes.c_void_p(0x10002)) == -4   # misaligned int32 array
    assert ragged(None, dims(batch=0)) == 0         # empty batch: nothing enqueued
    assert ragged(p, dims(heads=0)) == -2


def test_static_scratch_checks_sizes_first(lib):
    # the same code as ddtree_verify_attn for unsupported sizes, before any device query
    p = ctypes.c_void_p(0x10000)
    bad = dims(nodes=0)
    assert lib.ddtree_verify_attn_static_scratch(p, p, p, p, p, p, 0.1, p, p, ctypes.byref(bad), None) == -2
    assert lib.ddtree_verify_attn_static_scratch(p, p, p, p, p, p, 0.1, p, p, None, None) == -1
    assert lib.ddtree_verify_attn_static_scratch(p, p, p, p, p, p, 0.1, p, p, ctypes.byref(dims(batch=0)),
                                                 None) == 0


def test_static_scratch_without_sm103_is_a_device_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    p = ctypes.c_void_p(0x10000)
    assert lib.ddtree_verify_attn_static_scratch(p, p, p, p, p, p, 0.1, p, p, ctypes.byref(dims()), None) == -6
