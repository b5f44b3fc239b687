"""The C-ABI library builds, loads without a GPU and exports every symbol
that include/lsmmerge.h declares; host-side argument checks need no GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "lsmmerge.h")).read()
    return sorted(set(re.findall(r"LSM_API[^;(]*?\b(lsm_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from lsm_replacement_merge_gb300 import _build
    return ctypes.CDLL(_build.build())


def test_header_declares_the_hot_path_calls():
    names = _declared()
    for call in ("merge_path_partition", "merge_stable", "collision_mark", "rank_build",
                 "rank_query", "replacement_merge_compact", "fc_lengths_scan", "fc_emit"):
        assert "lsm_" + call in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_host_side_checks_without_gpu(lib):
    lib.lsm_status_string.restype = ctypes.c_char_p
    assert lib.lsm_status_string(0) == b"LSM_OK"
    assert lib.lsm_abi_version() == 101
    size = ctypes.c_size_t(0)
    assert lib.lsm_workspace_size(1, 2, 1 << 26, 1 << 26, ctypes.byref(size)) == 0
    assert size.value > 0
    assert lib.lsm_workspace_size(1, 99, 10, 10, ctypes.byref(size)) == 2      # LSM_ERR_DTYPE
    assert lib.lsm_workspace_size(2, 0, -1, 10, ctypes.byref(size)) == 1       # LSM_ERR_ARG
    # argument errors are caught on the host before anything touches a device
    I = ctypes.c_int64
    assert lib.lsm_merge_stable(7, None, None, I(1), None, None, I(1), None, None, None,
                                ctypes.c_size_t(0), None) == 2
    assert lib.lsm_collision_mark(None, I(-1), None, I(0), None, None, None, ctypes.c_size_t(0),
                                  None) == 1
    assert lib.lsm_collision_mark(ctypes.c_void_p(16), I(1 << 31), ctypes.c_void_p(16), I(1),
                                  ctypes.c_void_p(16), ctypes.c_void_p(16), None,
                                  ctypes.c_size_t(0), None) == 3              # LSM_ERR_OVERFLOW
    assert lib.lsm_rank_build(ctypes.c_void_p(16), I(100), ctypes.c_void_p(16), ctypes.c_void_p(16),
                              ctypes.c_void_p(16), ctypes.c_size_t(0), None) == 6  # workspace
    assert lib.lsm_tune_merge(2, 8, 2, 1) == 1
    assert lib.lsm_tune_merge(2, 7, 2, 1) == 0
