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


def test_rank2048_host_checks_without_gpu(lib):
    I, P, S = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    size = ctypes.c_size_t(0)
    assert lib.lsm_workspace_size(8, 0, 12_000_000, 0, ctypes.byref(size)) == 0
    # one uint32 total per CTA of 256 blocks of 2048 bits, plus slack
    assert 4 * 23 <= size.value <= 4096
    assert lib.lsm_rank2048_build(P(16), I(-1), P(16), P(16), P(16), P(16), S(4096), None) == 1
    assert lib.lsm_rank2048_build(P(16), I(1 << 36), P(16), P(16), P(16), P(16), S(1 << 30),
                                  None) == 3
    assert lib.lsm_rank2048_build(P(20), I(100), P(16), P(16), P(16), P(16), S(4096), None) == 7
    assert lib.lsm_rank2048_build(P(16), I(100), P(16), P(16), P(16), P(16), S(1), None) == 6
    assert lib.lsm_rank2048_query(P(16), None, P(16), I(10), P(16), I(1), P(16), None) == 1
    assert lib.lsm_rank2048_query(P(16), P(16), P(16), I(10), P(16), I(0), P(16), None) == 0
    # the rank2048 compaction checks its arguments like the rank512 one
    assert lib.lsm_replacement_merge_compact_rank2048(I(10), I(10), P(16), P(16), None, P(16),
                                                      P(16), P(16), P(16), P(16), P(16), S(1 << 20),
                                                      None) == 1
    assert lib.lsm_replacement_merge_compact_rank2048(I(1 << 31), I(10), P(16), P(16), P(16),
                                                      P(16), P(16), P(16), P(16), P(16), P(16),
                                                      S(1 << 20), None) == 3


def test_ef_sizes_without_gpu(lib):
    import numpy as np
    import oracle
    out = (ctypes.c_int64 * 5)()
    for N, U in ((0, 0), (1, 5), (14, 1000), (15, 1000), (7_200_000, 2_500_000_000),
                 (100, (1 << 64) - 1)):
        assert lib.lsm_ef_sizes(ctypes.c_int64(N), ctypes.c_uint64(U), out) == 0
        assert tuple(out) == oracle.ef_sizes(N, U)
    assert lib.lsm_ef_sizes(ctypes.c_int64(-1), ctypes.c_uint64(0), out) == 1
    I, P = ctypes.c_int64, ctypes.c_void_p
    assert lib.lsm_fc_ef_build(None, I(10), ctypes.c_uint64(0), ctypes.c_uint64(0), P(8), P(8),
                               P(8), P(8), P(8), None) == 1
    assert lib.lsm_fc_ef_build(P(12), I(10), ctypes.c_uint64(0), ctypes.c_uint64(100), P(8),
                               P(8), P(8), P(8), P(8), None) == 7


def test_direct_scatter_host_checks_without_gpu(lib):
    I, P = ctypes.c_int64, ctypes.c_void_p
    args = [P(16), I(10), P(16), I(10), P(16), P(16), P(16), P(16), P(16), P(16), P(16), None]
    bad = list(args)
    bad[5] = None                                              # dir
    assert lib.lsm_replacement_direct_scatter(*bad) == 1
    bad = list(args)
    bad[1] = I(1 << 31)
    assert lib.lsm_replacement_direct_scatter(*bad) == 3
    bad = list(args)
    bad[2] = P(24)                                             # B misaligned
    assert lib.lsm_replacement_direct_scatter(*bad) == 7


def test_fused_host_checks_without_gpu(lib):
    I, P, S = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    size = ctypes.c_size_t(0)
    assert lib.lsm_workspace_size(9, 0, 12_000_000, 4_000_000, ctypes.byref(size)) == 0
    tiles = (16_000_000 + 2815) // 2816
    assert size.value >= 16 * tiles  # a co-rank and a state per tile
    args = [P(16), I(10), P(16), I(10), P(16), P(16), P(16), P(16), P(16), P(16), P(16), P(16),
            P(16), S(1 << 20), None]
    bad = list(args)
    bad[6] = None                                              # dir
    assert lib.lsm_replacement_merge_fused(*bad) == 1
    bad = list(args)
    bad[3] = I(1 << 31)
    assert lib.lsm_replacement_merge_fused(*bad) == 3
    bad = list(args)
    bad[8] = P(20)                                             # refs misaligned
    assert lib.lsm_replacement_merge_fused(*bad) == 7
    bad = list(args)
    bad[13] = S(8)
    assert lib.lsm_replacement_merge_fused(*bad) == 6


def test_bytefc_host_checks_without_gpu(lib):
    I, P, S, U = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint64
    fc = _FcInput(_Bytes(P(64), P(128)), _Bytes(P(64), P(128)), None, I(10),
                  _Bytes(P(64), P(128)), _Bytes(P(64), P(128)), None, I(10), None, None)
    assert lib.lsm_bytefc_lengths_scan(ctypes.byref(fc), P(16), I(-1), U(0), P(16), P(16),
                                       P(16), P(16), P(16), S(1 << 20), None) == 1
    assert lib.lsm_bytefc_lengths_scan(ctypes.byref(fc), P(16), I(21), U(0), P(16), P(16),
                                       P(16), P(16), P(16), S(1 << 20), None) == 3
    assert lib.lsm_bytefc_lengths_scan(ctypes.byref(fc), P(16), I(5), U(0), P(16), P(16),
                                       P(20), P(16), P(16), S(1 << 20), None) == 7
    assert lib.lsm_bytefc_emit(ctypes.byref(fc), P(16), I(5), U(0), P(16), P(16), P(16), None,
                               I(100), None) == 1


def test_merge_sort_host_checks_without_gpu(lib):
    I, P, S = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    sizes = {}
    for kt in (1, 2):
        for N in (1, 2816, 1 << 27):
            size = ctypes.c_size_t(0)
            assert lib.lsm_workspace_size(7, kt, N, 0, ctypes.byref(size)) == 0
            sizes[kt, N] = size.value
        # the alternate buffers: one key and one payload per element, at least
        assert sizes[kt, 1 << 27] >= (1 << 27) * (4 if kt == 1 else 8) + (1 << 27) * 4
    assert sizes[2, 1 << 27] > sizes[1, 1 << 27]
    size = ctypes.c_size_t(0)
    assert lib.lsm_workspace_size(7, 9, 10, 0, ctypes.byref(size)) == 2   # LSM_ERR_DTYPE
    assert lib.lsm_merge_sort(3, P(16), None, I(4), P(16), None, P(16), S(1 << 20), None) == 2
    assert lib.lsm_merge_sort(2, P(16), None, I(-1), P(16), None, P(16), S(1 << 20), None) == 1
    # payload in without payload out, and the reverse
    assert lib.lsm_merge_sort(2, P(16), P(16), I(4), P(16), None, P(16), S(1 << 20), None) == 1
    assert lib.lsm_merge_sort(2, P(16), None, I(4), P(16), P(16), P(16), S(1 << 20), None) == 1
    assert lib.lsm_merge_sort(2, P(16), None, I(1 << 41), P(16), None, P(16), S(1 << 20),
                              None) == 3                                   # LSM_ERR_OVERFLOW
    assert lib.lsm_merge_sort(2, P(24), None, I(4), P(16), None, P(16), S(1 << 20), None) == 7
    assert lib.lsm_merge_sort(2, P(16), None, I(4), P(16), None, P(16), S(8), None) == 6
    assert lib.lsm_merge_sort(2, None, None, I(0), None, None, None, S(0), None) == 0


class _Bytes(ctypes.Structure):
    _fields_ = [("arena", ctypes.c_void_p), ("off", ctypes.c_void_p)]


class _FcInput(ctypes.Structure):
    _fields_ = [("keyA", _Bytes), ("valA", _Bytes), ("tombA", ctypes.c_void_p), ("m", ctypes.c_int64),
                ("keyB", _Bytes), ("valB", _Bytes), ("tombB", ctypes.c_void_p), ("n", ctypes.c_int64),
                ("prefixA", ctypes.c_void_p), ("prefixB", ctypes.c_void_p)]


def test_prefix_table_checks_without_gpu(lib):
    # the key prefix tables: 16-byte aligned, and both or neither for the
    # lengths pass (an empty source needs none); caught on the host
    I, P, S = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    a = _Bytes(P(64), P(128))
    b = _Bytes(P(64), P(128))
    assert lib.lsm_collision_mark_str_prefix(ctypes.byref(a), I(10), ctypes.byref(b), I(10), P(16),
                                             P(16), P(24), P(32), P(16), S(1 << 20), None) == 7
    assert lib.lsm_collision_mark_str_prefix(ctypes.byref(a), I(-1), ctypes.byref(b), I(10), P(16),
                                             P(16), None, None, P(16), S(1 << 20), None) == 1

    def lengths(prefixA, prefixB, m=10, n=10):
        fc = _FcInput(_Bytes(P(64), P(128)), _Bytes(P(64), P(128)), None, I(m),
                      _Bytes(P(64), P(128)), _Bytes(P(64), P(128)), None, I(n),
                      P(prefixA) if prefixA else None, P(prefixB) if prefixB else None)
        return lib.lsm_fc_lengths_scan(ctypes.byref(fc), P(16), I(5), P(16), P(16), P(16), P(16),
                                       None, S(0), None)

    assert lengths(256, None) == 1          # one table for two non-empty sources
    assert lengths(None, 256) == 1
    assert lengths(264, 256) == 7           # not 16-byte aligned
    assert lengths(256, 264) == 7
    assert lengths(256, None, n=0) == 6     # an empty B needs no table: on to the workspace check
    assert lengths(None, None) == 6
