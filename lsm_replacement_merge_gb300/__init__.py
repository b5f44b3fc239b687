"""Python binding of liblsmmerge.so, the GB300 merge-path replacement merge.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels. Tensors are torch CUDA tensors (PyTorch provides device memory and
streams); each function passes their device pointers and the current CUDA
stream to the C entry point of the same name (``lsm_<name>`` in
``include/lsmmerge.h``) and raises ``LsmError`` on a non-zero status. Outputs
the caller does not pass are allocated with torch.

The library must be built first (``__graft_entry__.build()`` or
``lsm_replacement_merge_gb300.build()``); importing this package never falls
back to any other implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "liblsmmerge.so")

LSM_OK = 0
LSM_ERR_ARG = 1
LSM_ERR_DTYPE = 2
LSM_ERR_OVERFLOW = 3
LSM_ERR_CUDA = 4
LSM_ERR_TIMEOUT = 5
LSM_ERR_WORKSPACE = 6
LSM_ERR_ALIGN = 7
LSM_ERR_UNSORTED = 8
LSM_KEY_I32 = 1
LSM_KEY_U64 = 2
LSM_OP_MERGE_STABLE = 1
LSM_OP_COLLISION_MARK = 2
LSM_OP_COLLISION_MARK_STR = 3
LSM_OP_RANK_BUILD = 4
LSM_OP_REPLACEMENT_COMPACT = 5
LSM_OP_FC_LENGTHS_SCAN = 6
LSM_OP_MERGE_SORT = 7
LSM_OP_RANK2048_BUILD = 8
LSM_OP_REPLACEMENT_FUSED = 9
LSM_OP_REPLACEMENT_MERGE = 10
LSM_OP_REPLACEMENT_MERGE_STR = 11
REF_FROM_B = 0x80000000
ORD_DROPPED = 0xFFFFFFFF

_lock = threading.Lock()
_lib = None


class LsmError(RuntimeError):
    def __init__(self, name, status):
        self.status = status
        super().__init__("%s failed: %s" % (name, _status_string(status)))


class _Bytes(ctypes.Structure):
    _fields_ = [("arena", ctypes.c_void_p), ("off", ctypes.c_void_p)]


class _FcInput(ctypes.Structure):
    _fields_ = [("keyA", _Bytes), ("valA", _Bytes), ("tombA", ctypes.c_void_p), ("m", ctypes.c_int64),
                ("keyB", _Bytes), ("valB", _Bytes), ("tombB", ctypes.c_void_p), ("n", ctypes.c_int64),
                ("prefixA", ctypes.c_void_p), ("prefixB", ctypes.c_void_p)]


def build(force: bool = False) -> str:
    from . import _build
    return _build.build(force=force)


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("liblsmmerge.so is not built (%s); run __graft_entry__.build()"
                                   % LIB_PATH)
            L = ctypes.CDLL(LIB_PATH)
            P, I, S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
            sig = {
                "lsm_status_string": ([ctypes.c_int], ctypes.c_char_p),
                "lsm_abi_version": ([], ctypes.c_int),
                "lsm_get_device_status": ([P, ctypes.c_int, P], ctypes.c_int),
                "lsm_workspace_size": ([ctypes.c_int, ctypes.c_int, I, I, P], ctypes.c_int),
                "lsm_merge_path_partition": ([ctypes.c_int, P, I, P, I, I, P, P], ctypes.c_int),
                "lsm_merge_stable": ([ctypes.c_int, P, P, I, P, P, I, P, P, P, S, P], ctypes.c_int),
                "lsm_merge_sort": ([ctypes.c_int, P, P, I, P, P, P, S, P], ctypes.c_int),
                "lsm_collision_mark": ([P, I, P, I, P, P, P, S, P], ctypes.c_int),
                "lsm_collision_mark_str": ([P, I, P, I, P, P, P, S, P], ctypes.c_int),
                "lsm_collision_mark_str_prefix": ([P, I, P, I, P, P, P, P, P, S, P], ctypes.c_int),
                "lsm_rank_build": ([P, I, P, P, P, S, P], ctypes.c_int),
                "lsm_rank_query": ([P, P, I, P, I, P, P], ctypes.c_int),
                "lsm_rank2048_build": ([P, I, P, P, P, P, S, P], ctypes.c_int),
                "lsm_rank2048_query": ([P, P, P, I, P, I, P, P], ctypes.c_int),
                "lsm_replacement_merge_compact": ([I, I, P, P, P, P, P, P, P, P, S, P], ctypes.c_int),
                "lsm_replacement_merge_compact_rank2048": ([I, I, P, P, P, P, P, P, P, P, P, S, P],
                                                           ctypes.c_int),
                "lsm_replacement_direct_scatter": ([P, I, P, I, P, P, P, P, P, P, P, P],
                                                   ctypes.c_int),
                "lsm_replacement_merge_fused": ([P, I, P, I, P, P, P, P, P, P, P, P, P, S, P],
                                                ctypes.c_int),
                "lsm_replacement_merge": ([P, I, P, I, P, P, P, P, P, P, P, P, P, S, P],
                                          ctypes.c_int),
                "lsm_replacement_merge_str": ([P, I, P, I, P, P, P, P, P, P, P, P, P, P, P, S, P],
                                              ctypes.c_int),
                "lsm_replacement_materialize": ([P, P, P, I, P, P, P, I, P, P, P, P, P, P],
                                                ctypes.c_int),
                "lsm_fc_lengths_scan": ([P, P, I, P, P, P, P, P, S, P], ctypes.c_int),
                "lsm_fc_emit": ([P, P, I, P, P, P, P, I, P], ctypes.c_int),
                "lsm_ef_sizes": ([I, ctypes.c_uint64, P], ctypes.c_int),
                "lsm_bytefc_lengths_scan": ([P, P, I, ctypes.c_uint64, P, P, P, P, P, S, P],
                                            ctypes.c_int),
                "lsm_bytefc_emit": ([P, P, I, ctypes.c_uint64, P, P, P, P, I, P], ctypes.c_int),
                "lsm_bytefc_value_width": ([P, P, I, P, P], ctypes.c_int),
                "lsm_fc_ef_build": ([P, I, ctypes.c_uint64, ctypes.c_uint64, P, P, P, P, P, P],
                                    ctypes.c_int),
                "lsm_debug_timeout_probe": ([I, P], ctypes.c_int),
                "lsm_tune_merge": ([ctypes.c_int] * 4, ctypes.c_int),
                "lsm_tune_replace": ([ctypes.c_int] * 3, ctypes.c_int),
                "lsm_tune_replacement_merge": ([ctypes.c_int], ctypes.c_int),
                "lsm_set_profile_events": ([P, P], ctypes.c_int),
                "lsm_rank_build_noalloc": ([P, I, P, P, P], ctypes.c_int),
                "lsm_validate_sorted": ([ctypes.c_int, P, I, ctypes.c_int, P, P], ctypes.c_int),
                "lsm_validate_sorted_str": ([P, I, ctypes.c_uint64, ctypes.c_int, P, P],
                                            ctypes.c_int),
            }
            for name, (args, res) in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def _status_string(status):
    try:
        return lib().lsm_status_string(status).decode()
    except Exception:  # pragma: no cover - only while reporting another error
        return "status %d" % status


def _check(name, rc):
    if rc != LSM_OK:
        raise LsmError(name, rc)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor, got one on %s" % t.device)
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _key_type(t):
    if t.dtype == torch.int32:
        return LSM_KEY_I32
    if t.dtype in (torch.uint64, torch.int64):
        return LSM_KEY_U64
    raise TypeError("keys must be int32 or uint64 (int64 views are accepted), got %s" % t.dtype)


def _empty(n, dtype, device):
    return torch.empty(int(n), dtype=dtype, device=device)


# ---------------------------------------------------------------------------
# utilities
# ---------------------------------------------------------------------------
def abi_version() -> int:
    return lib().lsm_abi_version()


def workspace_size(op: int, m: int, n: int, key_type: int = LSM_KEY_U64) -> int:
    out = ctypes.c_size_t(0)
    _check("lsm_workspace_size", lib().lsm_workspace_size(op, key_type, m, n, ctypes.byref(out)))
    return out.value


def workspace(op: int, m: int, n: int, device, key_type: int = LSM_KEY_U64):
    return torch.empty(workspace_size(op, m, n, key_type), dtype=torch.uint8, device=device)


def get_device_status(reset: bool = False, stream=None) -> int:
    st = ctypes.c_int32(0)
    _check("lsm_get_device_status",
           lib().lsm_get_device_status(ctypes.byref(st), int(bool(reset)), _stream(stream)))
    return st.value


def set_profile_events(start=None, stop=None) -> None:
    """Time the next call's main kernel with two torch.cuda.Event objects
    (created with enable_timing=True); see lsm_set_profile_events."""
    for ev in (start, stop):
        if ev is not None and not ev.cuda_event:
            ev.record()  # torch creates the CUDA event lazily, at its first record
    sp = ctypes.c_void_p(start.cuda_event) if start is not None else None
    ep = ctypes.c_void_p(stop.cuda_event) if stop is not None else None
    _check("lsm_set_profile_events", lib().lsm_set_profile_events(sp, ep))


MERGE_CONFIGS = ((5, 2, 1), (7, 2, 1), (11, 2, 1), (15, 2, 1), (7, 4, 2), (11, 3, 2), (15, 2, 2),
                 (7, 3, 1))
DEFAULT_MERGE_CONFIG = (11, 2, 1)


REPLACE_VARIANTS = ((256, 11), (128, 23), (256, 23), (512, 11))
# (0, 0) selects the warp pipelines (the default); the rest the earlier
# block-synchronous tile pipelines, kept for comparison
DEFAULT_REPLACE_VARIANT = {0: (0, 0), 1: (0, 0)}  # kernel -> (threads, items)


def tune_replace(kernel: int, threads: int, items_per_thread: int) -> None:
    """Tile variant of collision_mark (kernel 0) or replacement_merge_compact (1)."""
    _check("lsm_tune_replace", lib().lsm_tune_replace(kernel, threads, items_per_thread))


DEFAULT_REPLACEMENT_MERGE_MODE = 0


def tune_replacement_merge(mode: int) -> None:
    """Form of replacement_merge: 0 = two tile pipelines (the default), 1 =
    the mark and the compaction in one kernel."""
    _check("lsm_tune_replacement_merge", lib().lsm_tune_replacement_merge(mode))


def tune_merge(key_type: int, items_per_thread: int, stages: int, out_tiles: int) -> None:
    _check("lsm_tune_merge", lib().lsm_tune_merge(key_type, items_per_thread, stages, out_tiles))


def debug_timeout_probe(limit_ns: int, stream=None) -> None:
    _check("lsm_debug_timeout_probe", lib().lsm_debug_timeout_probe(int(limit_ns), _stream(stream)))


# ---------------------------------------------------------------------------
# a1, a2: partition and stable merge
# ---------------------------------------------------------------------------
def merge_path_partition(A, B, items_per_tile: int, out_ij=None, stream=None):
    m, n = A.numel(), B.numel()
    G = (m + n + items_per_tile - 1) // items_per_tile
    if out_ij is None:
        out_ij = _empty(2 * (G + 1), torch.int64, A.device)
    _check("lsm_merge_path_partition",
           lib().lsm_merge_path_partition(_key_type(A), _ptr(A), m, _ptr(B), n, items_per_tile,
                                          _ptr(out_ij), _stream(stream)))
    return out_ij.view(G + 1, 2)


def merge_stable(A, B, Apay=None, Bpay=None, out_keys=None, out_pay=None, ws=None, stream=None):
    kt = _key_type(A)
    m, n = A.numel(), B.numel()
    dev = A.device
    if out_keys is None:
        out_keys = _empty(m + n, A.dtype, dev)
    if Apay is not None and out_pay is None:
        out_pay = _empty(m + n, torch.uint32, dev)
    if ws is None:
        ws = workspace(LSM_OP_MERGE_STABLE, m, n, dev, kt)
    _check("lsm_merge_stable",
           lib().lsm_merge_stable(kt, _ptr(A), _ptr(Apay), m, _ptr(B), _ptr(Bpay), n,
                                  _ptr(out_keys), _ptr(out_pay), _ptr(ws), ws.numel(),
                                  _stream(stream)))
    return out_keys, out_pay


def merge_sort(keys, pay=None, out_keys=None, out_pay=None, ws=None, stream=None):
    kt = _key_type(keys)
    N = keys.numel()
    dev = keys.device
    if out_keys is None:
        out_keys = _empty(N, keys.dtype, dev)
    if pay is not None and out_pay is None:
        out_pay = _empty(N, torch.uint32, dev)
    if ws is None:
        ws = workspace(LSM_OP_MERGE_SORT, N, 0, dev, kt)
    _check("lsm_merge_sort",
           lib().lsm_merge_sort(kt, _ptr(keys), _ptr(pay), N, _ptr(out_keys), _ptr(out_pay),
                                _ptr(ws), ws.numel(), _stream(stream)))
    return out_keys, out_pay


# ---------------------------------------------------------------------------
# a3 - a5: replacement merge
# ---------------------------------------------------------------------------
def collision_mark(A, B, C=None, lb_B=None, ws=None, stream=None):
    m, n = A.numel(), B.numel()
    dev = A.device
    if C is None:
        C = _empty((m + 31) // 32, torch.uint32, dev)
    if lb_B is None:
        lb_B = _empty(n, torch.uint32, dev)
    if ws is None:
        ws = workspace(LSM_OP_COLLISION_MARK, m, n, dev)
    _check("lsm_collision_mark",
           lib().lsm_collision_mark(_ptr(A), m, _ptr(B), n, _ptr(C), _ptr(lb_B), _ptr(ws),
                                    ws.numel(), _stream(stream)))
    return C, lb_B


class Bytes:
    """A CSR byte column on the device: arena (uint8, padded so that it stays
    readable to the next multiple of 8 bytes) and offsets (uint64[count+1])."""

    def __init__(self, arena, off):
        self.arena, self.off = arena, off

    @property
    def count(self):
        return self.off.numel() - 1

    @staticmethod
    def from_numpy(arena: np.ndarray, off: np.ndarray, device):
        size = int(len(arena))
        padded = np.zeros((size + 7) // 8 * 8 + 8, dtype=np.uint8)
        padded[:size] = arena
        return Bytes(torch.from_numpy(padded).to(device),
                     torch.from_numpy(np.ascontiguousarray(off, dtype=np.uint64)).to(device))

    def _c(self):
        return _Bytes(_ptr(self.arena), _ptr(self.off))


def validate_sorted(keys, strict: bool, d_first=None, stream=None):
    """lsm_validate_sorted: d_first (device int64[1]) = the first t whose pair
    (t, t+1) breaks the order, or -1; a violation also records
    LSM_ERR_UNSORTED in the device status word."""
    if d_first is None:
        d_first = _empty(1, torch.int64, keys.device)
    _check("lsm_validate_sorted",
           lib().lsm_validate_sorted(_key_type(keys), _ptr(keys) if keys.numel() else None,
                                     keys.numel(), int(bool(strict)), _ptr(d_first),
                                     _stream(stream)))
    return d_first


def validate_sorted_str(col: Bytes, strict: bool, arena_bytes=None, d_first=None, stream=None):
    """lsm_validate_sorted_str over a CSR byte column (arena_bytes defaults to
    the arena's readable length)."""
    if d_first is None:
        d_first = _empty(1, torch.int64, col.off.device)
    if arena_bytes is None:
        arena_bytes = col.arena.numel()
    c = col._c()
    _check("lsm_validate_sorted_str",
           lib().lsm_validate_sorted_str(ctypes.byref(c), col.count, int(arena_bytes),
                                         int(bool(strict)), _ptr(d_first), _stream(stream)))
    return d_first


def collision_mark_str(A: Bytes, B: Bytes, C=None, lb_B=None, ws=None, stream=None):
    m, n = A.count, B.count
    dev = A.off.device
    if C is None:
        C = _empty((m + 31) // 32, torch.uint32, dev)
    if lb_B is None:
        lb_B = _empty(n, torch.uint32, dev)
    if ws is None:
        ws = workspace(LSM_OP_COLLISION_MARK_STR, m, n, dev)
    a, b = A._c(), B._c()
    _check("lsm_collision_mark_str",
           lib().lsm_collision_mark_str(ctypes.byref(a), m, ctypes.byref(b), n, _ptr(C), _ptr(lb_B),
                                        _ptr(ws), ws.numel(), _stream(stream)))
    return C, lb_B


def collision_mark_str_prefix(A: Bytes, B: Bytes, C=None, lb_B=None, prefixA=None, prefixB=None,
                              ws=None, stream=None):
    """lsm_collision_mark_str_prefix: the string collision mark, and the key
    prefix tables (uint64[2 count] per source) that FcInput can carry.
    Returns (C, lb_B, prefixA, prefixB)."""
    m, n = A.count, B.count
    dev = A.off.device
    if C is None:
        C = _empty((m + 31) // 32, torch.uint32, dev)
    if lb_B is None:
        lb_B = _empty(n, torch.uint32, dev)
    if prefixA is None:
        prefixA = _empty(max(2 * m, 2), torch.uint64, dev)
    if prefixB is None:
        prefixB = _empty(max(2 * n, 2), torch.uint64, dev)
    if ws is None:
        ws = workspace(LSM_OP_COLLISION_MARK_STR, m, n, dev)
    a, b = A._c(), B._c()
    _check("lsm_collision_mark_str_prefix",
           lib().lsm_collision_mark_str_prefix(ctypes.byref(a), m, ctypes.byref(b), n, _ptr(C),
                                               _ptr(lb_B), _ptr(prefixA), _ptr(prefixB), _ptr(ws),
                                               ws.numel(), _stream(stream)))
    return C, lb_B, prefixA, prefixB


def replacement_merge_str(A: Bytes, B: Bytes, C=None, lb_B=None, prefixA=None, prefixB=None,
                          dir_=None, d_total=None, refs=None, ord_A=None, ord_B=None, d_count=None,
                          ws=None, stream=None, want_lb=True, want_prefix=True):
    """The whole replacement merge for string keys in one call
    (lsm_replacement_merge_str). Returns (C, lb_B, prefixA, prefixB, dir,
    d_total, refs, ord_A, ord_B, d_count); lb_B (want_lb=False) and the
    prefix tables (want_prefix=False) are None when not asked for."""
    m, n = A.count, B.count
    dev = A.off.device
    if C is None:
        C = _empty(max((m + 31) // 32, 4), torch.uint32, dev)
    if lb_B is None and want_lb:
        lb_B = _empty(max(n, 1), torch.uint32, dev)
    if prefixA is None and want_prefix:
        prefixA = _empty(max(2 * m, 2), torch.uint64, dev)
    if prefixB is None and want_prefix:
        prefixB = _empty(max(2 * n, 2), torch.uint64, dev)
    if dir_ is None:
        dir_ = _empty(3 * (m // 512 + 1), torch.uint32, dev)
    if d_total is None:
        d_total = _empty(1, torch.int64, dev)
    if refs is None:
        refs = _empty(max(m + n, 1), torch.uint32, dev)
    if ord_A is None:
        ord_A = _empty(max(m, 1), torch.uint32, dev)
    if ord_B is None:
        ord_B = _empty(max(n, 1), torch.uint32, dev)
    if d_count is None:
        d_count = _empty(1, torch.int64, dev)
    if ws is None:
        ws = workspace(LSM_OP_REPLACEMENT_MERGE_STR, m, n, dev)
    a, b = A._c(), B._c()
    _check("lsm_replacement_merge_str",
           lib().lsm_replacement_merge_str(
               ctypes.byref(a), m, ctypes.byref(b), n, _ptr(C) if m else None,
               _ptr(lb_B) if (n and lb_B is not None) else None,
               _ptr(prefixA) if prefixA is not None else None,
               _ptr(prefixB) if prefixB is not None else None, _ptr(dir_), _ptr(d_total),
               _ptr(refs), _ptr(ord_A) if m else None, _ptr(ord_B) if n else None, _ptr(d_count),
               _ptr(ws), ws.numel(), _stream(stream)))
    return C, lb_B, prefixA, prefixB, dir_, d_total, refs, ord_A, ord_B, d_count


def rank_build(C, m: int, dir_=None, d_total=None, ws=None, stream=None):
    dev = C.device
    if dir_ is None:
        dir_ = _empty(3 * (m // 512 + 1), torch.uint32, dev)
    if d_total is None:
        d_total = _empty(1, torch.int64, dev)
    if ws is None:
        ws = workspace(LSM_OP_RANK_BUILD, m, 0, dev)
    _check("lsm_rank_build",
           lib().lsm_rank_build(_ptr(C) if m else None, m, _ptr(dir_), _ptr(d_total), _ptr(ws),
                                ws.numel(), _stream(stream)))
    return dir_, d_total


def rank_build_noalloc(C, m: int, dir_=None, d_total=None, stream=None):
    """lsm_rank_build_noalloc: rank_build whose scratch is a static device
    array inside the library (m <= 2^29 - 1; calls on one device must not
    overlap). Outputs not passed in are allocated here by torch; the C entry
    point itself allocates nothing."""
    dev = C.device
    if dir_ is None:
        dir_ = _empty(3 * (m // 512 + 1), torch.uint32, dev)
    if d_total is None:
        d_total = _empty(1, torch.int64, dev)
    _check("lsm_rank_build_noalloc",
           lib().lsm_rank_build_noalloc(_ptr(C) if m else None, m, _ptr(dir_), _ptr(d_total),
                                        _stream(stream)))
    return dir_, d_total


def rank2048_build(C, m: int, dir_=None, epochs=None, d_total=None, ws=None, stream=None):
    dev = C.device
    if dir_ is None:
        dir_ = _empty(m // 2048 + 1, torch.uint64, dev)
    if epochs is None:
        epochs = _empty(m // (1 << 32) + 1, torch.uint64, dev)
    if d_total is None:
        d_total = _empty(1, torch.int64, dev)
    if ws is None:
        ws = workspace(LSM_OP_RANK2048_BUILD, m, 0, dev)
    _check("lsm_rank2048_build",
           lib().lsm_rank2048_build(_ptr(C), m, _ptr(dir_), _ptr(epochs), _ptr(d_total), _ptr(ws),
                                    ws.numel(), _stream(stream)))
    return dir_, epochs, d_total


def rank2048_query(C, dir_, epochs, m: int, pos, out=None, stream=None):
    if out is None:
        out = _empty(pos.numel(), torch.uint64, pos.device)
    _check("lsm_rank2048_query",
           lib().lsm_rank2048_query(_ptr(C), _ptr(dir_), _ptr(epochs), m, _ptr(pos), pos.numel(),
                                    _ptr(out), _stream(stream)))
    return out


def rank_query(C, dir_, m: int, pos, out=None, stream=None):
    q = pos.numel()
    if out is None:
        out = _empty(q, torch.uint32, pos.device)
    _check("lsm_rank_query",
           lib().lsm_rank_query(_ptr(C) if m else None, _ptr(dir_), m, _ptr(pos), q, _ptr(out),
                                _stream(stream)))
    return out


def replacement_merge_compact(m: int, n: int, C, dir_, lb_B, refs=None, ord_A=None, ord_B=None,
                              d_count=None, ws=None, stream=None):
    dev = dir_.device
    if refs is None:
        refs = _empty(max(m + n, 1), torch.uint32, dev)
    if ord_A is None:
        ord_A = _empty(m, torch.uint32, dev)
    if ord_B is None:
        ord_B = _empty(n, torch.uint32, dev)
    if d_count is None:
        d_count = _empty(1, torch.int64, dev)
    if ws is None:
        ws = workspace(LSM_OP_REPLACEMENT_COMPACT, m, n, dev)
    _check("lsm_replacement_merge_compact",
           lib().lsm_replacement_merge_compact(m, n, _ptr(C) if m else None, _ptr(dir_),
                                               _ptr(lb_B) if n else None, _ptr(refs),
                                               _ptr(ord_A) if m else None, _ptr(ord_B) if n else None,
                                               _ptr(d_count), _ptr(ws), ws.numel(), _stream(stream)))
    return refs, ord_A, ord_B, d_count


def replacement_merge(A, B, C=None, lb_B=None, dir_=None, d_total=None, refs=None,
                      ord_A=None, ord_B=None, d_count=None, ws=None, stream=None, want_lb=True):
    """The whole path in one call (lsm_replacement_merge). Returns (C, lb_B,
    dir, d_total, refs, ord_A, ord_B, d_count); with want_lb=False and no
    lb_B given the lower bounds are not written and lb_B is None."""
    m, n = A.numel(), B.numel()
    dev = A.device
    if C is None:
        C = _empty(max((m + 31) // 32, 4), torch.uint32, dev)
    if lb_B is None and want_lb:
        lb_B = _empty(n, torch.uint32, dev)
    if dir_ is None:
        dir_ = _empty(3 * (m // 512 + 1), torch.uint32, dev)
    if d_total is None:
        d_total = _empty(1, torch.int64, dev)
    if refs is None:
        refs = _empty(max(m + n, 1), torch.uint32, dev)
    if ord_A is None:
        ord_A = _empty(m, torch.uint32, dev)
    if ord_B is None:
        ord_B = _empty(n, torch.uint32, dev)
    if d_count is None:
        d_count = _empty(1, torch.int64, dev)
    if ws is None:
        ws = workspace(LSM_OP_REPLACEMENT_MERGE, m, n, dev)
    _check("lsm_replacement_merge",
           lib().lsm_replacement_merge(
               _ptr(A) if m else None, m, _ptr(B) if n else None, n, _ptr(C) if m else None,
               _ptr(lb_B) if (n and lb_B is not None) else None, _ptr(dir_), _ptr(d_total),
               _ptr(refs), _ptr(ord_A) if m else None, _ptr(ord_B) if n else None, _ptr(d_count),
               _ptr(ws), ws.numel(), _stream(stream)))
    return C, lb_B, dir_, d_total, refs, ord_A, ord_B, d_count


def replacement_merge_fused(A, B, C=None, lb_B=None, dir_=None, d_total=None, refs=None,
                            ord_A=None, ord_B=None, d_count=None, ws=None, stream=None):
    """Returns (C, lb_B, dir, d_total, refs, ord_A, ord_B, d_count)."""
    m, n = A.numel(), B.numel()
    dev = A.device
    if C is None:
        C = _empty(max((m + 31) // 32, 4), torch.uint32, dev)
    if lb_B is None:
        lb_B = _empty(n, torch.uint32, dev)
    if dir_ is None:
        dir_ = _empty(3 * (m // 512 + 1), torch.uint32, dev)
    if d_total is None:
        d_total = _empty(1, torch.int64, dev)
    if refs is None:
        refs = _empty(max(m + n, 1), torch.uint32, dev)
    if ord_A is None:
        ord_A = _empty(m, torch.uint32, dev)
    if ord_B is None:
        ord_B = _empty(n, torch.uint32, dev)
    if d_count is None:
        d_count = _empty(1, torch.int64, dev)
    if ws is None:
        ws = workspace(LSM_OP_REPLACEMENT_FUSED, m, n, dev)
    _check("lsm_replacement_merge_fused",
           lib().lsm_replacement_merge_fused(
               _ptr(A) if m else None, m, _ptr(B) if n else None, n, _ptr(C) if m else None,
               _ptr(lb_B) if n else None, _ptr(dir_), _ptr(d_total), _ptr(refs),
               _ptr(ord_A) if m else None, _ptr(ord_B) if n else None, _ptr(d_count), _ptr(ws),
               ws.numel(), _stream(stream)))
    return C, lb_B, dir_, d_total, refs, ord_A, ord_B, d_count


def replacement_direct_scatter(A, B, C, dir_, lb_B, refs=None, ord_A=None, ord_B=None,
                               d_count=None, stream=None):
    m, n = A.numel(), B.numel()
    dev = dir_.device
    if refs is None:
        refs = _empty(max(m + n, 1), torch.uint32, dev)
    if ord_A is None:
        ord_A = _empty(m, torch.uint32, dev)
    if ord_B is None:
        ord_B = _empty(n, torch.uint32, dev)
    if d_count is None:
        d_count = _empty(1, torch.int64, dev)
    _check("lsm_replacement_direct_scatter",
           lib().lsm_replacement_direct_scatter(
               _ptr(A) if m else None, m, _ptr(B) if n else None, n, _ptr(C) if m else None,
               _ptr(dir_), _ptr(lb_B) if n else None, _ptr(refs), _ptr(ord_A) if m else None,
               _ptr(ord_B) if n else None, _ptr(d_count), _stream(stream)))
    return refs, ord_A, ord_B, d_count


def replacement_merge_compact_rank2048(m: int, n: int, C, dir_, epochs, lb_B, refs=None,
                                       ord_A=None, ord_B=None, d_count=None, ws=None, stream=None):
    dev = dir_.device
    if refs is None:
        refs = _empty(max(m + n, 1), torch.uint32, dev)
    if ord_A is None:
        ord_A = _empty(m, torch.uint32, dev)
    if ord_B is None:
        ord_B = _empty(n, torch.uint32, dev)
    if d_count is None:
        d_count = _empty(1, torch.int64, dev)
    if ws is None:
        ws = workspace(LSM_OP_REPLACEMENT_COMPACT, m, n, dev)
    _check("lsm_replacement_merge_compact_rank2048",
           lib().lsm_replacement_merge_compact_rank2048(
               m, n, _ptr(C) if m else None, _ptr(dir_), _ptr(epochs), _ptr(lb_B) if n else None,
               _ptr(refs), _ptr(ord_A) if m else None, _ptr(ord_B) if n else None, _ptr(d_count),
               _ptr(ws), ws.numel(), _stream(stream)))
    return refs, ord_A, ord_B, d_count


def replacement_materialize(A, B, refs, d_count, valA=None, valB=None, tombA=None, tombB=None,
                            out_keys=None, out_vals=None, out_tomb=None, stream=None):
    """lsm_replacement_materialize: the survivors' keys, values (when valA and
    valB are given) and tombstone bits, in merged order, for the first
    d_count[0] refs. Returns (out_keys, out_vals, out_tomb)."""
    m, n = A.numel(), B.numel()
    dev = refs.device
    if out_keys is None:
        out_keys = _empty(max(m + n, 1), A.dtype, dev)
    if out_vals is None and valA is not None:
        out_vals = _empty(max(m + n, 1), torch.uint32, dev)
    if out_tomb is None:
        out_tomb = torch.zeros(max((m + n + 31) // 32, 1), dtype=torch.uint32, device=dev)
    _check("lsm_replacement_materialize",
           lib().lsm_replacement_materialize(_ptr(A) if m else None, _ptr(valA) if m else None,
                                             _ptr(tombA), m, _ptr(B) if n else None,
                                             _ptr(valB) if n else None, _ptr(tombB), n,
                                             _ptr(refs), _ptr(d_count), _ptr(out_keys),
                                             _ptr(out_vals), _ptr(out_tomb), _stream(stream)))
    return out_keys, out_vals, out_tomb


# ---------------------------------------------------------------------------
# a6, a7: front compression
# ---------------------------------------------------------------------------
class FcInput:
    """Keys, values and tombstone bitmaps of both sources, on the device, and
    optionally the key prefix tables from collision_mark_str_prefix."""

    def __init__(self, keyA: Bytes, valA: Bytes, tombA, keyB: Bytes, valB: Bytes, tombB,
                 prefixA=None, prefixB=None):
        self.keyA, self.valA, self.tombA = keyA, valA, tombA
        self.keyB, self.valB, self.tombB = keyB, valB, tombB
        self.prefixA, self.prefixB = prefixA, prefixB

    def _c(self):
        return _FcInput(self.keyA._c(), self.valA._c(), _ptr(self.tombA), self.keyA.count,
                        self.keyB._c(), self.valB._c(), _ptr(self.tombB), self.keyB.count,
                        _ptr(self.prefixA), _ptr(self.prefixB))


def fc_lengths_scan(fc: FcInput, refs, N: int, lcp=None, ctrl=None, rec_bits=None, bit_off=None,
                    ws=None, stream=None):
    dev = fc.keyA.off.device
    if lcp is None:
        lcp = _empty(N, torch.uint32, dev)
    if ctrl is None:
        ctrl = _empty(N, torch.uint32, dev)
    if rec_bits is None:
        rec_bits = _empty(N, torch.uint32, dev)
    if bit_off is None:
        bit_off = _empty(N + 1, torch.uint64, dev)
    if ws is None:
        ws = workspace(LSM_OP_FC_LENGTHS_SCAN, N, 0, dev)
    c = fc._c()
    _check("lsm_fc_lengths_scan",
           lib().lsm_fc_lengths_scan(ctypes.byref(c), _ptr(refs) if N else None, N,
                                     _ptr(lcp) if N else None, _ptr(ctrl) if N else None,
                                     _ptr(rec_bits) if N else None, _ptr(bit_off), _ptr(ws),
                                     ws.numel(), _stream(stream)))
    return lcp, ctrl, rec_bits, bit_off


def fc_emit(fc: FcInput, refs, N: int, lcp, ctrl, bit_off, nwords: int, payload=None, stream=None):
    dev = fc.keyA.off.device
    if payload is None:
        payload = _empty(max(nwords, 1), torch.uint32, dev)
    c = fc._c()
    _check("lsm_fc_emit",
           lib().lsm_fc_emit(ctypes.byref(c), _ptr(refs) if N else None, N,
                             _ptr(lcp) if N else None, _ptr(ctrl) if N else None, _ptr(bit_off),
                             _ptr(payload) if nwords else None, nwords, _stream(stream)))
    return payload


# ---------------------------------------------------------------------------
# f4: byte-profile front compression
# ---------------------------------------------------------------------------
def bytefc_lengths_scan(fc: FcInput, refs, N: int, W: int = 0, lcp=None, ctrl=None,
                        rec_bytes=None, byte_off=None, ws=None, stream=None):
    dev = refs.device
    if lcp is None:
        lcp = _empty(max(N, 1), torch.uint32, dev)
    if ctrl is None:
        ctrl = _empty(max(N, 1), torch.uint32, dev)
    if rec_bytes is None:
        rec_bytes = _empty(max(N, 1), torch.uint32, dev)
    if byte_off is None:
        byte_off = _empty(N + 1, torch.uint64, dev)
    if ws is None:
        ws = workspace(LSM_OP_FC_LENGTHS_SCAN, N, 0, dev)
    c = fc._c()
    _check("lsm_bytefc_lengths_scan",
           lib().lsm_bytefc_lengths_scan(ctypes.byref(c), _ptr(refs), N, W, _ptr(lcp), _ptr(ctrl),
                                         _ptr(rec_bytes), _ptr(byte_off), _ptr(ws), ws.numel(),
                                         _stream(stream)))
    return lcp, ctrl, rec_bytes, byte_off


def bytefc_value_width(fc: FcInput, refs, N: int, d_width=None, stream=None):
    """lsm_bytefc_value_width: device uint64[4] whose element 0 is the common
    encoded value width of the N merged records (1 + the value length when
    every record is present with one length, else 0)."""
    if d_width is None:
        d_width = _empty(4, torch.uint64, refs.device)
    c = fc._c()
    _check("lsm_bytefc_value_width",
           lib().lsm_bytefc_value_width(ctypes.byref(c), _ptr(refs) if N else None, N,
                                        _ptr(d_width), _stream(stream)))
    return d_width


def bytefc_emit(fc: FcInput, refs, N: int, lcp, ctrl, byte_off, nbytes: int, W: int = 0,
                payload=None, stream=None):
    if payload is None:
        payload = _empty(max(nbytes, 1), torch.uint8, refs.device)
    c = fc._c()
    _check("lsm_bytefc_emit",
           lib().lsm_bytefc_emit(ctypes.byref(c), _ptr(refs), N, W, _ptr(lcp), _ptr(ctrl),
                                 _ptr(byte_off), _ptr(payload), nbytes, _stream(stream)))
    return payload


# ---------------------------------------------------------------------------
# f2: Elias-Fano navigation over the record offsets
# ---------------------------------------------------------------------------
def ef_sizes(N: int, U: int):
    """(n, L, lows words, highs words, groups) for N records, last entry U."""
    out = (ctypes.c_int64 * 5)()
    _check("lsm_ef_sizes", lib().lsm_ef_sizes(N, U, out))
    return tuple(int(v) for v in out)


def fc_ef_build(bit_off, N: int, U: int, w: int = 0, lows=None, highs=None, samples=None,
                sparse=None, d_nsparse=None, stream=None):
    """U = bit_off[N] - N w, read by the caller. Returns (lows, highs, samples,
    sparse, d_nsparse); sparse holds n slots, the first d_nsparse of them used."""
    dev = bit_off.device
    n, L, nl, nh, G = ef_sizes(N, U)
    if lows is None:
        lows = _empty(max(nl, 1), torch.uint64, dev)
    if highs is None:
        highs = _empty(nh, torch.uint64, dev)
    if samples is None:
        samples = _empty(2 * G, torch.uint64, dev)
    if sparse is None:
        sparse = _empty(n, torch.uint64, dev)
    if d_nsparse is None:
        d_nsparse = _empty(1, torch.int64, dev)
    _check("lsm_fc_ef_build",
           lib().lsm_fc_ef_build(_ptr(bit_off), N, w, U, _ptr(lows), _ptr(highs), _ptr(samples),
                                 _ptr(sparse), _ptr(d_nsparse), _stream(stream)))
    return lows, highs, samples, sparse, d_nsparse
