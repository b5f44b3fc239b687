"""CPU oracle for the merge-path replacement merge -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The GPU library never does, and the two
share no code: this wrapper loads ``oracle.c`` (plain sequential C, compiled
here with gcc) and passes numpy arrays to it.

Each function below names the definition it implements; the C file carries
the full citations. Pins that tie the oracle to the pages (worked examples,
brute force, closed forms, invariants) live in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_build", "liblsmoracle.so")
_lock = threading.Lock()
_lib = None

REF_FROM_B = 0x80000000
ORD_DROPPED = 0xFFFFFFFF


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, portable flags)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared",
                           "-Wall", "-Wextra", "-o", tmp, _SRC])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int64
            U = ctypes.c_uint64
            for name in ("oracle_merge_i32", "oracle_merge_u64"):
                fn = getattr(_lib, name)
                fn.argtypes = [P, P, I, P, P, I, P, P, P]
                fn.restype = None
            for name in ("oracle_mergesort_pass_i32", "oracle_mergesort_pass_u64"):
                fn = getattr(_lib, name)
                fn.argtypes = [P, P, I, I, P, P]
                fn.restype = None
            for name in ("oracle_merge_sort_i32", "oracle_merge_sort_u64"):
                fn = getattr(_lib, name)
                fn.argtypes = [P, P, I, P, P]
                fn.restype = I
            for name in ("oracle_partition_i32", "oracle_partition_u64"):
                fn = getattr(_lib, name)
                fn.argtypes = [P, I, P, I, I, P]
                fn.restype = None
            _lib.oracle_replacement_u64.argtypes = [P, I, P, I, P, P, P, P, P]
            _lib.oracle_replacement_u64.restype = I
            _lib.oracle_replacement_str.argtypes = [P, P, I, P, P, I, P, P, P, P, P]
            _lib.oracle_replacement_str.restype = I
            _lib.oracle_materialize_u64.argtypes = [P, P, P, I, P, P, P, I, P, I, P, P, P]
            _lib.oracle_materialize_u64.restype = None
            _lib.oracle_rank_prefix.argtypes = [P, I, P]
            _lib.oracle_rank_prefix.restype = None
            _lib.oracle_rank512_dir.argtypes = [P, I, P]
            _lib.oracle_rank512_dir.restype = None
            _lib.oracle_rank2048_dir.argtypes = [P, I, P, P]
            _lib.oracle_rank2048_dir.restype = None
            _lib.oracle_rank2048_query.argtypes = [P, P, P, P, I, P]
            _lib.oracle_rank2048_query.restype = None
            _lib.oracle_rank_query.argtypes = [P, I, P, I, P]
            _lib.oracle_rank_query.restype = None
            _lib.oracle_ordinals_formula_u64.argtypes = [P, I, P, I, P, P, P, P]
            _lib.oracle_ordinals_formula_u64.restype = None
            _lib.oracle_fc_encode.argtypes = [P] * 10 + [P, I, P, P, P, P, P, I]
            _lib.oracle_fc_encode.restype = I
            _lib.oracle_fc_decode.argtypes = [P, U, I, P, U, P, P, U, P, P]
            _lib.oracle_fc_decode.restype = I
            _lib.oracle_ef_sizes.argtypes = [I, U, P]
            _lib.oracle_ef_sizes.restype = None
            _lib.oracle_ef_build.argtypes = [P, I, U, P, P, P, P]
            _lib.oracle_ef_build.restype = I
            _lib.oracle_leb128.argtypes = [U, P]
            _lib.oracle_leb128.restype = U
            _lib.oracle_bytefc_encode.argtypes = [P] * 10 + [P, I, U, P, P, P, P, P, I]
            _lib.oracle_bytefc_encode.restype = I
            _lib.oracle_bytefc_decode.argtypes = [P, U, I, U, P, U, P, P, U, P, P]
            _lib.oracle_bytefc_decode.restype = I
            _lib.oracle_eg0_len.argtypes = [U]
            _lib.oracle_eg0_len.restype = U
            _lib.oracle_eg0_bits.argtypes = [U, P]
            _lib.oracle_eg0_bits.restype = U
    return _lib


def _p(a):
    """Pointer to a C-contiguous numpy array (or NULL for None)."""
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be contiguous"
    return a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# Stable merge and co-rank
# --------------------------------------------------------------------------
def merge(A, B, Apay=None, Bpay=None, provenance=False):
    """Two-pointer stable merge, ties to A. Returns (keys, payload|None, prov|None).

    prov[k] = i for A[i], m + j for B[j]."""
    kind = _kind(A)
    A = _c(A, kind)
    B = _c(B, kind)
    m, n = len(A), len(B)
    out = np.empty(m + n, dtype=kind)
    has_pay = Apay is not None
    Apay = _c(Apay, np.uint32)
    Bpay = _c(Bpay, np.uint32)
    out_pay = np.empty(m + n, dtype=np.uint32) if has_pay else None
    prov = np.empty(m + n, dtype=np.int64) if provenance else None
    fn = _load().oracle_merge_i32 if kind == np.int32 else _load().oracle_merge_u64
    fn(_p(A), _p(Apay), m, _p(B), _p(Bpay), n, _p(out), _p(out_pay), _p(prov))
    return out, out_pay, prov


def partition(A, B, items_per_tile):
    """Co-rank (i, j) at k_g = min(g*D, m+n), g = 0..ceil((m+n)/D), by walking
    the merge. Returns an int64 array of shape (G+1, 2)."""
    kind = _kind(A)
    A = _c(A, kind)
    B = _c(B, kind)
    m, n = len(A), len(B)
    D = int(items_per_tile)
    G = (m + n + D - 1) // D
    out = np.empty((G + 1, 2), dtype=np.int64)
    fn = (_load().oracle_partition_i32 if kind == np.int32
          else _load().oracle_partition_u64)
    fn(_p(A), m, _p(B), n, D, _p(out))
    return out


def corank(A, B, k):
    """Number of A elements among the first k merge outputs (0 <= k <= m+n)."""
    if k == 0:
        return 0
    return int(partition(A, B, k)[1, 0])


def merge_sort_pass(keys, width, pay=None):
    """One bottom-up merge sort pass ([CH14] 14.2): adjacent runs of `width`
    merged pairwise, the left run first on ties. Returns (keys, payload|None)."""
    kind = _kind(keys)
    keys = _c(keys, kind)
    n = len(keys)
    pay = _c(pay, np.uint32)
    out = np.empty(n, dtype=kind)
    out_pay = np.empty(n, dtype=np.uint32) if pay is not None else None
    fn = (_load().oracle_mergesort_pass_i32 if kind == np.int32
          else _load().oracle_mergesort_pass_u64)
    fn(_p(keys), _p(pay), n, int(width), _p(out), _p(out_pay))
    return out, out_pay


def merge_sort(keys, pay=None):
    """Bottom-up merge sort ([CH14] 14.2), widths 1, 2, 4, ... Returns
    (keys, payload|None, passes)."""
    kind = _kind(keys)
    keys = _c(keys, kind)
    n = len(keys)
    pay = _c(pay, np.uint32)
    out = np.empty(n, dtype=kind)
    out_pay = np.empty(n, dtype=np.uint32) if pay is not None else None
    fn = (_load().oracle_merge_sort_i32 if kind == np.int32
          else _load().oracle_merge_sort_u64)
    passes = fn(_p(keys), _p(pay), n, _p(out), _p(out_pay))
    if passes < 0:
        raise MemoryError("oracle merge sort: scratch allocation failed")
    return out, out_pay, int(passes)


def _kind(A):
    dt = np.asarray(A).dtype
    if dt == np.int32:
        return np.int32
    if dt == np.uint64:
        return np.uint64
    raise TypeError("oracle keys must be int32 or uint64, got %s" % dt)


# --------------------------------------------------------------------------
# Replacement merge, rank, ordinals
# --------------------------------------------------------------------------
class Replacement:
    """Outputs of the sequential replacement walk."""

    def __init__(self, refs, C, lb_B, ord_A, ord_B, count):
        self.refs, self.C, self.lb_B = refs, C, lb_B
        self.ord_A, self.ord_B, self.count = ord_A, ord_B, count


def replacement_u64(A, B):
    A = _c(A, np.uint64)
    B = _c(B, np.uint64)
    m, n = len(A), len(B)
    refs = np.empty(m + n, dtype=np.uint32)
    C = np.zeros(max((m + 31) // 32, 0), dtype=np.uint32)
    lb_B = np.empty(n, dtype=np.uint32)
    ord_A = np.empty(m, dtype=np.uint32)
    ord_B = np.empty(n, dtype=np.uint32)
    cnt = _load().oracle_replacement_u64(_p(A), m, _p(B), n, _p(refs), _p(C),
                                         _p(lb_B), _p(ord_A), _p(ord_B))
    return Replacement(refs[:cnt].copy(), C, lb_B, ord_A, ord_B, int(cnt))


def materialize_u64(A, valA, tombA, B, valB, tombB, refs):
    """Keys, values and tombstone bits of the survivors refs names, in order
    (oracle_materialize_u64). A tombstone bitmap may be None."""
    A, B = _c(A, np.uint64), _c(B, np.uint64)
    valA, valB = _c(valA, np.uint32), _c(valB, np.uint32)
    tA, tB = _c(tombA, np.uint32), _c(tombB, np.uint32)
    refs = _c(refs, np.uint32)
    N = len(refs)
    keys = np.empty(N, dtype=np.uint64)
    vals = np.empty(N, dtype=np.uint32)
    tomb = np.zeros((N + 31) // 32, dtype=np.uint32)
    _load().oracle_materialize_u64(_p(A), _p(valA), _p(tA), len(A), _p(B), _p(valB), _p(tB),
                                   len(B), _p(refs), N, _p(keys), _p(vals), _p(tomb))
    return keys, vals, tomb


def replacement_str(Aarena, Aoff, Barena, Boff):
    Aarena = _c(Aarena, np.uint8)
    Barena = _c(Barena, np.uint8)
    Aoff = _c(Aoff, np.uint64)
    Boff = _c(Boff, np.uint64)
    m, n = len(Aoff) - 1, len(Boff) - 1
    refs = np.empty(m + n, dtype=np.uint32)
    C = np.zeros(max((m + 31) // 32, 0), dtype=np.uint32)
    lb_B = np.empty(n, dtype=np.uint32)
    ord_A = np.empty(m, dtype=np.uint32)
    ord_B = np.empty(n, dtype=np.uint32)
    cnt = _load().oracle_replacement_str(_p(Aarena), _p(Aoff), m, _p(Barena), _p(Boff), n,
                                         _p(refs), _p(C), _p(lb_B), _p(ord_A), _p(ord_B))
    return Replacement(refs[:cnt].copy(), C, lb_B, ord_A, ord_B, int(cnt))


def rank_prefix(C, m):
    C = _c(C, np.uint32)
    R = np.empty(m + 1, dtype=np.uint32)
    _load().oracle_rank_prefix(_p(C), m, _p(R))
    return R


def rank512_dir(C, m):
    C = _c(C, np.uint32)
    dir_ = np.empty(3 * (m // 512 + 1), dtype=np.uint32)
    _load().oracle_rank512_dir(_p(C), m, _p(dir_))
    return dir_


def rank2048_dir(C, m):
    """The rank2048 layout: (dir uint64[floor(m/2048)+1], epochs uint64[floor(m/2^32)+1])."""
    C = _c(C, np.uint32)
    dir_ = np.empty(m // 2048 + 1, dtype=np.uint64)
    epochs = np.empty(m // (1 << 32) + 1, dtype=np.uint64)
    _load().oracle_rank2048_dir(_p(C), m, _p(dir_), _p(epochs))
    return dir_, epochs


def rank2048_query(C, dir_, epochs, pos):
    """R(p) for each p by the rank2048 query procedure (uint64)."""
    C = _c(C, np.uint32)
    dir_ = _c(dir_, np.uint64)
    epochs = _c(epochs, np.uint64)
    pos = _c(pos, np.uint64)
    out = np.empty(len(pos), dtype=np.uint64)
    _load().oracle_rank2048_query(_p(C), _p(dir_), _p(epochs), _p(pos), len(pos), _p(out))
    return out


def rank_query(C, m, pos):
    C = _c(C, np.uint32)
    pos = _c(pos, np.uint32)
    out = np.empty(len(pos), dtype=np.uint32)
    _load().oracle_rank_query(_p(C), m, _p(pos), len(pos), _p(out))
    return out


def ordinals_formula_u64(A, B):
    """Path (a): independent lower bounds and the closed-form ordinals.
    Returns (C, lb_B, ord_A, ord_B)."""
    A = _c(A, np.uint64)
    B = _c(B, np.uint64)
    m, n = len(A), len(B)
    C = np.zeros(max((m + 31) // 32, 0), dtype=np.uint32)
    lb_B = np.empty(n, dtype=np.uint32)
    ord_A = np.empty(m, dtype=np.uint32)
    ord_B = np.empty(n, dtype=np.uint32)
    _load().oracle_ordinals_formula_u64(_p(A), m, _p(B), n, _p(C), _p(lb_B),
                                        _p(ord_A), _p(ord_B))
    return C, lb_B, ord_A, ord_B


# --------------------------------------------------------------------------
# Front compression
# --------------------------------------------------------------------------
def eg0_len(x: int) -> int:
    """E(x) as the oracle computes it."""
    return int(_load().oracle_eg0_len(x))


def eg0_bits(x: int) -> str:
    """The oracle's EG0 code word for x, as a '0'/'1' string."""
    words = np.zeros(8, dtype=np.uint32)
    nb = int(_load().oracle_eg0_bits(x, _p(words)))
    return "".join(str((int(words[t // 32]) >> (31 - t % 32)) & 1) for t in range(nb))


class FC:
    def __init__(self, lcp, ctrl, rec_bits, bit_off, payload, total_bits):
        self.lcp, self.ctrl, self.rec_bits = lcp, ctrl, rec_bits
        self.bit_off, self.payload, self.total_bits = bit_off, payload, total_bits


def fc_encode(keysA, valsA, tombA, keysB, valsB, tombB, refs, with_payload=True):
    """Sequential FC encoder. keysX / valsX are (arena uint8, offsets uint64);
    tombX is a uint32 bitmap or None. Returns an FC record."""
    refs = _c(refs, np.uint32)
    N = len(refs)
    ka, koa = _c(keysA[0], np.uint8), _c(keysA[1], np.uint64)
    kb, kob = _c(keysB[0], np.uint8), _c(keysB[1], np.uint64)
    va, voa = _c(valsA[0], np.uint8), _c(valsA[1], np.uint64)
    vb, vob = _c(valsB[0], np.uint8), _c(valsB[1], np.uint64)
    ta, tb = _c(tombA, np.uint32), _c(tombB, np.uint32)
    lcp = np.empty(N, dtype=np.uint32)
    ctrl = np.empty(N, dtype=np.uint32)
    rec = np.empty(N, dtype=np.uint32)
    off = np.empty(N + 1, dtype=np.uint64)
    lib = _load()
    args = [_p(ka), _p(koa), _p(va), _p(voa), _p(ta), _p(kb), _p(kob), _p(vb), _p(vob), _p(tb),
            _p(refs), N]
    total = lib.oracle_fc_encode(*args, _p(lcp), _p(ctrl), _p(rec), _p(off), None, 0)
    if total < 0:
        raise ValueError("FC record field exceeds 32 bits")
    payload = None
    if with_payload:
        nwords = (int(total) + 31) // 32
        payload = np.zeros(max(nwords, 1), dtype=np.uint32)[:nwords]
        t2 = lib.oracle_fc_encode(*args, None, None, None, None, _p(payload) if nwords else None,
                                  nwords)
        assert t2 == total
    return FC(lcp, ctrl, rec, off, payload, int(total))


def leb128(x):
    """Textbook unsigned LEB128 bytes of x."""
    out = np.zeros(10, dtype=np.uint8)
    n = _load().oracle_leb128(int(x), _p(out))
    return out[:n].tolist()


def bytefc_encode(keysA, valsA, tombA, keysB, valsB, tombB, refs, W=0, with_payload=True):
    """Sequential byte-profile FC encoder ([BP]). Returns an FC record whose
    rec_bits / bit_off / payload / total_bits hold record bytes, byte offsets,
    payload bytes (uint8) and the payload length in bytes."""
    refs = _c(refs, np.uint32)
    N = len(refs)
    ka, koa = _c(keysA[0], np.uint8), _c(keysA[1], np.uint64)
    kb, kob = _c(keysB[0], np.uint8), _c(keysB[1], np.uint64)
    va, voa = _c(valsA[0], np.uint8), _c(valsA[1], np.uint64)
    vb, vob = _c(valsB[0], np.uint8), _c(valsB[1], np.uint64)
    ta, tb = _c(tombA, np.uint32), _c(tombB, np.uint32)
    lcp = np.empty(N, dtype=np.uint32)
    ctrl = np.empty(N, dtype=np.uint32)
    rec = np.empty(N, dtype=np.uint32)
    off = np.empty(N + 1, dtype=np.uint64)
    lib = _load()
    args = [_p(ka), _p(koa), _p(va), _p(voa), _p(ta), _p(kb), _p(kob), _p(vb), _p(vob), _p(tb),
            _p(refs), N, int(W)]
    total = lib.oracle_bytefc_encode(*args, _p(lcp), _p(ctrl), _p(rec), _p(off), None, 0)
    if total < 0:
        raise ValueError("byte FC: a field exceeds 32 bits or a record breaks the common width")
    payload = None
    if with_payload:
        payload = np.zeros(max(int(total), 1), dtype=np.uint8)[:int(total)]
        t2 = lib.oracle_bytefc_encode(*args, None, None, None, None,
                                      _p(payload) if total else None, int(total))
        assert t2 == total
    return FC(lcp, ctrl, rec, off, payload, int(total))


def bytefc_value_width(valsA_off, tombA, valsB_off, tombB, refs):
    """The common encoded value width of the merged records ([BP] "Pipeline":
    the width is detected before sizing; 17 = a one-byte presence tag and 16
    value bytes): 1 + L when every record refs names is present and every one
    of their values has L bytes, else 0 (0 for no records). Plain loop over
    the records."""
    offs = (np.asarray(valsA_off, np.int64), np.asarray(valsB_off, np.int64))
    tombs = (tombA, tombB)
    length = None
    if len(refs) == 0:
        return 0
    for r in np.asarray(refs, np.uint32).tolist():
        src, idx = r >> 31, r & 0x7FFFFFFF
        t = tombs[src]
        if t is not None and len(t) and (int(t[idx // 32]) >> (idx % 32)) & 1:
            return 0
        L = int(offs[src][idx + 1] - offs[src][idx])
        if length is None:
            length = L
        elif L != length:
            return 0
    return 1 + length


def bytefc_decode(payload, N, W, key_cap, val_cap):
    """Independent byte-profile decoder. Returns (keys (arena, off), vals (arena, off), tombs)."""
    payload = _c(payload, np.uint8)
    key_ar = np.zeros(max(key_cap, 1), dtype=np.uint8)
    val_ar = np.zeros(max(val_cap, 1), dtype=np.uint8)
    key_off = np.empty(N + 1, dtype=np.uint64)
    val_off = np.empty(N + 1, dtype=np.uint64)
    tomb = np.zeros(max((N + 31) // 32, 1), dtype=np.uint32)
    rc = _load().oracle_bytefc_decode(_p(payload) if len(payload) else None, len(payload), N,
                                      int(W), _p(key_ar), key_cap, _p(key_off), _p(val_ar),
                                      val_cap, _p(val_off), _p(tomb))
    if rc != len(payload):
        raise ValueError("byte FC decode failed (%d)" % rc)
    return (key_ar, key_off), (val_ar, val_off), tomb


class EF:
    """Elias-Fano navigation sections over sampled record offsets."""

    def __init__(self, n, L, lows, highs, samples, sparse):
        self.n, self.L = n, L
        self.lows, self.highs, self.samples, self.sparse = lows, highs, samples, sparse


def ef_sizes(N, U):
    """(n, L, lows words, highs words, groups) for N records and last entry U."""
    out = np.empty(5, dtype=np.int64)
    _load().oracle_ef_sizes(int(N), int(U), _p(out))
    return tuple(int(v) for v in out)


def ef_build(bit_off, N, w=0):
    """EF sections over bit_off[0, 15, 30, ...] and bit_off[N], minus w per ordinal."""
    bit_off = _c(bit_off, np.uint64)
    U = int(bit_off[N]) - int(N) * int(w)
    n, L, nl, nh, G = ef_sizes(N, U)
    lows = np.zeros(max(nl, 1), dtype=np.uint64)
    highs = np.zeros(max(nh, 1), dtype=np.uint64)
    samples = np.zeros(2 * G, dtype=np.uint64)
    sparse = np.zeros(max(n, 1), dtype=np.uint64)
    ns = _load().oracle_ef_build(_p(bit_off), int(N), int(w), _p(lows), _p(highs), _p(samples),
                                 _p(sparse))
    return EF(n, L, lows[:nl], highs[:nh], samples, sparse[:ns])


def fc_decode(payload, total_bits, N, key_cap, val_cap):
    """Independent decoder. Returns (keys (arena, off), vals (arena, off), tomb bitmap)."""
    payload = _c(payload, np.uint32)
    key_ar = np.zeros(max(key_cap, 1), dtype=np.uint8)
    val_ar = np.zeros(max(val_cap, 1), dtype=np.uint8)
    key_off = np.empty(N + 1, dtype=np.uint64)
    val_off = np.empty(N + 1, dtype=np.uint64)
    tomb = np.zeros(max((N + 31) // 32, 1), dtype=np.uint32)
    rc = _load().oracle_fc_decode(_p(payload) if len(payload) else None, total_bits, N,
                                  _p(key_ar), key_cap, _p(key_off), _p(val_ar), val_cap,
                                  _p(val_off), _p(tomb))
    if rc < 0:
        raise ValueError("FC payload did not parse (code %d)" % rc)
    if rc != total_bits:
        raise ValueError("FC payload has %d trailing bits" % (total_bits - rc))
    return (key_ar[:int(key_off[-1])], key_off), (val_ar[:int(val_off[-1])], val_off), tomb
