"""Seeded synthetic inputs for the merge-path replacement merge.

This module draws, sorts and packs inputs; it holds none of the method's
arithmetic (no merge, no co-rank, no dedup, no rank, no encoding). Both the
CPU oracle and the GPU library consume exactly the arrays it returns. Every
generator uses numpy's PCG64 with a fixed seed, so the same call gives the
same bytes on every machine.

Workloads (the sizes are the defaults; every generator also takes smaller
sizes for the parity tests):

  merge_i32      sorted int32 keys drawn from [0, 4096) (heavy ties), each
                 with a uint32 payload holding its source index in A||B
  merge_u64      sorted uniform 64-bit keys, m = n = 2^26, same payload
  replace_u64    strictly sorted unique uint64 keys: A = 12,000,000 older
                 keys, B = 4,000,000 newer keys of which 25% are drawn from
                 A; uint32 values; 5% of B are tombstones
  replace_skewed A = 2^24 - 1 unique keys; B = 65,536 keys clustered in 64
                 windows of 1024 consecutive A positions, half of each
                 window's B keys drawn from A and half fresh keys inside it
  sort_u64       2^27 uniform 64-bit keys in input order, each with a uint32
                 payload holding its input position (the element count and
                 layout of the 2^26 + 2^26 merge's output)
  sort_i32       int32 keys uniform in a range (heavy ties when narrow), same
                 payload
  strings        4,000,000 unique byte-string keys per input built from a
                 prefix tree (fanout 16, depth 4, 2-byte edge labels) plus a
                 random 0-56 byte suffix; 20% of B's keys are A keys; values
                 of 0-16 bytes, 5% tombstones per input
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _raw_u64(rng: np.random.Generator, size: int) -> np.ndarray:
    return rng.bit_generator.random_raw(size).astype(np.uint64, copy=False)


# ---------------------------------------------------------------------------
# Stable-merge inputs
# ---------------------------------------------------------------------------
@dataclass
class MergeInput:
    A: np.ndarray
    B: np.ndarray
    Apay: np.ndarray
    Bpay: np.ndarray


def _source_index_payload(m: int, n: int):
    return (np.arange(m, dtype=np.uint32), (m + np.arange(n, dtype=np.int64)).astype(np.uint32))


def merge_i32(seed: int = 1, m: int = 4096, n: int = 4096, hi: int = 4096) -> MergeInput:
    """int32 keys uniform in [0, hi), sorted; payload = source index in A||B."""
    rng = _rng(seed)
    A = np.sort(rng.integers(0, hi, size=m, dtype=np.int32))
    B = np.sort(rng.integers(0, hi, size=n, dtype=np.int32))
    Apay, Bpay = _source_index_payload(m, n)
    return MergeInput(A, B, Apay, Bpay)


def merge_u64(seed: int = 2, m: int = 1 << 26, n: int = 1 << 26) -> MergeInput:
    """Uniform 64-bit keys, sorted; payload = source index in A||B."""
    rng = _rng(seed)
    A = np.sort(_raw_u64(rng, m))
    B = np.sort(_raw_u64(rng, n))
    Apay, Bpay = _source_index_payload(m, n)
    return MergeInput(A, B, Apay, Bpay)


# ---------------------------------------------------------------------------
# Merge-sort inputs (unsorted)
# ---------------------------------------------------------------------------
@dataclass
class SortInput:
    keys: np.ndarray   # unsorted keys
    pay: np.ndarray    # uint32 payload = input position


def sort_u64(seed: int = 6, N: int = 1 << 27) -> SortInput:
    """Uniform 64-bit keys in input order; payload = input position."""
    rng = _rng(seed)
    return SortInput(_raw_u64(rng, N), np.arange(N, dtype=np.uint32))


def sort_i32(seed: int = 7, N: int = 4096, lo: int = 0, hi: int = 4096) -> SortInput:
    """int32 keys uniform in [lo, hi) in input order (ties when the range is
    narrow); payload = input position."""
    rng = _rng(seed)
    return SortInput(rng.integers(lo, hi, size=N, dtype=np.int32), np.arange(N, dtype=np.uint32))


# ---------------------------------------------------------------------------
# Replacement-merge inputs (unique keys within each input)
# ---------------------------------------------------------------------------
@dataclass
class ReplaceInput:
    A: np.ndarray            # uint64[m], strictly increasing (older)
    B: np.ndarray            # uint64[n], strictly increasing (newer)
    valA: np.ndarray         # uint32[m]
    valB: np.ndarray         # uint32[n]
    tombB: np.ndarray        # uint32[ceil(n/32)] bitmap, bit j = B_j is a tombstone
    n_shared: int = 0        # how many B keys were drawn from A


def _sorted_unique(x: np.ndarray) -> np.ndarray:
    x = np.sort(x)
    if len(x) < 2:
        return x
    return x[np.concatenate([[True], x[1:] != x[:-1]])]


def _unique_pool(rng, count: int) -> np.ndarray:
    """`count` distinct uniform 64-bit keys, sorted."""
    pool = _sorted_unique(_raw_u64(rng, count))
    while len(pool) < count:
        pool = _sorted_unique(np.concatenate([pool, _raw_u64(rng, count - len(pool))]))
    return pool[:count]


def _bitmap(bits_set: np.ndarray, length: int) -> np.ndarray:
    words = np.zeros(max((length + 31) // 32, 0), dtype=np.uint32)
    if len(bits_set):
        np.bitwise_or.at(words, bits_set // 32, (np.uint32(1) << (bits_set % 32).astype(np.uint32)))
    return words


def replace_u64(seed: int = 3, m: int = 12_000_000, n: int = 4_000_000,
                shared_frac: float = 0.25, tomb_frac: float = 0.05) -> ReplaceInput:
    rng = _rng(seed)
    n_shared = min(int(round(n * shared_frac)), m)
    n_fresh = n - n_shared
    pool = _unique_pool(rng, m + n_fresh)
    perm = rng.permutation(m + n_fresh)
    A = np.sort(pool[perm[:m]])
    fresh = pool[perm[m:]]
    shared = A[rng.choice(m, size=n_shared, replace=False)] if n_shared else A[:0]
    B = np.sort(np.concatenate([fresh, shared]))
    valA = rng.integers(0, 2**32, size=m, dtype=np.uint32)
    valB = rng.integers(0, 2**32, size=n, dtype=np.uint32)
    n_tomb = int(round(n * tomb_frac))
    tomb_idx = np.sort(rng.choice(n, size=n_tomb, replace=False)) if n_tomb else np.zeros(0, np.int64)
    return ReplaceInput(A, B, valA, valB, _bitmap(tomb_idx.astype(np.int64), n), n_shared)


def replace_skewed(seed: int = 4, m: int = (1 << 24) - 1, windows: int = 64,
                   window: int = 1024, per_window_shared: int = 512,
                   per_window_fresh: int = 512, tomb_frac: float = 0.05) -> ReplaceInput:
    """B clustered in `windows` random windows of `window` consecutive A positions."""
    rng = _rng(seed)
    A = np.sort(_unique_pool(rng, m))
    slot = 2 * window
    n_slots = (m - window) // slot
    assert n_slots >= windows, "A too small for the requested windows"
    slots = np.sort(rng.choice(n_slots, size=windows, replace=False))
    starts = slots * slot + rng.integers(0, window, size=windows)
    parts = []
    n_shared = 0
    for s in starts:
        s = int(s)
        shared = A[s + rng.choice(window, size=per_window_shared, replace=False)]
        lo, hi = int(A[s]), int(A[s + window - 1])
        fresh = np.zeros(0, dtype=np.uint64)
        while len(fresh) < per_window_fresh:
            cand = (lo + 1 + (_raw_u64(rng, 2 * per_window_fresh) % np.uint64(hi - lo - 1))).astype(np.uint64)
            pos = np.searchsorted(A, cand)
            in_a = (pos < m) & (A[np.minimum(pos, m - 1)] == cand)
            fresh = _sorted_unique(np.concatenate([fresh, cand[~in_a]]))
        fresh = rng.permutation(fresh)[:per_window_fresh]
        parts.append(shared)
        parts.append(fresh)
        n_shared += per_window_shared
    B = np.sort(np.concatenate(parts)) if parts else np.zeros(0, np.uint64)
    n = len(B)
    valA = rng.integers(0, 2**32, size=m, dtype=np.uint32)
    valB = rng.integers(0, 2**32, size=n, dtype=np.uint32)
    n_tomb = int(round(n * tomb_frac))
    tomb_idx = np.sort(rng.choice(n, size=n_tomb, replace=False)) if n_tomb else np.zeros(0, np.int64)
    return ReplaceInput(A, B, valA, valB, _bitmap(tomb_idx.astype(np.int64), n), n_shared)


def replace_random_small(seed: int, m: int, n: int, shared: int, universe: int | None = None,
                         tomb_frac: float = 0.05) -> ReplaceInput:
    """Small unique-key inputs over a narrow universe (dense collisions)."""
    rng = _rng(seed)
    if universe is None:
        universe = max(4 * (m + n), 16)
    keys = rng.choice(universe, size=m + (n - shared), replace=False).astype(np.uint64)
    A = np.sort(keys[:m])
    fresh = keys[m:]
    sh = A[rng.choice(m, size=shared, replace=False)] if shared else A[:0]
    B = np.sort(np.concatenate([fresh, sh]))
    valA = rng.integers(0, 2**32, size=m, dtype=np.uint32)
    valB = rng.integers(0, 2**32, size=n, dtype=np.uint32)
    n_tomb = int(round(n * tomb_frac))
    tomb_idx = np.sort(rng.choice(n, size=n_tomb, replace=False)) if n_tomb else np.zeros(0, np.int64)
    return ReplaceInput(A, B, valA, valB, _bitmap(tomb_idx.astype(np.int64), n), shared)


# ---------------------------------------------------------------------------
# String-key inputs (CSR arenas: bytes + uint64 offsets[count+1])
# ---------------------------------------------------------------------------
@dataclass
class StringSide:
    key_arena: np.ndarray    # uint8
    key_off: np.ndarray      # uint64[count + 1]
    val_arena: np.ndarray    # uint8
    val_off: np.ndarray      # uint64[count + 1]
    tomb: np.ndarray         # uint32 bitmap, bit t = record t is a tombstone

    @property
    def count(self) -> int:
        return len(self.key_off) - 1

    def key(self, t: int) -> bytes:
        return bytes(self.key_arena[int(self.key_off[t]):int(self.key_off[t + 1])])

    def value(self, t: int):
        if (int(self.tomb[t // 32]) >> (t % 32)) & 1:
            return None
        return bytes(self.val_arena[int(self.val_off[t]):int(self.val_off[t + 1])])


@dataclass
class StringInput:
    A: StringSide
    B: StringSide
    n_shared: int = 0
    max_key: int = 64


def _lex_order(padded: np.ndarray, lengths: np.ndarray) -> np.ndarray:
    """Row order of zero-padded byte strings by (bytes, length): unsigned
    lexicographic order with a proper prefix first."""
    width = padded.shape[1]
    assert width % 8 == 0
    words = padded.reshape(len(padded), width // 8, 8)[:, :, ::-1].copy().view(np.uint64)[:, :, 0]
    cols = [lengths] + [words[:, w] for w in range(width // 8 - 1, -1, -1)]
    return np.lexsort(cols)


def _dedupe_sorted(padded, lengths):
    if len(lengths) == 0:
        return padded, lengths
    same = np.all(padded[1:] == padded[:-1], axis=1) & (lengths[1:] == lengths[:-1])
    keep = np.concatenate([[True], ~same])
    return padded[keep], lengths[keep]


def _pack(padded: np.ndarray, lengths: np.ndarray):
    mask = np.arange(padded.shape[1])[None, :] < lengths[:, None]
    arena = padded[mask]
    off = np.zeros(len(lengths) + 1, dtype=np.uint64)
    np.cumsum(lengths, out=off[1:])
    return np.ascontiguousarray(arena, dtype=np.uint8), off


def _values(rng, count: int, max_len: int, tomb_frac: float):
    lengths = rng.integers(0, max_len + 1, size=count).astype(np.int64)
    n_tomb = int(round(count * tomb_frac))
    tomb_idx = np.sort(rng.choice(count, size=n_tomb, replace=False)) if n_tomb else np.zeros(0, np.int64)
    lengths[tomb_idx] = 0
    off = np.zeros(count + 1, dtype=np.uint64)
    np.cumsum(lengths, out=off[1:])
    total = int(off[-1])
    arena = rng.bit_generator.random_raw((total + 7) // 8).view(np.uint8)[:total].copy()
    return arena, off, _bitmap(tomb_idx.astype(np.int64), count)


def strings(seed: int = 5, count: int = 4_000_000, shared_frac: float = 0.20,
            fanout: int = 16, depth: int = 4, label_bytes: int = 2,
            max_suffix: int = 56, max_value: int = 16, tomb_frac: float = 0.05,
            min_suffix: int = 0) -> StringInput:
    """Prefix-tree string keys; A and B each hold `count` unique keys."""
    rng = _rng(seed)
    prefix_len = depth * label_bytes
    width = prefix_len + max_suffix
    width8 = (width + 7) // 8 * 8
    # edge labels: each internal node has `fanout` distinct random labels
    n_leaves = fanout ** depth
    leaf_prefix = np.zeros((n_leaves, prefix_len), dtype=np.uint8)
    for level in range(depth):
        nodes = fanout ** level
        lab = np.empty((nodes, fanout), dtype=np.int64)
        for v in range(nodes):
            lab[v] = rng.choice(1 << (8 * label_bytes), size=fanout, replace=False)
        # leaf index -> its ancestor at this level and child slot
        leaf = np.arange(n_leaves)
        anc = leaf // fanout ** (depth - level)
        slot = (leaf // fanout ** (depth - level - 1)) % fanout
        val = lab[anc, slot]
        for b in range(label_bytes):
            leaf_prefix[:, level * label_bytes + b] = (val >> (8 * (label_bytes - 1 - b))) & 0xFF
    n_shared = int(round(count * shared_frac))
    need = 2 * count - n_shared
    padded = np.zeros((0, width8), dtype=np.uint8)
    lengths = np.zeros(0, dtype=np.int64)
    while len(lengths) < need:
        extra = need - len(lengths) + need // 50 + 16
        leaves = rng.integers(0, n_leaves, size=extra)
        suf = rng.integers(min_suffix, max_suffix + 1, size=extra)
        rows = np.zeros((extra, width8), dtype=np.uint8)
        rows[:, :prefix_len] = leaf_prefix[leaves]
        rnd = rng.bit_generator.random_raw((extra * max_suffix + 7) // 8).view(np.uint8)
        rnd = rnd[:extra * max_suffix].reshape(extra, max_suffix)
        keep = np.arange(max_suffix)[None, :] < suf[:, None]
        rows[:, prefix_len:prefix_len + max_suffix] = np.where(keep, rnd, 0)
        padded = np.concatenate([padded, rows])
        lengths = np.concatenate([lengths, prefix_len + suf])
        order = _lex_order(padded, lengths)
        padded, lengths = _dedupe_sorted(padded[order], lengths[order])
    # choose `need` distinct keys at random, then split into A-only, shared, B-only
    pick = np.sort(rng.choice(len(lengths), size=need, replace=False))
    padded, lengths = padded[pick], lengths[pick]
    role = rng.permutation(need)
    a_rows = np.sort(role[:count])
    b_fresh = role[count:]
    b_shared = a_rows[rng.choice(count, size=n_shared, replace=False)]
    b_rows = np.sort(np.concatenate([b_fresh, b_shared]))
    sides = []
    for rows in (a_rows, b_rows):
        arena, off = _pack(padded[rows], lengths[rows])
        varena, voff, tomb = _values(rng, len(rows), max_value, tomb_frac)
        sides.append(StringSide(arena, off, varena, voff, tomb))
    return StringInput(sides[0], sides[1], n_shared, width)


def strings_from_lists(keysA, keysB, valsA=None, valsB=None) -> StringInput:
    """Build a StringInput from explicit sorted byte strings. A value of None
    is a tombstone; missing value lists mean empty values."""
    def side(keys, vals):
        keys = [bytes(k) for k in keys]
        off = np.zeros(len(keys) + 1, dtype=np.uint64)
        off[1:] = np.cumsum([len(k) for k in keys]) if keys else []
        arena = np.frombuffer(b"".join(keys), dtype=np.uint8).copy()
        if vals is None:
            vals = [b""] * len(keys)
        tomb_idx = np.array([t for t, v in enumerate(vals) if v is None], dtype=np.int64)
        vb = [b"" if v is None else bytes(v) for v in vals]
        voff = np.zeros(len(vb) + 1, dtype=np.uint64)
        voff[1:] = np.cumsum([len(v) for v in vb]) if vb else []
        varena = np.frombuffer(b"".join(vb), dtype=np.uint8).copy()
        return StringSide(arena, off, varena, voff, _bitmap(tomb_idx, len(keys)))
    return StringInput(side(keysA, valsA), side(keysB, valsB), 0,
                       max([len(k) for k in list(keysA) + list(keysB)] + [0]))
