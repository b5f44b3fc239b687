"""GPU parity for the front-compression pass: lengths, bit offsets and the
word-owned payload emit, against the oracle's sequential encoder (bit-exact),
on refs produced by the GPU string replacement merge."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from tests.gpu_util import down, up  # noqa: E402
from tests.test_oracle_pins import _str_cases  # noqa: E402


@pytest.fixture(scope="module")
def lsm():
    import lsm_replacement_merge_gb300 as lsm
    lsm.lib()
    lsm.get_device_status(reset=True)
    yield lsm
    assert lsm.get_device_status() == lsm.LSM_OK


def device_input(lsm, s):
    dev = torch.device("cuda:0")
    def tomb(side):
        return up(side.tomb) if len(side.tomb) else None
    fc = lsm.FcInput(lsm.Bytes.from_numpy(s.A.key_arena, s.A.key_off, dev),
                     lsm.Bytes.from_numpy(s.A.val_arena, s.A.val_off, dev), tomb(s.A),
                     lsm.Bytes.from_numpy(s.B.key_arena, s.B.key_off, dev),
                     lsm.Bytes.from_numpy(s.B.val_arena, s.B.val_off, dev), tomb(s.B))
    return fc


def gpu_refs(lsm, fc):
    m, n = fc.keyA.count, fc.keyB.count
    C, lb = lsm.collision_mark_str(fc.keyA, fc.keyB)
    if m == 0:
        C = up(np.zeros(4, np.uint32))
    dir_, _ = lsm.rank_build(C, m)
    refs, _, _, cnt = lsm.replacement_merge_compact(m, n, C, dir_, lb)
    return refs, int(cnt.item())


def _prefix_table(arena, off):
    """Each key's bytes 0..7 and 8..15 as big-endian words, zero past its end
    (the definition the prefix tables follow), as uint64[2 count]."""
    off = np.asarray(off, dtype=np.int64)
    count = len(off) - 1
    if count <= 0:
        return np.zeros(0, np.uint64)
    lens = off[1:] - off[:-1]
    idx = off[:-1, None] + np.arange(16)[None, :]
    src = np.asarray(arena, dtype=np.uint8)
    safe = np.minimum(idx, max(len(src) - 1, 0))
    rows = np.where(np.arange(16)[None, :] < lens[:, None], src[safe] if len(src) else 0, 0)
    rows = np.ascontiguousarray(rows.astype(np.uint8))
    return rows.view(">u8").astype(np.uint64).reshape(-1)


def check_fc(lsm, s, extra_words=3):
    fc = device_input(lsm, s)
    if fc.keyA.count + fc.keyB.count == 0:
        return
    refs, N = gpu_refs(lsm, fc)
    r = oracle.replacement_str(s.A.key_arena, s.A.key_off, s.B.key_arena, s.B.key_off)
    assert N == r.count and np.array_equal(down(refs)[:N], r.refs)
    exp = oracle.fc_encode((s.A.key_arena, s.A.key_off), (s.A.val_arena, s.A.val_off),
                           s.A.tomb if len(s.A.tomb) else None,
                           (s.B.key_arena, s.B.key_off), (s.B.val_arena, s.B.val_off),
                           s.B.tomb if len(s.B.tomb) else None, r.refs)
    lcp, ctrl, rec, off = lsm.fc_lengths_scan(fc, refs, N)
    assert np.array_equal(down(lcp), exp.lcp)
    assert np.array_equal(down(ctrl), exp.ctrl)
    assert np.array_equal(down(rec), exp.rec_bits)
    assert np.array_equal(down(off), exp.bit_off)
    total = int(down(off[N:N + 1])[0])
    assert total == exp.total_bits
    nwords = (total + 31) // 32 + extra_words
    payload = lsm.fc_emit(fc, refs, N, lcp, ctrl, off, nwords)
    got = down(payload)[:nwords]
    assert np.array_equal(got[:len(exp.payload)], exp.payload)
    assert not got[len(exp.payload):].any()        # words past the payload are zero
    # the same through the key prefix tables that the string mark writes
    m, n = fc.keyA.count, fc.keyB.count
    C2, lb2, pA, pB = lsm.collision_mark_str_prefix(fc.keyA, fc.keyB)
    if m:
        assert np.array_equal(down(C2)[: (m + 31) // 32], r.C)
        assert np.array_equal(down(pA)[: 2 * m], _prefix_table(s.A.key_arena, s.A.key_off))
    if n:
        assert np.array_equal(down(lb2), r.lb_B)
        assert np.array_equal(down(pB)[: 2 * n], _prefix_table(s.B.key_arena, s.B.key_off))
    fcp = lsm.FcInput(fc.keyA, fc.valA, fc.tombA, fc.keyB, fc.valB, fc.tombB, pA, pB)
    lcp2, ctrl2, rec2, off2 = lsm.fc_lengths_scan(fcp, refs, N)
    assert np.array_equal(down(lcp2), exp.lcp)
    assert np.array_equal(down(ctrl2), exp.ctrl)
    assert np.array_equal(down(rec2), exp.rec_bits)
    assert np.array_equal(down(off2), exp.bit_off)
    payload2 = lsm.fc_emit(fcp, refs, N, lcp2, ctrl2, off2, nwords)
    assert np.array_equal(down(payload2)[:nwords], got)
    # the Elias-Fano navigation over the scanned offsets
    check_ef(lsm, off, N, exp.bit_off)
    return exp


def check_ef(lsm, d_off, N, want_off, w=0):
    """EF sections built on the GPU from d_off (device) against the oracle's
    built from want_off (the oracle's own offsets, equal to d_off)."""
    want = oracle.ef_build(want_off, N, w)
    U = int(want_off[N]) - N * w
    lows, highs, samples, sparse, ns = lsm.fc_ef_build(d_off, N, U, w)
    n, L, nl, nh, G = lsm.ef_sizes(N, U)
    assert (n, L) == (want.n, want.L)
    assert np.array_equal(down(lows)[:nl], want.lows)
    assert np.array_equal(down(highs)[:nh], want.highs)
    assert np.array_equal(down(samples), want.samples)
    k = int(ns.item())
    assert k == len(want.sparse) and np.array_equal(down(sparse)[:k], want.sparse)


def test_hand_derived_words(lsm, golden):
    g = golden("fc_hand_derived.txt")
    for name, val in (("one_tomb", None), ("one_empty", b"")):
        s = synth.strings_from_lists([bytes(g[name + "_key"])], [], [val], [])
        exp = check_fc(lsm, s, extra_words=0)
        assert exp.payload.tolist() == g[name + "_words"]
    s = synth.strings_from_lists([b"ab", b"ac"], [], [None, b"\xff"], [])
    assert check_fc(lsm, s, extra_words=5).payload.tolist() == g["two_words"]


@pytest.mark.parametrize("case", list(_str_cases()))
def test_small_cases(lsm, case):
    ka, kb = case
    rng = np.random.default_rng(len(ka) * 31 + len(kb))
    va = [None if rng.random() < 0.3 else bytes(rng.integers(0, 256, rng.integers(0, 5)).astype(np.uint8))
          for _ in ka]
    vb = [None if rng.random() < 0.3 else bytes(rng.integers(0, 256, rng.integers(0, 5)).astype(np.uint8))
          for _ in kb]
    check_fc(lsm, synth.strings_from_lists(ka, kb, va, vb))


def test_long_keys_and_values(lsm):
    rng = np.random.default_rng(7)
    base = bytes(rng.integers(0, 256, 300).astype(np.uint8))
    ka = sorted({base[:rng.integers(0, 300)] + bytes(rng.integers(0, 256, rng.integers(0, 40)).astype(np.uint8))
                 for _ in range(400)})
    kb = sorted(set(ka[::3]) | {base + b"\x00" * t for t in range(5)})
    va = [bytes(rng.integers(0, 256, rng.integers(0, 200)).astype(np.uint8)) for _ in ka]
    vb = [None if t % 4 == 0 else b"v" * (t % 37) for t in range(len(kb))]
    check_fc(lsm, synth.strings_from_lists(ka, kb, va, vb))


@pytest.mark.parametrize("seed,count", [(0, 200), (1, 5000), (2, 60000)])
def test_prefix_tree(lsm, seed, count):
    check_fc(lsm, synth.strings(seed=seed, count=count, fanout=8, depth=3, max_suffix=30))


def test_config_strings_4M(lsm):
    """The full string workload: 4,000,000 + 4,000,000 keys."""
    check_fc(lsm, synth.strings())


def test_many_tiny_records_per_run(lsm):
    # 3-byte keys sharing long prefixes, mostly tombstones: a dozen bits per
    # record, so one run of 8192 payload words holds ~20,000 records and its
    # metadata is staged in many chunks; words straddle chunk boundaries.
    ka = [int(x).to_bytes(3, "big") for x in range(0, 120000, 2)]
    kb = [int(x).to_bytes(3, "big") for x in range(1, 120000, 6)]
    va = [None if x % 7 else b"" for x in range(len(ka))]
    vb = [None if x % 5 else b"\x01" for x in range(len(kb))]
    check_fc(lsm, synth.strings_from_lists(ka, kb, va, vb))


def test_records_spanning_many_runs(lsm):
    # values of 40-100 KB: a record covers one or more runs of 8192 words, so
    # whole runs are composed from one record's value bytes
    rng = np.random.default_rng(21)
    ka = [b"k%04d" % t for t in range(0, 40, 2)]
    kb = [b"k%04d" % t for t in range(1, 40, 4)]
    va = [bytes(rng.integers(0, 256, int(rng.integers(40000, 100000))).astype(np.uint8)) if t % 3 == 0
          else b"x" for t in range(len(ka))]
    vb = [bytes(rng.integers(0, 256, 70001).astype(np.uint8)) if t % 2 else None
          for t in range(len(kb))]
    check_fc(lsm, synth.strings_from_lists(ka, kb, va, vb))
