"""GPU parity for the byte-profile front compression (C ABI vs oracle).

Bit-exact: byte LCPs, controls, record lengths, byte offsets and every
payload byte must equal the oracle's for the same merged records: the
hand-derived records, edge keys (empty, proper prefixes, long shared
prefixes, long values), the prefix-tree strings, the 4M + 4M string
workload and the common width 17 (a presence tag and sixteen value bytes)."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from tests.gpu_util import down, up  # noqa: E402
from tests.test_gpu_fc import _prefix_table, device_input, gpu_refs  # noqa: E402


@pytest.fixture(scope="module")
def lsm():
    import lsm_replacement_merge_gb300 as lsm
    lsm.lib()
    lsm.get_device_status(reset=True)
    yield lsm
    assert lsm.get_device_status() == lsm.LSM_OK


def check_bytefc(lsm, s, W=0):
    fc = device_input(lsm, s)
    if fc.keyA.count + fc.keyB.count == 0:
        return
    refs, N = gpu_refs(lsm, fc)
    r = oracle.replacement_str(s.A.key_arena, s.A.key_off, s.B.key_arena, s.B.key_off)
    assert N == r.count and np.array_equal(down(refs)[:N], r.refs)
    exp = oracle.bytefc_encode((s.A.key_arena, s.A.key_off), (s.A.val_arena, s.A.val_off),
                               s.A.tomb if len(s.A.tomb) else None,
                               (s.B.key_arena, s.B.key_off), (s.B.val_arena, s.B.val_off),
                               s.B.tomb if len(s.B.tomb) else None, r.refs, W=W)
    lcp, ctrl, rec, off = lsm.bytefc_lengths_scan(fc, refs, N, W)
    assert np.array_equal(down(lcp)[:N], exp.lcp)
    assert np.array_equal(down(ctrl)[:N], exp.ctrl)
    assert np.array_equal(down(rec)[:N], exp.rec_bits)
    assert np.array_equal(down(off), exp.bit_off)
    # the same lengths with the key prefix tables (the LCP from their first
    # 16 bytes), built on the host from their definition
    # (an empty source needs no table)
    if fc.keyA.count or fc.keyB.count:
        fc2 = device_input(lsm, s)
        if fc.keyA.count:
            fc2.prefixA = up(_prefix_table(s.A.key_arena, s.A.key_off))
        if fc.keyB.count:
            fc2.prefixB = up(_prefix_table(s.B.key_arena, s.B.key_off))
        lcp2, ctrl2, rec2, off2 = lsm.bytefc_lengths_scan(fc2, refs, N, W)
        assert np.array_equal(down(lcp2)[:N], exp.lcp)
        assert np.array_equal(down(ctrl2)[:N], exp.ctrl)
        assert np.array_equal(down(rec2)[:N], exp.rec_bits)
        assert np.array_equal(down(off2), exp.bit_off)
    total = exp.total_bits
    payload = lsm.bytefc_emit(fc, refs, N, lcp, ctrl, off, total + 5, W,
                              payload=torch.full((total + 5,), 0xEE, dtype=torch.uint8,
                                                 device="cuda"))
    got = down(payload)
    assert np.array_equal(got[:total], exp.payload)
    assert (got[total:] == 0xEE).all()  # nothing past the payload is written


def test_hand_derived(lsm, golden):
    g = golden("bytefc_hand_derived.txt")
    s = synth.strings_from_lists([b"ab", b"ac"], [b"ac"], [None, b"\xff"], [b"\xff"])
    check_bytefc(lsm, s)
    s = synth.strings_from_lists([b"A"], [], [bytes(range(16))], [])
    check_bytefc(lsm, s, W=17)
    assert len(g["w17_payload"]) == 20


def test_edge_keys(lsm):
    check_bytefc(lsm, synth.strings_from_lists(
        [b"", b"a", b"ab", b"abc" * 60, b"b"], [b"a", b"abd", b"c" * 300],
        [None, b"", b"x" * 200, b"y", None], [b"1", None, b""]))
    check_bytefc(lsm, synth.strings_from_lists([bytes([7]) * k for k in range(1, 70)], [],
                                               [None] * 69, []))


@pytest.mark.parametrize("seed,count", [(1, 2000), (2, 30000)])
def test_prefix_tree(lsm, seed, count):
    check_bytefc(lsm, synth.strings(seed=seed, count=count))


def test_common_width_17(lsm):
    rng = np.random.default_rng(4)
    keysA = sorted({bytes(rng.integers(0, 256, size=int(rng.integers(1, 20)), dtype=np.uint8))
                    for _ in range(3000)})
    keysB = sorted(set(keysA[::3]) | {bytes([200 + t % 50]) * (t % 7 + 1) for t in range(40)})
    valsA = [bytes(rng.integers(0, 256, size=16, dtype=np.uint8)) for _ in keysA]
    valsB = [bytes(rng.integers(0, 256, size=16, dtype=np.uint8)) for _ in keysB]
    check_bytefc(lsm, synth.strings_from_lists(keysA, keysB, valsA, valsB), W=17)


def test_config_strings_4M(lsm):
    check_bytefc(lsm, synth.strings())


def _width_inputs():
    rng = np.random.default_rng(9)
    keysA = sorted({bytes(rng.integers(0, 256, size=int(rng.integers(1, 12)), dtype=np.uint8))
                    for _ in range(5000)})
    v = lambda L: bytes(rng.integers(0, 256, size=L, dtype=np.uint8))  # noqa: E731
    # A varies: 16-byte values, some 5-byte values and some tombstones
    valsA = [None if t % 11 == 3 else v(5 if t % 7 == 2 else 16) for t in range(len(keysA))]
    odd = [k for k, x in zip(keysA, valsA) if x is None or len(x) != 16]
    # B replaces every odd A record (and adds fresh keys) with 16-byte values
    keysB = sorted(set(odd) | set(keysA[::17]) | {b"\xff" * (t % 5 + 13) for t in range(9)})
    valsB = [v(16) for _ in keysB]
    yield synth.strings_from_lists(keysA, keysB, valsA, valsB), 17
    # one B tombstone survives: no common width
    valsB2 = list(valsB)
    valsB2[len(valsB2) // 2] = None
    yield synth.strings_from_lists(keysA, keysB, valsA, valsB2), 0
    # one B value of 15 bytes: no common width
    valsB3 = list(valsB)
    valsB3[3] = v(15)
    yield synth.strings_from_lists(keysA, keysB, valsA, valsB3), 0


@pytest.mark.parametrize("case", range(3))
def test_value_width_detected(lsm, case):
    s, want = list(_width_inputs())[case]
    fc = device_input(lsm, s)
    refs, N = gpu_refs(lsm, fc)
    r = oracle.replacement_str(s.A.key_arena, s.A.key_off, s.B.key_arena, s.B.key_off)
    exp = oracle.bytefc_value_width(s.A.val_off, s.A.tomb, s.B.val_off, s.B.tomb, r.refs)
    assert exp == want
    W = int(down(lsm.bytefc_value_width(fc, refs, N))[0])
    assert W == exp
    # sized and emitted with the detected width, bit-exact against the oracle
    check_bytefc(lsm, s, W=W)


def test_width_errors_are_reported(lsm):
    # W = 17 over records that do not all have it: LSM_ERR_ARG in the device
    # status, for a surviving tombstone and for a 15-byte value
    for case in (1, 2):
        s, _ = list(_width_inputs())[case]
        fc = device_input(lsm, s)
        refs, N = gpu_refs(lsm, fc)
        lsm.get_device_status(reset=True)
        lsm.bytefc_lengths_scan(fc, refs, N, 17)
        assert lsm.get_device_status(reset=True) == lsm.LSM_ERR_ARG
        # the same through the key prefix tables (the flat lengths kernel)
        fc.prefixA = up(_prefix_table(s.A.key_arena, s.A.key_off)) if fc.keyA.count else None
        fc.prefixB = up(_prefix_table(s.B.key_arena, s.B.key_off)) if fc.keyB.count else None
        lsm.bytefc_lengths_scan(fc, refs, N, 17)
        assert lsm.get_device_status(reset=True) == lsm.LSM_ERR_ARG
    # an emit whose offsets do not match its records: reported, and nothing is
    # written past the buffer the caller gave
    s, _ = list(_width_inputs())[0]
    fc = device_input(lsm, s)
    refs, N = gpu_refs(lsm, fc)
    lcp, ctrl, rec, off = lsm.bytefc_lengths_scan(fc, refs, N, 17)
    assert lsm.get_device_status(reset=True) == lsm.LSM_OK
    bad = down(off).copy()
    bad[1:] -= 1  # every record one byte too short
    bad_off = up(bad)
    total = int(down(off)[N])
    buf = torch.full((total + 64,), 0xEE, dtype=torch.uint8, device="cuda")
    lsm.bytefc_emit(fc, refs, N, lcp, ctrl, bad_off, total, 17, payload=buf)
    assert lsm.get_device_status(reset=True) == lsm.LSM_ERR_ARG
    assert (down(buf)[total:] == 0xEE).all()
