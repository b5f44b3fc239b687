"""GPU parity for the string-key collision mark (and the key-free compaction
that follows it) against the oracle's string replacement walk, as separate
calls and as the whole path in one call (lsm_replacement_merge_str, whose
string mark also writes the merge bitmap and the compaction's co-ranks)."""
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


def run_str(lsm, s):
    dev = torch.device("cuda:0")
    A = lsm.Bytes.from_numpy(s.A.key_arena, s.A.key_off, dev)
    B = lsm.Bytes.from_numpy(s.B.key_arena, s.B.key_off, dev)
    m, n = A.count, B.count
    if m + n == 0:
        return None
    C, lb = lsm.collision_mark_str(A, B)
    if m == 0:
        C = up(np.zeros(4, np.uint32))
    dir_, _ = lsm.rank_build(C, m)
    refs, ordA, ordB, cnt = lsm.replacement_merge_compact(m, n, C, dir_, lb)
    N = int(cnt.item())
    return down(C)[: (m + 31) // 32], down(lb), down(refs)[:N], down(ordA), down(ordB)


def run_whole_str(lsm, s):
    """lsm_replacement_merge_str: the same outputs in one call, plus the
    directory, R(m), the count and the prefix tables."""
    dev = torch.device("cuda:0")
    A = lsm.Bytes.from_numpy(s.A.key_arena, s.A.key_off, dev)
    B = lsm.Bytes.from_numpy(s.B.key_arena, s.B.key_off, dev)
    m, n = A.count, B.count
    C, lb, pA, pB, dir_, tot, refs, ordA, ordB, cnt = lsm.replacement_merge_str(A, B)
    N = int(cnt.item())
    out = dict(C=down(C)[: (m + 31) // 32], lb=down(lb)[:n], refs=down(refs)[:N],
               ordA=down(ordA)[:m], ordB=down(ordB)[:n], dir=down(dir_), total=int(tot.item()),
               count=N, pA=down(pA)[: 2 * m], pB=down(pB)[: 2 * n])
    if m + n:
        # the prefix tables equal those of the separate mark call
        _, _, qA, qB = lsm.collision_mark_str_prefix(A, B)
        assert np.array_equal(out["pA"], down(qA)[: 2 * m])
        assert np.array_equal(out["pB"], down(qB)[: 2 * n])
    return out


def check(lsm, s):
    r = oracle.replacement_str(s.A.key_arena, s.A.key_off, s.B.key_arena, s.B.key_off)
    got = run_str(lsm, s)
    if got is None:
        assert r.count == 0
    else:
        C, lb, refs, ordA, ordB = got
        assert np.array_equal(C, r.C) and np.array_equal(lb, r.lb_B)
        assert np.array_equal(refs, r.refs)
        assert np.array_equal(ordA, r.ord_A) and np.array_equal(ordB, r.ord_B)
    # the whole path in one call, on the same input
    m = len(s.A.key_off) - 1
    w = run_whole_str(lsm, s)
    assert w["count"] == r.count and w["total"] == m + (len(s.B.key_off) - 1) - r.count
    assert np.array_equal(w["C"], r.C) and np.array_equal(w["lb"], r.lb_B)
    assert np.array_equal(w["refs"], r.refs)
    assert np.array_equal(w["ordA"], r.ord_A) and np.array_equal(w["ordB"], r.ord_B)
    assert np.array_equal(w["dir"], oracle.rank512_dir(r.C, m))


@pytest.mark.parametrize("case", list(_str_cases()))
def test_small_string_cases(lsm, case):
    check(lsm, synth.strings_from_lists(*case))


@pytest.mark.parametrize("seed,count", [(0, 500), (1, 3000), (2, 20000)])
def test_prefix_tree_strings(lsm, seed, count):
    check(lsm, synth.strings(seed=seed, count=count, fanout=8, depth=2, max_suffix=20))


def _stem_lists(seed, count):
    """Keys cut from one random 24-byte stem at every length 0..24, then
    tails of up to 12 bytes over {0, 1, 255}: many pairs agree on their first
    8 or 16 bytes, or differ only by trailing zero bytes, and lengths fall on
    both sides of the 8- and 16-byte word edges."""
    rng = np.random.default_rng(seed)
    stem = bytes(rng.integers(0, 256, size=24).astype(np.uint8))
    alphabet = np.array([0, 1, 255], dtype=np.uint8)
    pool = set()
    while len(pool) < count:
        cut = int(rng.integers(0, 25))
        tail = alphabet[rng.integers(0, 3, size=int(rng.integers(0, 13)))].tobytes()
        pool.add(stem[:cut] + tail)
    keys = sorted(pool)
    pick = rng.permutation(len(keys))
    A = sorted(keys[t] for t in pick[: len(keys) // 2])
    B = sorted(keys[t] for t in pick[len(keys) // 3:])
    return A, B


@pytest.mark.parametrize("seed,count", [(3, 700), (4, 6000)])
def test_keys_sharing_long_prefixes(lsm, seed, count):
    check(lsm, synth.strings_from_lists(*_stem_lists(seed, count)))


def test_keys_with_one_16_byte_prefix(lsm):
    # Every key is one 16-byte stem and an 8-byte big-endian counter: all
    # pairs agree on their first 16 bytes and on their length, so the order
    # comes from bytes 16..23 alone (A holds multiples of 2, B of 3).
    stem = bytes(range(40, 56))
    A = [stem + (2 * i).to_bytes(8, "big") for i in range(3000)]
    B = [stem + (3 * j).to_bytes(8, "big") for j in range(2000)]
    check(lsm, synth.strings_from_lists(A, B))


def test_config_strings_4M(lsm):
    check(lsm, synth.strings())


def test_whole_path_str_without_lower_bounds_or_tables(lsm):
    # lb_B and the prefix tables are optional on the whole path
    st = synth.strings(seed=9, count=5000, fanout=8, depth=2, max_suffix=20)
    dev = torch.device("cuda:0")
    A = lsm.Bytes.from_numpy(st.A.key_arena, st.A.key_off, dev)
    B = lsm.Bytes.from_numpy(st.B.key_arena, st.B.key_off, dev)
    r = oracle.replacement_str(st.A.key_arena, st.A.key_off, st.B.key_arena, st.B.key_off)
    C, lb, pA, pB, dir_, tot, refs, ordA, ordB, cnt = lsm.replacement_merge_str(
        A, B, want_lb=False, want_prefix=False)
    assert lb is None and pA is None and pB is None
    N = int(cnt.item())
    assert N == r.count
    assert np.array_equal(down(refs)[:N], r.refs)
    assert np.array_equal(down(ordA), r.ord_A) and np.array_equal(down(ordB), r.ord_B)
