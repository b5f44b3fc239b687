"""GPU parity for the string-key collision mark (and the key-free compaction
that follows it) against the oracle's string replacement walk."""
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


def check(lsm, s):
    got = run_str(lsm, s)
    r = oracle.replacement_str(s.A.key_arena, s.A.key_off, s.B.key_arena, s.B.key_off)
    if got is None:
        assert r.count == 0
        return
    C, lb, refs, ordA, ordB = got
    assert np.array_equal(C, r.C) and np.array_equal(lb, r.lb_B)
    assert np.array_equal(refs, r.refs)
    assert np.array_equal(ordA, r.ord_A) and np.array_equal(ordB, r.ord_B)


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
