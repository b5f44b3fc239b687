"""GPU parity for the rank2048 directory (C ABI vs oracle), bit-exact.

Every entry, every epoch and R(m) must equal the oracle's; the query must
equal the oracle's query at every position (EOF included) on the maps the
collision-bitmap page asks to probe (all-zero, all-one, sparse, near
31/32/33, 63/64/65, 511/512/513, 2047/2048/2049), on ragged sizes and on a
bitmap the size of the 12M-record replacement's. Past 2^32 bits an all-one
map checks the epochs against the closed form R(p) = p."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from tests.gpu_util import down, up  # noqa: E402


@pytest.fixture(scope="module")
def lsm():
    import lsm_replacement_merge_gb300 as lsm
    lsm.lib()
    lsm.get_device_status(reset=True)
    yield lsm
    assert lsm.get_device_status() == lsm.LSM_OK


def _maps():
    rng = np.random.default_rng(11)
    for m in (0, 1, 31, 32, 33, 63, 64, 65, 511, 512, 513, 2047, 2048, 2049, 4095, 4096, 4097,
              6144, 524287, 524288, 524289, 3_000_017):
        yield m, np.zeros(m, bool)
        yield m, np.ones(m, bool)
        sp = np.zeros(m, bool)
        for p in (0, 31, 32, 33, 63, 64, 65, 511, 512, 513, 2047, 2048, 2049, m - 1):
            if 0 <= p < m:
                sp[p] = True
        yield m, sp
        yield m, rng.random(m) < 0.3


def _pack(bits):
    return synth._bitmap(np.flatnonzero(bits).astype(np.int64), len(bits))


def _check(lsm, C, m):
    d_want, e_want = oracle.rank2048_dir(C, m)
    Cg = up(C) if len(C) else torch.zeros(4, dtype=torch.uint32, device="cuda")
    d, e, tot = lsm.rank2048_build(Cg, m)
    assert np.array_equal(down(d), d_want)
    assert np.array_equal(down(e), e_want)
    pos = np.arange(m + 1, dtype=np.uint64)
    if m > 200_000:
        pos = np.unique(np.concatenate([pos[:5000], pos[-5000:],
                                        np.random.default_rng(m).integers(0, m + 1, 20000)])
                        ).astype(np.uint64)
    want = oracle.rank2048_query(C, d_want, e_want, pos)
    assert int(tot.item()) == int(oracle.rank2048_query(C, d_want, e_want,
                                                        np.array([m], np.uint64))[0])
    got = lsm.rank2048_query(Cg, d, e, m, up(pos))
    assert np.array_equal(down(got), want)


@pytest.mark.parametrize("case", range(len(list(_maps()))))
def test_rank2048_maps(lsm, case):
    m, bits = list(_maps())[case]
    _check(lsm, _pack(bits), m)


def test_rank2048_replacement_sized_bitmap(lsm):
    # the collision bitmap of the 12M + 4M replacement: 12,000,000 bits, 1M set
    m = 12_000_000
    idx = np.sort(np.random.default_rng(3).choice(m, 1_000_000, replace=False))
    _check(lsm, synth._bitmap(idx.astype(np.int64), m), m)


def test_rank2048_epochs_past_2pow32(lsm):
    m = (1 << 32) + 5000
    nwords = (m + 31) // 32
    C32 = torch.full((nwords,), -1, dtype=torch.int32, device="cuda")
    C32[-1] = (1 << (m % 32)) - 1
    C = C32.view(torch.uint32)
    d, e, tot = lsm.rank2048_build(C, m)
    assert down(e).tolist() == [0, 1 << 32] and int(tot.item()) == m
    b = np.arange(m // 2048 + 1, dtype=np.uint64)
    start = 2048 * b
    rel = start & np.uint64(0xFFFFFFFF)
    pops = [np.minimum(np.maximum(np.int64(m) - (start.astype(np.int64) + 512 * r), 0), 512)
            .astype(np.uint64) for r in range(3)]
    want = rel | (pops[0] << np.uint64(32)) | (pops[1] << np.uint64(42)) | (pops[2] << np.uint64(52))
    assert np.array_equal(down(d), want)
    pos = np.array([0, 1, 511, 512, 2047, 2048, (1 << 32) - 1, 1 << 32, (1 << 32) + 1,
                    (1 << 32) + 1535, (1 << 32) + 2048, (1 << 32) + 4999, m], dtype=np.uint64)
    assert np.array_equal(down(lsm.rank2048_query(C, d, e, m, up(pos))), pos)
