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


# ---- the replacement pipeline reading R(i) from the rank2048 directory ------
from tests.test_oracle_pins import REPLACE_CASES  # noqa: E402


def _pipeline_2048(lsm, A, B):
    m, n = len(A), len(B)
    C, lb = lsm.collision_mark(up(A), up(B))
    if m == 0:
        C = torch.zeros(4, dtype=torch.uint32, device="cuda")
    d, e, tot = lsm.rank2048_build(C, m)
    refs, ordA, ordB, cnt = lsm.replacement_merge_compact_rank2048(m, n, C, d, e, lb)
    N = int(cnt.item())
    return dict(C=down(C)[:(m + 31) // 32], dir=down(d), epochs=down(e), total=int(tot.item()),
                refs=down(refs)[:N], ordA=down(ordA), ordB=down(ordB), count=N)


def _check_pipeline(got, A, B):
    r = oracle.replacement_u64(A, B)
    d, e = oracle.rank2048_dir(r.C, len(A))
    assert got["count"] == r.count
    assert np.array_equal(got["C"], r.C)
    assert got["total"] == len(A) + len(B) - r.count
    assert np.array_equal(got["dir"], d) and np.array_equal(got["epochs"], e)
    assert np.array_equal(got["refs"], r.refs)
    assert np.array_equal(got["ordA"], r.ord_A)
    assert np.array_equal(got["ordB"], r.ord_B)


@pytest.mark.parametrize("m,n,shared,universe", [c for c in REPLACE_CASES if c[0] + c[1] > 0] + [
    (20000, 7000, 7000, None), (100000, 100000, 50000, 250000), (300000, 2000, 1000, None),
    (2000, 300000, 2000, None)])
def test_rank2048_pipeline_parity(lsm, m, n, shared, universe):
    inp = synth.replace_random_small(seed=m * 7 + n + shared, m=m, n=n, shared=shared,
                                     universe=universe)
    _check_pipeline(_pipeline_2048(lsm, inp.A, inp.B), inp.A, inp.B)


def test_rank2048_pipeline_replace_12M_4M(lsm):
    inp = synth.replace_u64()
    _check_pipeline(_pipeline_2048(lsm, inp.A, inp.B), inp.A, inp.B)


def test_rank2048_pipeline_skewed_2pow24(lsm):
    inp = synth.replace_skewed()
    _check_pipeline(_pipeline_2048(lsm, inp.A, inp.B), inp.A, inp.B)
