"""GPU parity for the Elias-Fano navigation sections (C ABI vs oracle).

Bit-exact: lows, highs, sample pairs, sparse exceptions and their count must
equal the oracle's for the same offsets, here synthetic offset sequences
(the FC tests run the same check on the offsets the length scan produced):
sizes around the 15-record sampling and the 256-entry groups, a common value
width, repeated entries, and groups whose high span is exactly 4095 and 4096
bits (dense and sparse)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from tests.gpu_util import up  # noqa: E402
from tests.test_gpu_fc import check_ef  # noqa: E402


@pytest.fixture(scope="module")
def lsm():
    import lsm_replacement_merge_gb300 as lsm
    lsm.lib()
    lsm.get_device_status(reset=True)
    yield lsm
    assert lsm.get_device_status() == lsm.LSM_OK


def _offsets(rng, N, lo, hi):
    return np.concatenate([[0], np.cumsum(rng.integers(lo, hi, size=N))]).astype(np.uint64)


@pytest.mark.parametrize("N", [0, 1, 14, 15, 16, 29, 30, 31, 3839, 3840, 3841, 61440, 61455,
                               100_000, 1_000_003])
def test_ef_parity(lsm, N):
    rng = np.random.default_rng(N + 7)
    for lo, hi, w in ((3, 400, 0), (40, 60, 40), (1, 2, 1), (100, 100_000, 0)):
        off = _offsets(rng, N, lo, hi)
        check_ef(lsm, up(off), N, off, w)


def test_ef_sparse_threshold(lsm):
    for top in (3840, 3841):
        n = 4001
        x = np.zeros(n, dtype=np.uint64)
        x[1:255] = np.arange(1, 255)
        x[255:] = top
        off = np.concatenate([np.repeat(x[:-1], 15), [x[-1]]]).astype(np.uint64)
        check_ef(lsm, up(off), 15 * (n - 1), off)


def test_ef_many_sparse_groups(lsm):
    # offsets that jump by 2^40 every 300 records: most groups sparse
    N = 200_000
    rng = np.random.default_rng(1)
    steps = rng.integers(5, 50, size=N).astype(np.uint64)
    steps[::300] += np.uint64(1 << 40)
    off = np.concatenate([[0], np.cumsum(steps)]).astype(np.uint64)
    check_ef(lsm, up(off), N, off)


def test_ef_wrong_extent_is_reported(lsm):
    off = np.arange(0, 16 * 100, 16, dtype=np.uint64)
    N = len(off) - 1
    U = int(off[N]) + 1  # not bit_off[N]: recorded, nothing written out of bounds
    lsm.fc_ef_build(up(off), N, U)
    assert lsm.get_device_status(reset=True) == 1   # LSM_ERR_ARG, then cleared
