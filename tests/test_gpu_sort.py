"""GPU parity for the bottom-up merge sort (C ABI vs oracle).

Bit-exact: keys and payloads must equal the oracle's element by element; the
payload is each key's input position, so equal keys must keep input order.
Sizes span the block-sort tile (256 threads x 11 items = 2816 elements), so
that the CTA-local passes, several global passes and ragged last runs all
run. At the full workload size the result is checked by the properties that
define the stable sort: ascending keys, a payload that is a permutation of
the input positions, each key equal to the input key its payload names, and
increasing positions among equal keys."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from tests.gpu_util import down, up  # noqa: E402

TILE = 256 * 11


@pytest.fixture(scope="module")
def lsm():
    import lsm_replacement_merge_gb300 as lsm
    lsm.lib()
    lsm.get_device_status(reset=True)
    yield lsm
    assert lsm.get_device_status() == lsm.LSM_OK


def test_worked_example(lsm, golden):
    g = golden("mergesort_chapter14.txt")
    for dt in (np.int32, np.uint64):
        x = np.array(g["input"], dt)
        keys, _ = lsm.merge_sort(up(x))
        assert down(keys).tolist() == g["after_width_4"]
        keys, pay = lsm.merge_sort(up(x), up(np.arange(len(x), dtype=np.uint32)))
        assert down(keys).tolist() == g["after_width_4"]
        assert x[down(pay)].tolist() == g["after_width_4"]


SIZES = [1, 2, 11, 12, 255 * 11 + 3, TILE - 1, TILE, TILE + 1, 2 * TILE, 3 * TILE + 5,
         8 * TILE, 9 * TILE - 1, 100_003, 1_000_003]


@pytest.mark.parametrize("N", SIZES)
def test_sort_parity(lsm, N):
    cases = [synth.sort_i32(seed=N, N=N, hi=64),
             synth.sort_i32(seed=N + 1, N=N, lo=-2**31, hi=2**31 - 1),
             synth.sort_u64(seed=N + 2, N=N)]
    # u64 with ties too: the top bits only
    s = synth.sort_u64(seed=N + 3, N=N)
    cases.append(synth.SortInput(s.keys >> np.uint64(58), s.pay))
    for c in cases:
        want_k, want_p, _ = oracle.merge_sort(c.keys, c.pay)
        keys, pay = lsm.merge_sort(up(c.keys), up(c.pay))
        assert np.array_equal(down(keys), want_k)
        assert np.array_equal(down(pay), want_p)
        keys, none = lsm.merge_sort(up(c.keys))
        assert none is None and np.array_equal(down(keys), want_k)


def test_sort_already_sorted_and_reversed(lsm):
    N = 5 * TILE + 77
    for x in (np.arange(N, dtype=np.uint64), np.arange(N, dtype=np.uint64)[::-1].copy(),
              np.zeros(N, dtype=np.uint64)):
        pay = np.arange(N, dtype=np.uint32)
        want_k, want_p, _ = oracle.merge_sort(x, pay)
        keys, p = lsm.merge_sort(up(x), up(pay))
        assert np.array_equal(down(keys), want_k) and np.array_equal(down(p), want_p)


def test_sort_empty_and_argument_errors(lsm):
    e = torch.empty(0, dtype=torch.uint64, device="cuda")
    keys, _ = lsm.merge_sort(e)
    assert keys.numel() == 0
    x = up(np.arange(10, dtype=np.uint64))
    with pytest.raises(lsm.LsmError):
        lsm.merge_sort(x, ws=torch.empty(16, dtype=torch.uint8, device="cuda"))


def test_sort_full_size_properties(lsm):
    # the bench workload: 2^27 uniform uint64 keys with their input positions
    s = synth.sort_u64()
    N = len(s.keys)
    xk = up(s.keys)
    keys, pay = lsm.merge_sort(xk, up(s.pay))
    torch.cuda.synchronize()
    k = keys.view(torch.int64) ^ (-(2**63))  # order-preserving signed view of uint64
    assert bool((k[1:] >= k[:-1]).all())
    p = pay.view(torch.int32).to(torch.int64)
    assert bool((torch.bincount(p, minlength=N) == 1).all())
    assert bool((xk.view(torch.int64)[p] == keys.view(torch.int64)).all())
    eq = k[1:] == k[:-1]
    assert bool((p[1:][eq] > p[:-1][eq]).all())
