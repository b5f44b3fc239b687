"""GPU parity for the whole replacement merge in one call
(lsm_replacement_merge, in both its forms: the collision mark and the
compaction in one kernel with a lookback for R, and as two pipelines with
the rank512 build between them, the compaction's tiles on the mark's
diagonals) against the oracle, bit-exact: C, lb_B, the directory, R(m), refs, ordinals and the
count. Cases span several tiles with ragged tails, dense and sparse
collisions, A-only and B-only stretches, ties at every tile boundary (B equal
to A), single records, empty inputs and the two full-size workloads."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from tests.gpu_util import down, up  # noqa: E402
from tests.test_gpu_replace import check_against_oracle  # noqa: E402
from tests.test_oracle_pins import REPLACE_CASES  # noqa: E402


@pytest.fixture(scope="module")
def lsm_mod():
    import lsm_replacement_merge_gb300 as lsm
    lsm.lib()
    lsm.get_device_status(reset=True)
    yield lsm
    assert lsm.get_device_status() == lsm.LSM_OK


@pytest.fixture(params=[1, 0], ids=["one_kernel", "two_pipelines"])
def lsm(lsm_mod, request):
    # every test runs both forms of the call: the mark and the compaction in
    # one kernel, and as two pipelines
    lsm_mod.tune_replacement_merge(request.param)
    try:
        yield lsm_mod
        assert lsm_mod.get_device_status() == lsm_mod.LSM_OK
    finally:
        lsm_mod.tune_replacement_merge(lsm_mod.DEFAULT_REPLACEMENT_MERGE_MODE)


def run_whole(lsm, A, B, ws=None, want_lb=True):
    m, n = len(A), len(B)
    C, lb, dir_, tot, refs, ordA, ordB, cnt = lsm.replacement_merge(up(A), up(B), ws=ws,
                                                                    want_lb=want_lb)
    N = int(cnt.item())
    return dict(C=down(C)[:(m + 31) // 32], lb=None if lb is None else down(lb), dir=down(dir_),
                total=int(tot.item()), refs=down(refs)[:N], ordA=down(ordA), ordB=down(ordB),
                count=N)


@pytest.mark.parametrize("m,n,shared,universe", [c for c in REPLACE_CASES if c[0] + c[1] > 0] + [
    (20000, 7000, 7000, None), (7000, 20000, 7000, None), (100000, 100000, 50000, 250000),
    (300000, 2000, 1000, None), (2000, 300000, 2000, None), (1000000, 1000000, 1000000, None),
    (2816, 2816, 1000, None), (2815, 1, 1, None), (1, 5631, 1, None)])
def test_whole_path_parity(lsm, m, n, shared, universe):
    inp = synth.replace_random_small(seed=m * 13 + n + shared, m=m, n=n, shared=shared,
                                     universe=universe)
    check_against_oracle(run_whole(lsm, inp.A, inp.B), inp.A, inp.B)


def test_whole_path_single_record_edges(lsm):
    for A, B in (([5], [5]), ([5], [6]), ([6], [5]), ([], [1]), ([1], []), ([1, 2, 3], [0, 2, 4]),
                 ([0, 2**64 - 1], [2**64 - 1]), ([0], [0, 2**64 - 1])):
        A = np.array(A, np.uint64)
        B = np.array(B, np.uint64)
        check_against_oracle(run_whole(lsm, A, B), A, B)


def test_whole_path_empty(lsm):
    e = up(np.zeros(0, np.uint64))
    C, lb, dir_, tot, refs, ordA, ordB, cnt = lsm.replacement_merge(e, e)
    assert int(cnt.item()) == 0 and int(tot.item()) == 0
    assert down(dir_).tolist() == [0, 0, 0]


def test_whole_path_clustered(lsm):
    # B dense inside a few windows of A (long A-only stretches between them)
    sk = synth.replace_skewed(seed=44, m=300000, windows=16, window=1024, per_window_shared=512,
                              per_window_fresh=512)
    check_against_oracle(run_whole(lsm, sk.A, sk.B), sk.A, sk.B)
    # |A| = 0 against the clustered B, and A alone
    e = np.zeros(0, np.uint64)
    check_against_oracle(run_whole(lsm, e, sk.B), e, sk.B)
    check_against_oracle(run_whole(lsm, sk.A, e), sk.A, e)


def test_whole_path_replace_12M_4M(lsm):
    inp = synth.replace_u64()
    check_against_oracle(run_whole(lsm, inp.A, inp.B), inp.A, inp.B)


def test_whole_path_skewed_2pow24(lsm):
    inp = synth.replace_skewed()
    check_against_oracle(run_whole(lsm, inp.A, inp.B), inp.A, inp.B)


def test_whole_path_twice_reuses_workspace(lsm):
    # a workspace left by an earlier call (other sizes) must not leak into the next
    ws = lsm.workspace(lsm.LSM_OP_REPLACEMENT_MERGE, 300000, 300000, torch.device("cuda"))
    for seed, (m, n, shared) in enumerate(((300000, 300000, 100000), (200000, 50000, 40000))):
        inp = synth.replace_random_small(seed=seed + 77, m=m, n=n, shared=shared)
        check_against_oracle(run_whole(lsm, inp.A, inp.B, ws=ws), inp.A, inp.B)


def test_whole_path_equals_separate_calls(lsm):
    # the three separate calls (each with its own partition) give the same bytes
    inp = synth.replace_random_small(seed=5, m=400000, n=150000, shared=60000)
    m, n = len(inp.A), len(inp.B)
    whole = run_whole(lsm, inp.A, inp.B)
    C, lb = lsm.collision_mark(up(inp.A), up(inp.B))
    dir_, tot = lsm.rank_build(C, m)
    refs, ordA, ordB, cnt = lsm.replacement_merge_compact(m, n, C, dir_, lb)
    N = int(cnt.item())
    assert N == whole["count"]
    assert np.array_equal(down(C)[:(m + 31) // 32], whole["C"])
    assert np.array_equal(down(lb), whole["lb"])
    assert np.array_equal(down(refs)[:N], whole["refs"])
    assert np.array_equal(down(ordA), whole["ordA"]) and np.array_equal(down(ordB), whole["ordB"])
    r = oracle.replacement_u64(inp.A, inp.B)
    assert N == r.count


@pytest.mark.parametrize("m,n,shared", [(20000, 7000, 7000), (300000, 300000, 100000),
                                        (2816, 2816, 1000), (0, 5000, 0), (5000, 0, 0)])
def test_whole_path_without_lower_bounds(lsm, m, n, shared):
    # lb_B is scratch on the whole path: a null lb_B leaves it unwritten and
    # every other output unchanged
    inp = synth.replace_random_small(seed=m + 3 * n + shared, m=m, n=n, shared=shared)
    got = run_whole(lsm, inp.A, inp.B, want_lb=False)
    assert got["lb"] is None
    check_against_oracle(got, inp.A, inp.B)


def test_whole_path_without_lower_bounds_12M_4M(lsm):
    inp = synth.replace_u64()
    check_against_oracle(run_whole(lsm, inp.A, inp.B, want_lb=False), inp.A, inp.B)
