"""GPU parity for the replacement merge: collision bitmap and lower bounds,
rank512 directory and queries, and the compaction into survivor refs and
ordinals (C ABI vs oracle, bit-exact)."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from tests.gpu_util import down, up  # noqa: E402
from tests.test_oracle_pins import REPLACE_CASES, _maps, _pack  # noqa: E402


@pytest.fixture(scope="module")
def lsm():
    import lsm_replacement_merge_gb300 as lsm
    lsm.lib()
    lsm.get_device_status(reset=True)
    yield lsm
    assert lsm.get_device_status() == lsm.LSM_OK


def run_pipeline(lsm, A, B):
    m, n = len(A), len(B)
    C, lb = lsm.collision_mark(up(A), up(B))
    dir_, tot = lsm.rank_build(C, m)
    refs, ordA, ordB, cnt = lsm.replacement_merge_compact(m, n, C, dir_, lb)
    N = int(cnt.item())
    return dict(C=down(C), lb=down(lb), dir=down(dir_), total=int(tot.item()), refs=down(refs)[:N],
                ordA=down(ordA), ordB=down(ordB), count=N)


def check_against_oracle(got, A, B):
    r = oracle.replacement_u64(A, B)
    m = len(A)
    assert got["count"] == r.count
    assert np.array_equal(got["C"], r.C)
    if got["lb"] is not None:
        assert np.array_equal(got["lb"], r.lb_B)
    assert got["total"] == len(A) + len(B) - r.count
    assert np.array_equal(got["dir"], oracle.rank512_dir(r.C, m))
    assert np.array_equal(got["refs"], r.refs)
    assert np.array_equal(got["ordA"], r.ord_A)
    assert np.array_equal(got["ordB"], r.ord_B)


@pytest.mark.parametrize("m,n,shared,universe", REPLACE_CASES + [
    (20000, 7000, 7000, None), (7000, 20000, 7000, None), (100000, 100000, 50000, 250000),
    (300000, 2000, 1000, None), (2000, 300000, 2000, None)])
def test_replacement_pipeline_parity(lsm, m, n, shared, universe):
    if m + n == 0:
        C, lb = lsm.collision_mark(up(np.zeros(0, np.uint64)), up(np.zeros(0, np.uint64)))
        dir_, tot = lsm.rank_build(C, 0)
        refs, _, _, cnt = lsm.replacement_merge_compact(0, 0, C, dir_, lb)
        assert int(cnt.item()) == 0 and int(tot.item()) == 0
        assert down(dir_).tolist() == [0, 0, 0]
        return
    inp = synth.replace_random_small(seed=m * 7 + n + shared, m=m, n=n, shared=shared,
                                     universe=universe)
    check_against_oracle(run_pipeline(lsm, inp.A, inp.B), inp.A, inp.B)


def test_single_record_edges(lsm):
    A = synth.replace_u64(seed=40, m=5000, n=10).A
    for B in (A[2500:2501].copy(), np.array([A[2500] + np.uint64(1)], np.uint64),
              A[:1].copy(), A[-1:].copy()):
        check_against_oracle(run_pipeline(lsm, A, B), A, B)
    # |A| = 0 against a clustered B
    sk = synth.replace_skewed(seed=41, m=60000, windows=8, window=512, per_window_shared=200,
                              per_window_fresh=100)
    check_against_oracle(run_pipeline(lsm, np.zeros(0, np.uint64), sk.B), np.zeros(0, np.uint64), sk.B)
    check_against_oracle(run_pipeline(lsm, sk.A, np.zeros(0, np.uint64)), sk.A, np.zeros(0, np.uint64))


@pytest.mark.parametrize("m,kind,bits", list(_maps()))
def test_rank_build_and_query_every_position(lsm, m, kind, bits):
    C = _pack(bits)
    Cd = up(C) if len(C) else up(np.zeros(4, np.uint32))
    dir_, tot = lsm.rank_build(Cd, m)
    R = oracle.rank_prefix(C, m)
    assert np.array_equal(down(dir_), oracle.rank512_dir(C, m))
    assert int(tot.item()) == int(R[m])
    pos = np.arange(m + 1, dtype=np.uint32)
    got = down(lsm.rank_query(Cd, dir_, m, up(pos)))
    assert np.array_equal(got, R)


def test_rank_query_out_of_range_sets_status(lsm):
    C = _pack(np.ones(100, bool))
    dir_, _ = lsm.rank_build(up(C), 100)
    out = down(lsm.rank_query(up(C), dir_, 100, up(np.array([100, 101], np.uint32))))
    assert out.tolist() == [100, 0xFFFFFFFF]
    assert lsm.get_device_status(reset=True) == 1   # LSM_ERR_ARG, then cleared


def test_config_replace_12M_4M(lsm):
    inp = synth.replace_u64()
    check_against_oracle(run_pipeline(lsm, inp.A, inp.B), inp.A, inp.B)


def test_config_skewed_2pow24(lsm):
    inp = synth.replace_skewed()
    check_against_oracle(run_pipeline(lsm, inp.A, inp.B), inp.A, inp.B)


def test_timeout_probe_reports_and_context_survives(lsm):
    lsm.get_device_status(reset=True)
    lsm.debug_timeout_probe(2_000_000)          # 2 ms wait on a flag nothing sets
    assert lsm.get_device_status(reset=True) == lsm.LSM_ERR_TIMEOUT
    A = np.arange(0, 100, 2, dtype=np.uint64)
    B = np.arange(0, 100, 3, dtype=np.uint64)
    check_against_oracle(run_pipeline(lsm, A, B), A, B)


def test_compact_rejects_lb_that_is_not_a_lower_bound_array(lsm):
    # An lb_B that no collision mark could have produced (unsorted values)
    # gives B records slots that collide or leave the tile: the kernel skips
    # those tiles and records LSM_ERR_ARG; the context stays usable.
    rng = np.random.default_rng(11)
    m, n = 50000, 20000
    A = np.arange(m, dtype=np.uint64) * 3
    C = np.zeros((m + 31) // 32, np.uint32)
    dir_, _ = lsm.rank_build(up(C), m)
    lb = rng.integers(0, m + 1, n, dtype=np.uint64).astype(np.uint32)
    lsm.replacement_merge_compact(m, n, up(C), dir_, up(lb))
    assert lsm.get_device_status(reset=True) == 1   # LSM_ERR_ARG, then cleared
    B = np.arange(n, dtype=np.uint64) * 5 + 1
    check_against_oracle(run_pipeline(lsm, A, B), A, B)


@pytest.mark.parametrize("kernel", [0, 1])
@pytest.mark.parametrize("variant", [(256, 11), (128, 23), (256, 23), (512, 11)])
def test_every_tile_variant_matches_oracle(lsm, kernel, variant):
    inp = synth.replace_random_small(seed=41 + kernel, m=300000, n=100000, shared=25000,
                                     universe=None)
    lsm.tune_replace(kernel, *variant)
    try:
        check_against_oracle(run_pipeline(lsm, inp.A, inp.B), inp.A, inp.B)
    finally:
        lsm.tune_replace(kernel, *lsm.DEFAULT_REPLACE_VARIANT[kernel])


def _materialize_check(lsm, A, B, valA, valB, tombA, tombB):
    m, n = len(A), len(B)
    Cd, lb = lsm.collision_mark(up(A), up(B))
    dir_, _ = lsm.rank_build(Cd, m)
    refs, _, _, cnt = lsm.replacement_merge_compact(m, n, Cd, dir_, lb)
    N = int(cnt.item())
    keys, vals, tomb = lsm.replacement_materialize(
        up(A), up(B), refs, cnt, valA=up(valA), valB=up(valB),
        tombA=None if tombA is None else up(tombA), tombB=None if tombB is None else up(tombB))
    r = oracle.replacement_u64(A, B)
    ek, ev, et = oracle.materialize_u64(A, valA, tombA, B, valB, tombB, r.refs)
    assert N == r.count
    assert np.array_equal(down(keys)[:N], ek)
    assert np.array_equal(down(vals)[:N], ev)
    assert np.array_equal(down(tomb)[:(N + 31) // 32], et)


@pytest.mark.parametrize("m,n,shared,universe", REPLACE_CASES + [(300000, 100000, 25000, None)])
def test_materialize_parity(lsm, m, n, shared, universe):
    if m + n == 0:
        return
    inp = synth.replace_random_small(seed=m * 3 + n + shared, m=m, n=n, shared=shared,
                                     universe=universe)
    rng = np.random.default_rng(m + 7 * n)
    tA = synth._bitmap(np.nonzero(rng.random(m) < 0.1)[0].astype(np.int64), m)
    tB = synth._bitmap(np.nonzero(rng.random(n) < 0.1)[0].astype(np.int64), n)
    _materialize_check(lsm, inp.A, inp.B, inp.valA, inp.valB, tA if m else None,
                       tB if n else None)


def test_materialize_without_values_or_tombstones(lsm):
    inp = synth.replace_random_small(seed=5, m=5000, n=3000, shared=1000)
    m, n = len(inp.A), len(inp.B)
    Cd, lb = lsm.collision_mark(up(inp.A), up(inp.B))
    dir_, _ = lsm.rank_build(Cd, m)
    refs, _, _, cnt = lsm.replacement_merge_compact(m, n, Cd, dir_, lb)
    keys, vals, tomb = lsm.replacement_materialize(up(inp.A), up(inp.B), refs, cnt)
    r = oracle.replacement_u64(inp.A, inp.B)
    ek, _, _ = oracle.materialize_u64(inp.A, inp.valA, None, inp.B, inp.valB, None, r.refs)
    assert vals is None
    assert np.array_equal(down(keys)[:r.count], ek)
    assert not down(tomb)[:(r.count + 31) // 32].any()


def test_config_replace_12M_4M_materialized(lsm):
    inp = synth.replace_u64()
    _materialize_check(lsm, inp.A, inp.B, inp.valA, inp.valB, None, inp.tombB)


def test_materialize_rejects_a_ref_past_its_input(lsm):
    A = np.arange(100, dtype=np.uint64)
    B = np.arange(100, 150, dtype=np.uint64)
    refs = np.array([0, 1, 99, 100, LSM_REF_FROM_B_PY | 49, LSM_REF_FROM_B_PY | 50], np.uint32)
    cnt = torch.tensor([len(refs)], dtype=torch.int64, device="cuda")
    keys, _, _ = lsm.replacement_materialize(up(A), up(B), up(refs), cnt)
    assert lsm.get_device_status(reset=True) == 1   # LSM_ERR_ARG, then cleared
    got = down(keys)
    assert got[0] == 0 and got[1] == 1 and got[2] == 99 and got[4] == 149


LSM_REF_FROM_B_PY = 0x80000000


# ---- the tiled direct scatter path ([CB] "The three experimental paths") ----
def run_direct_scatter(lsm, A, B):
    m, n = len(A), len(B)
    dA, dB = up(A), up(B)
    C, lb = lsm.collision_mark(dA, dB)
    if m == 0:
        C = up(np.zeros(4, np.uint32))
    dir_, _ = lsm.rank_build(C, m)
    refs, ordA, ordB, cnt = lsm.replacement_direct_scatter(dA, dB, C, dir_, lb)
    N = int(cnt.item())
    return dict(refs=down(refs)[:N], ordA=down(ordA), ordB=down(ordB), count=N)


def check_scatter(got, A, B):
    r = oracle.replacement_u64(A, B)
    assert got["count"] == r.count
    assert np.array_equal(got["refs"], r.refs)
    assert np.array_equal(got["ordA"], r.ord_A)
    assert np.array_equal(got["ordB"], r.ord_B)


@pytest.mark.parametrize("m,n,shared,universe", [c for c in REPLACE_CASES if c[0] + c[1] > 0] + [
    (20000, 7000, 7000, None), (7000, 20000, 7000, None), (100000, 100000, 50000, 250000),
    (300000, 2000, 1000, None), (2000, 300000, 2000, None)])
def test_direct_scatter_parity(lsm, m, n, shared, universe):
    inp = synth.replace_random_small(seed=m * 7 + n + shared, m=m, n=n, shared=shared,
                                     universe=universe)
    check_scatter(run_direct_scatter(lsm, inp.A, inp.B), inp.A, inp.B)


def test_direct_scatter_replace_12M_4M(lsm):
    inp = synth.replace_u64()
    check_scatter(run_direct_scatter(lsm, inp.A, inp.B), inp.A, inp.B)


def test_direct_scatter_skewed_2pow24(lsm):
    inp = synth.replace_skewed()
    check_scatter(run_direct_scatter(lsm, inp.A, inp.B), inp.A, inp.B)


# ---- the fused pass: mark, rank, ordinals and refs in one call ----------------
def run_fused(lsm, A, B):
    m, n = len(A), len(B)
    C, lb, dir_, tot, refs, ordA, ordB, cnt = lsm.replacement_merge_fused(up(A), up(B))
    N = int(cnt.item())
    return dict(C=down(C)[:(m + 31) // 32], lb=down(lb), dir=down(dir_), total=int(tot.item()),
                refs=down(refs)[:N], ordA=down(ordA), ordB=down(ordB), count=N)


@pytest.mark.parametrize("m,n,shared,universe", REPLACE_CASES + [
    (20000, 7000, 7000, None), (7000, 20000, 7000, None), (100000, 100000, 50000, 250000),
    (300000, 2000, 1000, None), (2000, 300000, 2000, None), (1000000, 1000000, 1000000, None)])
def test_fused_parity(lsm, m, n, shared, universe):
    inp = synth.replace_random_small(seed=m * 7 + n + shared, m=m, n=n, shared=shared,
                                     universe=universe)
    check_against_oracle(run_fused(lsm, inp.A, inp.B), inp.A, inp.B)


def test_fused_single_record_edges(lsm):
    for A, B in (([5], [5]), ([5], [6]), ([6], [5]), ([], [1]), ([1], []), ([1, 2, 3], [0, 2, 4])):
        A = np.array(A, np.uint64)
        B = np.array(B, np.uint64)
        check_against_oracle(run_fused(lsm, A, B), A, B)


def test_fused_empty(lsm):
    e = up(np.zeros(0, np.uint64))
    *_, refs, _, _, cnt = lsm.replacement_merge_fused(e, e)
    assert int(cnt.item()) == 0


def test_fused_replace_12M_4M(lsm):
    inp = synth.replace_u64()
    check_against_oracle(run_fused(lsm, inp.A, inp.B), inp.A, inp.B)


def test_fused_skewed_2pow24(lsm):
    inp = synth.replace_skewed()
    check_against_oracle(run_fused(lsm, inp.A, inp.B), inp.A, inp.B)


def test_fused_twice_reuses_workspace(lsm):
    # the tile states are cleared by each call's partition: a workspace left
    # by an earlier call (other sizes) must not leak into the next one
    ws = lsm.workspace(lsm.LSM_OP_REPLACEMENT_FUSED, 300000, 300000, torch.device("cuda"))
    for seed, (m, n, shared) in enumerate(((300000, 300000, 100000), (200000, 50000, 40000))):
        inp = synth.replace_random_small(seed=seed + 99, m=m, n=n, shared=shared)
        C, lb, dir_, tot, refs, ordA, ordB, cnt = lsm.replacement_merge_fused(up(inp.A), up(inp.B),
                                                                            ws=ws)
        N = int(cnt.item())
        got = dict(C=down(C)[:(m + 31) // 32], lb=down(lb), dir=down(dir_), total=int(tot.item()),
                   refs=down(refs)[:N], ordA=down(ordA), ordB=down(ordB), count=N)
        check_against_oracle(got, inp.A, inp.B)
