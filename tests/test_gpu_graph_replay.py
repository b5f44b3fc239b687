"""Calls captured in a CUDA graph and replayed on new inputs, and calls whose
workspace holds stale words, against the oracle, bit-exact: the whole
replacement step (u64, both forms, and strings), the standalone rank
builds, the stable merge, the merge sort and the FC lengths scan + emit.

The single-launch rank builds (rank512 and rank2048) and the one-kernel
replacement merge find their prefixes by a decoupled lookback over per-CTA
state words kept in the caller's workspace. Each call zeroes those words
before the kernel that reads them runs: the co-rank partition that starts the
whole path clears them, and a standalone build issues a memset on its
stream. So a replay reads nothing that an earlier replay published, and a
workspace whose words look like published states (the previous contents of a
recycled allocation) changes nothing."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from tests.gpu_util import down, up  # noqa: E402
from tests.test_gpu_replace import check_against_oracle  # noqa: E402

# A word that reads as "published, inclusive prefix 5" to a lookback.
STALE_STATE = np.uint64((1 << 32) | (1 << 31) | 5)


@pytest.fixture(scope="module")
def lsm():
    import lsm_replacement_merge_gb300 as lsm
    lsm.lib()
    lsm.get_device_status(reset=True)
    yield lsm
    assert lsm.get_device_status() == lsm.LSM_OK
    lsm.tune_replacement_merge(lsm.DEFAULT_REPLACEMENT_MERGE_MODE)


def _stale(nbytes):
    """A workspace filled with words that look like published lookback states."""
    words = (nbytes + 7) // 8
    t = up(np.full(words, STALE_STATE, np.uint64).view(np.int64))
    return t.view(torch.uint8)[:nbytes]


def _capture(fn):
    """Run fn once on a side stream (first-call queries), then capture it."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


# ---- u64 whole path ------------------------------------------------------------------

M, N, SHARED = 300_001, 120_007, 40_000


@pytest.mark.parametrize("mode", [0, 1], ids=["two_pipelines", "one_kernel"])
def test_whole_path_graph_replay(lsm, mode):
    lsm.tune_replacement_merge(mode)
    try:
        dev = torch.device("cuda:0")
        A = torch.empty(M, dtype=torch.uint64, device=dev)
        B = torch.empty(N, dtype=torch.uint64, device=dev)
        first = synth.replace_random_small(seed=500, m=M, n=N, shared=SHARED)
        A.copy_(up(first.A))
        B.copy_(up(first.B))
        ws = _stale(lsm.workspace_size(lsm.LSM_OP_REPLACEMENT_MERGE, M, N))
        out = lsm.replacement_merge(A, B, ws=ws)
        C, lb, dir_, tot, refs, ordA, ordB, cnt = out

        def call():
            lsm.replacement_merge(A, B, C=C, lb_B=lb, dir_=dir_, d_total=tot, refs=refs,
                                  ord_A=ordA, ord_B=ordB, d_count=cnt, ws=ws)

        g = _capture(call)
        for seed in (501, 502, 503):
            inp = synth.replace_random_small(seed=seed, m=M, n=N, shared=SHARED - 7 * (seed - 500))
            A.copy_(up(inp.A))
            B.copy_(up(inp.B))
            g.replay()
            torch.cuda.synchronize()
            k = int(cnt.item())
            got = dict(C=down(C)[:(M + 31) // 32], lb=down(lb), dir=down(dir_),
                       total=int(tot.item()), refs=down(refs)[:k], ordA=down(ordA),
                       ordB=down(ordB), count=k)
            check_against_oracle(got, inp.A, inp.B)
        assert lsm.get_device_status() == lsm.LSM_OK
    finally:
        lsm.tune_replacement_merge(lsm.DEFAULT_REPLACEMENT_MERGE_MODE)


@pytest.mark.parametrize("mode", [0, 1], ids=["two_pipelines", "one_kernel"])
def test_whole_path_stale_workspace(lsm, mode):
    lsm.tune_replacement_merge(mode)
    try:
        inp = synth.replace_random_small(seed=510, m=M, n=N, shared=SHARED)
        ws = _stale(lsm.workspace_size(lsm.LSM_OP_REPLACEMENT_MERGE, M, N))
        C, lb, dir_, tot, refs, ordA, ordB, cnt = lsm.replacement_merge(up(inp.A), up(inp.B),
                                                                        ws=ws)
        k = int(cnt.item())
        check_against_oracle(dict(C=down(C)[:(M + 31) // 32], lb=down(lb), dir=down(dir_),
                                  total=int(tot.item()), refs=down(refs)[:k], ordA=down(ordA),
                                  ordB=down(ordB), count=k), inp.A, inp.B)
    finally:
        lsm.tune_replacement_merge(lsm.DEFAULT_REPLACEMENT_MERGE_MODE)


# ---- standalone rank builds ------------------------------------------------------------

def _bitmap(seed, m, density):
    rng = np.random.default_rng(seed)
    return synth._bitmap(np.flatnonzero(rng.random(m) < density).astype(np.int64), m)


@pytest.mark.parametrize("m", [1, 5000, 2_000_003])
def test_rank_build_graph_replay(lsm, m):
    C = up(_bitmap(520, m, 0.3))
    ws = _stale(lsm.workspace_size(lsm.LSM_OP_RANK_BUILD, m, 0))
    dir_, tot = lsm.rank_build(C, m, ws=ws)
    g = _capture(lambda: lsm.rank_build(C, m, dir_=dir_, d_total=tot, ws=ws))
    for seed, density in ((521, 0.05), (522, 0.9), (523, 0.5)):
        bits = _bitmap(seed, m, density)
        C[:len(bits)].copy_(up(bits))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(down(dir_), oracle.rank512_dir(bits, m))
        assert int(tot.item()) == int(np.unpackbits(bits.view(np.uint8),
                                                    bitorder="little")[:m].sum())
    assert lsm.get_device_status() == lsm.LSM_OK


@pytest.mark.parametrize("m", [1, 5000, 2_000_003])
def test_rank2048_build_graph_replay(lsm, m):
    C = up(_bitmap(530, m, 0.3))
    ws = _stale(lsm.workspace_size(lsm.LSM_OP_RANK2048_BUILD, m, 0))
    dir_, ep, tot = lsm.rank2048_build(C, m, ws=ws)
    g = _capture(lambda: lsm.rank2048_build(C, m, dir_=dir_, epochs=ep, d_total=tot, ws=ws))
    for seed, density in ((531, 0.05), (532, 0.9), (533, 0.5)):
        bits = _bitmap(seed, m, density)
        C[:len(bits)].copy_(up(bits))
        g.replay()
        torch.cuda.synchronize()
        d_want, e_want = oracle.rank2048_dir(bits, m)
        assert np.array_equal(down(dir_), d_want)
        assert np.array_equal(down(ep), e_want)
        assert int(tot.item()) == int(oracle.rank2048_query(bits, d_want, e_want,
                                                            np.array([m], np.uint64))[0])
    assert lsm.get_device_status() == lsm.LSM_OK


# ---- string whole path ---------------------------------------------------------------

SM, SN, SSHARED = 40_000, 15_000, 6_000


def _str_lists(seed):
    """Sorted unique byte keys of mixed length over a small alphabet (long
    shared prefixes), SM for A and SN for B with SSHARED in both."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, 41, size=3 * (SM + SN))
    pool = sorted({bytes(rng.integers(97, 101, size=int(k), dtype=np.uint8)) for k in lens})
    assert len(pool) >= SM + SN
    pick = rng.permutation(len(pool))
    a_idx = np.sort(pick[:SM])
    fresh = pick[SM:SM + SN - SSHARED]
    b_idx = np.sort(np.concatenate([rng.choice(a_idx, SSHARED, replace=False), fresh]))
    return [pool[i] for i in a_idx], [pool[i] for i in b_idx]


def test_whole_path_str_graph_replay(lsm):
    dev = torch.device("cuda:0")
    cap = 64 * (SM + SN) + 64  # arena capacity: 40-byte keys at most, padded
    arenaA = torch.zeros(cap, dtype=torch.uint8, device=dev)
    arenaB = torch.zeros(cap, dtype=torch.uint8, device=dev)
    offA = torch.zeros(SM + 1, dtype=torch.uint64, device=dev)
    offB = torch.zeros(SN + 1, dtype=torch.uint64, device=dev)
    A, B = lsm.Bytes(arenaA, offA), lsm.Bytes(arenaB, offB)

    def load(seed):
        s = synth.strings_from_lists(*_str_lists(seed))
        for arena, off, side in ((arenaA, offA, s.A), (arenaB, offB, s.B)):
            arena.zero_()
            arena[:len(side.key_arena)].copy_(up(side.key_arena))
            off.copy_(up(side.key_off))
        return s

    load(540)
    ws = _stale(lsm.workspace_size(lsm.LSM_OP_REPLACEMENT_MERGE_STR, SM, SN))
    outs = lsm.replacement_merge_str(A, B, ws=ws)
    C, lb, pA, pB, dir_, tot, refs, ordA, ordB, cnt = outs

    def call():
        lsm.replacement_merge_str(A, B, C=C, lb_B=lb, prefixA=pA, prefixB=pB, dir_=dir_,
                                  d_total=tot, refs=refs, ord_A=ordA, ord_B=ordB, d_count=cnt,
                                  ws=ws)

    g = _capture(call)
    for seed in (541, 542, 543):
        s = load(seed)
        g.replay()
        torch.cuda.synchronize()
        r = oracle.replacement_str(s.A.key_arena, s.A.key_off, s.B.key_arena, s.B.key_off)
        k = int(cnt.item())
        assert k == r.count and int(tot.item()) == SM + SN - r.count
        assert np.array_equal(down(C)[:(SM + 31) // 32], r.C)
        assert np.array_equal(down(lb)[:SN], r.lb_B)
        assert np.array_equal(down(refs)[:k], r.refs)
        assert np.array_equal(down(ordA)[:SM], r.ord_A)
        assert np.array_equal(down(ordB)[:SN], r.ord_B)
        assert np.array_equal(down(dir_), oracle.rank512_dir(r.C, SM))
    assert lsm.get_device_status() == lsm.LSM_OK


# ---- the other calls: stable merge, merge sort, FC lengths + emit --------------------

def test_merge_stable_graph_replay(lsm):
    m, n = 200_003, 150_001
    dev = torch.device("cuda:0")
    A = torch.empty(m, dtype=torch.uint64, device=dev)
    B = torch.empty(n, dtype=torch.uint64, device=dev)
    Ap = up(np.arange(m, dtype=np.uint32))
    Bp = up((m + np.arange(n)).astype(np.uint32))

    def load(seed, hi):
        rng = np.random.default_rng(seed)
        a = np.sort(rng.integers(0, hi, size=m, dtype=np.uint64))
        b = np.sort(rng.integers(0, hi, size=n, dtype=np.uint64))
        A.copy_(up(a))
        B.copy_(up(b))
        return a, b

    load(550, 1 << 40)
    ws = _stale(lsm.workspace_size(lsm.LSM_OP_MERGE_STABLE, m, n))
    keys, pay = lsm.merge_stable(A, B, Ap, Bp, ws=ws)
    g = _capture(lambda: lsm.merge_stable(A, B, Ap, Bp, keys, pay, ws))
    for seed, hi in ((551, 1 << 63), (552, 64), (553, 1 << 20)):  # ties in the second
        a, b = load(seed, hi)
        g.replay()
        torch.cuda.synchronize()
        ok, okp, _ = oracle.merge(a, b, np.arange(m, dtype=np.uint32),
                                  (m + np.arange(n)).astype(np.uint32))
        assert np.array_equal(down(keys), ok) and np.array_equal(down(pay), okp)
    assert lsm.get_device_status() == lsm.LSM_OK


def test_merge_sort_graph_replay(lsm):
    N = 300_007
    dev = torch.device("cuda:0")
    keys_in = torch.empty(N, dtype=torch.uint64, device=dev)
    pay_in = up(np.arange(N, dtype=np.uint32))

    def load(seed):
        s = synth.sort_u64(seed=seed, N=N)
        k = s.keys >> np.uint64(seed % 7 * 8)  # more ties from seed to seed
        keys_in.copy_(up(k))
        return k

    load(560)
    ws = _stale(lsm.workspace_size(lsm.LSM_OP_MERGE_SORT, N, 0))
    out_k, out_p = lsm.merge_sort(keys_in, pay_in, ws=ws)
    g = _capture(lambda: lsm.merge_sort(keys_in, pay_in, out_k, out_p, ws))
    for seed in (561, 562, 563):
        k = load(seed)
        g.replay()
        torch.cuda.synchronize()
        want_k, want_p, _ = oracle.merge_sort(k, np.arange(N, dtype=np.uint32))
        assert np.array_equal(down(out_k), want_k) and np.array_equal(down(out_p), want_p)
    assert lsm.get_device_status() == lsm.LSM_OK


def test_fc_lengths_and_emit_graph_replay(lsm):
    """The FC lengths scan and emit captured once and replayed after the
    value bytes change in place (same extents, so the same lengths and a
    different payload)."""
    from tests.test_gpu_fc import device_input, gpu_refs
    s = synth.strings(seed=570, count=30000, fanout=8, depth=3, max_suffix=30)
    fc = device_input(lsm, s)
    refs, N = gpu_refs(lsm, fc)
    r = oracle.replacement_str(s.A.key_arena, s.A.key_off, s.B.key_arena, s.B.key_off)
    ws = _stale(lsm.workspace_size(lsm.LSM_OP_FC_LENGTHS_SCAN, N, 0))
    lcp, ctrl, rec, off = lsm.fc_lengths_scan(fc, refs, N, ws=ws)
    nwords = (int(down(off[N:N + 1])[0]) + 31) // 32
    payload = lsm.fc_emit(fc, refs, N, lcp, ctrl, off, nwords)

    def call():
        lsm.fc_lengths_scan(fc, refs, N, lcp, ctrl, rec, off, ws)
        lsm.fc_emit(fc, refs, N, lcp, ctrl, off, nwords, payload)

    g = _capture(call)
    rng = np.random.default_rng(571)
    for _ in range(3):
        for side, dev_arena in ((s.A, fc.valA.arena), (s.B, fc.valB.arena)):
            side.val_arena[:] = rng.integers(0, 256, len(side.val_arena)).astype(np.uint8)
            dev_arena[:len(side.val_arena)].copy_(up(side.val_arena))
        g.replay()
        torch.cuda.synchronize()
        exp = oracle.fc_encode((s.A.key_arena, s.A.key_off), (s.A.val_arena, s.A.val_off),
                               s.A.tomb if len(s.A.tomb) else None,
                               (s.B.key_arena, s.B.key_off), (s.B.val_arena, s.B.val_off),
                               s.B.tomb if len(s.B.tomb) else None, r.refs)
        assert np.array_equal(down(off), exp.bit_off)
        assert np.array_equal(down(payload)[:len(exp.payload)], exp.payload)
    assert lsm.get_device_status() == lsm.LSM_OK
