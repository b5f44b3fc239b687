"""GPU checks past 2^31 elements, where 64-bit index arithmetic matters.

The oracle cannot run at these sizes in seconds, so the results are checked
by properties that pin them down exactly (merge) or against closed forms
built from library routines on the GPU (replacement). Each test needs tens
of GB of device memory and skips itself when the device has less free."""
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from tests.gpu_util import dev  # noqa: E402

LSM_REF_FROM_B = 0x80000000
LSM_ORD_DROPPED = 0xFFFFFFFF


@pytest.fixture(scope="module")
def lsm():
    import lsm_replacement_merge_gb300 as lsm
    lsm.lib()
    lsm.get_device_status(reset=True)
    yield lsm
    assert lsm.get_device_status() == lsm.LSM_OK


def _need(gib):
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info()
    if free < gib << 30:
        pytest.skip("needs %d GiB of free device memory" % gib)


def _u32(t):
    """uint32 tensor -> int64 values."""
    return t.view(torch.int32).to(torch.int64) & 0xFFFFFFFF


def test_stable_merge_beyond_2pow31_elements(lsm):
    # The output is the stable merge exactly when (1) keys are nondecreasing,
    # (2) each output key is the input element its payload names, (3) the
    # payloads are a permutation of the input positions and (4) equal keys
    # keep increasing payloads (A's indices precede B's, m + j).
    _need(96)
    m, n = (1 << 30) + 12345, (1 << 30) - 777
    total = m + n
    assert total > (1 << 31)
    g = torch.Generator(device=dev()).manual_seed(5)
    A = torch.sort(torch.randint(0, 1 << 62, (m,), device=dev(), generator=g))[0]
    B = torch.randint(0, 1 << 62, (n,), device=dev(), generator=g)
    B[::3] = A[torch.randint(0, m, ((n + 2) // 3,), device=dev(), generator=g)]  # ties with A
    B = torch.sort(B)[0]
    Ap = torch.arange(m, device=dev(), dtype=torch.int64).to(torch.int32).view(torch.uint32)
    Bp = torch.arange(m, total, device=dev(), dtype=torch.int64).to(torch.int32).view(torch.uint32)
    keys, pay = lsm.merge_stable(A, B, Ap, Bp)
    del Ap, Bp
    torch.cuda.synchronize()
    assert bool((keys[1:] >= keys[:-1]).all())
    p = _u32(pay)
    del pay
    src = torch.cat([A, B])
    del A, B
    assert bool((src[p] == keys).all())
    del src
    seen = torch.zeros(total, dtype=torch.bool, device=dev())
    seen[p] = True
    assert bool(seen.all())
    del seen
    eq = keys[1:] == keys[:-1]
    assert int(eq.sum()) > 0
    assert bool((p[1:][eq] > p[:-1][eq]).all())


def test_replacement_beyond_2pow31_elements(lsm):
    # A_i = 3 i and B_j = 2 j + 1: B_j collides with A exactly when 2 j + 1 is
    # a multiple of 3. Expected values from library routines on the GPU:
    # lower bounds by searchsorted, ranks by a cumulative sum, and the refs by
    # scattering each record to its ordinal.
    _need(110)
    m, n = (5 << 28) + 7, (1 << 30) - 3
    total = m + n
    assert total > (1 << 31)
    A = torch.arange(m, device=dev(), dtype=torch.int64) * 3
    B = torch.arange(n, device=dev(), dtype=torch.int64) * 2 + 1
    C, lb = lsm.collision_mark(A, B)
    dir_, tot = lsm.rank_build(C, m)
    refs, ordA, ordB, cnt = lsm.replacement_merge_compact(m, n, C, dir_, lb)
    torch.cuda.synchronize()
    # lower bounds of B in A, and the collision bits
    lb_exp = torch.searchsorted(A, B)
    assert bool((_u32(lb) == lb_exp).all())
    hit = (lb_exp < m) & (A[lb_exp.clamp(max=m - 1)] == B)
    col = torch.zeros(m, dtype=torch.bool, device=dev())
    col[lb_exp[hit]] = True
    del hit
    words = (m + 31) // 32
    bits = torch.zeros(words * 32, dtype=torch.int64, device=dev())
    bits[:m] = col.to(torch.int64)
    weights = torch.bitwise_left_shift(torch.ones(32, dtype=torch.int64, device=dev()),
                                       torch.arange(32, device=dev()))
    C_exp = (bits.view(words, 32) * weights).sum(dim=1)
    del bits
    assert bool((_u32(C) == C_exp).all())
    del C_exp
    # ranks, count and ordinals
    R = torch.zeros(m + 1, dtype=torch.int64, device=dev())
    R[1:] = torch.cumsum(col.to(torch.int64), 0)
    N = total - int(R[m])
    assert int(tot.item()) == int(R[m]) and int(cnt.item()) == N
    lbA = torch.searchsorted(B, A)
    iA = torch.arange(m, device=dev(), dtype=torch.int64)
    ordA_exp = torch.where(col, torch.full_like(iA, LSM_ORD_DROPPED), iA + lbA - R[:m])
    del lbA
    assert bool((_u32(ordA) == ordA_exp).all())
    jB = torch.arange(n, device=dev(), dtype=torch.int64)
    ordB_exp = jB + lb_exp - R[lb_exp]
    assert bool((_u32(ordB) == ordB_exp).all())
    del R, lb_exp
    refs_exp = torch.empty(N, dtype=torch.int64, device=dev())
    keep = ~col
    refs_exp[ordA_exp[keep]] = iA[keep]
    refs_exp[ordB_exp] = jB + LSM_REF_FROM_B
    assert bool((_u32(refs[:N]) == refs_exp).all())


@pytest.mark.parametrize("mode", [0, 1], ids=["two_pipelines", "one_kernel"])
def test_whole_path_beyond_2pow31_elements(lsm, mode):
    # The whole-path call (lsm_replacement_merge) on the same 2.4 G records,
    # both forms, equal to the separate calls, which the test above checks
    # against closed forms: positions past 2^31 in the merge bitmap, the
    # co-ranks, the lookback and the outputs.
    _need(100)
    m, n = (5 << 28) + 7, (1 << 30) - 3
    A = torch.arange(m, device=dev(), dtype=torch.int64) * 3
    B = torch.arange(n, device=dev(), dtype=torch.int64) * 2 + 1
    C, lb = lsm.collision_mark(A, B)
    dir_, tot = lsm.rank_build(C, m)
    refs, ordA, ordB, cnt = lsm.replacement_merge_compact(m, n, C, dir_, lb)
    del lb
    lsm.tune_replacement_merge(mode)
    try:
        Cw, lbw, dirw, totw, refsw, ordAw, ordBw, cntw = lsm.replacement_merge(A, B, want_lb=False)
    finally:
        lsm.tune_replacement_merge(lsm.DEFAULT_REPLACEMENT_MERGE_MODE)
    torch.cuda.synchronize()
    assert lbw is None
    N = int(cnt.item())
    assert int(cntw.item()) == N and int(totw.item()) == int(tot.item())
    words = (m + 31) // 32

    def same(x, y):  # bitwise equality of two uint32 tensors
        return bool((x.view(torch.int32) == y.view(torch.int32)).all())

    assert same(Cw[:words], C[:words]) and same(dirw, dir_)
    assert same(ordAw, ordA) and same(ordBw, ordB)
    assert same(refsw[:N], refs[:N])


def _eg0_len(x):
    import numpy as np
    return 2 * (np.floor(np.log2(x.astype(np.float64) + 1)).astype(np.int64)) + 1


def test_fc_payload_beyond_2pow32_bits(lsm):
    # 532,480 records with 8-byte keys 0, 1, 2, ... (A the even ones, B the
    # odd ones) and 1 KB values: a 4.36 Gbit payload. With consecutive integer
    # keys every length is a closed form (the LCP of r-1 and r is 63 minus the
    # trailing zeros of r); the payload is checked by decoding records at the
    # start, across bit 2^32 and at the end with a plain bit reader.
    import numpy as np
    _need(8)
    h = (1 << 18) + 4096
    N = 2 * h
    d = dev()

    def side(par, mul, add):
        keys = (np.arange(h, dtype=np.uint64) * 2 + par).astype(">u8").view(np.uint8)
        kb = lsm.Bytes.from_numpy(keys, np.arange(h + 1, dtype=np.uint64) * 8, d)
        t = torch.arange(h, device=d, dtype=torch.int64)[:, None]
        b = torch.arange(1024, device=d, dtype=torch.int64)[None, :]
        arena = torch.zeros(h * 1024 + 8, dtype=torch.uint8, device=d)
        arena[:h * 1024] = ((t * mul + b * 7 + add) & 255).to(torch.uint8).reshape(-1)
        voff = (torch.arange(h + 1, device=d, dtype=torch.int64) * 1024).view(torch.uint64)
        return kb, lsm.Bytes(arena, voff)

    kA, vA = side(0, 131, 0)
    kB, vB = side(1, 29, 5)
    tomb_rec = (np.arange(h) % 97) == 3  # A records t with t % 97 == 3
    tw = np.zeros((h + 31) // 32, dtype=np.uint32)
    for t in np.nonzero(tomb_rec)[0]:
        tw[t // 32] |= np.uint32(1 << (t % 32))
    fc = lsm.FcInput(kA, vA, torch.from_numpy(tw).to(d), kB, vB, None)
    C, lb = lsm.collision_mark_str(kA, kB)
    dir_, _ = lsm.rank_build(C, h)
    refs, _, _, cnt = lsm.replacement_merge_compact(h, h, C, dir_, lb)
    assert int(cnt.item()) == N
    r = np.arange(N, dtype=np.int64)
    refs_exp = np.where(r % 2 == 1, LSM_REF_FROM_B, 0) | (r >> 1)
    assert np.array_equal(_u32(refs[:N]).cpu().numpy(), refs_exp)
    lcp, ctrl, rec, off = lsm.fc_lengths_scan(fc, refs, N)
    # closed forms
    x = np.maximum((r - 1) ^ r, 1)
    l_exp = np.where(r == 0, 0, 64 - (np.floor(np.log2(x.astype(np.float64))).astype(np.int64) + 1))
    c_exp = np.where(r % 15 == 0, 1 + l_exp, 64 - l_exp)
    dd = 64 - l_exp
    tomb = (r % 2 == 0) & tomb_rec[r >> 1]
    v = np.where(tomb, 1, 1 + _eg0_len(np.array([1024]))[0] + 8 * 1024)
    rec_exp = _eg0_len(c_exp) + _eg0_len(dd) + dd + v
    off_exp = np.zeros(N + 1, dtype=np.int64)
    off_exp[1:] = np.cumsum(rec_exp)
    total = int(off_exp[N])
    assert total > (1 << 32)
    assert np.array_equal(_u32(lcp).cpu().numpy(), l_exp)
    assert np.array_equal(_u32(ctrl).cpu().numpy(), c_exp)
    assert np.array_equal(_u32(rec).cpu().numpy(), rec_exp)
    assert np.array_equal(off.view(torch.int64).cpu().numpy(), off_exp)
    nwords = (total + 31) // 32 + 3
    words = _u32(lsm.fc_emit(fc, refs, N, lcp, ctrl, off, nwords)).cpu().numpy().astype(np.uint64)
    assert not words[(total + 31) // 32:].any()
    if total % 32:
        assert int(words[total // 32]) & ((1 << (32 - total % 32)) - 1) == 0

    def bits(p, k):  # k <= 32 stream bits from p, as an integer
        q, s = p >> 5, p & 31
        w = (int(words[q]) << 32) | (int(words[q + 1]) if q + 1 < len(words) else 0)
        return (w >> (64 - s - k)) & ((1 << k) - 1)

    def eg0(p):
        z = 0
        while bits(p + z, 1) == 0:
            z += 1
        return bits(p + z, z + 1) - 1, p + 2 * z + 1

    cross = int(np.searchsorted(off_exp, 1 << 32, side="right")) - 1
    sample = sorted(set([0, 1, 2, 14, 15, 16, 1000] + list(range(cross - 2, cross + 4))
                        + [N - 2, N - 1]))
    for i in sample:
        p = int(off_exp[i])
        c, p = eg0(p)
        assert c == c_exp[i]
        dlen, p = eg0(p)
        assert dlen == dd[i]
        key = 0
        for q in range(0, dlen, 32):
            k = min(32, dlen - q)
            key = (key << k) | bits(p + q, k)
        assert key == i & ((1 << dlen) - 1)
        p += dlen
        if tomb[i]:
            assert bits(p, 1) == 0
            p += 1
        else:
            assert bits(p, 1) == 1
            vlen, p = eg0(p + 1)
            assert vlen == 1024
            t = i >> 1
            mul, add = (131, 0) if i % 2 == 0 else (29, 5)
            for b in range(0, 1024, 4):
                exp = 0
                for u in range(4):
                    exp = (exp << 8) | ((t * mul + (b + u) * 7 + add) & 255)
                assert bits(p + 8 * b, 32) == exp
            p += 8 * 1024
        assert p == off_exp[i + 1]
