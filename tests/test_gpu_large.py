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
