"""lsm_rank_build_noalloc: the rank512 build without a workspace.

Some callers cannot allocate device memory when they call into the library
(for example a latency-critical path that forbids cudaMalloc after start-up,
or a plug-in whose host program owns all device memory). This entry point
keeps its scratch in a static device array inside the library. The tests
call it through the C ABI and check the directory and R(m) against the
oracle, and against lsm_rank_build, on calls in a row with different sizes,
so that contents left in the shared array by one call cannot leak into the
next; one call uses the whole array (m = 2^29 - 1, the documented limit) and
one size past it must be refused. The file sorts last so that a run which
stops at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MAX_M = (1 << 29) - 1  # the static scratch covers 4096 CTAs x 256 blocks x 512 bits


def _bitmap(m, density, seed):
    rng = np.random.default_rng(seed)
    bits = rng.random(m) < density
    words = np.zeros(max((m + 31) // 32, 1), dtype=np.uint32)
    idx = np.flatnonzero(bits)
    np.bitwise_or.at(words, idx // 32, (np.uint32(1) << (idx % 32).astype(np.uint32)))
    return words


def _random_words(m, seed):
    # a uniformly random bitmap (density 1/2) with the bits past m cleared
    rng = np.random.default_rng(seed)
    w = rng.integers(0, 2**32, max((m + 31) // 32, 1), dtype=np.uint64).astype(np.uint32)
    if m % 32:
        w[(m - 1) // 32] &= np.uint32((1 << (m % 32)) - 1)
    w[(m + 31) // 32:] = 0
    return w


def _noalloc(lsm, C, m, dir_out, tot_out, stream=True):
    return lsm.lib().lsm_rank_build_noalloc(
        ctypes.c_void_p(C.data_ptr()), m, ctypes.c_void_p(dir_out.data_ptr()),
        ctypes.c_void_p(tot_out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream) if stream else None)


def test_noalloc_rank_build_matches_oracle_and_workspace_version():
    import lsm_replacement_merge_gb300 as lsm
    dev = torch.device("cuda:0")
    # calls in a row: a large bitmap, a small one, then the largest allowed
    cases = ((3_000_017, 0.4, 0), (70_001, 0.02, 1), (MAX_M, None, 2))
    for m, density, seed in cases:
        Cn = _bitmap(m, density, seed) if density is not None else _random_words(m, seed)
        C = torch.from_numpy(Cn).to(dev)
        dir_na = torch.full((3 * (m // 512 + 1),), 0xFFFFFFFF, dtype=torch.uint32, device=dev)
        tot_na = torch.full((1,), -1, dtype=torch.int64, device=dev)
        assert _noalloc(lsm, C, m, dir_na, tot_na) == lsm.LSM_OK
        torch.cuda.synchronize()
        got = dir_na.cpu().numpy()
        # the oracle's directory, built bit by bit from R(i)
        assert np.array_equal(got, oracle.rank512_dir(Cn, m))
        # R(m) against a library popcount of the bitmap
        assert int(tot_na.item()) == int(np.unpackbits(Cn.view(np.uint8)).sum())
        if m <= 3_000_017:
            R = oracle.rank_prefix(Cn, m)
            assert int(tot_na.item()) == int(R[m])
            # the workspace version agrees too
            dir_ref, tot_ref = lsm.rank_build(C, m)
            assert np.array_equal(got, dir_ref.cpu().numpy())
            assert int(tot_ref.item()) == int(tot_na.item())
        del C, dir_na, tot_na
        torch.cuda.empty_cache()


def test_noalloc_rank_build_rejects_oversized_input():
    import lsm_replacement_merge_gb300 as lsm
    dev = torch.device("cuda:0")
    C = torch.zeros(16, dtype=torch.uint32, device=dev)
    d = torch.zeros(16, dtype=torch.uint32, device=dev)
    t = torch.zeros(1, dtype=torch.int64, device=dev)
    rc = lsm.lib().lsm_rank_build_noalloc(ctypes.c_void_p(C.data_ptr()), MAX_M + 1,
                                          ctypes.c_void_p(d.data_ptr()),
                                          ctypes.c_void_p(t.data_ptr()), None)
    assert rc == lsm.LSM_ERR_OVERFLOW  # beyond the static scratch: nothing launched
    assert int(t.item()) == 0 and int(d.sum().item()) == 0
