"""lsm_rank_build_noalloc: the rank512 build without a workspace.

Some callers cannot allocate device memory when they call into the library
(for example a latency-critical path that forbids cudaMalloc after start-up,
or a plug-in whose host program owns all device memory). This entry point
keeps its scratch in a static device array inside the library. The test
calls it through the C ABI and checks it against lsm_rank_build, on two calls
in a row with different sizes, so that contents left in the shared array by
the first call cannot leak into the second. The file sorts last so that a
run which stops at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _bitmap(m, density, seed):
    rng = np.random.default_rng(seed)
    bits = rng.random(m) < density
    words = np.zeros(max((m + 31) // 32, 1), dtype=np.uint32)
    idx = np.flatnonzero(bits)
    np.bitwise_or.at(words, idx // 32, (np.uint32(1) << (idx % 32).astype(np.uint32)))
    return words


def test_noalloc_rank_build_matches_workspace_version_twice():
    import lsm_replacement_merge_gb300 as lsm
    dev = torch.device("cuda:0")
    # two calls in a row: a large bitmap, then a smaller one
    for call, (m, density) in enumerate(((3_000_017, 0.4), (70_001, 0.02))):
        C = torch.from_numpy(_bitmap(m, density, seed=call)).to(dev)
        dir_ref, tot_ref = lsm.rank_build(C, m)
        dir_na = torch.empty_like(dir_ref)
        tot_na = torch.empty_like(tot_ref)
        rc = lsm.lib().lsm_rank_build_noalloc(
            ctypes.c_void_p(C.data_ptr()), m, ctypes.c_void_p(dir_na.data_ptr()),
            ctypes.c_void_p(tot_na.data_ptr()),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == lsm.LSM_OK
        torch.cuda.synchronize()
        assert np.array_equal(dir_na.cpu().numpy(), dir_ref.cpu().numpy())
        assert int(tot_na.item()) == int(tot_ref.item())


def test_noalloc_rank_build_rejects_oversized_input():
    import lsm_replacement_merge_gb300 as lsm
    dev = torch.device("cuda:0")
    C = torch.zeros(16, dtype=torch.uint32, device=dev)
    d = torch.zeros(16, dtype=torch.uint32, device=dev)
    t = torch.zeros(1, dtype=torch.int64, device=dev)
    rc = lsm.lib().lsm_rank_build_noalloc(ctypes.c_void_p(C.data_ptr()), 1 << 29,
                                          ctypes.c_void_p(d.data_ptr()),
                                          ctypes.c_void_p(t.data_ptr()), None)
    assert rc == 3  # LSM_ERR_OVERFLOW: beyond the static scratch
