"""GPU tests of the sortedness validators (lsm_validate_sorted,
lsm_validate_sorted_str): the first violating pair against a plain Python
scan of the same host-built input, LSM_ERR_UNSORTED in the device status
word, and a context that stays usable afterwards ("Everett: byte-profile GPU
merge", "Pipeline": inputs are otherwise trusted)."""
import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from tests.gpu_util import up  # noqa: E402


@pytest.fixture()
def lsm():
    import lsm_replacement_merge_gb300 as lsm
    lsm.lib()
    lsm.get_device_status(reset=True)
    yield lsm
    lsm.get_device_status(reset=True)


def first_violation(keys, strict):
    for t in range(len(keys) - 1):
        if (keys[t] >= keys[t + 1]) if strict else (keys[t] > keys[t + 1]):
            return t
    return -1


def run(lsm, keys, strict):
    lsm.get_device_status(reset=True)
    d = lsm.validate_sorted(up(keys), strict)
    got = int(d.item())
    status = lsm.get_device_status(reset=True)
    return got, status


@pytest.mark.parametrize("dtype", [np.uint64, np.int32])
def test_sorted_inputs_pass(lsm, dtype):
    rng = np.random.default_rng(1)
    info = np.iinfo(dtype)
    keys = np.sort(rng.integers(info.min, info.max, 1_000_003, dtype=dtype, endpoint=True))
    uniq = np.unique(keys)
    for k, strict in ((keys, False), (uniq, True), (uniq, False)):
        assert run(lsm, k, strict) == (-1, lsm.LSM_OK)
    for k in (keys[:0], keys[:1]):
        assert run(lsm, k, True) == (-1, lsm.LSM_OK)


@pytest.mark.parametrize("dtype", [np.uint64, np.int32])
def test_violations_found(lsm, dtype):
    rng = np.random.default_rng(2)
    info = np.iinfo(dtype)
    base = np.unique(rng.integers(info.min, info.max, 700_001, dtype=dtype, endpoint=True))
    n = len(base)
    cases = []
    k = base.copy()
    k[[n // 2, 3 * n // 4]] = k[[3 * n // 4, n // 2]]  # two swapped keys
    cases.append((k, False))
    k = base.copy()
    k[n - 1] = k[n - 2]  # a duplicate at the very end: fine unless strict
    cases.append((k, True))
    cases.append((k, False))
    k = base.copy()
    k[0] = k[1]  # a duplicate at the start
    cases.append((k, True))
    k = base[::-1].copy()  # descending
    cases.append((k, False))
    if dtype == np.int32:  # signed order: -1 after +1 is a violation
        cases.append((np.array([-5, -1, 1, -1, 7], dtype=np.int32), False))
    for k, strict in cases:
        want = first_violation(k.tolist(), strict)
        got, status = run(lsm, k, strict)
        assert got == want
        assert status == (lsm.LSM_ERR_UNSORTED if want >= 0 else lsm.LSM_OK)


def _col(lsm, keys, dev):
    s = synth.strings_from_lists(keys, [])
    return lsm.Bytes.from_numpy(s.A.key_arena, s.A.key_off, dev)


def test_string_order(lsm):
    dev = torch.device("cuda:0")
    s = synth.strings(seed=21, count=20000, fanout=4, depth=4)
    col = lsm.Bytes.from_numpy(s.A.key_arena, s.A.key_off, dev)
    lsm.get_device_status(reset=True)
    assert int(lsm.validate_sorted_str(col, True).item()) == -1
    assert lsm.get_device_status(reset=True) == lsm.LSM_OK
    cases = [
        ([b"a", b"ab", b"b"], True, -1),
        ([b"ab", b"a"], False, 0),              # a proper prefix sorts first
        ([b"", b"", b"x"], True, 0),            # duplicate empty keys
        ([b"", b"", b"x"], False, -1),
        ([b"x" * 40 + b"a", b"x" * 40 + b"b", b"x" * 40 + b"a"], False, 1),  # past 16 bytes
        ([b"\x00", b"\x00\x00", b"\xff", b"\x7f"], True, 2),  # unsigned byte order
    ]
    for keys, strict, want in cases:
        got = int(lsm.validate_sorted_str(_col(lsm, keys, dev), strict).item())
        status = lsm.get_device_status(reset=True)
        assert got == want
        assert status == (lsm.LSM_ERR_UNSORTED if want >= 0 else lsm.LSM_OK)


def test_string_malformed_offsets_are_reported_not_read(lsm):
    dev = torch.device("cuda:0")
    col = _col(lsm, [b"apple", b"banana", b"cherry", b"date"], dev)
    off = col.off.cpu().numpy().copy()
    # offsets going backwards at key 2, and an end past the arena
    bad = off.copy()
    bad[2] = bad[1] - 1
    col.off = torch.from_numpy(bad).to(dev)
    assert int(lsm.validate_sorted_str(col, True).item()) == 0
    assert lsm.get_device_status(reset=True) == lsm.LSM_ERR_UNSORTED
    bad = off.copy()
    bad[4] = 10 ** 12
    col.off = torch.from_numpy(bad).to(dev)
    assert int(lsm.validate_sorted_str(col, True).item()) == 2
    assert lsm.get_device_status(reset=True) == lsm.LSM_ERR_UNSORTED
    # a single key whose end lies past the arena
    one = _col(lsm, [b"solo"], dev)
    one.off = torch.tensor([0, 10 ** 9], dtype=torch.uint64, device=dev)
    assert int(lsm.validate_sorted_str(one, True).item()) == 0
    assert lsm.get_device_status(reset=True) == lsm.LSM_ERR_UNSORTED
    # the context is still usable
    col.off = torch.from_numpy(off).to(dev)
    assert int(lsm.validate_sorted_str(col, True).item()) == -1
    assert lsm.get_device_status(reset=True) == lsm.LSM_OK
