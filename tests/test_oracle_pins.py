"""Pins for the CPU oracle: page examples, brute force, closed forms, invariants.

Nothing here touches a GPU or the CUDA library. Each test ties the oracle to
something other than itself: a value printed on a page (tests/golden), a
textbook routine (a stable sort, a cumulative sum, a Python dict applied in
chronological order, Python big-int arithmetic), or an invariant the pages
state.
"""
import itertools

import numpy as np
import pytest

import oracle
import synth


# ---------------------------------------------------------------------------
# Stable merge and co-rank
# ---------------------------------------------------------------------------
def test_worked_example_merge_and_crossings(golden):
    g = golden("merge_path_worked_example.txt")
    for dt in (np.int32, np.uint64):
        a, b = np.array(g["a"], dt), np.array(g["b"], dt)
        keys, _, prov = oracle.merge(a, b, provenance=True)
        assert keys.tolist() == g["merged"]
        assert [int(p < len(a)) for p in prov] == g["path_takes_a"]
        assert oracle.corank(a, b, g["corank_k"][0]) == g["corank_i"][0]
        for k, i in zip(g["crossing_k"], g["crossing_i"]):
            assert oracle.corank(a, b, k) == i
        part = oracle.partition(a, b, 2)
        assert part[:, 0].tolist() == g["crossing_i"]
        assert (part.sum(axis=1)).tolist() == g["crossing_k"]


def test_chapter14_coranks(golden):
    g = golden("corank_chapter14.txt")
    A, B = np.array(g["A"], np.int32), np.array(g["B"], np.int32)
    for k, i, j in zip(g["k"], g["i"], g["j"]):
        assert (oracle.corank(A, B, k), k - oracle.corank(A, B, k)) == (i, j)
    assert oracle.merge(A, B)[0].tolist() == g["merged"]


def test_corank_trap(golden):
    g = golden("corank_trap.txt")
    assert oracle.corank(np.array(g["a"], np.int32), np.array(g["b"], np.int32),
                         g["k"][0]) == g["i"][0]


def test_tie_provenance(golden):
    g = golden("tie_provenance.txt")
    a, b = np.array(g["a"], np.int32), np.array(g["b"], np.int32)
    keys, _, prov = oracle.merge(a, b, provenance=True)
    assert keys.tolist() == g["values"]
    assert prov.tolist() == g["provenance"]
    assert oracle.corank(a, b, g["k"][0]) == g["i"][0]
    # the page's point: the wrong split has the same values, other provenance
    src = np.concatenate([a, b])
    assert src[g["wrong_provenance"]].tolist() == g["values"]
    assert g["wrong_provenance"] != prov.tolist()


def _brute_coranks(A, B):
    """Co-rank at every k from Python's stable sort of tagged elements."""
    tagged = sorted([(int(x), 0) for x in A] + [(int(x), 1) for x in B],
                    key=lambda t: (t[0], t[1]))
    out = [0]
    for _, src in tagged:
        out.append(out[-1] + (src == 0))
    return out


def _sorted_sequences(alphabet, max_len):
    for length in range(max_len + 1):
        yield from itertools.combinations_with_replacement(alphabet, length)


@pytest.mark.parametrize("dt", [np.int32, np.uint64])
def test_corank_brute_force_all_small(dt):
    seqs = list(_sorted_sequences(range(4), 4))
    for sa in seqs:
        A = np.array(sa, dt)
        for sb in seqs:
            B = np.array(sb, dt)
            part = oracle.partition(A, B, 1)
            assert part[:, 0].tolist() == _brute_coranks(A, B), (sa, sb)
            assert (part.sum(axis=1) == np.arange(len(A) + len(B) + 1)).all()


@pytest.mark.parametrize("m,n", [(0, 0), (0, 9), (9, 0), (1, 1), (7, 100), (5000, 3001),
                                 (4096, 4096)])
def test_merge_matches_stable_sort(m, n):
    rng = np.random.default_rng(m * 7919 + n)
    for dt, hi in ((np.int32, 64), (np.int32, 1 << 30), (np.uint64, 1 << 62)):
        A = np.sort(rng.integers(-hi if dt == np.int32 else 0, hi, size=m).astype(dt))
        B = np.sort(rng.integers(-hi if dt == np.int32 else 0, hi, size=n).astype(dt))
        Apay = rng.integers(0, 2**32, size=m, dtype=np.uint32)
        Bpay = rng.integers(0, 2**32, size=n, dtype=np.uint32)
        keys, pay, prov = oracle.merge(A, B, Apay, Bpay, provenance=True)
        cat = np.concatenate([A, B])
        order = np.argsort(cat, kind="stable")
        assert (keys == cat[order]).all()
        assert (pay == np.concatenate([Apay, Bpay])[order]).all()
        assert (prov == order).all()
        # partition entries agree with the stable-sort order at every tile cut
        D = 37
        part = oracle.partition(A, B, D)
        for g, (i, j) in enumerate(part):
            k = min(g * D, m + n)
            assert i + j == k and int((order[:k] < m).sum()) == i


# ---------------------------------------------------------------------------
# Bottom-up merge sort ([CH14] 14.2)
# ---------------------------------------------------------------------------
def test_mergesort_worked_example(golden):
    g = golden("mergesort_chapter14.txt")
    for dt in (np.int32, np.uint64):
        x = np.array(g["input"], dt)
        for w in (1, 2, 4):
            x, _ = oracle.merge_sort_pass(x, w)
            assert x.tolist() == g["after_width_%d" % w]
        keys, _, passes = oracle.merge_sort(np.array(g["input"], dt))
        assert keys.tolist() == g["after_width_4"] and passes == g["passes"][0]
    # the section's pair view: position 5 of the width-2 pass belongs to the
    # pair starting at 4, whose output is the merge of its two runs alone
    x1 = np.array(g["after_width_1"], np.int32)
    x2, _ = oracle.merge_sort_pass(x1, 2)
    p0, loc = g["pair_view_pair_start"][0], g["pair_view_local"][0]
    assert p0 + loc == g["pair_view_position"][0]
    pair = oracle.merge(x1[p0:p0 + 2], x1[p0 + 2:p0 + 4])[0]
    assert x2[p0:p0 + 4].tolist() == pair.tolist()


@pytest.mark.parametrize("n", [0, 1, 2, 3, 7, 8, 9, 1000, 4096, 4097, 30011])
def test_mergesort_matches_stable_sort(n):
    rng = np.random.default_rng(n + 17)
    for dt, lo, hi in ((np.int32, -8, 8), (np.int32, -2**31, 2**31 - 1),
                       (np.uint64, 0, 2**64 - 1), (np.uint64, 0, 5)):
        keys = rng.integers(lo, hi, size=n, dtype=np.int64 if dt == np.int32 else np.uint64,
                            endpoint=True).astype(dt)
        pay = np.arange(n, dtype=np.uint32)
        out, out_pay, passes = oracle.merge_sort(keys, pay)
        order = np.argsort(keys, kind="stable")
        assert (out == keys[order]).all()
        assert (out_pay == order).all()
        assert passes == (0 if n <= 1 else int(np.ceil(np.log2(n))))


def test_mergesort_brute_force_small():
    # every sequence of length <= 6 over {0, 1, 2}: the oracle's keys and
    # input positions against Python's stable sort of (key, position)
    for n in range(7):
        for seq in itertools.product(range(3), repeat=n):
            keys = np.array(seq, dtype=np.int32)
            out, pay, _ = oracle.merge_sort(keys, np.arange(n, dtype=np.uint32))
            want = sorted(range(n), key=lambda t: seq[t])
            assert pay.tolist() == want and out.tolist() == [seq[t] for t in want]


def test_mergesort_pass_keeps_a_lone_tail_run():
    # n = 7 at width 4: one pair [0, 8) clipped to 7 merges runs [0,4) and
    # [4,7); at width 8 the whole array is a lone run and is copied
    x = np.array([0, 1, 7, 9, 1, 2, 7], np.int32)
    y, p = oracle.merge_sort_pass(x, 8, np.arange(7, dtype=np.uint32))
    assert y.tolist() == x.tolist() and p.tolist() == list(range(7))
    y, p = oracle.merge_sort_pass(x, 4, np.arange(7, dtype=np.uint32))
    assert y.tolist() == [0, 1, 1, 2, 7, 7, 9]
    assert p.tolist() == [0, 1, 4, 5, 2, 6, 3]  # equal keys: left run first


# ---------------------------------------------------------------------------
# Replacement merge
# ---------------------------------------------------------------------------
def _chronological(A_keys, B_keys):
    """Apply A then B to a dict: the newer record replaces the older one."""
    d = {}
    for i, k in enumerate(A_keys):
        d[k] = (0, i)
    for j, k in enumerate(B_keys):
        d[k] = (1, j)
    return [(src << 31) | idx for _, (src, idx) in sorted(d.items())]


REPLACE_CASES = [  # (m, n, shared, universe)
    (0, 0, 0, 16), (0, 5, 0, 16), (5, 0, 0, 16), (1, 1, 1, 4), (1, 1, 0, 4),
    (64, 64, 64, 64 * 2), (64, 64, 0, 400), (33, 17, 9, 80), (1000, 300, 150, None),
    (513, 2049, 513, 4000), (2048, 2048, 1024, 5000),
]


@pytest.mark.parametrize("m,n,shared,universe", REPLACE_CASES)
def test_replacement_vs_chronological_map(m, n, shared, universe):
    inp = synth.replace_random_small(seed=m * 31 + n + shared, m=m, n=n, shared=shared,
                                     universe=universe)
    A, B = inp.A, inp.B
    r = oracle.replacement_u64(A, B)
    assert r.refs.tolist() == _chronological(A.tolist(), B.tolist())
    in_b = set(B.tolist())
    C_expected = synth._bitmap(np.array([i for i, k in enumerate(A.tolist()) if k in in_b],
                                        dtype=np.int64), m)
    assert (r.C == C_expected).all()


@pytest.mark.parametrize("m,n,shared,universe", REPLACE_CASES)
def test_replacement_invariants_and_formula_ordinals(m, n, shared, universe):
    inp = synth.replace_random_small(seed=m + 3 * n + shared, m=m, n=n, shared=shared,
                                     universe=universe)
    A, B = inp.A, inp.B
    r = oracle.replacement_u64(A, B)
    popc = int(sum(bin(int(w)).count("1") for w in r.C))
    assert r.count == m + n - popc == m + n - shared
    keys = np.array([B[x & 0x7FFFFFFF] if x >> 31 else A[x] for x in r.refs], np.uint64)
    assert (keys[1:] > keys[:-1]).all()
    assert sorted(int(x & 0x7FFFFFFF) for x in r.refs if x >> 31) == list(range(n))
    # the walk's ordinals and the closed forms (independent lower bounds) agree
    C2, lb2, ordA2, ordB2 = oracle.ordinals_formula_u64(A, B)
    assert (C2 == r.C).all() and (lb2 == r.lb_B).all()
    assert (ordA2 == r.ord_A).all() and (ordB2 == r.ord_B).all()
    # unique and gap-free over count slots
    live = np.concatenate([r.ord_A[r.ord_A != oracle.ORD_DROPPED], r.ord_B]).astype(np.int64)
    assert sorted(live.tolist()) == list(range(r.count))
    # lower bounds against numpy's searchsorted
    assert (r.lb_B == np.searchsorted(A, B, side="left")).all()


@pytest.mark.parametrize("m,n,shared,universe", REPLACE_CASES)
def test_materialized_survivors_vs_chronological_map(m, n, shared, universe):
    # Apply A then B, each record (key, value, tombstone), to a dict: the
    # surviving records in key order are the materialized output.
    inp = synth.replace_random_small(seed=m * 5 + n + 7 * shared, m=m, n=n, shared=shared,
                                     universe=universe)
    rng = np.random.default_rng(m + n + shared)
    valA = rng.integers(0, 2**32, m, dtype=np.uint32)
    valB = rng.integers(0, 2**32, n, dtype=np.uint32)
    tA = rng.random(m) < 0.2
    tB = rng.random(n) < 0.2
    tombA = synth._bitmap(np.nonzero(tA)[0].astype(np.int64), m)
    tombB = synth._bitmap(np.nonzero(tB)[0].astype(np.int64), n)
    d = {}
    for i, k in enumerate(inp.A.tolist()):
        d[k] = (int(valA[i]), bool(tA[i]))
    for j, k in enumerate(inp.B.tolist()):
        d[k] = (int(valB[j]), bool(tB[j]))
    items = sorted(d.items())
    r = oracle.replacement_u64(inp.A, inp.B)
    keys, vals, tomb = oracle.materialize_u64(inp.A, valA, tombA, inp.B, valB, tombB, r.refs)
    assert keys.tolist() == [k for k, _ in items]
    assert vals.tolist() == [v for _, (v, _) in items]
    flags = [bool((int(tomb[t // 32]) >> (t % 32)) & 1) for t in range(len(items))]
    assert flags == [f for _, (_, f) in items]
    if len(items) % 32:  # bits past the last record are zero
        assert int(tomb[-1]) >> (len(items) % 32) == 0


def test_replacement_skewed_generator_small():
    inp = synth.replace_skewed(seed=4, m=40000, windows=4, window=256,
                               per_window_shared=128, per_window_fresh=128)
    r = oracle.replacement_u64(inp.A, inp.B)
    assert r.count == len(inp.A) + len(inp.B) - inp.n_shared
    assert r.refs.tolist() == _chronological(inp.A.tolist(), inp.B.tolist())


def _str_cases():
    yield [b"", b"a", b"ab", b"abc"], [b"ab", b"b"]
    yield [b"\x00", b"\x00\x00", b"\xff"], [b"", b"\x00", b"\x00\x01", b"\xff\xff"]
    yield [], [b"x"]
    yield [b"x"], []
    yield [], []
    rng = np.random.default_rng(11)
    pool = sorted({bytes(rng.integers(0, 3, size=rng.integers(0, 5)).astype(np.uint8))
                   for _ in range(300)})
    pick = rng.permutation(len(pool))
    A = sorted(pool[t] for t in pick[: len(pool) // 2])
    B = sorted(set(pool[t] for t in pick[len(pool) // 3:]))
    yield A, B


@pytest.mark.parametrize("case", list(_str_cases()))
def test_replacement_str_vs_chronological_map(case):
    ka, kb = case
    s = synth.strings_from_lists(ka, kb)
    r = oracle.replacement_str(s.A.key_arena, s.A.key_off, s.B.key_arena, s.B.key_off)
    assert r.refs.tolist() == _chronological(ka, kb)
    assert r.count == len(r.refs)


def _side_keys(side):
    off = side.key_off.astype(np.int64)
    return [side.key_arena[off[t]:off[t + 1]].tobytes() for t in range(len(off) - 1)]


def _str_bitmap_cases():
    for ka, kb in _str_cases():
        yield synth.strings_from_lists(ka, kb)
    # stems: B keys that extend, shorten or equal A keys by one byte
    yield synth.strings_from_lists(
        [b"ab", b"abc", b"abd", b"b", b"b\x00\x00", b"ba"],
        [b"a", b"ab", b"abb", b"abc\x00", b"abd", b"b\x00", b"ba", b"bb"])
    # prefix-tree keys as in the string workload, small: shared 8-byte stems,
    # keys longer than the 16-byte prefix cache, 20 % of B drawn from A
    yield synth.strings(seed=17, count=3000, fanout=4, depth=4)
    yield synth.strings(seed=18, count=2000, fanout=2, depth=4, max_suffix=40, min_suffix=12)


@pytest.mark.parametrize("s", list(_str_bitmap_cases()))
def test_replacement_str_bitmap_and_lower_bounds(s):
    # C and lb_B of the string walk against Python's own byte order: bisect_left
    # over the sorted bytes list of A gives each B key's lower bound, and a set
    # membership test gives the collision bit of each A key ("Everett:
    # collision bitmap and rank experiment", "Corrected record ordinals").
    import bisect
    ka, kb = _side_keys(s.A), _side_keys(s.B)
    assert ka == sorted(ka) and kb == sorted(kb)
    r = oracle.replacement_str(s.A.key_arena, s.A.key_off, s.B.key_arena, s.B.key_off)
    lb = [bisect.bisect_left(ka, k) for k in kb]
    assert r.lb_B.tolist() == lb
    in_b = set(kb)
    hit = np.array([t for t, k in enumerate(ka) if k in in_b], dtype=np.int64)
    assert (r.C == synth._bitmap(hit, len(ka))).all()
    # the ordinals by the closed forms, with R(i) counted from the membership test
    R = np.concatenate([[0], np.cumsum([k in in_b for k in ka])]).astype(np.int64)
    ordA = [oracle.ORD_DROPPED if ka[t] in in_b else t + bisect.bisect_left(kb, ka[t]) - R[t]
            for t in range(len(ka))]
    ordB = [j + lb[j] - R[lb[j]] for j in range(len(kb))]
    assert r.ord_A.tolist() == ordA and r.ord_B.tolist() == ordB


# ---------------------------------------------------------------------------
# Rank and the rank512 directory
# ---------------------------------------------------------------------------
def _maps():
    rng = np.random.default_rng(5)
    for m in (0, 1, 31, 32, 33, 63, 64, 65, 511, 512, 513, 2047, 2048, 2049, 5000):
        for kind in ("zero", "one", "sparse", "random"):
            if kind == "zero":
                bits = np.zeros(m, bool)
            elif kind == "one":
                bits = np.ones(m, bool)
            elif kind == "sparse":
                bits = np.zeros(m, bool)
                for p in (0, 31, 32, 33, 63, 64, 65, 511, 512, 513, 2047, 2048, m - 1):
                    if 0 <= p < m:
                        bits[p] = True
            else:
                bits = rng.random(m) < 0.3
            yield m, kind, bits


def _pack(bits):
    return synth._bitmap(np.flatnonzero(bits).astype(np.int64), len(bits))


@pytest.mark.parametrize("m,kind,bits", list(_maps()))
def test_rank_prefix_and_directory(m, kind, bits):
    C = _pack(bits)
    R = oracle.rank_prefix(C, m)
    expect = np.concatenate([[0], np.cumsum(bits)]).astype(np.uint32)
    assert (R == expect).all()
    # The directory answers R(p) at every p in [0, m] by the page's query:
    # block prefix + packed 9-bit sub-prefix + at most one preceding 32-bit
    # word + the masked current word.
    d = oracle.rank512_dir(C, m)
    assert len(d) == 3 * (m // 512 + 1)
    for p in range(m + 1):
        b, s = p // 512, (p % 512) // 64
        r = int(d[3 * b])
        if s:
            packed = int(d[3 * b + 1]) | (int(d[3 * b + 2]) << 32)
            r += (packed >> (9 * (s - 1))) & 0x1FF
        w = p // 32
        if p % 64 >= 32:
            r += bin(int(C[w - 1])).count("1")
        if p % 32:
            r += bin(int(C[w]) & ((1 << (p % 32)) - 1)).count("1")
        assert r == expect[p], (m, kind, p)
    q = np.arange(m + 1, dtype=np.uint32)
    assert (oracle.rank_query(C, m, q) == expect).all()


def _maps2048():
    yield from _maps()
    rng = np.random.default_rng(6)
    for m in (4095, 4096, 4097, 6143, 6144, 6145, 10000):
        yield m, "one", np.ones(m, bool)
        yield m, "random", rng.random(m) < 0.5


@pytest.mark.parametrize("m,kind,bits", list(_maps2048()))
def test_rank2048_directory(m, kind, bits):
    C = _pack(bits)
    expect = np.concatenate([[0], np.cumsum(bits)]).astype(np.uint64)
    d, ep = oracle.rank2048_dir(C, m)
    assert len(d) == m // 2048 + 1 and len(ep) == 1 and ep[0] == 0
    # the fields: relative count at the block start, then the populations of
    # the block's first three 512-bit runs, ten bits each
    for b in range(len(d)):
        e = int(d[b])
        assert e & 0xFFFFFFFF == expect[2048 * b]
        for r in range(3):
            lo, hi = min(2048 * b + 512 * r, m), min(2048 * b + 512 * (r + 1), m)
            assert (e >> (32 + 10 * r)) & 0x3FF == int(bits[lo:hi].sum())
        assert e >> 62 == 0
    # the query procedure answers R(p) at every position, EOF included
    q = np.arange(m + 1, dtype=np.uint64)
    assert (oracle.rank2048_query(C, d, ep, q) == expect).all()


def test_rank2048_epochs_past_2pow32():
    # all ones past one epoch: R(p) = p, the second epoch holds 2^32 and its
    # first entry counts from zero again
    m = (1 << 32) + 5000
    C = np.full((m + 31) // 32, 0xFFFFFFFF, dtype=np.uint32)
    C[-1] = (1 << (m % 32)) - 1
    d, ep = oracle.rank2048_dir(C, m)
    assert ep.tolist() == [0, 1 << 32]
    b = (1 << 32) // 2048
    assert int(d[b]) & 0xFFFFFFFF == 0 and int(d[b - 1]) & 0xFFFFFFFF == (1 << 32) - 2048
    pos = np.array([0, 1, (1 << 32) - 1, 1 << 32, (1 << 32) + 1, (1 << 32) + 2047,
                    (1 << 32) + 2048, (1 << 32) + 4999, m], dtype=np.uint64)
    assert (oracle.rank2048_query(C, d, ep, pos) == pos).all()


# ---------------------------------------------------------------------------
# Front compression
# ---------------------------------------------------------------------------
def test_eg0_closed_form_and_textbook_code():
    xs = list(range(1 << 16)) + [(1 << s) + d for s in range(16, 21) for d in (-2, -1, 0, 1)]
    xs += np.random.default_rng(3).integers(0, 1 << 20, size=2000).tolist()
    for x in xs:
        z = (x + 1).bit_length() - 1            # floor(log2(x+1))
        textbook = "0" * z + bin(x + 1)[2:]     # order-0 Exp-Golomb code word
        assert oracle.eg0_len(x) == 2 * z + 1 == len(textbook)
    for x in xs[:4096:7] + xs[-50:]:
        z = (x + 1).bit_length() - 1
        assert oracle.eg0_bits(x) == "0" * z + bin(x + 1)[2:]


def _encode_strings(s, refs):
    return oracle.fc_encode((s.A.key_arena, s.A.key_off), (s.A.val_arena, s.A.val_off), s.A.tomb,
                            (s.B.key_arena, s.B.key_off), (s.B.val_arena, s.B.val_off), s.B.tomb,
                            refs)


def test_fc_hand_derived(golden):
    g = golden("fc_hand_derived.txt")
    for name, val in (("one_tomb", None), ("one_empty", b"")):
        s = synth.strings_from_lists([bytes(g[name + "_key"])], [], [val], [])
        fc = _encode_strings(s, np.array([0], np.uint32))
        assert fc.total_bits == g[name + "_bits"][0]
        assert fc.payload.tolist() == g[name + "_words"]
    s = synth.strings_from_lists([b"ab", b"ac"], [], [None, b"\xff"], [])
    fc = _encode_strings(s, np.array([0, 1], np.uint32))
    assert fc.total_bits == g["two_bits"][0]
    assert fc.lcp.tolist() == g["two_lcp"]
    assert fc.ctrl.tolist() == g["two_ctrl"]
    assert fc.rec_bits.tolist() == g["two_rec_bits"]
    assert fc.payload.tolist() == g["two_words"]


def _bit_lcp(x: bytes, y: bytes) -> int:
    """Leading equal bits of two byte strings, clamped to the shorter one."""
    n = min(len(x), len(y))
    if n == 0:
        return 0
    a = int.from_bytes(x[:n], "big")
    b = int.from_bytes(y[:n], "big")
    return 8 * n - (a ^ b).bit_length()


def _check_fc_roundtrip(s):
    r = oracle.replacement_str(s.A.key_arena, s.A.key_off, s.B.key_arena, s.B.key_off)
    fc = _encode_strings(s, r.refs)
    N = r.count
    keys = [s.B.key(x & 0x7FFFFFFF) if x >> 31 else s.A.key(x) for x in r.refs]
    vals = [s.B.value(x & 0x7FFFFFFF) if x >> 31 else s.A.value(x) for x in r.refs]
    assert int(fc.bit_off[N]) == fc.total_bits == int(fc.rec_bits.astype(np.int64).sum())
    assert (np.diff(fc.bit_off.astype(np.int64)) == fc.rec_bits).all()
    for i in range(N):
        assert fc.lcp[i] == (0 if i == 0 else _bit_lcp(keys[i - 1], keys[i]))
        if i > 0:
            assert 8 * len(keys[i]) - fc.lcp[i] >= 1       # strictly increasing keys
    if N:
        assert fc.ctrl[0] == 1
    key_cap = sum(len(k) for k in keys)
    val_cap = sum(len(v) for v in vals if v is not None)
    (ka, ko), (va, vo), tomb = oracle.fc_decode(fc.payload, fc.total_bits, N, key_cap, val_cap)
    for i in range(N):
        assert bytes(ka[int(ko[i]):int(ko[i + 1])]) == keys[i]
        is_tomb = (int(tomb[i // 32]) >> (i % 32)) & 1
        assert bool(is_tomb) == (vals[i] is None)
        if vals[i] is not None:
            assert bytes(va[int(vo[i]):int(vo[i + 1])]) == vals[i]
    return fc


def test_fc_roundtrip_edge_keys():
    ka = [b"", b"\x00", b"\x00\x00", b"\x00\x01", b"\x7f", b"\x80", b"ab", b"abc", b"abd",
          b"b" * 40, b"b" * 41, b"\xff" * 3]
    kb = [b"\x00", b"\x00\x00\x00", b"abc", b"b" * 40 + b"\x01", b"\xff\xff"]
    va = [None, b"", b"\x01", None, b"xyz", b"", b"\x00" * 16, None, b"q", b"", None, b"z"]
    vb = [None, b"new", None, b"", b"\xff" * 16]
    _check_fc_roundtrip(synth.strings_from_lists(ka, kb, va, vb))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_fc_roundtrip_prefix_tree(seed):
    s = synth.strings(seed=seed, count=700, fanout=4, depth=2, max_suffix=12)
    fc = _check_fc_roundtrip(s)
    # restarts every 15 records: c_i = 1 + l_i there
    assert fc.ctrl[15] == 1 + fc.lcp[15] and fc.ctrl[30] == 1 + fc.lcp[30]


def test_synth_is_deterministic():
    a = synth.replace_u64(seed=9, m=1000, n=300)
    b = synth.replace_u64(seed=9, m=1000, n=300)
    assert (a.A == b.A).all() and (a.B == b.B).all() and (a.tombB == b.tombB).all()
    assert len(np.unique(a.A)) == 1000 and len(np.intersect1d(a.A, a.B)) == a.n_shared
    s1 = synth.strings(seed=9, count=300, fanout=4, depth=2, max_suffix=6)
    s2 = synth.strings(seed=9, count=300, fanout=4, depth=2, max_suffix=6)
    assert (s1.A.key_arena == s2.A.key_arena).all() and (s1.B.key_off == s2.B.key_off).all()


# ---------------------------------------------------------------------------
# Elias-Fano navigation over record offsets ([GC])
# ---------------------------------------------------------------------------
def _bits_le(words, nbits):
    """Bits 0..nbits-1 of a uint64 array, bit t in word t/64 at position t%64."""
    b = np.unpackbits(np.asarray(words, dtype="<u8").view(np.uint8), bitorder="little")
    return b[:nbits], b[nbits:]


def _ef_expect(bit_off, N, w):
    ords = list(range(0, N, 15)) + [N]
    return [int(bit_off[o]) - o * w for o in ords]


def _check_ef(bit_off, N, w=0):
    x = _ef_expect(bit_off, N, w)
    ef = oracle.ef_build(bit_off, N, w)
    n, L, U = len(x), ef.L, x[-1]
    assert ef.n == n
    # L: the largest L with n 2^L <= U, or 0
    assert (n << L) <= U < (n << (L + 1)) if L else U < 2 * n
    # lows: x mod 2^L at [sL, sL + L), nothing past nL
    lo, pad = _bits_le(ef.lows, n * L)
    assert not pad.any() and len(ef.lows) == (n * L + 63) // 64
    for s_ in range(n):
        v = sum(int(lo[s_ * L + b]) << b for b in range(L))
        assert v == x[s_] & ((1 << L) - 1)
    # highs: one set bit per entry, x recovered from its position
    nh = (U >> L) + n
    hi, pad = _bits_le(ef.highs, nh)
    assert not pad.any() and len(ef.highs) == (nh + 63) // 64
    h = np.flatnonzero(hi)
    assert len(h) == n
    for s_ in range(n):
        assert ((int(h[s_]) - s_) << L) | (x[s_] & ((1 << L) - 1)) == x[s_]
    # samples and sparse exceptions, group by group
    e = 0
    exc = []
    for g in range((n + 255) // 256):
        first, last = 256 * g, min(256 * g + 255, n - 1)
        sp = int(h[last] - h[first]) >= 4096
        assert int(ef.samples[2 * g]) == h[first]
        assert int(ef.samples[2 * g + 1]) == (e << 1) | int(sp)
        if sp:
            exc += [int(v) for v in h[first:last + 1]]
            e += last - first + 1
    assert [int(v) for v in ef.sparse] == exc
    return ef


def _offsets(rng, N, lo, hi):
    return np.concatenate([[0], np.cumsum(rng.integers(lo, hi, size=N))]).astype(np.uint64)


@pytest.mark.parametrize("N", [0, 1, 14, 15, 16, 29, 30, 31, 3839, 3840, 3841, 100_000])
def test_ef_sections_decode(N):
    rng = np.random.default_rng(N + 5)
    _check_ef(_offsets(rng, N, 3, 400), N)
    # a common value width w: every record at least w bits long
    _check_ef(_offsets(rng, N, 40, 60), N, w=40)
    _check_ef(_offsets(rng, N, 1, 2), N, w=1)  # every x equal: repeated entries


def test_ef_sparse_threshold_exact():
    # 4001 entries; group 0 climbs to x_255 and everything after repeats it,
    # so L = 0 and group 0 spans x_255 + 255 high positions
    for top, sparse in ((3840, False), (3841, True)):
        n = 4001
        x = np.zeros(n, dtype=np.uint64)
        x[1:255] = np.arange(1, 255)
        x[255:] = top
        N = 15 * (n - 1)
        bit_off = np.repeat(x[:-1], 15)
        bit_off = np.concatenate([bit_off, [x[-1]]]).astype(np.uint64)
        ef = _check_ef(bit_off, N)
        assert ef.L == 0 and (int(ef.samples[1]) & 1) == int(sparse)
        assert len(ef.sparse) == (256 if sparse else 0)


def test_ef_over_an_fc_scan():
    # the sequence the FC length scan produces for the prefix-tree keys
    s = synth.strings(seed=9, count=3000)
    r = oracle.replacement_str(s.A.key_arena, s.A.key_off, s.B.key_arena, s.B.key_off)
    fc = _encode_strings(s, r.refs)
    _check_ef(fc.bit_off, r.count)


# ---------------------------------------------------------------------------
# Byte-profile front compression ([BP] "Pipeline")
# ---------------------------------------------------------------------------
def test_leb128_standard_values():
    # unsigned LEB128 as the DWARF standard defines and tabulates it
    table = {0: [0x00], 1: [0x01], 2: [0x02], 127: [0x7F], 128: [0x80, 0x01],
             129: [0x81, 0x01], 130: [0x82, 0x01], 12857: [0xB9, 0x64],
             624485: [0xE5, 0x8E, 0x26], (1 << 32) - 1: [0xFF, 0xFF, 0xFF, 0xFF, 0x0F]}
    for x, want in table.items():
        assert oracle.leb128(x) == want
    # every x decodes back (seven bits per byte, low group first) and only
    # the last byte lacks the continuation bit
    for x in list(range(1 << 15)) + [(1 << k) + d for k in range(15, 63) for d in (-1, 0, 1)]:
        b = oracle.leb128(x)
        assert sum((v & 0x7F) << (7 * t) for t, v in enumerate(b)) == x
        assert all(v & 0x80 for v in b[:-1]) and not b[-1] & 0x80
        assert len(b) == max(1, (x.bit_length() + 6) // 7)


def test_bytefc_hand_derived(golden):
    g = golden("bytefc_hand_derived.txt")
    s = synth.strings_from_lists([b"ab", b"ac"], [], [None, b"\xff"], [])
    refs = np.array([0, 1], np.uint32)
    fc = oracle.bytefc_encode((s.A.key_arena, s.A.key_off), (s.A.val_arena, s.A.val_off),
                              s.A.tomb, (s.B.key_arena, s.B.key_off),
                              (s.B.val_arena, s.B.val_off), s.B.tomb, refs)
    assert fc.lcp.tolist() == g["two_keys_lcp"] and fc.ctrl.tolist() == g["two_keys_ctrl"]
    assert fc.rec_bits.tolist() == g["two_keys_rec"]
    assert fc.payload.tolist() == g["two_keys_payload"]
    s = synth.strings_from_lists([b"A"], [], [bytes(range(16))], [])
    fc = oracle.bytefc_encode((s.A.key_arena, s.A.key_off), (s.A.val_arena, s.A.val_off),
                              s.A.tomb, (s.B.key_arena, s.B.key_off),
                              (s.B.val_arena, s.B.val_off), s.B.tomb,
                              np.array([0], np.uint32), W=17)
    assert fc.payload.tolist() == g["w17_payload"]


def _byte_lcp(x: bytes, y: bytes) -> int:
    n = 0
    while n < min(len(x), len(y)) and x[n] == y[n]:
        n += 1
    return n


def _check_bytefc_roundtrip(s, W=0):
    r = oracle.replacement_str(s.A.key_arena, s.A.key_off, s.B.key_arena, s.B.key_off)
    N = r.count
    fc = oracle.bytefc_encode((s.A.key_arena, s.A.key_off), (s.A.val_arena, s.A.val_off),
                              s.A.tomb if len(s.A.tomb) else None,
                              (s.B.key_arena, s.B.key_off), (s.B.val_arena, s.B.val_off),
                              s.B.tomb if len(s.B.tomb) else None, r.refs, W=W)
    keys = [s.B.key(x & 0x7FFFFFFF) if x >> 31 else s.A.key(x) for x in r.refs]
    vals = [s.B.value(x & 0x7FFFFFFF) if x >> 31 else s.A.value(x) for x in r.refs]
    assert int(fc.bit_off[N]) == fc.total_bits == int(fc.rec_bits.astype(np.int64).sum())
    for i in range(N):
        p = 0 if i == 0 else _byte_lcp(keys[i - 1], keys[i])
        assert fc.lcp[i] == p
        assert fc.ctrl[i] == (1 + p if i % 15 == 0 else len(keys[i - 1]) - p)
        v = 1 if vals[i] is None else (W if W else 1 + len(oracle.leb128(len(vals[i]))) + len(vals[i]))
        assert fc.rec_bits[i] == (len(oracle.leb128(int(fc.ctrl[i]))) +
                                  len(oracle.leb128(len(keys[i]) - p)) + len(keys[i]) - p + v)
    key_cap = sum(len(k) for k in keys)
    val_cap = sum(len(v) for v in vals if v is not None)
    (ka, ko), (va, vo), tomb = oracle.bytefc_decode(fc.payload, N, W, key_cap, val_cap)
    for i in range(N):
        assert bytes(ka[int(ko[i]):int(ko[i + 1])]) == keys[i]
        assert bool((int(tomb[i // 32]) >> (i % 32)) & 1) == (vals[i] is None)
        if vals[i] is not None:
            assert bytes(va[int(vo[i]):int(vo[i + 1])]) == vals[i]
    return fc


@pytest.mark.parametrize("seed", [1, 2])
def test_bytefc_roundtrip_prefix_tree(seed):
    _check_bytefc_roundtrip(synth.strings(seed=seed, count=2000))


def test_bytefc_roundtrip_edges_and_common_width():
    _check_bytefc_roundtrip(synth.strings_from_lists(
        [b"", b"a", b"ab", b"abc" * 60, b"b"], [b"a", b"abd", b"c" * 300],
        [None, b"", b"x" * 200, b"y", None], [b"1", None, b""]))
    rng = np.random.default_rng(4)
    keysA = sorted({bytes(rng.integers(0, 256, size=int(rng.integers(1, 20)), dtype=np.uint8))
                    for _ in range(300)})
    keysB = sorted(set(keysA[::3]) | {bytes([200 + t % 50]) * (t % 7 + 1) for t in range(40)})
    valsA = [bytes(rng.integers(0, 256, size=16, dtype=np.uint8)) for _ in keysA]
    valsB = [bytes(rng.integers(0, 256, size=16, dtype=np.uint8)) for _ in keysB]
    s = synth.strings_from_lists(keysA, keysB, valsA, valsB)
    _check_bytefc_roundtrip(s, W=17)


def _width_case(keysA, valsA, keysB, valsB):
    s = synth.strings_from_lists(keysA, keysB, valsA, valsB)
    r = oracle.replacement_str(s.A.key_arena, s.A.key_off, s.B.key_arena, s.B.key_off)
    return oracle.bytefc_value_width(s.A.val_off, s.A.tomb, s.B.val_off, s.B.tomb, r.refs)


def test_bytefc_value_width_special_cases():
    v16, v15 = b"v" * 16, b"w" * 15
    # every survivor present with sixteen value bytes: width 17 ([BP] "Pipeline")
    assert _width_case([b"a", b"b"], [v16, v16], [b"c"], [v16]) == 17
    # a tombstone or a value of another length anywhere: no common width
    assert _width_case([b"a", b"b"], [v16, None], [b"c"], [v16]) == 0
    assert _width_case([b"a", b"b"], [v16, v15], [b"c"], [v16]) == 0
    # the odd records replaced by newer ones of the common length: width 17
    assert _width_case([b"a", b"b", b"c"], [v16, v15, None], [b"b", b"c"], [v16, v16]) == 17
    # a newer tombstone survives and breaks it
    assert _width_case([b"a", b"b"], [v16, v16], [b"b"], [None]) == 0
    # empty values make width 1 (the tag alone); no records, no width
    assert _width_case([b"a"], [b""], [b"b"], [b""]) == 1
    assert _width_case([], [], [], []) == 0
