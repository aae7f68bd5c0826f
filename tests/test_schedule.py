"""Host-side checks of the prefix pass's schedule (no GPU): the planner's choice
between fixed-length key splits and key-range groups, and the units of the groups.

Key-range groups lay the requests' 64-key steps end to end and cut them into G
equal ranges; the pairs of group g compute every row tile over range g, one unit
per request it touches, and a request's piece k (its k-th range) goes to split
slot k.  The expected units here are built from that definition directly, step by
step, and compared with the library's enumeration, which the kernels share.
"""
import ctypes

import numpy as np
import pytest

from speculative_decoding_tree_05_gb300 import ddtree

STEP = 64


@pytest.fixture(scope="module")
def lib():
    L = ddtree.lib()
    L.ddtree_internal_group_unit.restype = ctypes.c_int
    L.ddtree_internal_group_unit.argtypes = [ctypes.POINTER(ctypes.c_int32), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int32)]
    return L


def plan(lib, sm_count=152, **kw):
    return ddtree.plan(ddtree.make_dims(**kw), sm_count, library=lib)


def lib_units(lib, lens, max_len, G):
    arr = (ctypes.c_int32 * len(lens))(*[int(x) for x in lens])
    out = (ctypes.c_int32 * 4)()
    units = {}
    for g in range(G):
        units[g] = []
        for idx in range(len(lens) + 2):
            if not lib.ddtree_internal_group_unit(arr, len(lens), max_len, G, g, idx, out):
                break
            units[g].append(tuple(out))
        else:
            raise AssertionError("a group has more units than requests")
    pieces = []
    for b in range(len(lens)):
        lib.ddtree_internal_group_unit(arr, len(lens), max_len, G, -1, b, out)
        pieces.append(out[0])
    return units, pieces


def expected_units(lens, max_len, G):
    """The definition, one step at a time: owner group of each step, then maximal runs."""
    G0 = G
    L = [min(max(int(x), 0), max_len) for x in lens]
    seq = [(b, s) for b in range(len(L)) for s in range(-(-L[b] // STEP))]  # steps end to end
    K = len(seq)
    G = min(G, K)  # with fewer steps than groups, one step for each of the first K groups
    owner = [0] * K
    for g in range(G):
        for x in range(g * K // G, (g + 1) * K // G):
            owner[x] = g
    units = {g: [] for g in range(G)}
    first_group = {}
    for x, (b, s) in enumerate(seq):
        first_group.setdefault(b, owner[x])
        g = owner[x]
        u = units[g]
        if u and u[-1][0] == b:
            u[-1][2] = min(L[b], (s + 1) * STEP)
        else:
            u.append([b, s * STEP, min(L[b], (s + 1) * STEP), g - first_group[b]])
    pieces = [len({owner[x] for x, (bb, _) in enumerate(seq) if bb == b}) for b in range(len(L))]
    return {g: [tuple(u) for u in units.get(g, [])] for g in range(G0)}, pieces


CASES = [
    ([48985, 63695, 45409, 37138, 95408, 45001, 112679, 51321], 131072, 15),  # a batch of mixed lengths
    ([4096, 131072], 131072, 38),
    ([1, 2, 63, 64, 65, 0, 129], 200, 5),        # ragged tails, an empty request
    ([0, 0, 0], 10, 4),                          # nothing to do
    ([100, 0, 300], 300, 16),                    # more groups than steps: some groups are empty
    ([-5, 70, 999], 128, 3),                     # out-of-range lengths are clamped like the kernels do
    ([64] * 64, 64, 76),                         # 64 one-step requests
]


@pytest.mark.parametrize("lens,max_len,G", CASES)
def test_group_units_match_the_definition(lib, lens, max_len, G):
    got, pieces = lib_units(lib, lens, max_len, G)
    want, want_pieces = expected_units(lens, max_len, G)
    assert got == want
    assert pieces == want_pieces


def test_group_units_cover_every_key_once(lib):
    rng = np.random.default_rng(7)
    for _ in range(40):
        B = int(rng.integers(2, 65))
        max_len = int(rng.integers(1, 5000))
        lens = rng.integers(0, max_len + 1, B)
        G = int(rng.integers(1, 80))
        units, pieces = lib_units(lib, lens, max_len, G)
        seen = [np.zeros(int(x), np.int32) for x in lens]
        slots = [set() for _ in lens]
        steps = []
        for g, us in units.items():
            n = 0
            for b, kb, ke, piece in us:
                assert 0 <= kb < ke <= lens[b] and kb % STEP == 0
                seen[b][kb:ke] += 1
                assert piece not in slots[b]
                slots[b].add(piece)
                n += -(-(ke - kb) // STEP)
            steps.append(n)
        assert all((s == 1).all() for s in seen)                      # every key exactly once
        assert all(slots[b] == set(range(pieces[b])) for b in range(B))  # pieces 0 .. n-1, each once
        used = [n for n in steps if n > 0] or [0]
        assert max(used) - min(used) <= 1                              # equal shares of the steps
        assert sum(n > 0 for n in steps) == min(G, sum(-(-int(x) // STEP) for x in lens))  # no empty group while steps remain


def test_planner_takes_groups_for_a_mixed_batch(lib):
    # 8 requests, 33 nodes x 16 heads (5 row tiles), prefixes of 37k..113k keys: 15 groups of 5 pairs
    lens = [48985, 63695, 45409, 37138, 95408, 45001, 112679, 51321]
    p = plan(lib, batch=8, nodes=33, heads=16, pool_slots=8 << 20, slot_stride=max(lens), max_prefix_len=max(lens),
             prefix_len_sum=sum(lens))
    assert p["row_tiles"] == 5 and p["groups"] == 15


@pytest.mark.parametrize("kw", [
    dict(batch=1, nodes=65, heads=128, pool_slots=2 << 20, slot_stride=65536, max_prefix_len=65536),  # one request
    dict(batch=1, nodes=9, heads=16, pool_slots=4 << 20, slot_stride=185000, max_prefix_len=185000),
    dict(batch=2, nodes=65, heads=128, pool_slots=2 << 20, slot_stride=8192, max_prefix_len=8192),  # 65 tiles each
    dict(batch=65, nodes=9, heads=16, pool_slots=1 << 20, slot_stride=4096, max_prefix_len=4096),   # over 64 requests
])
def test_planner_keeps_splits(lib, kw):
    assert plan(lib, **kw)["groups"] == 0


def test_planner_long_first_split_for_one_request_with_many_tiles(lib):
    # 65 row tiles of one 65536-key request on 76 pairs: the 65 first units take 882 steps while the
    # 11 free pairs run the 65 second units of 142 steps, six each (888 step times against 6 x 153)
    p = plan(lib, batch=1, nodes=65, heads=128, pool_slots=2 << 20, slot_stride=65536, max_prefix_len=65536)
    assert p["groups"] == 0 and p["splits"] == 2
    assert (p["chunk0"], p["chunk"]) == (882 * STEP, 142 * STEP)
    assert p["chunk0"] + p["chunk"] == 65536


@pytest.mark.parametrize("kw,splits", [
    (dict(batch=1, nodes=65, heads=16, pool_slots=1 << 20, slot_stride=8192, max_prefix_len=8192), 8),
    (dict(batch=1, nodes=9, heads=16, pool_slots=4 << 20, slot_stride=185000, max_prefix_len=185000), 38),
])
def test_planner_equal_splits_when_tiles_are_few(lib, kw, splits):
    p = plan(lib, **kw)
    assert p["groups"] == 0 and p["splits"] == splits and p["chunk0"] == p["chunk"]
