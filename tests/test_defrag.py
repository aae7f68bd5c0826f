"""Host-side defragmentation policy: fragmentation metric, sorted free list, compaction plan."""
import numpy as np
import pytest

from speculative_decoding_tree_05_gb300 import defrag
from speculative_decoding_tree_05_gb300 import workloads as wl


def test_contiguous_runs_and_fragmentation():
    assert defrag.contiguous_runs([5, 6, 7, 10, 11, 3]).tolist() == [3, 2, 1]
    assert defrag.contiguous_runs([]).tolist() == []
    f = defrag.fragmentation([5, 6, 7, 10, 11, 3], step=2)
    # steps (5,6) contiguous, (7,10) not, (11,3) not
    assert f["runs"] == 3 and f["keys"] == 6 and f["contiguous_steps"] == pytest.approx(1 / 3)
    g = defrag.fragmentation(np.arange(100, 100 + 3 * 64 + 5))
    assert g["runs"] == 1 and g["contiguous_steps"] == 1.0
    # one break inside the second step only
    s = np.arange(1000, 1000 + 3 * 64)
    s[64 + 10:] += 7
    h = defrag.fragmentation(s)
    assert h["runs"] == 2 and h["contiguous_steps"] == pytest.approx(2 / 3)


def test_sorted_free_list():
    fl = defrag.SortedFreeList(32)
    assert fl.free_count == 31 and fl.alloc(3).tolist() == [1, 2, 3]
    fl.release([2])
    assert fl.alloc(2).tolist() == [2, 4]          # lowest free slots first
    with pytest.raises(ValueError):
        fl.release([5])                               # already free
    fl = defrag.SortedFreeList(32, free_slots=[3, 4, 9, 10, 11, 12, 20])
    assert fl.find_run(3) == 9 and fl.find_run(5) == -1 and fl.find_run(1) == 3
    assert fl.take_run(10, 2).tolist() == [10, 11]
    assert fl.free.tolist() == [3, 4, 9, 12, 20]
    with pytest.raises(ValueError):
        fl.take_run(3, 3)                             # 5 is not free
    with pytest.raises(MemoryError):
        fl.alloc(6)
    with pytest.raises(ValueError):
        defrag.SortedFreeList(8, free_slots=[0, 1])   # slot 0 is the pad slot


def test_plan_compaction_moves_fragmented_requests_to_disjoint_runs():
    rng = np.random.default_rng(7)
    pool = 1 << 15
    fifo = wl.churned_allocator(rng, pool, keep_free=12000, max_alloc=512)
    lens = [3000, 0, 1200, 700, 64]
    tables = [fifo.alloc(L) for L in lens]
    assert defrag.fragmentation(tables[0])["contiguous_steps"] < 1.0
    # the churned pool is the lower half of a pool twice as large whose upper half is free
    big = 2 * pool
    free = defrag.SortedFreeList(big, free_slots=np.concatenate(list(fifo.segments) + [np.arange(pool, big)]))
    assert free.find_run(sum(lens)) >= pool
    free_before = free.free_count
    live = np.concatenate([t for t in tables if t.size])
    # a host stand-in for the pool rows: each slot's row holds its own id
    rows = np.arange(big, dtype=np.int64)[:, None] * np.array([[1, -1, 3]])
    plan = defrag.plan_compaction(tables, lens, free)
    assert len(plan.requests) == len(plan.dst_start)
    dsts = []
    for b, s in zip(plan.requests, plan.dst_start):
        run = np.arange(s, s + lens[b])
        assert s >= 1 and run[-1] < big
        assert np.intersect1d(run, live).size == 0   # never overwrites a live row (in-place safe)
        dsts.append(run)
    if dsts:
        allr = np.concatenate(dsts)
        assert np.unique(allr).size == allr.size     # runs are pairwise disjoint
    assert free.free_count == free_before - sum(lens[b] for b in plan.requests)
    # the copy (what ddtree.kv_compact does on the device) and the table rewrite
    new_tables = [t.copy() for t in tables]
    for b, s in zip(plan.requests, plan.dst_start):
        rows[s:s + lens[b]] = rows[tables[b]]
        new_tables[b] = np.arange(s, s + lens[b])
    for b, L in enumerate(lens):
        if L:
            assert np.array_equal(rows[new_tables[b]][:, 0], tables[b])  # same logical rows
    defrag.finish_compaction(plan, tables, lens, free)
    assert free.free_count == free_before
    for b in plan.requests:
        f = defrag.fragmentation(new_tables[b])
        assert f["runs"] == 1 and f["contiguous_steps"] == 1.0
    # every fragmented request was moved (the free upper half fits them all)
    moved = set(plan.requests.tolist())
    for b, L in enumerate(lens):
        if L and defrag.fragmentation(tables[b])["contiguous_steps"] < 1.0:
            assert b in moved


# ----------------------------------------------------------------------------- kv_compact aliasing validator

def _check(slot_idx, prefix_len, dst_start, pool=1000, same_pool=True, tree=None):
    from speculative_decoding_tree_05_gb300 import build, ddtree
    build.build()
    return ddtree.kv_compact_check(np.asarray(slot_idx), np.asarray(prefix_len), np.asarray(dst_start), pool,
                                   same_pool=same_pool, tree_slot_idx=tree)


def test_compact_check_accepts_disjoint_plan():
    assert _check([[5, 9, 7], [1, 2, 3]], [3, 3], [100, 200]) == (0, -1)


def test_compact_check_rejects_destination_over_live_source():
    # request 1's source slot 101 lies in request 0's destination [100, 103)
    assert _check([[5, 9, 7], [101, 2, 3]], [3, 3], [100, 200]) == (-7, 101)


def test_compact_check_allows_rows_already_in_place():
    assert _check([[100, 101, 7]], [3], [100]) == (0, -1)


def test_compact_check_rejects_overlapping_destinations():
    assert _check([[5, 9, 7], [1, 2, 3]], [3, 3], [100, 102]) == (-7, 102)


def test_compact_check_rejects_destination_outside_pool():
    assert _check([[5, 9, 7]], [3], [998], pool=1000)[0] == -7


def test_compact_check_two_pools_ignore_sources():
    assert _check([[100, 9, 7]], [3], [99], same_pool=False) == (0, -1)
    assert _check([[100, 9, 7]], [3], [99], same_pool=True) == (-7, 100)


def test_compact_check_protects_tree_rows():
    assert _check([[5, 9, 7]], [3], [100], tree=[[50, 102]]) == (-7, 102)
    assert _check([[5, 9, 7]], [3], [100], tree=[[50, 103]]) == (0, -1)


def test_compact_check_accepts_the_defrag_plan():
    # the planner's in-place plan for a churned pool satisfies the contract
    w = wl.make_workload("tiny", batch=3, prefix=("list", 700, 300, 900), nodes=9, heads=2, pool_slots=1 << 14,
                         slots="churn")
    used = w.used_slots()
    free = np.setdiff1d(np.arange(1, w.pool_slots), used)
    plan = defrag.plan_compaction(w.slot_idx, w.prefix_len, defrag.SortedFreeList(w.pool_slots, free))
    assert len(plan.requests) > 0
    r = plan.requests
    rc, bad = _check(w.slot_idx[r], w.prefix_len[r], plan.dst_start, pool=w.pool_slots, tree=w.tree_slot_idx[r])
    assert rc == 0, bad
    # a plan that puts a request's destination over its own live rows (shifted by 3) is caught
    bad_start = plan.dst_start.copy()
    bad_start[0] = int(w.slot_idx[r[0], 5]) - 3
    rc, bad = _check(w.slot_idx[r], w.prefix_len[r], bad_start, pool=w.pool_slots)
    assert rc == -7
