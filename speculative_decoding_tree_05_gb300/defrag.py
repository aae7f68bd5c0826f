"""Host-side defragmentation policy for a page_size=1 KV slot pool.

With one token per slot, a free list churned by serving hands a long request
scattered slots, and every verify step then gathers its prefix row by row.  The
pages propose keeping the free list sorted and compacting a request's rows into
one contiguous run ("The Architecture Detective: Uncovering FlashMLA's
Potential for Blackwell DDTree Verification", sections "The Message in Full"
and "Defragmentation: Separating Signal from Noise").  This module is that
policy on the host:

* `fragmentation` measures a slot table: runs of consecutive slots, and the
  share of 64-key steps whose slots are all consecutive (such a step is loaded
  by the prefix kernel as tiled TMA boxes instead of a row gather);
* `SortedFreeList` keeps the free slots in ascending order, so an allocation
  takes the lowest free slots and a contiguous run can be found first-fit;
* `plan_compaction` picks, for fragmented requests, a free contiguous run to
  move them to.  The runs come from the free list, so they are disjoint from
  every live slot and from each other, which is what an in-place
  `ddtree_kv_compact` (kv_dst == kv_src) requires; the device copy itself is
  the library's kernel.
"""
from __future__ import annotations

import dataclasses

import numpy as np

STEP_KEYS = 64  # keys per prefix-kernel step


def contiguous_runs(slots) -> np.ndarray:
    """Lengths of the maximal runs s, s+1, s+2, ... in a slot table (in order)."""
    s = np.asarray(slots, dtype=np.int64)
    if s.size == 0:
        return np.zeros(0, dtype=np.int64)
    breaks = np.nonzero(np.diff(s) != 1)[0]
    edges = np.concatenate([[0], breaks + 1, [s.size]])
    return np.diff(edges)


def fragmentation(slots, step: int = STEP_KEYS) -> dict:
    """Runs of consecutive slots and the share of full `step`-key steps that are contiguous."""
    s = np.asarray(slots, dtype=np.int64)
    runs = contiguous_runs(s)
    full = s.size // step
    if full:
        blocks = s[: full * step].reshape(full, step)
        contiguous = np.all(np.diff(blocks, axis=1) == 1, axis=1)
        frac = float(contiguous.mean())
    else:
        frac = 1.0 if s.size else 0.0
    return {"keys": int(s.size), "runs": int(runs.size),
            "mean_run": float(runs.mean()) if runs.size else 0.0,
            "contiguous_steps": frac}


class SortedFreeList:
    """Free slots of a pool kept in ascending order (slot 0 is never free: it is the pad slot)."""

    def __init__(self, pool_slots: int, free_slots=None):
        self.pool_slots = int(pool_slots)
        if free_slots is None:
            self.free = np.arange(1, pool_slots, dtype=np.int64)
        else:
            f = np.unique(np.asarray(free_slots, dtype=np.int64))
            if f.size and (f[0] < 1 or f[-1] >= pool_slots):
                raise ValueError("free slots must lie in [1, pool_slots)")
            self.free = f

    @property
    def free_count(self) -> int:
        return int(self.free.size)

    def alloc(self, n: int) -> np.ndarray:
        """The n lowest free slots, ascending."""
        if n > self.free.size:
            raise MemoryError(f"alloc({n}) with {self.free.size} free slots")
        out, self.free = self.free[:n].copy(), self.free[n:]
        return out

    def find_run(self, n: int) -> int:
        """First slot of the lowest free run of at least n consecutive slots, or -1."""
        if n <= 0 or self.free.size < n:
            return -1
        runs = contiguous_runs(self.free)
        starts = np.concatenate([[0], np.cumsum(runs)[:-1]])
        fit = np.nonzero(runs >= n)[0]
        return int(self.free[starts[fit[0]]]) if fit.size else -1

    def take_run(self, start: int, n: int) -> np.ndarray:
        """Allocate the slots start .. start+n-1, which must all be free."""
        want = np.arange(start, start + n, dtype=np.int64)
        idx = np.searchsorted(self.free, want)
        if n and (idx[-1] >= self.free.size or not np.array_equal(self.free[idx], want)):
            raise ValueError("run is not free")
        self.free = np.delete(self.free, idx)
        return want

    def release(self, slots) -> None:
        s = np.asarray(slots, dtype=np.int64)
        if np.intersect1d(s, self.free).size:
            raise ValueError("double free")
        self.free = np.union1d(self.free, s)


@dataclasses.dataclass
class CompactionPlan:
    requests: np.ndarray   # indices of the requests to move
    dst_start: np.ndarray  # first destination slot of each (the run dst_start .. dst_start+L-1)


def plan_compaction(slot_tables, prefix_lens, free_list: SortedFreeList,
                    min_contiguous: float = 1.0) -> CompactionPlan:
    """Choose destination runs for requests whose prefix is not already contiguous.

    Longest requests first (they gain the most steps); a request whose
    `contiguous_steps` is at least `min_contiguous`, or for which no free run is
    long enough, stays.  The chosen runs are taken from `free_list`; the caller
    runs the copy (ddtree.kv_compact on the chosen rows, in place or into
    another pool) and then releases the old slots with `finish_compaction`.
    """
    lens = np.asarray(prefix_lens, dtype=np.int64)
    order = np.argsort(-lens, kind="stable")
    chosen, starts = [], []
    for b in order:
        L = int(lens[b])
        if L == 0:
            continue
        if fragmentation(np.asarray(slot_tables[b])[:L])["contiguous_steps"] >= min_contiguous:
            continue
        start = free_list.find_run(L)
        if start < 0:
            continue
        free_list.take_run(start, L)
        chosen.append(int(b))
        starts.append(start)
    return CompactionPlan(np.asarray(chosen, dtype=np.int64), np.asarray(starts, dtype=np.int64))


def finish_compaction(plan: CompactionPlan, old_slot_tables, prefix_lens, free_list: SortedFreeList) -> None:
    """After the copy: the moved requests' old slots go back to the free list."""
    for b in plan.requests:
        L = int(np.asarray(prefix_lens)[b])
        free_list.release(np.asarray(old_slot_tables[b])[:L])
