"""The defragmentation policy end to end on the GPU: plan on the host, copy in place on the device.

A churned pool gives each request scattered slots; `defrag.plan_compaction`
picks free contiguous runs, `ddtree.kv_compact` copies the rows into them in
the same pool (source and destination disjoint, as the plan guarantees), and
the verify call on the rewritten slot table must give bit-identical results
(the consecutive 64-key steps now go through the kernel's tiled-box loads).
"""
import numpy as np
import pytest

from speculative_decoding_tree_05_gb300 import defrag
from speculative_decoding_tree_05_gb300 import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _run(v, d, w):
    out, lse = v(d["q"], d["kv_pool"], d["slot_idx"], d["prefix_len"], d["tree_parent"], d["tree_slot_idx"],
                 w.sm_scale)
    torch.cuda.synchronize()
    return out, lse


def test_in_place_compaction_plan_keeps_results_bit_exact():
    from speculative_decoding_tree_05_gb300 import ddtree

    w = wl.make_workload("tiny", batch=3, prefix=("list", 5000, 3100, 1500), nodes=9, heads=16, max_depth=4,
                         pool_slots=1 << 16, slots="churn")
    d = wl.to_device(w, "cuda", poison=True)
    v = ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride, w.max_prefix_len)
    out0, lse0 = _run(v, d, w)
    assert v.status() == 0

    tables = [w.slot_idx[b, : int(w.prefix_len[b])].astype(np.int64) for b in range(w.batch)]
    assert all(defrag.fragmentation(t)["contiguous_steps"] < 1.0 for t in tables)
    used = np.concatenate(tables + [w.tree_slot_idx.reshape(-1).astype(np.int64)])
    free = defrag.SortedFreeList(w.pool_slots, free_slots=np.setdiff1d(np.arange(1, w.pool_slots), used))
    plan = defrag.plan_compaction(tables, w.prefix_len, free)
    assert sorted(plan.requests.tolist()) == [0, 1, 2]

    sel = torch.from_numpy(plan.requests).cuda()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    new_rows = ddtree.kv_compact(d["kv_pool"], d["kv_pool"], d["slot_idx"][sel].contiguous(), d["prefix_len"][sel],
                                 torch.from_numpy(plan.dst_start).cuda(), workspace=ws)
    assert ddtree.read_device_status(ws) == 0
    d["slot_idx"][sel] = new_rows
    defrag.finish_compaction(plan, tables, w.prefix_len, free)

    host_idx = d["slot_idx"].cpu().numpy()
    for k, b in enumerate(plan.requests):
        L = int(w.prefix_len[b])
        assert np.array_equal(host_idx[b, :L], np.arange(plan.dst_start[k], plan.dst_start[k] + L))
        f = defrag.fragmentation(host_idx[b, :L])
        assert f["runs"] == 1 and f["contiguous_steps"] == 1.0
        rows = d["kv_pool"][torch.from_numpy(host_idx[b, :L]).long().cuda()].view(torch.int16).cpu().numpy()
        assert np.array_equal(rows.view(np.uint16), w.kv_prefix_bits[b])
    out1, lse1 = _run(v, d, w)
    assert v.status() == 0
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)
