"""A verify call captured in a CUDA graph replays to the same bits as direct calls.

The verify call must be capturable in a CUDA graph ("The Art of Systematic
Investigation", section "Input Knowledge Required to Understand This Message";
"The Anatomy of a Kernel Investigation", section "Conclusion"): the library
allocates nothing, never synchronises and puts all work (a status memset, the
prefix pass, the tail/merge kernel as its programmatic dependent) on the
caller's stream.  A replay must also read the live contents of the captured
buffers, so the test rewrites q and the slot table in place between replays.
"""
import numpy as np
import pytest

from speculative_decoding_tree_05_gb300 import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _args(d, w):
    return (d["q"], d["kv_pool"], d["slot_idx"], d["prefix_len"], d["tree_parent"], d["tree_slot_idx"], w.sm_scale)


def test_verify_call_replays_in_cuda_graph():
    from speculative_decoding_tree_05_gb300 import ddtree

    kw = dict(prefix=(4099,), nodes=33, heads=16, max_depth=6, max_branch=4, pool_slots=1 << 16)
    w = wl.make_workload("tiny", **kw)
    d = wl.to_device(w, "cuda", poison=True)
    v = ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride, w.max_prefix_len)
    shape = (w.batch, w.nodes, w.heads, wl.D_V)
    out_g = torch.empty(shape, dtype=torch.float32, device="cuda")
    lse_g = torch.empty(shape[:3], dtype=torch.float32, device="cuda")

    # first call outside any capture: per-device set-up (kernel attributes, driver entry point)
    v(*_args(d, w), out=out_g, lse=lse_g)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        v(*_args(d, w), out=out_g, lse=lse_g)
    out_g.zero_()
    lse_g.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert v.status() == 0
    out_d, lse_d = v(*_args(d, w))
    torch.cuda.synchronize()
    assert torch.equal(out_g, out_d) and torch.equal(lse_g, lse_d)

    # new contents in the captured buffers: another seed's q, and the same prefix rows moved
    # to other slots of the pool (the graph must gather through the rewritten table)
    w2 = wl.make_workload("tiny", seed=12345, **kw)
    d["q"].copy_(wl.to_device(w2, "cuda", poison=True)["q"])
    L = int(w.prefix_len[0])
    old = d["slot_idx"][0, :L].long()
    used = torch.zeros(w.pool_slots, dtype=torch.bool, device="cuda")
    used[old] = True
    used[d["tree_slot_idx"].reshape(-1).long()] = True
    used[0] = True
    free = torch.nonzero(~used).reshape(-1)[:L]
    assert free.numel() == L
    d["kv_pool"][free] = d["kv_pool"][old]
    d["slot_idx"][0, :L] = free.to(torch.int32)
    g.replay()
    torch.cuda.synchronize()
    assert v.status() == 0
    out_d2, lse_d2 = v(*_args(d, w))
    torch.cuda.synchronize()
    assert torch.equal(out_g, out_d2) and torch.equal(lse_g, lse_d2)
    assert not torch.equal(out_d2, out_d)  # the new q really changed the result
    assert np.isfinite(out_g.cpu().numpy()).all()


def test_group_plan_replays_in_cuda_graph():
    # a batch whose prefix pass runs as key-range groups (the persistent group kernel) captured and
    # replayed: the same bits as a direct call, also after new prefix lengths are written in place
    # (the groups are recomputed on the device from prefix_len at every replay)
    from speculative_decoding_tree_05_gb300 import ddtree

    rng = np.random.default_rng(21)
    lens = rng.integers(0, 3000, 64)
    w = wl.make_workload("tiny", batch=64, prefix=("list", *(int(x) for x in lens)), nodes=3, heads=16,
                         max_depth=3, max_branch=0, pool_slots=1 << 18, slots="churn")
    d = wl.to_device(w, "cuda", poison=True)
    v = ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride, w.max_prefix_len)
    assert ddtree.plan(v.dims)["groups"] > 0
    shape = (w.batch, w.nodes, w.heads, wl.D_V)
    out_g = torch.empty(shape, dtype=torch.float32, device="cuda")
    lse_g = torch.empty(shape[:3], dtype=torch.float32, device="cuda")
    v(*_args(d, w), out=out_g, lse=lse_g)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        v(*_args(d, w), out=out_g, lse=lse_g)
    for step in range(2):
        if step == 1:
            # shorter prefixes, written into the captured length array (the slot rows stay valid)
            d["prefix_len"].copy_(torch.div(d["prefix_len"], 2, rounding_mode="floor"))
        out_g.zero_()
        lse_g.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert v.status() == 0
        out_d, lse_d = v(*_args(d, w))
        torch.cuda.synchronize()
        assert torch.equal(out_g, out_d) and torch.equal(lse_g, lse_d)
