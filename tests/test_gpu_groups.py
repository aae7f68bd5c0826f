"""The prefix pass by key-range groups on the GPU (batches of 2..64 requests).

For such a batch the planner may lay the requests' 64-key steps end to end and
give each group of row_tiles CTA pairs an equal share of them (every pair one
row tile of the share, one unit per request it touches, the units back to back
on the same barriers); the merge then takes each request's pieces.  Each case
asserts that the plan really uses groups and compares every element with the
fp64 oracle: empty, one-key and one-step requests, requests spread over many
groups, groups spanning many requests, fewer steps than groups, ragged trees,
and queries scaled so that the units are rerun with 20-bit exchange mantissas.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import compare, require_cuda
from speculative_decoding_tree_05_gb300 import ddtree, workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    require_cuda()
    from speculative_decoding_tree_05_gb300 import build
    build.build()
    ddtree.lib()


def _args(d, w):
    return (d["q"], d["kv_pool"], d["slot_idx"], d["prefix_len"], d["tree_parent"], d["tree_slot_idx"], w.sm_scale)


def _verifier(w, hint=True):
    return ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride, w.max_prefix_len,
                           prefix_len_sum=int(w.prefix_len.sum()) if hint else 0)


def _mixed_lengths(n, seed):
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, 4000, n)
    lens[:6] = (0, 1, 63, 64, 65, 3999)  # empty, one key, ragged and exact single steps
    return tuple(int(x) for x in lens)


CASES = {
    # 64 requests x 48 rows (one row tile): 76 groups, several requests per group
    "many_small": dict(batch=64, prefix=("list", *_mixed_lengths(64, 1)), nodes=3, heads=16),
    # 6 requests x 528 rows (five row tiles): 15 groups of 5 pairs, requests spread over many groups
    "mixed_528": dict(batch=6, prefix=("list", 12000, 800, 0, 12000, 5000, 12000), nodes=33, heads=16),
    # 30 requests x 144 rows: 38 groups of 2 pairs
    "thirty_144": dict(batch=30, prefix=("list", *(3000,) * 30), nodes=9, heads=16),
}


def _workload(name, **extra):
    kw = dict(max_depth=6, max_branch=0, pool_slots=1 << 18, slots="churn")
    kw.update(CASES[name])
    kw.update(extra)
    return wl.make_workload("tiny", **kw)


@pytest.mark.parametrize("name", sorted(CASES))
def test_groups_every_element(name):
    w = _workload(name)
    v = _verifier(w)
    assert ddtree.plan(v.dims)["groups"] > 0
    d = wl.to_device(w, "cuda", poison=True)
    out, lse = v(*_args(d, w))
    assert v.status() == 0
    ref_o, ref_l, st = oracle.verify_workload(w)
    assert st == 0
    compare(out, lse, ref_o, ref_l)
    # bitwise reproducible, and independent of where the rows sit in the pool
    out2, lse2 = v(*_args(d, w))
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    del d
    wc = _workload(name, slots="contiguous")
    dc = wl.to_device(wc, "cuda", poison=True)
    out3, lse3 = v(*_args(dc, wc))
    assert v.status() == 0 and torch.equal(out, out3) and torch.equal(lse, lse3)


def test_groups_with_fewer_steps_than_groups():
    # 64 requests of at most 100 keys under a loose bound of 4000: the plan takes 76 groups for what
    # could be 64 x 63 steps, the requests hold 64 steps, and only that many groups get one
    lens = [0, 1, 63, 64, 65, 100] + [int(x) for x in np.random.default_rng(3).integers(0, 41, 58)]
    w = wl.make_workload("tiny", batch=64, prefix=("list", *lens), nodes=3, heads=16, max_depth=3, max_branch=0,
                         pool_slots=1 << 15, slots="churn")
    bound = 4000
    v = ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, bound, bound)
    steps = sum(-(-x // 64) for x in lens)
    assert ddtree.plan(v.dims)["groups"] > steps
    d = wl.to_device(w, "cuda", poison=True)
    slots = torch.zeros((w.batch, bound), dtype=torch.int32, device="cuda")  # rows padded to the bound
    slots[:, :w.slot_stride] = d["slot_idx"]
    d["slot_idx"] = slots
    out, lse = v(*_args(d, w))
    assert v.status() == 0
    ref_o, ref_l, _ = oracle.verify_workload(w)
    compare(out, lse, ref_o, ref_l)


def test_groups_ragged_trees():
    w = _workload("many_small")
    v = _verifier(w)
    assert ddtree.plan(v.dims)["groups"] > 0
    d = wl.to_device(w, "cuda", poison=True)
    tree_len = np.asarray([(b * 7) % 4 for b in range(w.batch)], np.int32)  # 0 .. 3 active nodes
    out, lse = v(*_args(d, w), tree_len=torch.from_numpy(tree_len).cuda())
    assert v.status() == 0
    ref_o, ref_l, _ = oracle.verify_workload(w)
    o = out.cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    for b, tl in enumerate(tree_len):
        if tl:
            compare(out[b, :tl], lse[b, :tl], ref_o[b, :tl], ref_l[b, :tl])
        assert np.all(o[b, tl:] == 0.0) and np.all(np.isneginf(l[b, tl:]))


def test_groups_rerun_with_wide_mantissas():
    # queries scaled by 8: partial scores of tens of log2 units, so units rerun with 20-bit mantissas
    # (continuing the barrier phases of the units before them)
    w = _workload("mixed_528")
    w.q_bits = wl.pow2_scaled_bits(w.q_bits, 3)
    v = _verifier(w)
    assert ddtree.plan(v.dims)["groups"] > 0
    d = wl.to_device(w, "cuda", poison=True)
    out, lse = v(*_args(d, w))
    assert v.status() == 0
    ref_o, ref_l, _ = oracle.verify_workload(w)
    compare(out, lse, ref_o, ref_l)


def test_fused_launch_on_a_group_plan():
    # the single fused launch keeps fixed-length key splits; it must agree with the oracle too
    w = _workload("mixed_528")
    v = _verifier(w)
    d = wl.to_device(w, "cuda", poison=True)
    out, lse = v(*_args(d, w), phase="fused")
    assert v.status() == 0
    ref_o, ref_l, _ = oracle.verify_workload(w)
    compare(out, lse, ref_o, ref_l)


def test_groups_clamp_and_report_prefix_lens_above_the_bound():
    # a bound below some requests' lengths: the group kernel and the merge clamp those requests to the
    # bound (the status word says so), and every row matches the oracle on the clamped lengths
    w = _workload("many_small")
    bound = 3000
    v = ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride, bound)
    assert ddtree.plan(v.dims)["groups"] > 0 and int(w.prefix_len.max()) > bound
    d = wl.to_device(w, "cuda", poison=True)
    out, lse = v(*_args(d, w))
    assert v.status() == ddtree.STATUS_BAD_PREFIX
    pool, si, ts = w.compact_host_pool()
    clamped = np.minimum(w.prefix_len, bound).astype(w.prefix_len.dtype)
    ref_o, ref_l, st = oracle.verify_attn(w.q_bits, pool, si, clamped, w.tree_parent, ts, w.sm_scale)
    assert st == 0
    compare(out, lse, ref_o, ref_l)
