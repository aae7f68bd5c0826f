"""Ragged trees on the GPU: requests with different node counts in one call.

The pages' trees range from 9 to 65 nodes per request ("The Art of Systematic
Investigation", section "Input Knowledge Required to Understand This Message",
item 1); `ddtree_verify_attn_ragged` takes the node count of each request.
Active rows are compared with the fp64 oracle (the request cut to its
tree_len nodes), inactive rows must be exactly out = 0, lse = -inf, and a
call whose tree_len is T everywhere must give the bits of the uniform call.
Also the multi-request 128-head x 65-node case, on sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_05_gb300 import ddtree, workloads as wl

pytestmark = pytest.mark.gpu

OUT_MAX, OUT_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_tree_05_gb300 import build
    build.build()
    ddtree.lib()


def _args(d, w):
    return (d["q"], d["kv_pool"], d["slot_idx"], d["prefix_len"], d["tree_parent"], d["tree_slot_idx"], w.sm_scale)


def _check_active(out, lse, ref_o, ref_l, tree_len):
    o = out.cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    for b, tl in enumerate(tree_len):
        tl = int(min(max(tl, 0), o.shape[1]))
        if tl:
            e_o = np.abs(o[b, :tl] - ref_o[b, :tl])
            e_l = np.abs(l[b, :tl] - ref_l[b, :tl])
            assert np.isfinite(o[b, :tl]).all() and np.isfinite(l[b, :tl]).all()
            assert e_o.max() <= OUT_MAX and e_o.mean() <= OUT_MEAN and e_l.max() <= LSE_MAX, \
                (b, e_o.max(), e_o.mean(), e_l.max())
        assert np.all(o[b, tl:] == 0.0) and np.all(np.isneginf(l[b, tl:]))


def test_ragged_batch_against_oracle():
    w = wl.make_workload("tiny", batch=4, prefix=("list", 3000, 0, 700, 1500), nodes=33, heads=16, max_depth=6,
                         pool_slots=1 << 16, slots="churn")
    d = wl.to_device(w, "cuda", poison=True)
    v = ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride, w.max_prefix_len)
    # 528 / 16 / 272 / 144 active rows: skipped tiles, one-node trees and ragged last tiles
    tree_len = np.asarray([33, 1, 17, 9], np.int32)
    out, lse = v(*_args(d, w), tree_len=torch.from_numpy(tree_len).cuda())
    torch.cuda.synchronize()
    assert v.status() == 0
    pool, si, ts = w.compact_host_pool()
    ref_o, ref_l, st = oracle.verify_attn_ragged(w.q_bits, pool, si, w.prefix_len, w.tree_parent, ts, w.sm_scale,
                                                 tree_len)
    assert st == 0
    _check_active(out, lse, ref_o, ref_l, tree_len)


def test_ragged_full_length_equals_uniform_call_bitwise():
    w = wl.make_workload("tiny", batch=2, prefix=("list", 2500, 900), nodes=17, heads=8, pool_slots=1 << 15)
    d = wl.to_device(w, "cuda", poison=True)
    v = ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride, w.max_prefix_len)
    out_u, lse_u = v(*_args(d, w))
    tl = torch.full((w.batch,), w.nodes, dtype=torch.int32, device="cuda")
    out_r, lse_r = v(*_args(d, w), tree_len=tl)
    torch.cuda.synchronize()
    assert v.status() == 0
    assert torch.equal(out_u, out_r) and torch.equal(lse_u, lse_r)


def test_ragged_tree_len_out_of_range_is_clamped_and_reported():
    w = wl.make_workload("tiny", batch=2, prefix=("list", 400, 300), nodes=9, heads=4, pool_slots=1 << 13)
    d = wl.to_device(w, "cuda", poison=True)
    v = ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride, w.max_prefix_len)
    out_c, lse_c = v(*_args(d, w), tree_len=torch.tensor([9, 0], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert v.status() == 0
    out_b, lse_b = v(*_args(d, w), tree_len=torch.tensor([20, -3], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert v.status() == ddtree.STATUS_BAD_TREE_LEN
    assert torch.equal(out_b, out_c) and torch.equal(lse_b, lse_c)
    assert bool(torch.all(out_b[1] == 0)) and bool(torch.all(torch.isneginf(lse_b[1])))


def test_multi_request_128_heads_65_nodes_sampled():
    """Two requests of 65 nodes x 128 heads (8320 rows each: 65 row tiles per request)."""
    w = wl.make_workload("tiny", batch=2, prefix=("list", 4100, 2049), nodes=65, heads=128, max_depth=8,
                         max_branch=4, pool_slots=1 << 16, slots="churn")
    d = wl.to_device(w, "cuda", poison=True)
    v = ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride, w.max_prefix_len)
    out, lse = v(*_args(d, w))
    torch.cuda.synchronize()
    assert v.status() == 0
    rng = np.random.default_rng(5)
    R = w.rows_per_request
    rows = np.unique(np.concatenate([b * R + rng.choice(R, 40, replace=False) for b in range(w.batch)]
                                    + [np.asarray([0, R - 1, R, 2 * R - 1])]))
    ref_o, ref_l, st = oracle.verify_workload(w, rows=rows)
    assert st == 0
    o = out.reshape(-1, wl.D_V)[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
    l = lse.reshape(-1)[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
    e_o, e_l = np.abs(o - ref_o), np.abs(l - ref_l)
    assert e_o.max() <= OUT_MAX and e_o.mean() <= OUT_MEAN and e_l.max() <= LSE_MAX, (e_o.max(), e_l.max())


def test_prefix_len_sum_hint_changes_only_the_split():
    """The host-side sum of the prefix lengths steers the split length of a batch
    of mixed lengths; the result matches the oracle with and without it."""
    w = wl.make_workload("tiny", batch=4, prefix=("list", 20000, 700, 6000, 150), nodes=9, heads=16,
                         pool_slots=1 << 16, slots="churn")
    d = wl.to_device(w, "cuda", poison=True)
    pool, si, ts = w.compact_host_pool()
    ref_o, ref_l, st = oracle.verify_attn(w.q_bits, pool, si, w.prefix_len, w.tree_parent, ts, w.sm_scale)
    assert st == 0
    for hint in (0, int(w.prefix_len.sum())):
        v = ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride, w.max_prefix_len,
                            prefix_len_sum=hint)
        out, lse = v(*_args(d, w))
        torch.cuda.synchronize()
        assert v.status() == 0
        _check_active(out, lse, ref_o, ref_l, [w.nodes] * w.batch)
