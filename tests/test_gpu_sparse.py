"""GPU parity of the sparse-index variant (ddtree_verify_attn_sparse) against the fp64 oracle.

Each tree node lists the pool slots of its keys (-1 = no key; a slot listed
twice counts twice); all heads of the node attend to them.  Compared element by
element with oracle.verify_sparse at the parity tolerances (out max-abs <= 2e-2,
mean-abs <= 2e-3, lse abs <= 1e-3), plus: an empty list gives out = 0 and
lse = -inf, a bad slot is left out and flagged while -1 is not, and lists that
name a node's visible set reproduce the dense verify call.
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


def run_sparse(w, idx, d=None):
    d = wl.to_device(w, "cuda", poison=True) if d is None else d
    v = ddtree.SparseVerifier(w.batch, w.nodes, w.heads, w.pool_slots, idx.shape[2])
    out, lse = v(d["q"], d["kv_pool"], torch.from_numpy(idx).cuda(), w.sm_scale)
    return out, lse, v.status(), d


def oracle_sparse(w, idx):
    pool, _, _ = w.compact_host_pool()
    return oracle.verify_sparse(w.q_bits, pool, wl.compact_indices(w, idx), w.sm_scale)


@pytest.mark.parametrize("kw,topk", [
    (dict(batch=2, prefix=("list", 900, 400), nodes=9, heads=16), 700),     # -1s and repeats, 11 steps
    (dict(batch=1, prefix=(3000,), nodes=3, heads=128), 2048),              # a full 128-row tile per node
    (dict(batch=1, prefix=(200,), nodes=5, heads=20), 33),                  # below one step; 20 heads
])
def test_sparse_every_element(kw, topk):
    w = wl.make_workload("tiny", pool_slots=1 << 16, slots="churn", **kw)
    idx = wl.sparse_indices(w, topk)
    out, lse, st, _ = run_sparse(w, idx)
    assert st == 0
    ref_o, ref_l, ost = oracle_sparse(w, idx)
    assert ost == 0
    compare(out, lse, ref_o, ref_l)


def test_sparse_empty_list_and_status():
    w = wl.make_workload("tiny", batch=1, prefix=(300,), nodes=4, heads=16, pool_slots=1 << 16)
    idx = wl.sparse_indices(w, 130)
    idx[0, 1] = -1                                   # node 1 has no key
    out, lse, st, d = run_sparse(w, idx)
    assert st == 0                                   # -1 is not a bad slot
    assert torch.all(lse[0, 1] == -float("inf")) and torch.all(out[0, 1] == 0)
    ref_o, ref_l, _ = oracle_sparse(w, idx)
    keep = [0, 2, 3]
    compare(out[:, keep], lse[:, keep], ref_o[:, keep], ref_l[:, keep])
    bad = idx.copy()
    bad[0, 2, 5] = w.pool_slots + 3                  # outside the pool: left out and flagged
    out2, lse2, st2, _ = run_sparse(w, bad, d)
    assert st2 & ddtree.STATUS_BAD_SLOT
    pool, _, _ = w.compact_host_pool()
    cidx = wl.compact_indices(w, idx)
    cidx[0, 2, 5] = -1                               # the oracle leaves the same key out
    ref_o2, ref_l2, _ = oracle.verify_sparse(w.q_bits, pool, cidx, w.sm_scale)
    compare(out2[:, keep], lse2[:, keep], ref_o2[:, keep], ref_l2[:, keep])


def test_sparse_lists_of_the_visible_set_match_dense_verify():
    # the pages' observation: a sparse call can express the tree mask when each list names the
    # whole prefix plus the node's ancestors and itself
    w = wl.make_workload("tiny", batch=2, prefix=("list", 700, 250), nodes=9, heads=16, pool_slots=1 << 16)
    lists = []
    for b in range(w.batch):
        anc = oracle._ancestors_by_descent(list(w.tree_parent[b]))
        for t in range(w.nodes):
            lists.append(list(w.slot_idx[b, :w.prefix_len[b]]) + [int(w.tree_slot_idx[b, u]) for u in sorted(anc[t])])
    topk = max(len(x) for x in lists)
    idx = np.asarray([x + [-1] * (topk - len(x)) for x in lists], np.int32).reshape(w.batch, w.nodes, topk)
    out_s, lse_s, st, d = run_sparse(w, idx)
    assert st == 0
    v = ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride, w.max_prefix_len)
    out_d, lse_d = v(d["q"], d["kv_pool"], d["slot_idx"], d["prefix_len"], d["tree_parent"], d["tree_slot_idx"],
                     w.sm_scale)
    ref_o, ref_l, _ = oracle.verify_workload(w)
    compare(out_s, lse_s, ref_o, ref_l)
    compare(out_d, lse_d, ref_o, ref_l)
