"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Tolerances (bf16 inputs, fp32 accumulation): out max-abs <= 2e-2 and
mean-abs <= 2e-3, lse abs <= 1e-3, over every element.  Every configuration,
including the full-size ones (c3: 8320 rows over a 65536-key prefix; c4: 144
rows over 185000 keys; c5: 8 requests, 4224 rows, ~540k keys), is compared on
every row; a fast variant on sampled rows stays for quick runs.  Properties
that hold at any size are checked too (finite outputs, determinism, layout
invariance, bit-exact compaction).  Unused pool slots hold NaN, so a gather
from a wrong slot shows up as NaN.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
from parity_util import compare, require_cuda, run_gpu as _run_gpu
from speculative_decoding_tree_05_gb300 import ddtree, workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    require_cuda()
    from speculative_decoding_tree_05_gb300 import build
    build.build()
    ddtree.lib()


def run_gpu(w, poison=True, dev=None):
    out, lse, status, d, _ = _run_gpu(w, poison=poison, dev=dev)
    return out, lse, status, d


@functools.lru_cache(maxsize=None)
def oracle_full(name):
    """fp64 oracle of a whole named configuration (every row), computed once per module."""
    return oracle.verify_workload(wl.make_workload(name))


def sample_rows(w, n_per_tile=3, seed=0):
    """Rows of every request: a few per 128-row tile, plus first and last row."""
    rng = np.random.default_rng(seed)
    R = w.rows_per_request
    rows = []
    for b in range(w.batch):
        base = b * R
        for t0 in range(0, R, 128):
            t1 = min(R, t0 + 128)
            rows.extend(base + rng.choice(np.arange(t0, t1), size=min(n_per_tile, t1 - t0), replace=False))
        rows.extend([base, base + R - 1])
    return np.unique(np.asarray(rows, np.int64))


# ----------------------------------------------------------------------------- small cases, every element

def test_tiny_full():
    w = wl.make_workload("tiny")
    out, lse, st, _ = run_gpu(w)
    assert st == 0
    ref_o, ref_l, _ = oracle.verify_workload(w)
    compare(out, lse, ref_o, ref_l)


def test_c2_full():
    w = wl.make_workload("c2")
    out, lse, st, _ = run_gpu(w)
    assert st == 0
    ref_o, ref_l, _ = oracle.verify_workload(w)
    compare(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("prefix,nodes,heads,tree", [
    ((0,), 9, 16, "random"),          # tree only
    ((1,), 1, 1, "chain"),            # single key + single node
    ((31,), 5, 3, "random"),          # ragged below one key step
    ((33,), 65, 2, "random"),         # one step + 1 key; 130 rows -> ragged second tile
    ((1000,), 128, 1, "random"),      # maximum node count
    ((517, 0, 64), 7, 20, "chain"),   # ragged batch incl. an empty prefix
    ((3000,), 17, 8, "random"),       # 136 rows: tile of 128 + 8
])
def test_edge_cases(prefix, nodes, heads, tree):
    w = wl.make_workload("tiny", batch=len(prefix), prefix=("list", *prefix), nodes=nodes, heads=heads, tree=tree,
                         max_depth=8, max_branch=0, pool_slots=1 << 16, slots="churn")
    out, lse, st, _ = run_gpu(w)
    assert st == 0
    ref_o, ref_l, _ = oracle.verify_workload(w)
    compare(out, lse, ref_o, ref_l)


def test_deterministic_and_layout_invariant():
    kw = dict(prefix=(4099,), nodes=33, heads=16, max_depth=6, max_branch=4, pool_slots=1 << 16)
    w = wl.make_workload("tiny", **kw)
    o1, l1, _, d = run_gpu(w)
    o2, l2, _, _ = run_gpu(w, dev=d)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    wc = wl.make_workload("tiny", slots="contiguous", **kw)
    o3, l3, _, _ = run_gpu(wc)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


# ----------------------------------------------------------------------------- device-side validation

def test_bad_slot_is_masked_and_reported():
    w = wl.make_workload("tiny", prefix=(300,))
    d = wl.to_device(w, "cuda")
    d["slot_idx"][0, 77] = w.pool_slots + 12     # corrupted after upload: the kernels must mask them
    d["tree_slot_idx"][0, 3] = -5
    out, lse, st, _ = run_gpu(w, dev=d)
    assert st & ddtree.STATUS_BAD_SLOT
    pool, si, ts = w.compact_host_pool()
    si[0, 77] = pool.shape[0] + 12     # the oracle leaves the same keys out
    ts[0, 3] = -5
    ref_o, ref_l, ost = oracle.verify_attn(w.q_bits, pool, si, w.prefix_len, w.tree_parent, ts, w.sm_scale)
    assert ost & oracle.BAD_SLOT
    compare(out, lse, ref_o, ref_l)


def test_bad_parent_is_ignored_and_reported():
    w = wl.make_workload("tiny")
    w.tree_parent[0, 5] = 7            # forward link: not an earlier node
    out, lse, st, _ = run_gpu(w)
    assert st & ddtree.STATUS_BAD_PARENT
    ref_o, ref_l, ost = oracle.verify_workload(w)
    assert ost & oracle.BAD_PARENT
    compare(out, lse, ref_o, ref_l)


def test_prefix_len_above_bound_is_reported():
    w = wl.make_workload("tiny")
    d = wl.to_device(w, "cuda")
    v = ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride, max_prefix_len=200)
    v(d["q"], d["kv_pool"], d["slot_idx"], d["prefix_len"], d["tree_parent"], d["tree_slot_idx"], w.sm_scale)
    assert v.status() & ddtree.STATUS_BAD_PREFIX


def test_host_errors_on_gpu():
    w = wl.make_workload("tiny")
    d = wl.to_device(w, "cuda")
    v = ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride)
    small = ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride)
    small.workspace = small.workspace[:100]
    with pytest.raises(ddtree.DDTError) as e:
        small(d["q"], d["kv_pool"], d["slot_idx"], d["prefix_len"], d["tree_parent"], d["tree_slot_idx"], 0.1)
    assert e.value.code == -3
    assert ddtree.workspace_bytes(v.dims) > 0


# ----------------------------------------------------------------------------- full-size configurations

@pytest.mark.parametrize("name", ["c3", "c4", "c5"])
def test_full_size_every_element(name):
    w = wl.make_workload(name)
    out, lse, st, d = run_gpu(w)
    assert st == 0
    ref_o, ref_l, ost = oracle_full(name)
    assert ost == 0
    compare(out, lse, ref_o, ref_l)
    if name == "c3":
        # same logical data on contiguous slots: bitwise identical results
        del d
        wc = wl.make_workload(name, slots="contiguous")
        oc, lc, stc, _ = run_gpu(wc)
        assert stc == 0 and torch.equal(out, oc) and torch.equal(lse, lc)


@pytest.mark.parametrize("name", ["c3", "c4", "c5"])
def test_full_size_sampled_fast(name):
    # quick variant: rows spread over every tile, computed one by one by the oracle
    w = wl.make_workload(name)
    out, lse, st, _ = run_gpu(w)
    assert st == 0 and torch.isfinite(out).all() and torch.isfinite(lse).all()
    rows = sample_rows(w, n_per_tile=2 if name == "c3" else 4)
    ref_o, ref_l, _ = oracle.verify_workload(w, rows=rows)
    compare(out, lse, ref_o, ref_l, rows=rows)


def test_c5_compaction_bit_exact():
    w = wl.make_workload("c5")
    d = wl.to_device(w, "cuda", poison=True)
    out1, lse1, st, _ = run_gpu(w, dev=d)
    assert st == 0
    # destination: one contiguous run per request in a fresh pool
    starts = np.concatenate([[1], 1 + np.cumsum(w.prefix_len[:-1].astype(np.int64))])
    dst_pool = torch.full_like(d["kv_pool"].view(torch.int16), wl.BF16_NAN).view(torch.bfloat16)
    ts = d["tree_slot_idx"].reshape(-1).long()
    free_tail = int(starts[-1] + w.prefix_len[-1])
    assert free_tail <= w.pool_slots
    # the tree rows move above the compacted runs
    new_tree = torch.arange(free_tail, free_tail + w.batch * w.nodes, dtype=torch.int32, device="cuda")
    dst_pool[new_tree.long()] = d["kv_pool"][ts]
    dst_start = torch.from_numpy(starts).cuda()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    new_idx = ddtree.kv_compact(d["kv_pool"], dst_pool, d["slot_idx"], d["prefix_len"], dst_start, workspace=ws)
    assert ddtree.read_device_status(ws) == 0
    for b in range(w.batch):
        L = int(w.prefix_len[b])
        s0 = int(starts[b])
        assert torch.equal(new_idx[b, :L].cpu(), torch.arange(s0, s0 + L, dtype=torch.int32))
        got = dst_pool[s0:s0 + L].view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, w.kv_prefix_bits[b])
    d2 = dict(d, kv_pool=dst_pool, slot_idx=new_idx, tree_slot_idx=new_tree.view(w.batch, w.nodes))
    out2, lse2, st2, _ = run_gpu(w, dev=d2)
    assert st2 == 0
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    ref_o, ref_l, _ = oracle_full("c5")
    compare(out2, lse2, ref_o, ref_l)


# ----------------------------------------------------------------------------- fused launch vs the two phases

@pytest.mark.parametrize("kw", [
    dict(),                                                                   # tiny
    dict(prefix=(4099,), nodes=33, heads=16, max_depth=6, max_branch=4, pool_slots=1 << 16),
    dict(batch=3, prefix=("list", 700, 0, 2000), nodes=17, heads=20, pool_slots=1 << 16, slots="churn"),
])
def test_fused_launch_equals_the_two_phases(kw):
    # ddtree_verify_attn_fused runs one persistent kernel with the merge of each row tile done by the
    # pair that finishes its last split; the two phase entry points run the prefix pass and the
    # tail/merge kernel separately.  Same arithmetic, so the same bits.
    w = wl.make_workload("tiny", **kw)
    d = wl.to_device(w, "cuda", poison=True)
    v = ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride, w.max_prefix_len)
    args = (d["q"], d["kv_pool"], d["slot_idx"], d["prefix_len"], d["tree_parent"], d["tree_slot_idx"], w.sm_scale)
    o1, l1 = v(*args, phase="fused")
    assert v.status() == 0
    o2, l2 = v(*args, phase="prefix")
    o2, l2 = v(*args, out=o2, lse=l2, phase="merge")
    assert v.status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ref_o, ref_l, _ = oracle.verify_workload(w)
    compare(o1, l1, ref_o, ref_l)


@pytest.mark.parametrize("name", ["c3", "c5"])
def test_fused_launch_full_size(name):
    # multi-wave configurations of the single fused launch: every element against the oracle, and the
    # same bits as the two-launch path where that path uses the same fixed-length key splits (c3; the
    # batch of c5 is divided by key-range groups there, which cut the keys elsewhere)
    w = wl.make_workload(name)
    d = wl.to_device(w, "cuda", poison=True)
    v = ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride, w.max_prefix_len)
    args = (d["q"], d["kv_pool"], d["slot_idx"], d["prefix_len"], d["tree_parent"], d["tree_slot_idx"], w.sm_scale)
    o1, l1 = v(*args, phase="fused")
    assert v.status() == 0
    o2, l2 = v(*args, phase="prefix")
    o2, l2 = v(*args, out=o2, lse=l2, phase="merge")
    assert v.status() == 0
    ref_o, ref_l, _ = oracle_full(name)
    compare(o1, l1, ref_o, ref_l)
    if ddtree.plan(v.dims)["groups"] == 0:
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    else:
        compare(o2, l2, ref_o, ref_l)


# ----------------------------------------------------------------------------- long first split

@pytest.mark.parametrize("length", [4096, 3900, 3840, 3841])
def test_long_first_split_edges(length):
    # 65 row tiles of one request under a bound of 4096 keys: the plan makes split 0 3840 keys long
    # and split 1 256.  Prefixes that end inside split 0, at its end, and one key into split 1 (the
    # merge must count 1, 1 and 2 splits) against the oracle, every element.
    w = wl.make_workload("tiny", prefix=(length,), nodes=65, heads=128, max_depth=8, max_branch=4,
                         pool_slots=1 << 14, slots="churn")
    bound = 4096
    v = ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, bound, bound)
    p = ddtree.plan(v.dims)
    assert (p["groups"], p["splits"], p["chunk0"], p["chunk"]) == (0, 2, 3840, 256)
    d = wl.to_device(w, "cuda", poison=True)
    slots = torch.zeros((1, bound), dtype=torch.int32, device="cuda")  # the slot row padded to the bound
    slots[:, :w.slot_stride] = d["slot_idx"]
    d["slot_idx"] = slots
    out, lse = v(d["q"], d["kv_pool"], d["slot_idx"], d["prefix_len"], d["tree_parent"], d["tree_slot_idx"],
                 w.sm_scale)
    assert v.status() == 0
    ref_o, ref_l, _ = oracle.verify_workload(w)
    compare(out, lse, ref_o, ref_l)
