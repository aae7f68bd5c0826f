"""GPU parity on the method's closed cases and at large score magnitudes.

Every case runs through the C ABI and is compared element by element with the
fp64 oracle (whose own pins cover the same closed forms on the CPU):
  decode          one tree node: ordinary single-query decode attention
  chain           a chain tree: causal attention over prefix + chain
  star            every node sees the prefix, the root and itself
  identical_keys  every prefix row the same: equal scores
  dominant_key    each query is 4x one key row: that key outweighs the rest by ~160 nats
  tree_only_deep  empty prefix, 128-node chain
  q_x4, q_x8      queries scaled by 4 and 8: partial scores of tens of log2 units,
                  where a 16-bit exchange of the pair's partial scores exceeds the
                  1e-3 lse tolerance
  growing_scores  scores rise by ~2 nats per 64-key step, so the running max keeps
                  growing inside a key split and the lazy O rescale runs repeatedly
A test build of the library (short wait limits, test hooks) checks that the lazy
rescale really runs on the growing case, that units whose partial scores
outgrow 16-bit exchange mantissas are rerun with 20-bit ones (and N(0,1) data
never is), and that a bounded wait which runs out reports DDT_STATUS_TIMEOUT
and leaves the context usable.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import build_and_load, compare, require_cuda, run_gpu
from speculative_decoding_tree_05_gb300 import ddtree, workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    require_cuda()
    build_and_load()


@pytest.fixture(scope="module")
def testhooks():
    return build_and_load("testhooks")


@pytest.mark.parametrize("kind", sorted(wl.CLOSED_CASES))
def test_closed_case_every_element(kind):
    w = wl.closed_case(kind)
    out, lse, st, _, _ = run_gpu(w)
    assert st == 0
    ref_o, ref_l, ost = oracle.verify_workload(w)
    assert ost == 0
    compare(out, lse, ref_o, ref_l)


def test_dominant_key_output_is_that_keys_value():
    # the closed form itself, on the GPU: out ~= v of the chosen key (its weight is 1 - e^-100s)
    w = wl.closed_case("dominant_key")
    out, lse, st, _, _ = run_gpu(w)
    assert st == 0
    ref_o, _, _ = oracle.verify_workload(w)
    assert np.abs(out.cpu().numpy() - ref_o).max() <= 2e-2


def test_lazy_rescale_runs_and_matches(testhooks):
    w = wl.closed_case("growing_scores")
    out, lse, st, _, v = run_gpu(w, library=testhooks)
    assert st == 0
    rescales = int(v.workspace[4:8].view(torch.int32).item())
    assert rescales > 0, "the growing-score case never rescaled O"
    ref_o, ref_l, _ = oracle.verify_workload(w)
    compare(out, lse, ref_o, ref_l)
    # the product build gives the same bits (the counter is the only difference)
    out2, lse2, st2, _, _ = run_gpu(w)
    assert st2 == 0 and torch.equal(out, out2) and torch.equal(lse, lse2)


def _reruns(v):
    return int(v.workspace[8:12].view(torch.int32).item())


@pytest.mark.parametrize("kind", ["q_x4", "q_x8", "dominant_key", "growing_scores"])
def test_large_scores_rerun_with_wide_exchange(testhooks, kind):
    w = wl.closed_case(kind)
    out, lse, st, _, v = run_gpu(w, library=testhooks)
    assert st == 0 and _reruns(v) > 0
    ref_o, ref_l, _ = oracle.verify_workload(w)
    compare(out, lse, ref_o, ref_l)


def test_unit_scale_scores_never_rerun(testhooks):
    w = wl.make_workload("c2")
    _, _, st, _, v = run_gpu(w, library=testhooks)
    assert st == 0 and _reruns(v) == 0


def test_timeout_is_reported_and_the_next_call_is_correct(testhooks):
    w = wl.make_workload("tiny", prefix=(1000,))
    d = wl.to_device(w, "cuda", poison=True)
    testhooks.ddtree_test_set_drop_step(2)        # no loads for step 2 of every unit: its waits run out
    try:
        _, _, st, _, _ = run_gpu(w, dev=d, library=testhooks)
    finally:
        testhooks.ddtree_test_set_drop_step(-1)
    assert st & ddtree.STATUS_TIMEOUT
    out, lse, st, _, _ = run_gpu(w, dev=d, library=testhooks)
    assert st == 0
    ref_o, ref_l, _ = oracle.verify_workload(w)
    compare(out, lse, ref_o, ref_l)


def test_timeout_in_a_key_range_group_plan(testhooks):
    # the same under the key-range group schedule: a pair's units run back to back on one set of
    # barriers, so after a wait runs out in one unit both CTAs of the pair must stop together
    rng = np.random.default_rng(11)
    lens = rng.integers(0, 3000, 64)
    lens[:4] = (0, 1, 64, 2999)
    w = wl.make_workload("tiny", batch=64, prefix=("list", *(int(x) for x in lens)), nodes=3, heads=16,
                         max_depth=3, max_branch=0, pool_slots=1 << 18, slots="churn")
    assert ddtree.plan(ddtree.make_dims(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride,
                                        w.max_prefix_len))["groups"] > 0
    d = wl.to_device(w, "cuda", poison=True)
    testhooks.ddtree_test_set_drop_step(2)
    try:
        _, _, st, _, _ = run_gpu(w, dev=d, library=testhooks)
    finally:
        testhooks.ddtree_test_set_drop_step(-1)
    assert st & ddtree.STATUS_TIMEOUT
    out, lse, st, _, _ = run_gpu(w, dev=d, library=testhooks)
    assert st == 0
    ref_o, ref_l, _ = oracle.verify_workload(w)
    compare(out, lse, ref_o, ref_l)


def test_group_plan_reruns_with_wide_exchange(testhooks):
    # queries scaled by 8 under the key-range group schedule: units rerun with 20-bit mantissas inside
    # the persistent group kernel (the test build counts the reruns), and the product build agrees
    rng = np.random.default_rng(12)
    lens = rng.integers(500, 3000, 64)
    w = wl.make_workload("tiny", batch=64, prefix=("list", *(int(x) for x in lens)), nodes=3, heads=16,
                         max_depth=3, max_branch=0, pool_slots=1 << 18, slots="churn")
    w.q_bits = wl.pow2_scaled_bits(w.q_bits, 3)
    assert ddtree.plan(ddtree.make_dims(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride,
                                        w.max_prefix_len))["groups"] > 0
    d = wl.to_device(w, "cuda", poison=True)
    out, lse, st, _, v = run_gpu(w, dev=d, library=testhooks)
    assert st == 0 and _reruns(v) > 0
    ref_o, ref_l, _ = oracle.verify_workload(w)
    compare(out, lse, ref_o, ref_l)
    out2, lse2, st2, _, _ = run_gpu(w, dev=d)
    assert st2 == 0 and torch.equal(out, out2) and torch.equal(lse, lse2)


def test_timeout_under_the_fused_launch(testhooks):
    # the single fused launch: after a wait runs out, the pair stops claiming units (its barriers'
    # phases are unknown), the status word says TIMEOUT, and the next call is correct
    w = wl.make_workload("tiny", prefix=(3000,), nodes=33, heads=16, max_depth=6, max_branch=4,
                         pool_slots=1 << 16, slots="churn")
    d = wl.to_device(w, "cuda", poison=True)
    v = ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride, w.max_prefix_len,
                        library=testhooks)
    args = (d["q"], d["kv_pool"], d["slot_idx"], d["prefix_len"], d["tree_parent"], d["tree_slot_idx"], w.sm_scale)
    testhooks.ddtree_test_set_drop_step(2)
    try:
        v(*args, phase="fused")
        st = v.status()
    finally:
        testhooks.ddtree_test_set_drop_step(-1)
    assert st & ddtree.STATUS_TIMEOUT
    out, lse = v(*args, phase="fused")
    assert v.status() == 0
    ref_o, ref_l, _ = oracle.verify_workload(w)
    compare(out, lse, ref_o, ref_l)
