"""The no-allocation verify entry point (ddtree_verify_attn_static_scratch).

Callers that cannot allocate device memory at call time (allocator or memory
pool callbacks, plugins limited to the buffers their host framework gives them)
use this entry point, whose scratch is a fixed array inside the library.  The
test calls it through the C ABI twice in a row and compares each result with
the regular entry point's: both run the same plan and kernels, so the results
must be bitwise equal (stricter than the parity tolerances of the other GPU
tests).  It also checks that sizes needing more scratch than the array holds are
rejected.  It is collected last so a stop-at-first-failure run has already run
everything else, and it passes alone in a fresh process too.
"""
import ctypes

import numpy as np
import pytest
import torch

from speculative_decoding_tree_05_gb300 import ddtree, workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_tree_05_gb300 import build
    build.build()
    ddtree.lib()


CASES = {
    "tiny": dict(),
    # 1 request, prefix 4099 (ragged last step), 33 nodes x 16 heads: scratch well inside the 32 MiB array
    "mid": dict(prefix=(4099,), nodes=33, heads=16, max_depth=6, max_branch=4, pool_slots=1 << 16),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_static_scratch_matches_regular_entry_point(case):
    w = wl.make_workload("tiny", **CASES[case])
    dims = ddtree.make_dims(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride, w.max_prefix_len)
    assert 0 < ddtree.workspace_bytes(dims) <= (32 << 20)
    d = wl.to_device(w, "cuda", poison=True)
    args = (d["q"], d["kv_pool"], d["slot_idx"], d["prefix_len"], d["tree_parent"], d["tree_slot_idx"], w.sm_scale)
    ref_o, ref_l = ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride, w.max_prefix_len)(*args)
    for _ in range(2):  # two calls in a row share (and reuse) the static array
        out = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_l, float("nan"))
        ddtree.verify_attn_static_scratch(*args, out=out, lse=lse, max_prefix_len=w.max_prefix_len)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all() and torch.isfinite(lse).all()
        assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)


def test_static_scratch_rejects_sizes_beyond_the_array():
    w = wl.make_workload("tiny")
    d = wl.to_device(w, "cuda")
    big = ddtree.make_dims(1, 65, 128, w.pool_slots, 1 << 20, 1 << 20)   # far more than 32 MiB of partials
    assert ddtree.workspace_bytes(big) > (32 << 20)
    out = torch.empty((1, 65, 128, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((1, 65, 128), dtype=torch.float32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = ddtree.lib().ddtree_verify_attn_static_scratch(p(d["q"]), p(d["kv_pool"]), p(d["slot_idx"]),
                                                         p(d["prefix_len"]), p(d["tree_parent"]),
                                                         p(d["tree_slot_idx"]), 0.1, p(out), p(lse),
                                                         ctypes.byref(big), None)
    assert rc == -3
