"""Helpers shared by the GPU parity tests (not collected by pytest).

Tolerances (bf16 inputs, fp32 accumulation): out max-abs <= 2e-2 and
mean-abs <= 2e-3, lse abs <= 1e-3 against the fp64 oracle.
"""
import numpy as np
import torch

from speculative_decoding_tree_05_gb300 import ddtree, workloads as wl

OUT_MAX, OUT_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


def run_gpu(w, poison=True, dev=None, library=None):
    """One verify call through the C ABI; returns (out, lse, status, device tensors, verifier)."""
    d = wl.to_device(w, "cuda", poison=poison) if dev is None else dev
    v = ddtree.Verifier(w.batch, w.nodes, w.heads, w.pool_slots, w.slot_stride, w.max_prefix_len, library=library)
    out, lse = v(d["q"], d["kv_pool"], d["slot_idx"], d["prefix_len"], d["tree_parent"], d["tree_slot_idx"],
                 w.sm_scale)
    status = v.status()
    return out, lse, status, d, v


def compare(out, lse, ref_o, ref_l, rows=None):
    """Element-by-element comparison with the oracle; returns (out max, out mean, lse max) errors."""
    o = out.reshape(-1, wl.D_V).cpu().numpy().astype(np.float64)
    l = lse.reshape(-1).cpu().numpy().astype(np.float64)
    if rows is not None:
        o, l = o[rows], l[rows]
    ref_o = ref_o.reshape(-1, wl.D_V)
    ref_l = ref_l.reshape(-1)
    assert np.isfinite(o).all() and np.isfinite(l).all()
    e_o = np.abs(o - ref_o)
    e_l = np.abs(l - ref_l)
    msg = f"out max {e_o.max():.3e} mean {e_o.mean():.3e} lse max {e_l.max():.3e}"
    assert e_o.max() <= OUT_MAX and e_o.mean() <= OUT_MEAN and e_l.max() <= LSE_MAX, msg
    return e_o.max(), e_o.mean(), e_l.max()


def build_and_load(variant="release"):
    from speculative_decoding_tree_05_gb300 import build
    path = build.build(variant=variant)
    return ddtree.lib() if variant == "release" else ddtree.load(path)


def require_cuda():
    import pytest
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
