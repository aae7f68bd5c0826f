"""Seeded input generators: trees, allocator churn, bf16 rounding, determinism."""
import numpy as np
import pytest
import torch

from speculative_decoding_tree_05_gb300 import workloads as wl


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10.0 ** rng.integers(-20, 20, 100000),
                        np.asarray([0.0, -0.0, 1.0, np.inf, -np.inf, 3.0e38], np.float32)]).astype(np.float32)
    ours = wl.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = wl.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


@pytest.mark.parametrize("depth,branch", [(4, 0), (8, 4), (6, 4), (2, 2)])
def test_random_tree_respects_caps(depth, branch):
    rng = np.random.default_rng(1)
    for _ in range(20):
        n = int(rng.integers(1, 40 if branch == 0 or depth > 2 else 7))
        p = wl.random_tree(rng, n, depth, branch)
        assert p[0] == -1 and all(0 <= p[i] < i for i in range(1, n))
        assert wl.tree_depths(p).max(initial=0) <= depth
        if branch:
            assert np.bincount(p[1:], minlength=n).max(initial=0) <= branch


def test_allocator_semantics():
    """alloc takes the head of the free list, free appends in the freed order."""
    a = wl.FreeListAllocator(10)
    assert list(a.alloc(3)) == [1, 2, 3]
    x = a.alloc(2)
    assert list(x) == [4, 5]
    a.free(np.asarray([3, 1, 2]))
    assert list(a.alloc(4)) == [6, 7, 8, 9]
    assert list(a.alloc(3)) == [3, 1, 2]
    with pytest.raises(MemoryError):
        a.alloc(1)


def test_churn_scatters_and_stays_valid():
    rng = np.random.default_rng(2)
    a = wl.churned_allocator(rng, 1 << 16, keep_free=1 << 13, max_alloc=512)
    s = a.alloc(4000)
    assert len(np.unique(s)) == 4000 and s.min() >= 1 and s.max() < (1 << 16)
    contiguous = np.mean(np.diff(s) == 1)
    assert contiguous < 0.995  # churned slots are not one contiguous run


@pytest.mark.parametrize("layout", ["perm", "churn", "contiguous"])
def test_workload_layouts(layout):
    w = wl.make_workload("tiny", slots=layout)
    used = w.used_slots()
    assert len(np.unique(used)) == len(used) and used.min() >= 1 and used.max() < w.pool_slots
    if layout == "contiguous":
        assert np.array_equal(used, np.arange(1, 1 + len(used)))
    w2 = wl.make_workload("tiny", slots="contiguous")
    assert np.array_equal(w.q_bits, w2.q_bits) and np.array_equal(w.kv_tree_bits, w2.kv_tree_bits)


def test_workload_is_seeded():
    a, b = wl.make_workload("tiny"), wl.make_workload("tiny")
    assert np.array_equal(a.q_bits, b.q_bits) and np.array_equal(a.slot_idx, b.slot_idx)
    assert np.array_equal(a.tree_parent, b.tree_parent)
    c = wl.make_workload("tiny", seed=7)
    assert not np.array_equal(a.q_bits, c.q_bits)


def test_config_shapes_without_values():
    """Structure of every named config (values are generated on demand elsewhere)."""
    for name, cfg in wl.CONFIGS.items():
        assert cfg.nodes <= 128
    w = wl.make_workload("tiny")
    assert w.q_bits.shape == (1, 9, 16, 576) and w.prefix_len[0] == 256
    assert wl.tree_depths(w.tree_parent[0]).max() <= 4


def test_work_formulas_count_active_rows_only():
    """FLOPs 2*T*H*L*(576+512) and bytes per request; ragged trees count their active nodes."""
    w = wl.make_workload("tiny", batch=3, prefix=("list", 100, 0, 37), nodes=5, heads=2, pool_slots=1 << 10)
    L = w.prefix_len.astype(np.int64)
    assert w.flops() == 2 * 5 * 2 * int(L.sum()) * 1088
    assert w.kv_bytes() == (int(L.sum()) + 3 * 5) * 1152
    rows = 3 * 5 * 2
    assert w.algorithmic_bytes() == w.kv_bytes() + int(L.sum()) * 4 + 3 * 5 * 8 + rows * (1152 + 2048 + 4)
    w.tree_len = np.asarray([5, 1, 7], np.int32)      # 7 is clamped to T = 5
    t = np.asarray([5, 1, 5])
    assert w.active_nodes().tolist() == t.tolist()
    assert w.flops() == 2 * 2 * int((t * L).sum()) * 1088
    assert w.kv_bytes() == (int(L.sum()) + int(t.sum())) * 1152
    rows = int(t.sum()) * 2
    assert w.algorithmic_bytes() == w.kv_bytes() + int(L.sum()) * 4 + int(t.sum()) * 8 + rows * (1152 + 2048 + 4)
