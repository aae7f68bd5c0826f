"""Pins for the CPU oracle, independent of the oracle's own code.

Each pin checks the oracle against something the pages or mathematics fix:
hand-derived visibility sets (tests/golden), PyTorch's scaled_dot_product_attention
in fp64 for the cases that reduce to textbook attention (single node = decode,
chain = causal, star), closed forms (identical keys, a dominant key, a sparse
worked example), invariants (inclusion-exclusion of softmax normalisers, joint
permutation of pool rows and slot indices, compaction) and an independently
written NumPy brute force.  The sparse-index variant is pinned against the
dense oracle (lists naming each node's visible keys), against closed forms
(-1 padding and list order change nothing; listing every key twice adds ln 2 to
the lse; an empty list gives -inf) and against its own NumPy brute force.  A mutation test plants plausible mistakes in copies
of the oracle's C source and checks that the pins catch every one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_05_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "visibility_trees.json")
D, DV = wl.D_QK, wl.D_V


def bf64(bits):
    return torch.from_numpy(wl.bf16_bits_to_f32(bits).astype(np.float64))


def case(seed, T=5, H=2, L=(7,), parent=None, N=96):
    """Tiny random inputs with distinct slots for every prefix and tree row."""
    rng = np.random.Generator(np.random.PCG64(seed))
    B = len(L)
    q = wl.normal_bf16(rng, (B, T, H, D))
    pool = wl.normal_bf16(rng, (N, D))
    stride = max(1, max(L))
    perm = rng.permutation(N).astype(np.int32)
    slot_idx = np.zeros((B, stride), np.int32)
    tree_slot = np.zeros((B, T), np.int32)
    off = 0
    for b in range(B):
        slot_idx[b, :L[b]] = perm[off:off + L[b]]
        off += L[b]
        tree_slot[b] = perm[off:off + T]
        off += T
    if parent is None:
        parent = np.stack([wl.random_tree(rng, T, 3, 0) for _ in range(B)])
    parent = np.broadcast_to(np.asarray(parent, np.int32), (B, T)).copy()
    return dict(q_bits=q, pool_bits=pool, slot_idx=slot_idx, prefix_len=np.asarray(L, np.int32),
                tree_parent=parent, tree_slot_idx=tree_slot, sm_scale=1.0 / math.sqrt(192.0))


def run(c, lib, **kw):
    args = dict(c)
    args.update(kw)
    return oracle.verify_attn(args["q_bits"], args["pool_bits"], args["slot_idx"], args["prefix_len"],
                              args["tree_parent"], args["tree_slot_idx"], args["sm_scale"], lib=lib)


def sdpa_rows(c, b, t, visible_cols):
    """fp64 torch SDPA for node t of request b over the listed key columns (prefix j, tree L+u)."""
    L = int(c["prefix_len"][b])
    rows = [int(c["slot_idx"][b, j]) if j < L else int(c["tree_slot_idx"][b, j - L]) for j in visible_cols]
    k = bf64(c["pool_bits"][rows])                      # [n, D]
    q = bf64(c["q_bits"][b, t])                         # [H, D]
    out = torch.nn.functional.scaled_dot_product_attention(
        q[None, :, None, :], k[None, None].expand(1, q.shape[0], -1, -1),
        k[None, None, :, :DV].expand(1, q.shape[0], -1, -1), scale=c["sm_scale"])
    lse = torch.logsumexp(torch.matmul(q, k.T) * c["sm_scale"], dim=-1)
    return out[0, :, 0].numpy(), lse.numpy()


# ----------------------------------------------------------------------------- pins (lib -> raise on failure)

def pin_golden_visibility(lib):
    g = json.load(open(GOLDEN))
    for cs in g["cases"]:
        p = np.asarray(cs["parent"], np.int32)
        vis = np.zeros((len(p), len(p)), np.uint8)
        st = lib.oracle_tree_visibility(oracle._ptr(p), len(p), oracle._ptr(vis))
        assert st == 0, cs["name"]
        for t, exp in enumerate(cs["visible"]):
            assert sorted(np.nonzero(vis[t])[0].tolist()) == exp, (cs["name"], t)
    for cs in g["invalid"]:
        p = np.asarray(cs["parent"], np.int32)
        vis = np.zeros((len(p), len(p)), np.uint8)
        assert lib.oracle_tree_visibility(oracle._ptr(p), len(p), oracle._ptr(vis)) & oracle.BAD_PARENT


def pin_single_node_is_decode(lib):
    c = case(11, T=1, H=3, L=(13,), parent=[-1])
    out, lse, st = run(c, lib)
    assert st == 0
    ref_o, ref_l = sdpa_rows(c, 0, 0, list(range(14)))
    np.testing.assert_allclose(out[0, 0], ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], ref_l, rtol=0, atol=1e-12)


def pin_chain_is_causal(lib):
    T, L = 6, 9
    c = case(12, T=T, H=2, L=(L,), parent=wl.chain_tree(T))
    out, lse, st = run(c, lib)
    assert st == 0
    rows = [int(x) for x in c["slot_idx"][0, :L]] + [int(x) for x in c["tree_slot_idx"][0]]
    k = bf64(c["pool_bits"][rows])
    q = bf64(c["q_bits"][0]).permute(1, 0, 2)            # [H, T, D]
    mask = torch.ones(T, L + T, dtype=torch.bool).tril(diagonal=L)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q[None], k[None, None].expand(1, 2, -1, -1), k[None, None, :, :DV].expand(1, 2, -1, -1),
        attn_mask=mask, scale=c["sm_scale"])[0].permute(1, 0, 2)
    np.testing.assert_allclose(out[0], ref.numpy(), rtol=0, atol=1e-12)


def pin_prefix_free_chain_is_causal(lib):
    T = 7
    c = case(13, T=T, H=2, L=(0,), parent=wl.chain_tree(T))
    out, lse, st = run(c, lib)
    k = bf64(c["pool_bits"][c["tree_slot_idx"][0]])
    q = bf64(c["q_bits"][0]).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q[None], k[None, None].expand(1, 2, -1, -1), k[None, None, :, :DV].expand(1, 2, -1, -1),
        is_causal=True, scale=c["sm_scale"])[0].permute(1, 0, 2)
    np.testing.assert_allclose(out[0], ref.numpy(), rtol=0, atol=1e-12)


def pin_star_tree(lib):
    T, L = 6, 5
    c = case(14, T=T, H=2, L=(L,), parent=[-1] + [0] * (T - 1))
    out, lse, st = run(c, lib)
    for t in range(T):
        cols = list(range(L)) + sorted({L, L + t})
        ref_o, ref_l = sdpa_rows(c, 0, t, cols)
        np.testing.assert_allclose(out[0, t], ref_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[0, t], ref_l, rtol=0, atol=1e-12)


def pin_identical_keys(lib):
    """All rows equal to one row r: s = scale*q.r for every key, so lse = s + ln(#visible), out = r[:512]."""
    T, L = 7, 11
    parent = np.asarray([-1, 0, 1, 2, 1, 0, 5], np.int32)
    c = case(15, T=T, H=2, L=(L,), parent=parent)
    r = c["pool_bits"][3].copy()
    c["pool_bits"][:] = r
    out, lse, st = run(c, lib)
    depth = wl.tree_depths(parent)
    rf = wl.bf16_bits_to_f32(r).astype(np.float64)
    for t in range(T):
        for h in range(2):
            qv = wl.bf16_bits_to_f32(c["q_bits"][0, t, h]).astype(np.float64)
            s = c["sm_scale"] * float(np.dot(qv, rf))
            assert abs(lse[0, t, h] - (s + math.log(L + depth[t] + 1))) < 1e-11
            np.testing.assert_allclose(out[0, t, h], rf[:DV], rtol=0, atol=1e-12)


def pin_dominant_key(lib):
    """q = 4 * k_j for one visible key j: its score exceeds the rest by >100, out = v_j."""
    T, L = 4, 10
    c = case(16, T=T, H=2, L=(L,), parent=[-1, 0, 1, 1])
    for t, j_row in [(0, int(c["slot_idx"][0, 6])), (3, int(c["tree_slot_idx"][0, 1]))]:
        kf = wl.bf16_bits_to_f32(c["pool_bits"][j_row])
        c["q_bits"][0, t, 0] = wl.f32_to_bf16_bits(4.0 * kf)
    out, lse, st = run(c, lib)
    for t, j_row in [(0, int(c["slot_idx"][0, 6])), (3, int(c["tree_slot_idx"][0, 1]))]:
        v = wl.bf16_bits_to_f32(c["pool_bits"][j_row][:DV]).astype(np.float64)
        np.testing.assert_allclose(out[0, t, 0], v, rtol=0, atol=1e-30 + 1e-12)


def pin_worked_example(lib):
    """Sparse rows with small integers; expected values written in closed form.

    Prefix keys p0, p1 and tree nodes 0 (root), 1, 2 with parent = [-1, 0, 0].
    q = e_0 + e_520, sm_scale = 1, so s = row[0] + row[520]; v = row[0:512].
    """
    T, L, N = 3, 2, 8
    pool = np.zeros((N, D), np.float32)
    # slot: (row[0], row[1], row[520])
    vals = {5: (1, 10, 0), 2: (2, 20, -1), 7: (0, 30, 0), 1: (3, 40, 1), 4: (-1, 50, 2)}
    for slot, (a, b_, r) in vals.items():
        pool[slot, 0], pool[slot, 1], pool[slot, 520] = a, b_, r
    q = np.zeros((1, T, 1, D), np.float32)
    q[..., 0] = 1
    q[..., 520] = 1
    c = dict(q_bits=wl.f32_to_bf16_bits(q), pool_bits=wl.f32_to_bf16_bits(pool),
             slot_idx=np.asarray([[5, 2]], np.int32), prefix_len=np.asarray([L], np.int32),
             tree_parent=np.asarray([[-1, 0, 0]], np.int32), tree_slot_idx=np.asarray([[7, 1, 4]], np.int32),
             sm_scale=1.0)
    out, lse, st = run(c, lib)
    e = math.e
    # node 0 sees p0 (s=1), p1 (s=1), root (s=0)
    z0 = e + e + 1
    assert abs(lse[0, 0, 0] - math.log(z0)) < 1e-12
    assert abs(out[0, 0, 0, 0] - (1 * e + 2 * e + 0) / z0) < 1e-12
    assert abs(out[0, 0, 0, 1] - (10 * e + 20 * e + 30) / z0) < 1e-12
    assert np.all(out[0, 0, 0, 2:] == 0) and abs(out[0, 0, 0, 520 - 512]) == 0
    # node 1 also sees itself (s=4); node 2 sees itself (s=1) and not node 1
    z1 = e + e + 1 + e ** 4
    assert abs(lse[0, 1, 0] - math.log(z1)) < 1e-12
    assert abs(out[0, 1, 0, 1] - (10 * e + 20 * e + 30 + 40 * e ** 4) / z1) < 1e-12
    z2 = e + e + 1 + e
    assert abs(lse[0, 2, 0] - math.log(z2)) < 1e-12
    assert abs(out[0, 2, 0, 0] - (1 * e + 2 * e + 0 - 1 * e) / z2) < 1e-12


def pin_inclusion_exclusion(lib):
    """Z(A+B+X) = Z(A+X) + Z(B+X) - Z(X) and the same for Z*out, with X the tree part.

    A = prefix[:6], B = prefix[6:], X = tree-only (prefix_len 0): three separate oracle calls.
    """
    T, L = 5, 14
    c = case(17, T=T, H=2, L=(L,))
    o_all, l_all, _ = run(c, lib)
    c_a = dict(c, prefix_len=np.asarray([6], np.int32))
    c_b = dict(c, slot_idx=np.ascontiguousarray(c["slot_idx"][:, 6:]), prefix_len=np.asarray([L - 6], np.int32))
    c_x = dict(c, prefix_len=np.asarray([0], np.int32))
    (o_a, l_a, _), (o_b, l_b, _), (o_x, l_x, _) = run(c_a, lib), run(c_b, lib), run(c_x, lib)
    ref = l_all
    z = np.exp(l_a - ref) + np.exp(l_b - ref) - np.exp(l_x - ref)
    np.testing.assert_allclose(z, 1.0, rtol=0, atol=1e-12)
    zo = (np.exp(l_a - ref)[..., None] * o_a + np.exp(l_b - ref)[..., None] * o_b
          - np.exp(l_x - ref)[..., None] * o_x)
    np.testing.assert_allclose(zo, o_all, rtol=0, atol=1e-11)


def pin_joint_permutation(lib):
    c = case(18, T=6, H=2, L=(9, 4))
    out, lse, _ = run(c, lib)
    rng = np.random.default_rng(5)
    perm = rng.permutation(c["pool_bits"].shape[0])     # new slot of old row r is perm[r]
    pool2 = np.empty_like(c["pool_bits"])
    pool2[perm] = c["pool_bits"]
    c2 = dict(c, pool_bits=pool2, slot_idx=perm[c["slot_idx"]].astype(np.int32),
              tree_slot_idx=perm[c["tree_slot_idx"]].astype(np.int32))
    out2, lse2, _ = run(c2, lib)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def pin_bruteforce(lib):
    for seed, L, T, H in [(21, (7,), 5, 2), (22, (0, 12), 9, 3), (23, (16, 3, 1), 4, 1)]:
        c = case(seed, T=T, H=H, L=L)
        out, lse, st = run(c, lib)
        assert st == 0
        bo, bl = oracle.brute_force(c["q_bits"], c["pool_bits"], c["slot_idx"], c["prefix_len"],
                                    c["tree_parent"], c["tree_slot_idx"], c["sm_scale"])
        np.testing.assert_allclose(out, bo, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, bl, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------- sparse-index variant

def sparse_lists(c, extra=0, seed=0):
    """Index lists that spell out each node's visible set: its request's prefix slots, then the slots of
    the node and its ancestors (found by descent in the NumPy reading, not by the C oracle's walk),
    padded with `extra` -1 entries; all lists are cut to one length with -1."""
    B, T = c["tree_parent"].shape
    lists = []
    for b in range(B):
        L = int(c["prefix_len"][b])
        anc = oracle._ancestors_by_descent(list(c["tree_parent"][b]))
        for t in range(T):
            lists.append(list(c["slot_idx"][b, :L]) + [int(c["tree_slot_idx"][b, u]) for u in sorted(anc[t])]
                         + [-1] * extra)
    topk = max(len(x) for x in lists)
    return np.asarray([x + [-1] * (topk - len(x)) for x in lists], np.int32).reshape(B, T, topk)


def pin_sparse_equals_dense(lib):
    # a list that names exactly a node's visible keys is dense verify attention
    for seed, T, H, L in ((41, 5, 2, (7, 3)), (42, 9, 3, (0, 12))):
        c = case(seed, T=T, H=H, L=L)
        o_d, l_d, st = run(c, lib)
        assert st == 0
        o_s, l_s, st_s = oracle.verify_sparse(c["q_bits"], c["pool_bits"], sparse_lists(c, extra=3),
                                              c["sm_scale"], lib=lib)
        assert st_s == 0
        np.testing.assert_allclose(o_s, o_d, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l_s, l_d, rtol=0, atol=1e-12)


def pin_sparse_padding_order_duplicates(lib):
    rng = np.random.Generator(np.random.PCG64(43))
    c = case(43, T=4, H=3, L=(11,), N=60)
    idx = rng.integers(0, 60, size=(1, 4, 9)).astype(np.int32)
    o, l, _ = oracle.verify_sparse(c["q_bits"], c["pool_bits"], idx, c["sm_scale"], lib=lib)
    # -1 entries anywhere and any order: the same attention
    padded = np.concatenate([idx, np.full((1, 4, 5), -1, np.int32)], axis=2)
    shuffled = np.stack([np.stack([rng.permutation(padded[0, t]) for t in range(4)])])
    o2, l2, st = oracle.verify_sparse(c["q_bits"], c["pool_bits"], shuffled, c["sm_scale"], lib=lib)
    assert st == 0
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l, rtol=0, atol=1e-12)
    # every key listed twice: each weight doubles, so lse gains ln 2 and out is unchanged
    o3, l3, _ = oracle.verify_sparse(c["q_bits"], c["pool_bits"], np.concatenate([idx, idx], axis=2),
                                     c["sm_scale"], lib=lib)
    np.testing.assert_allclose(o3, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l3, l + math.log(2.0), rtol=0, atol=1e-12)


def pin_sparse_empty_list(lib):
    c = case(44, T=3, H=2, L=(5,), N=40)
    idx = np.asarray([[[3, 7, -1], [-1, -1, -1], [9, -1, 9]]], np.int32)
    o, l, st = oracle.verify_sparse(c["q_bits"], c["pool_bits"], idx, c["sm_scale"], lib=lib)
    assert st == 0
    assert np.all(l[0, 1] == -np.inf) and np.all(o[0, 1] == 0.0)
    assert np.isfinite(l[0, 0]).all() and np.isfinite(l[0, 2]).all()
    # a single (twice-listed) key: out is that key's value row
    np.testing.assert_allclose(o[0, 2], np.broadcast_to(wl.bf16_bits_to_f32(c["pool_bits"][9, :DV]), (2, DV)),
                               rtol=0, atol=1e-12)


def pin_sparse_bruteforce(lib):
    rng = np.random.Generator(np.random.PCG64(45))
    c = case(45, T=6, H=3, L=(4, 2), N=70)
    idx = rng.integers(-1, 70, size=(2, 6, 13)).astype(np.int32)
    o, l, st = oracle.verify_sparse(c["q_bits"], c["pool_bits"], idx, c["sm_scale"], lib=lib)
    bo, bl = oracle.brute_force_sparse(c["q_bits"], c["pool_bits"], idx, c["sm_scale"])
    assert st == 0
    np.testing.assert_allclose(o, bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, bl, rtol=0, atol=1e-12)


def test_sparse_bad_slot_is_left_out_and_flagged():
    c = case(46, T=2, H=2, L=(3,), N=30)
    good = np.asarray([[[4, 5, -1], [6, -1, -1]]], np.int32)
    bad = np.asarray([[[4, 5, 30], [6, -7, -1]]], np.int32)
    o1, l1, s1 = oracle.verify_sparse(c["q_bits"], c["pool_bits"], good, c["sm_scale"])
    o2, l2, s2 = oracle.verify_sparse(c["q_bits"], c["pool_bits"], bad, c["sm_scale"])
    assert s1 == 0 and s2 & oracle.BAD_SLOT
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


INDEPENDENT_PINS = [pin_golden_visibility, pin_single_node_is_decode, pin_chain_is_causal,
                    pin_prefix_free_chain_is_causal, pin_star_tree, pin_identical_keys, pin_dominant_key,
                    pin_worked_example, pin_inclusion_exclusion, pin_joint_permutation,
                    pin_sparse_equals_dense, pin_sparse_padding_order_duplicates, pin_sparse_empty_list]
ALL_PINS = INDEPENDENT_PINS + [pin_bruteforce, pin_sparse_bruteforce]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.load())


# ----------------------------------------------------------------------------- host behaviour

def test_bad_slot_is_masked_and_flagged():
    c = case(31, T=4, H=2, L=(8,))
    c_bad = dict(c, slot_idx=c["slot_idx"].copy())
    c_bad["slot_idx"][0, 3] = c["pool_bits"].shape[0] + 5
    out, lse, st = run(c_bad, oracle.load())
    assert st & oracle.BAD_SLOT
    keep = [j for j in range(8) if j != 3]
    c_ref = dict(c, slot_idx=np.ascontiguousarray(c["slot_idx"][:, keep]), prefix_len=np.asarray([7], np.int32))
    out_r, lse_r, st_r = run(c_ref, oracle.load())
    assert st_r == 0
    np.testing.assert_allclose(out, out_r, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_r, rtol=0, atol=1e-13)


def test_row_subset_equals_full():
    c = case(32, T=5, H=3, L=(6, 2))
    out, lse, _ = run(c, oracle.load())
    rows = np.asarray([0, 7, 29, 16], np.int64)
    o2, l2, _ = oracle.verify_attn(c["q_bits"], c["pool_bits"], c["slot_idx"], c["prefix_len"],
                                   c["tree_parent"], c["tree_slot_idx"], c["sm_scale"], rows=rows)
    assert np.array_equal(o2, out.reshape(-1, DV)[rows])
    assert np.array_equal(l2, lse.reshape(-1)[rows])


def test_kv_compact_oracle():
    c = case(33, T=3, H=2, L=(6, 5), N=64)
    dst_start = np.asarray([40, 50], np.int64)
    pool2, si2, st = oracle.kv_compact(c["pool_bits"], c["slot_idx"], c["prefix_len"], dst_start)
    assert st == 0
    for b in range(2):
        for j in range(int(c["prefix_len"][b])):
            assert si2[b, j] == dst_start[b] + j
            assert np.array_equal(pool2[dst_start[b] + j], c["pool_bits"][c["slot_idx"][b, j]])
    o1, l1, _ = run(c, oracle.load())
    o2, l2, _ = run(dict(c, pool_bits=pool2, slot_idx=si2), oracle.load())
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_workload_compact_pool_matches_full_pool():
    w = wl.make_workload("tiny")
    full = np.full((w.pool_slots, D), wl.BF16_NAN, np.uint16)
    full[w.slot_idx[0, :w.prefix_len[0]]] = w.kv_prefix_bits[0]
    full[w.tree_slot_idx[0]] = w.kv_tree_bits[0]
    o1, l1, s1 = oracle.verify_attn(w.q_bits, full, w.slot_idx, w.prefix_len, w.tree_parent,
                                    w.tree_slot_idx, w.sm_scale)
    o2, l2, s2 = oracle.verify_workload(w)
    assert s1 == 0 and s2 == 0
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    assert np.isfinite(o1).all()


# ----------------------------------------------------------------------------- mutations

MUTATIONS = {
    "drop self from the tree mask": ("vis[(size_t)t * T + u] = 1;", "if (u != t) vis[(size_t)t * T + u] = 1;"),
    "stop the ancestor walk below the root": ("      u = p;\n", "      u = (p == 0) ? -1 : p;\n"),
    "drop the last prefix key": ("for (int j = 0; j < L; ++j) m[j] = 1;", "for (int j = 0; j < L; ++j) m[j] = (j + 1 < L);"),
    "drop the rope term": ("for (int d = 0; d < d_qk; ++d) dot", "for (int d = 0; d < d_v; ++d) dot"),
    "v from the wrong dims": ("o[e] += p * bf16_value(kv[j][e]);", "o[e] += p * bf16_value(kv[j][e + (d_qk - d_v)]);"),
    "log base 2 for the lse": ("double l = smax + log(z);", "double l = smax + log2(z);"),
    "scale divides": ("s[j] = sm_scale * dot;", "s[j] = dot / sm_scale;"),
    "unshifted normaliser": ("if (m[j]) z += exp(s[j] - smax);", "if (m[j]) z += exp(s[j]);"),
    "tree key of the query node": (": tree_slot_idx[(int64_t)b * T + (j - L)];", ": tree_slot_idx[(int64_t)b * T + t];"),
    "neighbouring head's query": ("const uint16_t* qrow = q + row * d_qk;", "const uint16_t* qrow = q + (row ^ 1) * d_qk;"),
    "bad parent not reported": ("status |= ORACLE_BAD_PARENT;", "status |= 0;"),
    "sparse: last listed key dropped": ("for (int k = 0; k < topk; ++k) {", "for (int k = 0; k + 1 < topk; ++k) {"),
    "sparse: -1 read as slot 0": ("const int64_t slot = list[k];", "const int64_t slot = list[k] == -1 ? 0 : list[k];"),
    "sparse: heads share the node's first query": ("const uint16_t* query = q + row * (int64_t)d_qk;",
                                                   "const uint16_t* query = q + (row - row % H) * (int64_t)d_qk;"),
    "sparse: weights not normalised": ("const double weight = exp(score[n] - log_norm);",
                                       "const double weight = exp(score[n] - best);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(oracle.SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name!r} not unique"
    mut_src = tmp_path / "mutant.c"
    mut_src.write_text(src.replace(old, new))
    so = oracle.build(str(mut_src), str(tmp_path / "libmutant.so"), extra_flags=("-DMUTANT",))
    lib = oracle.load(so)
    caught = []
    for pin in INDEPENDENT_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"mutation {name!r} passed every independent pin"


# ----------------------------------------------------------------------------- ragged trees

def test_ragged_rows_equal_the_full_tree_rows():
    """Nodes are in topological order, so a node's ancestors precede it: cutting
    a request's tree after tree_len nodes leaves every kept row unchanged (the
    visibility rule of "The Art of Systematic Investigation", section "Input
    Knowledge Required to Understand This Message", item 1), and the cut rows
    are reported as out = 0, lse = -inf."""
    c = case(41, T=7, H=2, L=(9, 0, 5))
    lib = oracle.load()
    out_u, lse_u, st_u = run(c, lib)
    tree_len = np.asarray([7, 1, 4], np.int32)
    out_r, lse_r, st_r = oracle.verify_attn_ragged(c["q_bits"], c["pool_bits"], c["slot_idx"], c["prefix_len"],
                                                   c["tree_parent"], c["tree_slot_idx"], c["sm_scale"], tree_len,
                                                   lib=lib)
    assert st_u == 0 and st_r == 0
    for b, tl in enumerate(tree_len):
        np.testing.assert_allclose(out_r[b, :tl], out_u[b, :tl], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse_r[b, :tl], lse_u[b, :tl], rtol=0, atol=1e-13)
        assert np.all(out_r[b, tl:] == 0.0) and np.all(np.isneginf(lse_r[b, tl:]))


def test_ragged_matches_brute_force_on_the_cut_tree():
    """The ragged result against the independent NumPy brute force run on each
    request cut to its tree_len nodes."""
    c = case(42, T=6, H=2, L=(5, 3))
    tree_len = np.asarray([3, 6], np.int32)
    out_r, lse_r, st = oracle.verify_attn_ragged(c["q_bits"], c["pool_bits"], c["slot_idx"], c["prefix_len"],
                                                 c["tree_parent"], c["tree_slot_idx"], c["sm_scale"], tree_len)
    assert st == 0
    for b, tl in enumerate(tree_len):
        ob, lb = oracle.brute_force(c["q_bits"][b:b + 1, :tl], c["pool_bits"], c["slot_idx"][b:b + 1],
                                    c["prefix_len"][b:b + 1], c["tree_parent"][b:b + 1, :tl],
                                    c["tree_slot_idx"][b:b + 1, :tl], c["sm_scale"])
        np.testing.assert_allclose(out_r[b, :tl], ob[0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse_r[b, :tl], lb[0], rtol=0, atol=1e-12)


def test_ragged_tree_len_is_clamped_and_flagged():
    c = case(43, T=4, H=1, L=(3, 2))
    full = oracle.verify_attn_ragged(c["q_bits"], c["pool_bits"], c["slot_idx"], c["prefix_len"], c["tree_parent"],
                                     c["tree_slot_idx"], c["sm_scale"], np.asarray([4, 0], np.int32))
    bad = oracle.verify_attn_ragged(c["q_bits"], c["pool_bits"], c["slot_idx"], c["prefix_len"], c["tree_parent"],
                                    c["tree_slot_idx"], c["sm_scale"], np.asarray([9, -2], np.int32))
    assert full[2] == 0 and bad[2] == oracle.BAD_TREE_LEN
    assert np.array_equal(full[0], bad[0]) and np.array_equal(full[1], bad[1])
