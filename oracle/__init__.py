"""CPU oracle for DDTree verify attention (MLA 576/512) -- test infrastructure only.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py`
may import this package.  It shares nothing with the CUDA library: the C file
next to this one is compiled by gcc into its own shared object, and the NumPy
brute force below is an independent second reading of the same definition.

Contents
  build()                 compile ddtree_oracle.c -> _build/libddtree_oracle.so (gcc, OpenMP)
  verify_attn(...)        fp64 verify attention via the C oracle (all rows or a row subset)
  verify_attn_ragged(...) the same for requests with tree_len[b] <= T active nodes each
  tree_visibility(parent) the tree part of the visibility mask, via the C oracle
  kv_compact(...)         row-copy compaction via the C oracle
  verify_sparse(...)      fp64 sparse-index variant: each node lists its key slots (-1 = none)
  brute_force(...)        NumPy fp64 re-derivation for tiny inputs (independent code path)
  brute_force_sparse(...) the same for the sparse-index variant

The definition both follow: every tree node sees the whole prefix and, among the
tree nodes, its ancestors and itself ("The Art of Systematic Investigation",
section "Input Knowledge Required to Understand This Message"; "The Architecture
Detective: Uncovering FlashMLA's Potential for Blackwell DDTree Verification",
sections "The Message in Full" and "Assumptions and Their Validity");
scores are sm_scale * q.k over 576 dims, values are the first 512 dims of the
same latent row, lse is the natural log of the softmax normaliser.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ddtree_oracle.c")
LIB = os.path.join(HERE, "_build", "libddtree_oracle.so")

BAD_SLOT = 1
BAD_PARENT = 2
BAD_ARGS = 4
BAD_TREE_LEN = 16

_lib = None


def build(src: str = SRC, out: str = LIB, extra_flags=()) -> str:
    """Compile the C oracle with gcc (-O2, OpenMP).  Rebuilds when the source is newer."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src) and not extra_flags:
        return out
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", *extra_flags, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def load(path: str | None = None):
    """Load (building if needed) the oracle library; a path loads a separately built variant."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    lib = ctypes.CDLL(path or build())
    p = ctypes.c_void_p
    lib.oracle_verify_attn.restype = ctypes.c_int
    lib.oracle_verify_attn.argtypes = [p, p, ctypes.c_int64, p, ctypes.c_int64, p, p, p, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_double, p, ctypes.c_int64, p, p]
    lib.oracle_tree_visibility.restype = ctypes.c_int
    lib.oracle_tree_visibility.argtypes = [p, ctypes.c_int, p]
    lib.oracle_verify_sparse.restype = ctypes.c_int
    lib.oracle_verify_sparse.argtypes = [p, p, ctypes.c_int64, p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_double, p, p]
    lib.oracle_kv_compact.restype = ctypes.c_int
    lib.oracle_kv_compact.argtypes = [p, p, ctypes.c_int64, p, ctypes.c_int64, p, p, ctypes.c_int,
                                      ctypes.c_int, p]
    if path is None:
        _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def verify_attn(q_bits, pool_bits, slot_idx, prefix_len, tree_parent, tree_slot_idx, sm_scale,
                rows=None, lib=None):
    """fp64 verify attention.

    q_bits uint16 [B,T,H,Dqk] (bf16 bits), pool_bits uint16 [N,Dqk], slot_idx int32 [B,stride],
    prefix_len int32 [B], tree_parent int32 [B,T], tree_slot_idx int32 [B,T].
    Returns (out fp64 [n,Dv] or [B,T,H,Dv], lse fp64 [n] or [B,T,H], status bits).
    D_v is fixed at D_qk - 64 (the latent part), as in the MLA absorbed form.
    """
    lib = lib or load()
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    pool = np.ascontiguousarray(pool_bits, dtype=np.uint16)
    B, T, H, dqk = q.shape
    dv = dqk - 64
    si = np.ascontiguousarray(slot_idx, dtype=np.int32).reshape(B, -1)
    pl = np.ascontiguousarray(prefix_len, dtype=np.int32)
    tp = np.ascontiguousarray(tree_parent, dtype=np.int32)
    ts = np.ascontiguousarray(tree_slot_idx, dtype=np.int32)
    if rows is None:
        n = B * T * H
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = len(rows_arr)
    out = np.zeros((n, dv), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    st = lib.oracle_verify_attn(_ptr(q), _ptr(pool), pool.shape[0], _ptr(si), si.shape[1], _ptr(pl),
                                _ptr(tp), _ptr(ts), B, T, H, dqk, dv, float(sm_scale),
                                None if rows_arr is None else _ptr(rows_arr), n, _ptr(out), _ptr(lse))
    if rows is None:
        out = out.reshape(B, T, H, dv)
        lse = lse.reshape(B, T, H)
    return out, lse, st


def verify_attn_ragged(q_bits, pool_bits, slot_idx, prefix_len, tree_parent, tree_slot_idx, sm_scale, tree_len,
                       lib=None):
    """fp64 verify attention for a batch whose request b has tree_len[b] active nodes.

    Request b is the request alone with T = tree_len[b] (its first tree_len[b]
    nodes; nodes are in topological order, so every ancestor of an active node
    is active); rows of nodes t >= tree_len[b] get out = 0, lse = -inf.  Values
    of tree_len outside [0, T] are clamped and set BAD_TREE_LEN.  Arrays keep
    their [B, T] shapes.
    """
    q = np.asarray(q_bits)
    B, T, H, dqk = q.shape
    dv = dqk - 64
    out = np.zeros((B, T, H, dv), dtype=np.float64)
    lse = np.full((B, T, H), -np.inf, dtype=np.float64)
    st = 0
    si = np.asarray(slot_idx).reshape(B, -1)
    for b in range(B):
        tl = int(tree_len[b])
        if tl < 0 or tl > T:
            st |= BAD_TREE_LEN
            tl = min(max(tl, 0), T)
        if tl == 0:
            continue
        o, l, s_b = verify_attn(q[b:b + 1, :tl], pool_bits, si[b:b + 1], np.asarray(prefix_len)[b:b + 1],
                                np.asarray(tree_parent)[b:b + 1, :tl], np.asarray(tree_slot_idx)[b:b + 1, :tl],
                                sm_scale, lib=lib)
        out[b, :tl] = o[0]
        lse[b, :tl] = l[0]
        st |= s_b
    return out, lse, st


def verify_workload(w, rows=None, lib=None):
    """Oracle on a workload, through its compact host pool (used rows only)."""
    pool, si, ts = w.compact_host_pool()
    return verify_attn(w.q_bits, pool, si, w.prefix_len, w.tree_parent, ts, w.sm_scale, rows=rows, lib=lib)


def verify_sparse(q_bits, pool_bits, indices, sm_scale, lib=None):
    """fp64 sparse-index verify attention.

    q_bits uint16 [B,T,H,Dqk], pool_bits uint16 [N,Dqk], indices int32 [B,T,topk] (-1 = no key).
    Returns (out fp64 [B,T,H,Dv], lse fp64 [B,T,H], status bits).
    """
    lib = lib or load()
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    pool = np.ascontiguousarray(pool_bits, dtype=np.uint16)
    B, T, H, dqk = q.shape
    dv = dqk - 64
    idx = np.ascontiguousarray(indices, dtype=np.int32).reshape(B, T, -1)
    topk = idx.shape[2]
    out = np.zeros((B, T, H, dv), dtype=np.float64)
    lse = np.zeros((B, T, H), dtype=np.float64)
    st = lib.oracle_verify_sparse(_ptr(q), _ptr(pool), pool.shape[0], _ptr(idx), topk, B, T, H, dqk, dv,
                                  float(sm_scale), _ptr(out), _ptr(lse))
    return out, lse, st


def tree_visibility(parent) -> tuple:
    lib = load()
    p = np.ascontiguousarray(parent, dtype=np.int32)
    T = len(p)
    vis = np.zeros((T, T), dtype=np.uint8)
    st = lib.oracle_tree_visibility(_ptr(p), T, _ptr(vis))
    return vis.astype(bool), st


def kv_compact(src_bits, slot_idx, prefix_len, dst_start, dst_bits=None):
    """Returns (dst pool, slot_idx_out, status); dst defaults to a copy of src."""
    lib = load()
    src = np.ascontiguousarray(src_bits, dtype=np.uint16)
    dst = src.copy() if dst_bits is None else np.ascontiguousarray(dst_bits, dtype=np.uint16).copy()
    si = np.ascontiguousarray(slot_idx, dtype=np.int32)
    out = si.copy()
    pl = np.ascontiguousarray(prefix_len, dtype=np.int32)
    ds = np.ascontiguousarray(dst_start, dtype=np.int64)
    st = lib.oracle_kv_compact(_ptr(src), _ptr(dst), src.shape[0], _ptr(si), si.shape[1], _ptr(pl),
                               _ptr(ds), si.shape[0], src.shape[1], _ptr(out))
    return dst, out, st


# ----------------------------------------------------------------------------- independent brute force

def _bf16(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(
        np.float64)


def _ancestors_by_descent(parent):
    """anc[t] = set of nodes whose subtree contains t, found by walking down from each node."""
    T = len(parent)
    children = [[] for _ in range(T)]
    for i in range(1, T):
        children[parent[i]].append(i)
    anc = [set() for _ in range(T)]
    for u in range(T):
        stack = [u]
        while stack:
            x = stack.pop()
            anc[x].add(u)
            stack.extend(children[x])
    return anc


def brute_force(q_bits, pool_bits, slot_idx, prefix_len, tree_parent, tree_slot_idx, sm_scale):
    """NumPy fp64 verify attention for tiny, valid inputs, written apart from the C oracle:
    subtree descent for the mask, a dense score matrix, logaddexp reduction for the lse."""
    q = _bf16(q_bits)
    pool = _bf16(pool_bits)
    B, T, H, dqk = q.shape
    dv = dqk - 64
    out = np.zeros((B, T, H, dv))
    lse = np.zeros((B, T, H))
    for b in range(B):
        L = int(prefix_len[b])
        keys = np.concatenate([pool[np.asarray(slot_idx[b][:L], dtype=np.int64)],
                               pool[np.asarray(tree_slot_idx[b], dtype=np.int64)]], axis=0)
        anc = _ancestors_by_descent(list(tree_parent[b]))
        for t in range(T):
            cols = list(range(L)) + [L + u for u in sorted(anc[t])]
            k = keys[cols]
            scores = (q[b, t] @ k.T) * sm_scale          # [H, n]
            lse_bt = np.logaddexp.reduce(scores, axis=1)
            w = np.exp(scores - lse_bt[:, None])
            out[b, t] = w @ k[:, :dv]
            lse[b, t] = lse_bt
    return out, lse


def brute_force_sparse(q_bits, pool_bits, indices, sm_scale):
    """NumPy fp64 sparse-index attention for tiny, valid inputs (every listed value is -1 or a pool row):
    dense scores over the listed rows, logaddexp reduction."""
    q = _bf16(q_bits)
    pool = _bf16(pool_bits)
    B, T, H, dqk = q.shape
    dv = dqk - 64
    idx = np.asarray(indices).reshape(B, T, -1)
    out = np.zeros((B, T, H, dv))
    lse = np.full((B, T, H), -np.inf)
    for b in range(B):
        for t in range(T):
            keys = pool[[int(s) for s in idx[b, t] if s != -1]]
            if len(keys) == 0:
                continue
            scores = (q[b, t] @ keys.T) * sm_scale
            l = np.logaddexp.reduce(scores, axis=1)
            out[b, t] = np.exp(scores - l[:, None]) @ keys[:, :dv]
            lse[b, t] = l
    return out, lse
