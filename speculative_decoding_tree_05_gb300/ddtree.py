"""Thin ctypes binding of include/ddtree.h: argument marshalling only.

Every step of the computation runs in the CUDA library (lib/libddtree.so).
PyTorch only provides device memory and the current stream.  If the library is
missing this module raises at import-time use; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "libddtree.so")

D_QK = 576
D_V = 512

DDT_OK = 0
ERRORS = {-1: "DDT_ERR_NULL", -2: "DDT_ERR_DIMS", -3: "DDT_ERR_WORKSPACE", -4: "DDT_ERR_ALIGN",
          -5: "DDT_ERR_LAUNCH", -6: "DDT_ERR_DEVICE", -7: "DDT_ERR_ALIAS"}
STATUS_BAD_SLOT = 1
STATUS_BAD_PARENT = 2
STATUS_BAD_PREFIX = 4
STATUS_TIMEOUT = 8
STATUS_BAD_TREE_LEN = 16

EXPORTS = ("ddtree_verify_workspace_bytes", "ddtree_verify_attn", "ddtree_verify_attn_fused",
           "ddtree_verify_attn_ragged",
           "ddtree_verify_prefix_phase",
           "ddtree_verify_merge_phase", "ddtree_verify_attn_static_scratch", "ddtree_kv_compact",
           "ddtree_kv_compact_check", "ddtree_verify_sparse_workspace_bytes", "ddtree_verify_attn_sparse",
           "ddtree_read_device_status", "ddtree_status_string")


class DDTError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {ERRORS.get(code, code)} ({status_string(code)})")
        self.code = code


class Dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_nodes", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("slot_stride", ctypes.c_int32), ("pool_slots", ctypes.c_int64),
                ("max_prefix_len", ctypes.c_int32), ("prefix_len_sum", ctypes.c_int32)]


_lib = None


def load(path: str):
    """Load a build of the library from `path` and declare its C signatures.

    lib() loads the product build; tests also load the test-hooks build this way.
    """
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing (run __graft_entry__.build())")
    L = ctypes.CDLL(path)
    vp, i32p = ctypes.c_void_p, ctypes.c_void_p
    L.ddtree_verify_workspace_bytes.restype = ctypes.c_size_t
    L.ddtree_verify_workspace_bytes.argtypes = [ctypes.POINTER(Dims)]
    for fn in ("ddtree_verify_attn", "ddtree_verify_attn_fused", "ddtree_verify_prefix_phase",
               "ddtree_verify_merge_phase"):
        if not hasattr(L, fn):   # builds that predate an entry point
            continue
        f = getattr(L, fn)
        f.restype = ctypes.c_int
        f.argtypes = [vp, vp, i32p, i32p, i32p, i32p, ctypes.c_float, vp, vp, ctypes.POINTER(Dims), vp,
                      ctypes.c_size_t, vp]
    L.ddtree_verify_attn_ragged.restype = ctypes.c_int
    L.ddtree_verify_attn_ragged.argtypes = [vp, vp, i32p, i32p, i32p, i32p, i32p, ctypes.c_float, vp, vp,
                                            ctypes.POINTER(Dims), vp, ctypes.c_size_t, vp]
    L.ddtree_verify_attn_static_scratch.restype = ctypes.c_int
    L.ddtree_verify_attn_static_scratch.argtypes = [vp, vp, i32p, i32p, i32p, i32p, ctypes.c_float, vp, vp,
                                                    ctypes.POINTER(Dims), vp]
    L.ddtree_kv_compact.restype = ctypes.c_int
    L.ddtree_kv_compact.argtypes = [vp, vp, i32p, i32p, vp, i32p, ctypes.POINTER(Dims), vp, vp]
    if hasattr(L, "ddtree_kv_compact_check"):   # absent from builds that predate the validator
        L.ddtree_kv_compact_check.restype = ctypes.c_int
        L.ddtree_kv_compact_check.argtypes = [vp, vp, vp, vp, ctypes.POINTER(Dims), ctypes.c_int32,
                                              ctypes.POINTER(ctypes.c_int64)]
    if hasattr(L, "ddtree_verify_attn_sparse"):
        L.ddtree_verify_sparse_workspace_bytes.restype = ctypes.c_size_t
        L.ddtree_verify_sparse_workspace_bytes.argtypes = [ctypes.POINTER(Dims)]
        L.ddtree_verify_attn_sparse.restype = ctypes.c_int
        L.ddtree_verify_attn_sparse.argtypes = [vp, vp, i32p, ctypes.c_float, vp, vp, ctypes.POINTER(Dims), vp,
                                                ctypes.c_size_t, vp]
    if hasattr(L, "ddtree_internal_plan"):
        L.ddtree_internal_plan.restype = ctypes.c_int
        L.ddtree_internal_plan.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, ctypes.POINTER(ctypes.c_int32)]
    L.ddtree_read_device_status.restype = ctypes.c_int
    L.ddtree_read_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int32), vp]
    L.ddtree_status_string.restype = ctypes.c_char_p
    L.ddtree_status_string.argtypes = [ctypes.c_int]
    return L


def lib():
    """Load lib/libddtree.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        _lib = load(LIB_PATH)
    return _lib


def status_string(code: int) -> str:
    return lib().ddtree_status_string(int(code)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def make_dims(batch, nodes, heads, pool_slots, slot_stride, max_prefix_len, prefix_len_sum=0) -> Dims:
    """prefix_len_sum: optional host-side sum of the prefix lengths (0: unknown); it only steers the split."""
    return Dims(int(batch), int(nodes), int(heads), int(slot_stride), int(pool_slots), int(max_prefix_len),
                int(prefix_len_sum))


def workspace_bytes(dims: Dims) -> int:
    return int(lib().ddtree_verify_workspace_bytes(ctypes.byref(dims)))


def plan(dims: Dims, sm_count: int | None = None, library=None) -> dict:
    """The schedule the library picks for these sizes: row tiles, key splits (keys of split 0 and of
    each later split), or key-range groups (groups > 0).  sm_count: the device's SM count (default: the current device's)."""
    if sm_count is None:
        import torch
        sm_count = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    out = (ctypes.c_int32 * 5)()
    _check((library or lib()).ddtree_internal_plan(ctypes.byref(dims), int(sm_count), out), "ddtree_internal_plan")
    return dict(row_tiles=out[0], splits=out[1], chunk0=out[4], chunk=out[2], groups=out[3])


def _check(rc, what):
    if rc != DDT_OK:
        raise DDTError(rc, what)


class Verifier:
    """Holds a workspace sized for one set of dims and runs verify calls with it.

    q [B,T,H,576] bf16, kv_pool [N,576] bf16, slot_idx [B,stride] int32, prefix_len [B] int32,
    tree_parent [B,T] int32, tree_slot_idx [B,T] int32 -- all CUDA tensors.
    """

    def __init__(self, batch, nodes, heads, pool_slots, slot_stride, max_prefix_len=None, device=None,
                 prefix_len_sum=0, library=None):
        import torch
        self.lib = lib() if library is None else library
        self.dims = make_dims(batch, nodes, heads, pool_slots, slot_stride,
                              slot_stride if max_prefix_len is None else max_prefix_len, prefix_len_sum)
        self.device = torch.device("cuda") if device is None else torch.device(device)
        with torch.cuda.device(self.device):
            n = int(self.lib.ddtree_verify_workspace_bytes(ctypes.byref(self.dims)))
            if n == 0:
                raise DDTError(-2, "ddtree_verify_workspace_bytes")
            self.workspace = torch.empty(n, dtype=torch.uint8, device=self.device)

    def __call__(self, q, kv_pool, slot_idx, prefix_len, tree_parent, tree_slot_idx, sm_scale, out=None,
                 lse=None, stream=None, phase="all", tree_len=None):
        """phase: "all" (ddtree_verify_attn), "fused" (ddtree_verify_attn_fused: always one launch),
        "prefix" or "merge" (the two-launch path's halves).

        tree_len: optional int32 [B] CUDA tensor of active nodes per request
        (ddtree_verify_attn_ragged; phase must be "all").
        """
        import torch
        B, T, H, D = q.shape
        if out is None:
            out = torch.empty((B, T, H, D_V), dtype=torch.float32, device=q.device)
        if lse is None:
            lse = torch.empty((B, T, H), dtype=torch.float32, device=q.device)
        if tree_len is not None:
            if phase != "all":
                raise ValueError("ragged trees run as one call (phase='all')")
            rc = self.lib.ddtree_verify_attn_ragged(_ptr(q), _ptr(kv_pool), _ptr(slot_idx), _ptr(prefix_len),
                                                 _ptr(tree_parent), _ptr(tree_slot_idx), _ptr(tree_len),
                                                 float(sm_scale), _ptr(out), _ptr(lse), ctypes.byref(self.dims),
                                                 _ptr(self.workspace), self.workspace.numel(), _stream(stream))
            _check(rc, "ddtree_verify_attn_ragged")
            return out, lse
        fn = {"all": "ddtree_verify_attn", "fused": "ddtree_verify_attn_fused", "prefix": "ddtree_verify_prefix_phase",
              "merge": "ddtree_verify_merge_phase"}[phase]
        rc = getattr(self.lib, fn)(_ptr(q), _ptr(kv_pool), _ptr(slot_idx), _ptr(prefix_len), _ptr(tree_parent),
                                _ptr(tree_slot_idx), float(sm_scale), _ptr(out), _ptr(lse),
                                ctypes.byref(self.dims), _ptr(self.workspace), self.workspace.numel(),
                                _stream(stream))
        _check(rc, fn)
        return out, lse

    def status(self, stream=None) -> int:
        return read_device_status(self.workspace, stream, library=self.lib)


def verify_attn(q, kv_pool, slot_idx, prefix_len, tree_parent, tree_slot_idx, sm_scale, max_prefix_len=None,
                out=None, lse=None, stream=None):
    """One-off verify call (allocates its own workspace); returns (out, lse)."""
    B, T, H, _ = q.shape
    v = Verifier(B, T, H, kv_pool.shape[0], slot_idx.shape[1], max_prefix_len, device=q.device)
    return v(q, kv_pool, slot_idx, prefix_len, tree_parent, tree_slot_idx, sm_scale, out, lse, stream)


class SparseVerifier:
    """Sparse-index verify attention: node (b, t) attends to the pool rows its index list names.

    indices [B, T, topk] int32 CUDA tensor (-1 = no key); q [B, T, H, 576] bf16; a workspace is
    held for one set of sizes.
    """

    def __init__(self, batch, nodes, heads, pool_slots, topk, device=None, library=None):
        import torch
        self.lib = lib() if library is None else library
        self.dims = make_dims(batch, nodes, heads, pool_slots, topk, topk)
        self.device = torch.device("cuda") if device is None else torch.device(device)
        with torch.cuda.device(self.device):
            n = int(self.lib.ddtree_verify_sparse_workspace_bytes(ctypes.byref(self.dims)))
            if n == 0:
                raise DDTError(-2, "ddtree_verify_sparse_workspace_bytes")
            self.workspace = torch.empty(n, dtype=torch.uint8, device=self.device)

    def __call__(self, q, kv_pool, indices, sm_scale, out=None, lse=None, stream=None):
        import torch
        B, T, H, _ = q.shape
        if out is None:
            out = torch.empty((B, T, H, D_V), dtype=torch.float32, device=q.device)
        if lse is None:
            lse = torch.empty((B, T, H), dtype=torch.float32, device=q.device)
        rc = self.lib.ddtree_verify_attn_sparse(_ptr(q), _ptr(kv_pool), _ptr(indices), float(sm_scale), _ptr(out),
                                                _ptr(lse), ctypes.byref(self.dims), _ptr(self.workspace),
                                                self.workspace.numel(), _stream(stream))
        _check(rc, "ddtree_verify_attn_sparse")
        return out, lse

    def status(self, stream=None) -> int:
        return read_device_status(self.workspace, stream, library=self.lib)


def verify_attn_static_scratch(q, kv_pool, slot_idx, prefix_len, tree_parent, tree_slot_idx, sm_scale, out,
                               lse, max_prefix_len=None, stream=None):
    """Verify attention with the library's fixed scratch array (no allocation in the call).

    For callers that cannot allocate device memory at call time; out and lse
    are caller-provided.  Calls must not overlap on the GPU (they share the array).
    """
    B, T, H, _ = q.shape
    stride = slot_idx.shape[1]
    dims = make_dims(B, T, H, kv_pool.shape[0], stride, stride if max_prefix_len is None else max_prefix_len)
    rc = lib().ddtree_verify_attn_static_scratch(_ptr(q), _ptr(kv_pool), _ptr(slot_idx), _ptr(prefix_len),
                                                 _ptr(tree_parent), _ptr(tree_slot_idx), float(sm_scale), _ptr(out),
                                                 _ptr(lse), ctypes.byref(dims), _stream(stream))
    _check(rc, "ddtree_verify_attn_static_scratch")
    return out, lse


def kv_compact_check(slot_idx, prefix_len, dst_start, pool_slots, same_pool=True, tree_slot_idx=None,
                     max_prefix_len=None):
    """Host-side check of kv_compact's aliasing contract (numpy arrays or CPU tensors).

    Returns (code, first offending slot or -1); code is DDT_OK or DDT_ERR_ALIAS (-7).
    """
    import numpy as np
    si = np.ascontiguousarray(np.asarray(slot_idx), dtype=np.int32)
    pl = np.ascontiguousarray(np.asarray(prefix_len), dtype=np.int32)
    ds = np.ascontiguousarray(np.asarray(dst_start), dtype=np.int64)
    B, stride = si.shape
    T = 1
    ts = None
    if tree_slot_idx is not None:
        ts = np.ascontiguousarray(np.asarray(tree_slot_idx), dtype=np.int32)
        T = ts.shape[1]
    dims = make_dims(B, T, 1, pool_slots, stride, stride if max_prefix_len is None else max_prefix_len)
    bad = ctypes.c_int64(-1)
    p = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    rc = lib().ddtree_kv_compact_check(p(si), p(pl), p(ds), p(ts), ctypes.byref(dims), int(bool(same_pool)),
                                       ctypes.byref(bad))
    return int(rc), int(bad.value)


def kv_compact(kv_src, kv_dst, slot_idx, prefix_len, dst_start, slot_idx_out=None, max_prefix_len=None,
               workspace=None, stream=None, validate=False, tree_slot_idx=None):
    """Copy each request's prefix rows to dst_start[b] + j; returns slot_idx_out.

    validate=True first runs kv_compact_check on host copies of the tables (a
    debug option: it synchronises with the device) and raises DDTError if the
    aliasing contract is broken.
    """
    import torch
    B, stride = slot_idx.shape
    if validate:
        rc, bad = kv_compact_check(slot_idx.cpu().numpy(), prefix_len.cpu().numpy(), dst_start.cpu().numpy(),
                                   kv_src.shape[0], same_pool=kv_src.data_ptr() == kv_dst.data_ptr(),
                                   tree_slot_idx=None if tree_slot_idx is None else tree_slot_idx.cpu().numpy(),
                                   max_prefix_len=max_prefix_len)
        if rc != DDT_OK:
            raise DDTError(rc, f"kv_compact_check (slot {bad})")
    if slot_idx_out is None:
        slot_idx_out = slot_idx.clone()
    if workspace is None:
        workspace = torch.empty(256, dtype=torch.uint8, device=slot_idx.device)
    dims = make_dims(B, 1, 1, kv_src.shape[0], stride, stride if max_prefix_len is None else max_prefix_len)
    rc = lib().ddtree_kv_compact(_ptr(kv_src), _ptr(kv_dst), _ptr(slot_idx), _ptr(prefix_len), _ptr(dst_start),
                                 _ptr(slot_idx_out), ctypes.byref(dims), _ptr(workspace), _stream(stream))
    _check(rc, "ddtree_kv_compact")
    return slot_idx_out


def read_device_status(workspace, stream=None, library=None) -> int:
    st = ctypes.c_int32(0)
    rc = (lib() if library is None else library).ddtree_read_device_status(_ptr(workspace), ctypes.byref(st), _stream(stream))
    _check(rc, "ddtree_read_device_status")
    return int(st.value)
