/*
 * ddtree.h -- C ABI of the DDTree verify-attention library for one GB300 (sm_103a).
 *
 * Operation ("The Architecture Detective: Uncovering FlashMLA's Potential for
 * Blackwell DDTree Verification", sections "The Message in Full" and "The
 * Discovery: FlashMLA's Hidden Capabilities"; "The Art of Systematic
 * Investigation", section "Input Knowledge Required to Understand This
 * Message"): in speculative decoding with a draft tree, every tree node of a
 * request is verified in one pass.  Each node's query attends to
 *   (a) the request's whole shared prefix, read through a page_size=1 token-slot
 *       table from a KV pool whose slots may be scattered, with no causal limit
 *       among the queries, and
 *   (b) among the tree nodes, only its ancestors and itself.
 * The attention is MLA in absorbed form: one KV head whose rows are 576 bf16
 * values (512 latent + 64 rope dims, 1152 bytes per slot); scores are
 * sm_scale * q.k over all 576 dims, values are the first 512 dims of the same row.
 *
 * Conventions for every entry point:
 *   - All buffers are caller-owned device memory unless stated otherwise.  The
 *     library allocates nothing, keeps no state between calls and never
 *     synchronises the stream (except ddtree_read_device_status, which says so).
 *   - All work is enqueued on `stream`; a call returns without waiting for it.
 *   - Host-side checks return a negative DDT_ERR_* code before anything is
 *     enqueued.  Problems that only the device can see (a slot index outside the
 *     pool, a parent entry that is not a valid earlier node, a prefix length out
 *     of range) never fault: the offending key or link is left out of the
 *     attention and a bit is OR-ed into a status word in the workspace, which
 *     ddtree_read_device_status returns.  The status word is cleared at the start
 *     of every call that takes the workspace.
 *   - Device pointers must be 16-byte aligned; bf16 is IEEE bfloat16.
 */
#ifndef DDTREE_H_
#define DDTREE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DDT_API __attribute__((visibility("default")))
#else
#define DDT_API
#endif

/* Same type as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* ddt_stream_t;

/* Host-side return codes. */
#define DDT_OK 0
#define DDT_ERR_NULL (-1)      /* a required pointer is NULL */
#define DDT_ERR_DIMS (-2)      /* unsupported sizes (see ddt_dims) */
#define DDT_ERR_WORKSPACE (-3) /* workspace smaller than ddtree_verify_workspace_bytes() */
#define DDT_ERR_ALIGN (-4)     /* a device pointer is not 16-byte aligned */
#define DDT_ERR_LAUNCH (-5)    /* a kernel launch or CUDA runtime call failed */
#define DDT_ERR_DEVICE (-6)    /* the current device is not an sm_103 GPU */
#define DDT_ERR_ALIAS (-7)     /* ddtree_kv_compact_check: destinations overlap or cover a live row */

/* Device status bits (ddtree_read_device_status). */
#define DDT_STATUS_BAD_SLOT 1      /* a slot index outside [0, pool_slots): key left out */
#define DDT_STATUS_BAD_PARENT 2    /* tree_parent[b][0] != -1 or tree_parent[b][i] not in [0, i): link ignored */
#define DDT_STATUS_BAD_PREFIX 4    /* prefix_len[b] outside [0, max_prefix_len]: clamped */
#define DDT_STATUS_TIMEOUT 8       /* a bounded on-chip wait gave up; outputs are not valid */
#define DDT_STATUS_BAD_TREE_LEN 16 /* tree_len[b] outside [0, num_nodes]: clamped */

/*
 * Sizes of one call.  Fixed by the library: D_qk = 576, D_v = 512.
 *   batch          B in [0, 65535] requests
 *   num_nodes      T in [1, 128] tree nodes per request (node 0 is the root)
 *   num_heads      H in [1, 1024] query heads (all share the single latent KV head)
 *   pool_slots     N >= 1 rows in the KV pool
 *   slot_stride    row stride (in entries) of slot_idx, >= max_prefix_len
 *   max_prefix_len upper bound on every prefix_len[b]; it sizes the workspace
 *                  and the launch.
 *   prefix_len_sum optional host-side hint: the sum of prefix_len over the
 *                  batch, or 0 if unknown.  It only steers the choice of the
 *                  key-split length (with 0 the planner assumes every request
 *                  is max_prefix_len long, which over-counts the work units of
 *                  a batch of mixed lengths and picks longer splits than
 *                  needed); results are correct for any value.  The workspace
 *                  size depends on it, so query ddtree_verify_workspace_bytes
 *                  with the same dims that the calls use.
 * The key-range split of each request depends only on these sizes, the
 * device's SM count and prefix_len[b], never on slot addresses, so results are
 * bitwise reproducible and identical for any slot layout of the same logical
 * data.
 */
typedef struct {
  int32_t batch;
  int32_t num_nodes;
  int32_t num_heads;
  int32_t slot_stride;
  int64_t pool_slots;
  int32_t max_prefix_len;
  int32_t prefix_len_sum;
} ddt_dims;

/* Bytes of workspace ddtree_verify_attn needs for these sizes on the current
 * device (0 if the sizes are unsupported).  Needs a current CUDA device. */
DDT_API size_t ddtree_verify_workspace_bytes(const ddt_dims* dims);

/*
 * Verify attention for every (request b, node t, head h).
 *
 *   q             bf16 [B, T, H, 576], contiguous (row id (b*T + t)*H + h)
 *   kv_pool       bf16 [N, 576], one latent row per slot
 *   slot_idx      int32 [B, slot_stride]: request b's prefix position j lives in
 *                 slot slot_idx[b*slot_stride + j], for j < prefix_len[b]
 *   prefix_len    int32 [B], each in [0, max_prefix_len]
 *   tree_parent   int32 [B, T]: parent[b][0] = -1, parent[b][i] in [0, i)
 *                 (nodes in topological order)
 *   tree_slot_idx int32 [B, T]: slot holding node i's own latent row
 *   sm_scale      scale applied to q.k before the softmax
 *   out           fp32 [B, T, H, 512] (written)
 *   lse           fp32 [B, T, H] (written): natural log of the softmax normaliser
 *   workspace     device scratch of >= ddtree_verify_workspace_bytes(dims) bytes,
 *                 256-byte aligned; holds the per-split partial results and the
 *                 status word.  Calls sharing a workspace must not overlap.
 *
 * The prefix part is split-KV over each request's key range, all T*H rows of a
 * request contracted together on the tensor cores; the tree part applies the
 * ancestor rule; a log-sum-exp merge combines them.  The call enqueues a
 * workspace clear, the prefix pass and the tail/merge kernel (exactly
 * ddtree_verify_prefix_phase then ddtree_verify_merge_phase; the second kernel
 * starts as a programmatic dependent of the first).  The key ranges come from
 * the sizes and the SM count: key splits of every request (all of one length,
 * or, for one request whose row tiles leave CTA pairs free, a long first split
 * with short ones behind it for the free pairs), or, for a
 * batch of 2 to 64 requests whose row tiles fit at least twice on the GPU's
 * CTA pairs, key-range groups (the requests' keys laid end to end and cut into
 * equal shares, each computed by one group of pairs).  Capturable in a CUDA
 * graph.  B = 0 enqueues nothing and returns DDT_OK.
 */
DDT_API int ddtree_verify_attn(const void* q, const void* kv_pool, const int32_t* slot_idx,
                       const int32_t* prefix_len, const int32_t* tree_parent,
                       const int32_t* tree_slot_idx, float sm_scale, float* out, float* lse,
                       const ddt_dims* dims, void* workspace, size_t workspace_bytes,
                       ddt_stream_t stream);

/*
 * The same computation as ddtree_verify_attn, always as one launch ("The Art of
 * Systematic Investigation", section "Input Knowledge Required to Understand
 * This Message", item 5, and "The Anatomy of a Kernel Investigation", section
 * "Conclusion": the verify kernel is captured in a CUDA graph; here it is a
 * single node besides the workspace clear).  A persistent grid of CTA pairs
 * works through the (request, key split, 128-row tile) units; the pair that
 * finishes the last split of a (request, row tile) merges its rows (tree tail
 * and log-sum-exp merge), counted with an atomic in the workspace: nothing ever
 * waits on another pair.  Same arguments and checks as ddtree_verify_attn, and
 * the same bits wherever ddtree_verify_attn uses key splits (this
 * launch always does; with key-range groups the partial sums are cut at other
 * keys and the results agree within rounding).  It is slower than
 * ddtree_verify_attn's two launches (the
 * merges run on the pairs that finish row tiles, not on every SM), so it is for
 * callers that want the single launch.
 */
DDT_API int ddtree_verify_attn_fused(const void* q, const void* kv_pool, const int32_t* slot_idx,
                                     const int32_t* prefix_len, const int32_t* tree_parent,
                                     const int32_t* tree_slot_idx, float sm_scale, float* out, float* lse,
                                     const ddt_dims* dims, void* workspace, size_t workspace_bytes,
                                     ddt_stream_t stream);

/*
 * Ragged trees: the same call for a batch whose requests have different node
 * counts (the pages' trees range from 9 to 65 nodes per request; "The Art of
 * Systematic Investigation", section "Input Knowledge Required to Understand
 * This Message", item 1).  Request b has tree_len[b] active nodes, 0..T-1 of
 * its [T]-strided arrays; T = dims->num_nodes is the largest count and keeps
 * every array's shape and stride.
 *   tree_len   int32 [B] device, each in [0, T] (values outside are clamped and
 *              set DDT_STATUS_BAD_TREE_LEN)
 * Rows of active nodes get exactly what ddtree_verify_attn would give that
 * request alone with T = tree_len[b]; rows of inactive nodes (t >= tree_len[b])
 * get out = 0 and lse = -inf, and their parent, slot and q entries are never
 * read.  Tiles of inactive rows skip the prefix pass.  tree_len must not be
 * NULL when B > 0 (DDT_ERR_NULL).
 */
DDT_API int ddtree_verify_attn_ragged(const void* q, const void* kv_pool, const int32_t* slot_idx,
                                      const int32_t* prefix_len, const int32_t* tree_parent,
                                      const int32_t* tree_slot_idx, const int32_t* tree_len, float sm_scale,
                                      float* out, float* lse, const ddt_dims* dims, void* workspace,
                                      size_t workspace_bytes, ddt_stream_t stream);

/*
 * The two phases of ddtree_verify_attn, for callers that schedule them
 * separately (for example to overlap the second with other work, or to time
 * each).  ddtree_verify_attn is exactly: clear the status word, then
 * ddtree_verify_prefix_phase, then ddtree_verify_merge_phase, on one stream.
 *   prefix phase: split-KV attention of every row over its prefix keys; writes
 *                 one normalised partial (o, lse) per key split into the
 *                 workspace.  Clears the status word first.
 *   merge phase:  tree tail (ancestors and self) and the log-sum-exp merge of
 *                 the tail with the prefix partials; writes out and lse.
 * Both take the same arguments and checks as ddtree_verify_attn; the merge
 * phase must follow the prefix phase of the same call on the same workspace.
 */
DDT_API int ddtree_verify_prefix_phase(const void* q, const void* kv_pool, const int32_t* slot_idx,
                               const int32_t* prefix_len, const int32_t* tree_parent,
                               const int32_t* tree_slot_idx, float sm_scale, float* out, float* lse,
                               const ddt_dims* dims, void* workspace, size_t workspace_bytes,
                               ddt_stream_t stream);
DDT_API int ddtree_verify_merge_phase(const void* q, const void* kv_pool, const int32_t* slot_idx,
                              const int32_t* prefix_len, const int32_t* tree_parent,
                              const int32_t* tree_slot_idx, float sm_scale, float* out, float* lse,
                              const ddt_dims* dims, void* workspace, size_t workspace_bytes,
                              ddt_stream_t stream);

/*
 * Sparse-index variant ("The Architecture Detective: Uncovering FlashMLA's
 * Potential for Blackwell DDTree Verification", sections "The Message in Full"
 * and "The Discovery: FlashMLA's Hidden Capabilities": the sparse attention
 * call takes a fixed-length list of key indices per query, -1 marking an
 * invalid entry; the pages set it aside for this workload because every list
 * would have to name the whole prefix).  Each tree node lists its own keys:
 *   indices   int32 [B, T, topk] device, topk = dims->max_prefix_len; node (b, t)
 *             attends, for all its H heads, to the rows kv_pool[indices[b][t][i]]
 *             with indices[b][t][i] != -1.  A slot listed twice counts twice.
 *             Other values outside [0, pool_slots) are left out and set
 *             DDT_STATUS_BAD_SLOT.  A node with no key gets out = 0, lse = -inf.
 *   q, out, lse as in ddtree_verify_attn ([B, T, H, ...]); dims->batch = B,
 *   num_nodes = T, num_heads = H, pool_slots = N, max_prefix_len = topk
 *   (slot_stride and prefix_len_sum are ignored); B * T <= 65535.
 *   workspace >= ddtree_verify_sparse_workspace_bytes(dims).
 * There is no tree part: the lists are the whole visible set.  The work is
 * the prefix pass over each node's list (the node's H heads are the rows of
 * the contraction) and the log-sum-exp merge of its key splits.
 */
DDT_API size_t ddtree_verify_sparse_workspace_bytes(const ddt_dims* dims);
DDT_API int ddtree_verify_attn_sparse(const void* q, const void* kv_pool, const int32_t* indices, float sm_scale,
                                      float* out, float* lse, const ddt_dims* dims, void* workspace,
                                      size_t workspace_bytes, ddt_stream_t stream);

/*
 * KV compaction (defragmentation) of each request's prefix rows
 * ("The Anatomy of a Kernel Investigation", section "The Reasoning Process: A
 * Deep Dive", phase 3; "The Architecture Detective", section "Defragmentation:
 * Separating Signal from Noise"):
 *   kv_dst[dst_start[b] + j] = kv_src[slot_idx[b][j]]       (bit-exact row copy)
 *   slot_idx_out[b][j]       = dst_start[b] + j
 * for j < prefix_len[b].  Entries of slot_idx_out beyond prefix_len[b] are not
 * written.  kv_src and kv_dst both have dims->pool_slots rows and may be the
 * same pool only if no destination row [dst_start[b], dst_start[b]+prefix_len[b])
 * is a source row of any request (the caller's contract; ddtree_kv_compact
 * does not check it -- ddtree_kv_compact_check below does, on the host).
 *   dst_start   int64 [B] device
 *   workspace   >= 256 bytes, 256-byte aligned (status word; bad source or
 *               destination slots set DDT_STATUS_BAD_SLOT and skip the row)
 */
DDT_API int ddtree_kv_compact(const void* kv_src, void* kv_dst, const int32_t* slot_idx,
                      const int32_t* prefix_len, const int64_t* dst_start, int32_t* slot_idx_out,
                      const ddt_dims* dims, void* workspace, ddt_stream_t stream);

/*
 * Debug validator of ddtree_kv_compact's aliasing contract, run on HOST copies
 * of the tables before a compaction ("The Architecture Detective", section
 * "Defragmentation: Separating Signal from Noise": compacting live KV in place
 * is only safe if no copy overwrites a row that is still read).  Pure host code:
 * it needs no GPU and enqueues nothing.
 *   slot_idx       int32 [B, slot_stride] host, as passed to ddtree_kv_compact
 *   prefix_len     int32 [B] host, each in [0, max_prefix_len] (else DDT_ERR_DIMS)
 *   dst_start      int64 [B] host
 *   tree_slot_idx  int32 [B, num_nodes] host, or NULL: the requests' tree rows,
 *                  which an in-place compaction must not overwrite either
 *   same_pool      nonzero when kv_dst is kv_src (in-place compaction)
 *   bad_slot       optional out: the first offending slot, or -1
 * Returns DDT_OK when every destination range [dst_start[b], +prefix_len[b])
 * lies inside the pool and the ranges are pairwise disjoint, and, for
 * same_pool, no destination row is a source slot of any request (a row that
 * is already at its destination, slot_idx[b][j] == dst_start[b] + j, is
 * allowed) or a tree slot; DDT_ERR_ALIAS otherwise.
 */
DDT_API int ddtree_kv_compact_check(const int32_t* slot_idx, const int32_t* prefix_len, const int64_t* dst_start,
                                    const int32_t* tree_slot_idx, const ddt_dims* dims, int32_t same_pool,
                                    int64_t* bad_slot);

/*
 * Verify attention without any allocation, for callers that cannot allocate
 * device memory when they run it (for example code running inside a memory
 * pool or allocator callback, or a plugin that may only use the buffers its
 * host framework hands it).  The pages have no counterpart of this entry point.
 *
 * Same arguments and results as ddtree_verify_attn, minus the workspace: the
 * scratch lives in a fixed 32 MiB device array inside the library, which every
 * GPU that loads the library holds until the process exits.  Sizes whose
 * scratch (ddtree_verify_workspace_bytes) exceeds 32 MiB return
 * DDT_ERR_WORKSPACE before anything is enqueued.  The first call on each device
 * looks up the array's device address (once, with that device current).  That
 * lookup can be the moment CUDA loads the library's device code onto the device
 * and reserves the array (modules load lazily by default), so it may allocate:
 * make the first call on each device at start-up, outside any allocator
 * callback and before any stream capture; later calls allocate nothing.  Size,
 * device and pointer checks return the same codes as ddtree_verify_attn.
 * Every call shares the one array:
 * calls whose work overlaps on the GPU (on different streams, or from several
 * threads) race and must be serialised by the caller.  The device status word
 * of these calls is not readable by the caller.
 */
DDT_API int ddtree_verify_attn_static_scratch(const void* q, const void* kv_pool, const int32_t* slot_idx,
                                              const int32_t* prefix_len, const int32_t* tree_parent,
                                              const int32_t* tree_slot_idx, float sm_scale, float* out,
                                              float* lse, const ddt_dims* dims, ddt_stream_t stream);

/* Waits for `stream`, then copies the status word of the last call that used
 * `workspace` to *host_status.  Returns DDT_OK or DDT_ERR_*.  The kernels write
 * the word asynchronously on the stream the verify call was enqueued on, so
 * the read waits for that stream alone (not the whole device): work on other
 * streams keeps running. */
DDT_API int ddtree_read_device_status(const void* workspace, int32_t* host_status, ddt_stream_t stream);

/* Static text for a DDT_ERR_* return code. */
DDT_API const char* ddtree_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* DDTREE_H_ */
