// api.cu -- the extern "C" boundary: argument checks, workspace plan, launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <algorithm>
#include <climits>
#include <cstdint>
#include <mutex>
#include <utility>
#include <vector>
#include "../../include/ddtree.h"
#include "kernels.cuh"
#include "schedule.cuh"

namespace ddt {
namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kStatusBytes = 256;

struct DeviceInfo {
  int sm_count = 0;
  bool ok = false;      // sm_103 and kernels configured
};

DeviceInfo g_dev[kMaxDevices];
std::once_flag g_once[kMaxDevices];

// Per-device, once: check the architecture and opt the kernels into large
// shared memory on that device.
int device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DDT_ERR_DEVICE;
  std::call_once(g_once[dev], [dev] {
    DeviceInfo d;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        major == 10 && minor == 3 && configure_prefix() == cudaSuccess && configure_tail_merge() == cudaSuccess)
      d.ok = true;
    g_dev[dev] = d;
  });
  *out = g_dev[dev];
  return out->ok ? DDT_OK : DDT_ERR_DEVICE;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Plan {
  int rows = 0, row_tiles = 0, chunk0 = kKeysPerTile, chunk = kKeysPerTile, splits = 0;
  int groups = 0;  // > 0: the two-launch path divides the batch into this many key-range groups
  size_t cnt_off = 0, cnt_bytes = 0, lse_off = 0, o_off = 0, bytes = 0;
};

int check_dims(const ddt_dims* d) {
  if (!d) return DDT_ERR_NULL;
  if (d->batch < 0 || d->batch > 65535 || d->num_nodes < 1 || d->num_nodes > kMaxNodes || d->num_heads < 1 ||
      d->num_heads > 1024 ||
      d->pool_slots < 1 || d->pool_slots > (int64_t(1) << 31) || d->max_prefix_len < 0 ||
      d->slot_stride < d->max_prefix_len || d->slot_stride < 0)
    return DDT_ERR_DIMS;
  return DDT_OK;
}

// Key-range split of the prefix.  Depends only on the sizes and the SM count, so
// a repeated call (or a call on a compacted pool) splits identically.
int make_plan(const ddt_dims* d, int sm_count, Plan* plan) {
  int rc = check_dims(d);
  if (rc != DDT_OK) return rc;
  Plan p;
  p.rows = d->num_nodes * d->num_heads;
  p.row_tiles = (p.rows + kTileRows - 1) / kTileRows;
  const int64_t L = d->max_prefix_len;
  if (L > 0 && d->batch > 0) {
    // Pick the number of key splits s (each unit = one CTA pair on one
    // (request, row tile, split)) that minimises the modelled time
    //   waves(s) * (64-key steps per unit + kUnitOverheadSteps),
    // the overhead being a unit's fixed cost (pipeline fill, Q staging, the
    // write of its partial O) in step equivalents; among equal costs take the
    // fewest splits.  Splits are at least kMinChunk keys long.
    const int64_t pairs = sm_count >= 2 ? sm_count / 2 : 1;
    const int64_t per_split = int64_t(d->batch) * p.row_tiles;
    // Units that hold keys: without a hint every request is taken to be L
    // long; with the sum of the prefix lengths, a request has about
    // sum/chunk splits in all plus half a split each for its partial last one.
    const int64_t len_sum = d->prefix_len_sum > 0 ? std::min<int64_t>(d->prefix_len_sum, L * d->batch) : 0;
    const int64_t tiles = (L + kKeysPerTile - 1) / kKeysPerTile;
    const int64_t max_splits = std::max<int64_t>(1, std::min<int64_t>(64, (L + kMinChunk - 1) / kMinChunk));
    int64_t best = 1;
    int64_t best_cost = -1;
    for (int64_t s = 1; s <= max_splits; ++s) {
      const int64_t steps = (tiles + s - 1) / s;            // per unit
      const int64_t splits = (tiles + steps - 1) / steps;   // splits that actually hold keys
      int64_t units = per_split * splits;
      if (len_sum > 0) {
        const int64_t chunk_keys = steps * kKeysPerTile;
        units = std::min(units, p.row_tiles * ((len_sum + chunk_keys - 1) / chunk_keys + (d->batch + 1) / 2));
      }
      const int64_t waves = (units + pairs - 1) / pairs;
      const int64_t cost = waves * (steps + kUnitOverheadSteps);
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        best = s;
      }
    }
    int64_t chunk = (tiles + best - 1) / best * kKeysPerTile;
    p.chunk0 = p.chunk = static_cast<int>(chunk);
    // One request whose row tiles leave R pairs free (T < pairs): a long first
    // split A on T pairs while the R others take the T short second splits,
    // k = ceil(T / R) each.  Balanced when A + o = k (S - A + o) (S steps, o a
    // unit's fixed cost); taken when its modelled time is below the equal
    // splits'.  c3: 65 tiles on 76 pairs, 882 + 142 steps in 888 step times
    // against 6 waves of 147 (918).
    const int64_t T = p.row_tiles, R = pairs - T, o = kUnitOverheadSteps;
    if (d->batch == 1 && R > 0 && tiles > 1) {
      const int64_t k = (T + R - 1) / R;
      const int64_t A = std::min(tiles - 1, std::max<int64_t>(1, (k * (tiles + o) - o + k) / (k + 1)));
      const int64_t cost = std::max(A + o, k * (tiles - A + o));
      if (cost < best_cost) {
        p.chunk0 = static_cast<int>(A * kKeysPerTile);
        p.chunk = static_cast<int>((tiles - A) * kKeysPerTile);
      }
    }
    p.splits = split_count(static_cast<int>(L), p.chunk0, p.chunk);
    // Key-range groups (schedule.cuh) for a batch whose row tiles fit at least
    // twice into the pairs: groups of row_tiles pairs share the steps of all
    // requests evenly, whatever their lengths.  Modelled cost: the steps of one
    // group plus a unit's fixed cost per request it touches (one, plus the
    // request boundaries that fall into it).  Taken when it is below the
    // splits' cost.
    if (d->batch >= 2 && d->batch <= kMaxGroupBatch && 2 * int64_t(p.row_tiles) <= pairs) {
      const int64_t steps_all = len_sum > 0 ? (len_sum + kKeysPerTile - 1) / kKeysPerTile + d->batch / 2
                                            : int64_t(d->batch) * tiles;
      int64_t g = pairs / p.row_tiles;
      g = std::min(g, std::max<int64_t>(1, steps_all / (kMinChunk / kKeysPerTile)));
      const int64_t cost = (steps_all + g - 1) / g + kUnitOverheadSteps * (1 + (d->batch - 1 + g - 1) / g);
      if (cost < best_cost) p.groups = static_cast<int>(g);
    }
  }
  // split slots per request: the splits, or the pieces of the groups (at most one per group)
  const size_t part_rows = size_t(d->batch) * std::max(p.splits, p.groups) * p.row_tiles * kTileRows;
  // [status words | split arrivals per (request, row tile) | lse partials | o partials]
  p.cnt_off = kStatusBytes;
  p.cnt_bytes = size_t(d->batch) * p.row_tiles * sizeof(int32_t);
  p.lse_off = align_up(p.cnt_off + p.cnt_bytes, 256);
  p.o_off = align_up(p.lse_off + part_rows * sizeof(float), 256);
  p.bytes = p.o_off + part_rows * kDv * sizeof(float);
  *plan = p;
  return DDT_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// cuTensorMapEncodeTiled, fetched from the driver once (no link-time libcuda dependency).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// The pool as a 2-D bf16 tensor [rows][576] (1152-byte rows), box of box_cols
// columns x box_rows rows, 128-byte swizzle (64 columns) or 64-byte (32 columns).
bool encode_pool_map(CUtensorMap* m, const void* pool, int64_t rows, uint32_t box_cols, uint32_t box_rows) {
  const EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDqk), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kRowBytes)};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t elem_strides[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides, box, elem_strides,
            CU_TENSOR_MAP_INTERLEAVE_NONE, box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace ddt

using namespace ddt;

namespace ddt {
// Checks of a verify call that do not look at its pointers, in the order
// ddtree_verify_attn applies them: sizes, then the device; on success
// *workspace_bytes is the scratch the call needs (0 for an empty batch).
int verify_precheck(const ddt_dims* dims, size_t* workspace_bytes) {
  int rc = check_dims(dims);
  if (rc != DDT_OK) return rc;
  *workspace_bytes = 0;
  if (dims->batch == 0) return DDT_OK;
  DeviceInfo dev;
  if ((rc = device_info(&dev)) != DDT_OK) return rc;
  Plan plan;
  if ((rc = make_plan(dims, dev.sm_count, &plan)) != DDT_OK) return rc;
  *workspace_bytes = plan.bytes;
  return DDT_OK;
}
}  // namespace ddt

extern "C" size_t ddtree_verify_workspace_bytes(const ddt_dims* dims) {
  DeviceInfo dev;
  if (device_info(&dev) != DDT_OK) return 0;
  Plan plan;
  if (make_plan(dims, dev.sm_count, &plan) != DDT_OK) return 0;
  return plan.bytes;
}

namespace ddt {
namespace {

enum Phase : int { kPhasePrefix = 1, kPhaseMerge = 2, kPhaseFused = 4 };

// The fused launch's persistent grid: at most the CTA pairs that fit at once.
int fused_pairs(const DeviceInfo& dev) {
  const int pairs = fused_max_pairs();
  return pairs > 0 ? pairs : (dev.sm_count >= 2 ? dev.sm_count / 2 : 1);
}

// The sparse-index call as the dense machinery sees it: each (request, node)
// is a request of one node whose key list is its prefix (topk =
// max_prefix_len entries, every list full length, -1 = no key).  Returns
// DDT_ERR_DIMS when the flattened batch is too large.
int sparse_as_dense(const ddt_dims* d, ddt_dims* e) {
  int rc = check_dims(d);
  if (rc != DDT_OK) return rc;
  const int64_t batch = int64_t(d->batch) * d->num_nodes;
  if (batch > 65535) return DDT_ERR_DIMS;
  *e = *d;
  e->batch = static_cast<int32_t>(batch);
  e->num_nodes = 1;
  e->slot_stride = d->max_prefix_len;
  const int64_t keys = batch * d->max_prefix_len;
  e->prefix_len_sum = keys <= INT32_MAX ? static_cast<int32_t>(keys) : 0;
  return DDT_OK;
}

int verify_phases(int phases, const void* q, const void* kv_pool, const int32_t* slot_idx,
                  const int32_t* prefix_len, const int32_t* tree_parent, const int32_t* tree_slot_idx,
                  const int32_t* tree_len, float sm_scale, float* out, float* lse, const ddt_dims* dims,
                  void* workspace, size_t workspace_bytes, ddt_stream_t stream, bool sparse = false) {
  int rc = check_dims(dims);
  if (rc != DDT_OK) return rc;
  if (dims->batch == 0) return DDT_OK;
  if (!q || !kv_pool || !out || !lse || !workspace || (!slot_idx && dims->max_prefix_len > 0) ||
      (!sparse && (!prefix_len || !tree_parent || !tree_slot_idx)))
    return DDT_ERR_NULL;
  if (!aligned(q, 16) || !aligned(kv_pool, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
      !aligned(workspace, 256) || !aligned(slot_idx, 4) || !aligned(prefix_len, 4) ||
      !aligned(tree_parent, 4) || !aligned(tree_slot_idx, 4) || !aligned(tree_len, 4))
    return DDT_ERR_ALIGN;
  DeviceInfo dev;
  if ((rc = device_info(&dev)) != DDT_OK) return rc;
  Plan plan;
  if ((rc = make_plan(dims, dev.sm_count, &plan)) != DDT_OK) return rc;
  if (workspace_bytes < plan.bytes) return DDT_ERR_WORKSPACE;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  const float scale_log2 = sm_scale * 1.4426950408889634f;
  float* lse_part = reinterpret_cast<float*>(ws + plan.lse_off);
  float* o_part = reinterpret_cast<float*>(ws + plan.o_off);

  if (phases & (kPhasePrefix | kPhaseFused)) {
    // the status words and (fused) the split arrival counters start at zero
    const size_t clear = (phases & kPhaseFused) ? plan.cnt_off + plan.cnt_bytes : 4 * sizeof(int32_t);
    if (cudaMemsetAsync(status, 0, clear, s) != cudaSuccess) return DDT_ERR_LAUNCH;
    if (plan.splits > 0 || (phases & kPhaseFused)) {
      PrefixParams pp;
#ifdef DDT_TEST_HOOKS
      pp.test_drop_step = g_test_drop_step;
#endif
      // the 64-row box maps (steps of consecutive slots) only when the pool has 64 rows
      pp.block_loads = dims->pool_slots >= kKeysPerTile ? 1 : 0;
      if (!encode_pool_map(&pp.tmap_rows, kv_pool, dims->pool_slots, 64, 1) ||
          (pp.block_loads && (!encode_pool_map(&pp.tmap_block, kv_pool, dims->pool_slots, 64, kKeysPerTile) ||
                              !encode_pool_map(&pp.tmap_rope, kv_pool, dims->pool_slots, 32, kKeysPerTile))))
        return DDT_ERR_LAUNCH;
      pp.q = static_cast<const uint16_t*>(q);
      pp.kv = static_cast<const uint16_t*>(kv_pool);
      pp.slot_idx = slot_idx;
      pp.prefix_len = prefix_len;
      pp.pool_slots = dims->pool_slots;
      pp.slot_stride = dims->slot_stride;
      pp.sparse = sparse ? 1 : 0;
      pp.rows = plan.rows;
      pp.heads = dims->num_heads;
      pp.nodes = dims->num_nodes;
      pp.tree_len = tree_len;
      pp.row_tiles = plan.row_tiles;
      pp.chunk0 = plan.chunk0;
      pp.chunk = plan.chunk;
      pp.max_splits = std::max(plan.splits, plan.groups);
      pp.batch = dims->batch;
      pp.groups = (phases & kPhaseFused) || sparse ? 0 : plan.groups;
      pp.max_prefix_len = dims->max_prefix_len;
      pp.scale_log2 = scale_log2;
      pp.o_part = o_part;
      pp.lse_part = lse_part;
      pp.status = status;
      if (phases & kPhaseFused) {
        FusedParams fp;
        fp.pre = pp;
        fp.tree_parent = tree_parent;
        fp.tree_slot_idx = tree_slot_idx;
        fp.out = out;
        fp.lse = lse;
        fp.arrivals = reinterpret_cast<int32_t*>(ws + plan.cnt_off);
        fp.splits = plan.splits > 0 ? plan.splits : 1;  // an empty prefix still has a (tail-only) unit per tile
        const int64_t units = int64_t(dims->batch) * fp.splits * plan.row_tiles;
        if (units > INT32_MAX) return DDT_ERR_DIMS;
        fp.units = static_cast<int32_t>(units);
        int pairs = fused_pairs(dev);
        if (pairs > fp.units) pairs = fp.units;
        if (launch_fused(fp, pairs, s) != cudaSuccess) return DDT_ERR_LAUNCH;
        return DDT_OK;
      }
      if (launch_prefix(pp, dims->batch, plan.splits, s) != cudaSuccess) return DDT_ERR_LAUNCH;
    }
  }
  if (phases & kPhaseMerge) {
    TailParams tp;
    tp.q = static_cast<const uint16_t*>(q);
    tp.kv = static_cast<const uint16_t*>(kv_pool);
    tp.prefix_len = prefix_len;
    tp.no_tail = sparse ? 1 : 0;
    tp.tree_parent = tree_parent;
    tp.tree_slot_idx = tree_slot_idx;
    tp.pool_slots = dims->pool_slots;
    tp.nodes = dims->num_nodes;
    tp.heads = dims->num_heads;
    tp.tree_len = tree_len;
    tp.heads_per_cta = dims->num_heads < 8 ? dims->num_heads : 8;
    tp.row_tiles = plan.row_tiles;
    tp.chunk0 = plan.chunk0;
    tp.chunk = plan.chunk;
    tp.max_splits = std::max(plan.splits, plan.groups);
    tp.batch = dims->batch;
    tp.groups = sparse ? 0 : plan.groups;
    tp.max_prefix_len = dims->max_prefix_len;
    tp.scale_log2 = scale_log2;
    tp.o_part = o_part;
    tp.lse_part = lse_part;
    tp.out = out;
    tp.lse = lse;
    tp.status = status;
    if (launch_tail_merge(tp, dims->batch, s) != cudaSuccess) return DDT_ERR_LAUNCH;
  }
  return DDT_OK;
}

}  // namespace
}  // namespace ddt

#define DDT_VERIFY_ARGS                                                                                     \
  const void *q, const void *kv_pool, const int32_t *slot_idx, const int32_t *prefix_len,                  \
      const int32_t *tree_parent, const int32_t *tree_slot_idx, float sm_scale, float *out, float *lse,      \
      const ddt_dims *dims, void *workspace, size_t workspace_bytes, ddt_stream_t stream
#define DDT_VERIFY_PASS                                                                                    \
  q, kv_pool, slot_idx, prefix_len, tree_parent, tree_slot_idx, nullptr, sm_scale, out, lse, dims, workspace, \
      workspace_bytes, stream

// Two launches (the prefix pass, then the tail/merge kernel as its programmatic
// dependent) measured faster than the single fused launch on every
// configuration: the merge then runs on every SM, overlapping the end of the
// prefix pass, instead of on the pair that finishes a row tile's last split.
extern "C" int ddtree_verify_attn(DDT_VERIFY_ARGS) {
  return verify_phases(kPhasePrefix | kPhaseMerge, DDT_VERIFY_PASS);
}
extern "C" int ddtree_verify_attn_fused(DDT_VERIFY_ARGS) { return verify_phases(kPhaseFused, DDT_VERIFY_PASS); }
extern "C" int ddtree_verify_attn_ragged(const void* q, const void* kv_pool, const int32_t* slot_idx,
                                         const int32_t* prefix_len, const int32_t* tree_parent,
                                         const int32_t* tree_slot_idx, const int32_t* tree_len, float sm_scale,
                                         float* out, float* lse, const ddt_dims* dims, void* workspace,
                                         size_t workspace_bytes, ddt_stream_t stream) {
  if (!tree_len && dims && dims->batch > 0) return DDT_ERR_NULL;
  return verify_phases(kPhasePrefix | kPhaseMerge, q, kv_pool, slot_idx, prefix_len, tree_parent, tree_slot_idx,
                       tree_len, sm_scale, out, lse, dims, workspace, workspace_bytes, stream);
}
extern "C" int ddtree_verify_prefix_phase(DDT_VERIFY_ARGS) { return verify_phases(kPhasePrefix, DDT_VERIFY_PASS); }

extern "C" size_t ddtree_verify_sparse_workspace_bytes(const ddt_dims* dims) {
  ddt_dims e;
  if (sparse_as_dense(dims, &e) != DDT_OK) return 0;
  return ddtree_verify_workspace_bytes(&e);
}

extern "C" int ddtree_verify_attn_sparse(const void* q, const void* kv_pool, const int32_t* indices, float sm_scale,
                                         float* out, float* lse, const ddt_dims* dims, void* workspace,
                                         size_t workspace_bytes, ddt_stream_t stream) {
  if (!dims) return DDT_ERR_NULL;
  ddt_dims e;
  const int rc = sparse_as_dense(dims, &e);
  if (rc != DDT_OK) return rc;
  return verify_phases(kPhasePrefix | kPhaseMerge, q, kv_pool, indices, nullptr, nullptr, nullptr, nullptr, sm_scale,
                       out, lse, &e, workspace, workspace_bytes, stream, true);
}
extern "C" int ddtree_verify_merge_phase(DDT_VERIFY_ARGS) { return verify_phases(kPhaseMerge, DDT_VERIFY_PASS); }

extern "C" int ddtree_kv_compact(const void* kv_src, void* kv_dst, const int32_t* slot_idx,
                                 const int32_t* prefix_len, const int64_t* dst_start, int32_t* slot_idx_out,
                                 const ddt_dims* dims, void* workspace, ddt_stream_t stream) {
  int rc = check_dims(dims);
  if (rc != DDT_OK) return rc;
  if (dims->batch == 0) return DDT_OK;
  if (!kv_src || !kv_dst || !prefix_len || !dst_start || !workspace ||
      ((!slot_idx || !slot_idx_out) && dims->max_prefix_len > 0))
    return DDT_ERR_NULL;
  if (!aligned(kv_src, 16) || !aligned(kv_dst, 16) || !aligned(workspace, 256) || !aligned(dst_start, 8) ||
      !aligned(slot_idx, 4) || !aligned(slot_idx_out, 4) || !aligned(prefix_len, 4))
    return DDT_ERR_ALIGN;
  DeviceInfo dev;
  if ((rc = device_info(&dev)) != DDT_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t* status = static_cast<int32_t*>(workspace);
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return DDT_ERR_LAUNCH;
  CompactParams cp;
  cp.src = static_cast<const uint16_t*>(kv_src);
  cp.dst = static_cast<uint16_t*>(kv_dst);
  cp.slot_idx = slot_idx;
  cp.prefix_len = prefix_len;
  cp.dst_start = dst_start;
  cp.slot_idx_out = slot_idx_out;
  cp.pool_slots = dims->pool_slots;
  cp.slot_stride = dims->slot_stride;
  cp.max_prefix_len = dims->max_prefix_len;
  cp.status = status;
  if (launch_kv_compact(cp, dims->batch, s) != cudaSuccess) return DDT_ERR_LAUNCH;
  return DDT_OK;
}

extern "C" int ddtree_kv_compact_check(const int32_t* slot_idx, const int32_t* prefix_len, const int64_t* dst_start,
                                       const int32_t* tree_slot_idx, const ddt_dims* dims, int32_t same_pool,
                                       int64_t* bad_slot) {
  int rc = check_dims(dims);
  if (rc != DDT_OK) return rc;
  if (bad_slot) *bad_slot = -1;
  const int B = dims->batch;
  if (B == 0) return DDT_OK;
  if (!prefix_len || !dst_start || (!slot_idx && dims->max_prefix_len > 0)) return DDT_ERR_NULL;
  auto fail = [&](int64_t slot) {
    if (bad_slot) *bad_slot = slot;
    return DDT_ERR_ALIAS;
  };
  // destination ranges: inside the pool and pairwise disjoint
  std::vector<std::pair<int64_t, int64_t>> dst;  // [begin, end)
  dst.reserve(B);
  for (int b = 0; b < B; ++b) {
    const int64_t L = prefix_len[b];
    if (L < 0 || L > dims->max_prefix_len) return DDT_ERR_DIMS;
    if (L == 0) continue;
    const int64_t d0 = dst_start[b];
    if (d0 < 0 || d0 + L > dims->pool_slots) return fail(d0 < 0 ? d0 : d0 + L - 1);
    dst.emplace_back(d0, d0 + L);
  }
  std::sort(dst.begin(), dst.end());
  for (size_t i = 1; i < dst.size(); ++i)
    if (dst[i].first < dst[i - 1].second) return fail(dst[i].first);
  if (!same_pool) return DDT_OK;
  // in place: no destination row may hold a live row that the copy (or a later
  // verify call) still reads, except a row that is already where it goes
  auto dst_hit = [&](int64_t slot) {
    auto it = std::upper_bound(dst.begin(), dst.end(), std::make_pair(slot, INT64_MAX));
    return it != dst.begin() && slot < std::prev(it)->second;
  };
  for (int b = 0; b < B; ++b) {
    const int32_t* row = slot_idx + static_cast<int64_t>(b) * dims->slot_stride;
    for (int32_t j = 0; j < prefix_len[b]; ++j) {
      const int64_t src = row[j];
      if (src == dst_start[b] + j) continue;  // already in place: the copy rewrites it with itself
      if (dst_hit(src)) return fail(src);
    }
    if (tree_slot_idx)
      for (int32_t u = 0; u < dims->num_nodes; ++u) {
        const int64_t t = tree_slot_idx[static_cast<int64_t>(b) * dims->num_nodes + u];
        if (dst_hit(t)) return fail(t);
      }
  }
  return DDT_OK;
}

extern "C" int ddtree_read_device_status(const void* workspace, int32_t* host_status, ddt_stream_t stream) {
  if (!workspace || !host_status) return DDT_ERR_NULL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return DDT_ERR_LAUNCH;
  if (cudaMemcpy(host_status, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DDT_ERR_LAUNCH;
  return DDT_OK;
}

// Host-side introspection of the schedule (not part of the public header; the
// CPU tests use it, no device is needed).
// The plan for these sizes on a device with sm_count SMs: out = {row tiles,
// key splits, keys of each later split, key-range groups (0: splits), keys of
// split 0}.
extern "C" __attribute__((visibility("default"))) int ddtree_internal_plan(const ddt_dims* dims, int sm_count,
                                                                           int32_t* out) {
  Plan plan;
  const int rc = make_plan(dims, sm_count, &plan);
  if (rc != DDT_OK) return rc;
  out[0] = plan.row_tiles;
  out[1] = plan.splits;
  out[2] = plan.chunk;
  out[3] = plan.groups;
  out[4] = plan.chunk0;
  return DDT_OK;
}

// Unit idx of key-range group g for host-side prefix lengths (clamped to
// [0, max_len] like the kernels do): out = {request, kbegin, kend, piece};
// returns 1, or 0 once the group has no more units.  With g < 0 it returns
// instead, in out[0], the number of pieces (split slots) of request idx.
extern "C" __attribute__((visibility("default"))) int ddtree_internal_group_unit(const int32_t* prefix_len, int batch,
                                                                                 int max_len, int groups, int g,
                                                                                 int idx, int32_t* out) {
  std::vector<int64_t> first(batch + 1, 0);
  std::vector<int> len(batch);
  for (int b = 0; b < batch; ++b) {
    const int L = prefix_len[b];
    len[b] = L < 0 ? 0 : (L > max_len ? max_len : L);
    first[b + 1] = first[b] + (len[b] + kKeysPerTile - 1) / kKeysPerTile;
  }
  const int64_t K = first[batch];
  auto off = [&](int r) { return first[r]; };
  auto steps = [&](int r) { return first[r + 1] - first[r]; };
  auto keys = [&](int r) { return len[r]; };
  if (g < 0) {
    out[0] = group_pieces(off(idx), steps(idx), K, groups);
    return 1;
  }
  return nth_group_unit(g, groups, K, batch, idx, off, steps, keys, &out[0], &out[1], &out[2], &out[3]) ? 1 : 0;
}

#ifdef DDT_TEST_HOOKS
// Test builds only (not part of the public header): make the prefix kernel's
// producers skip the loads of one step, so a bounded wait runs out.
int32_t ddt::g_test_drop_step = -1;
extern "C" __attribute__((visibility("default"))) void ddtree_test_set_drop_step(int32_t step) {
  ddt::g_test_drop_step = step;
}
#endif

extern "C" const char* ddtree_status_string(int code) {
  switch (code) {
    case DDT_OK: return "ok";
    case DDT_ERR_NULL: return "a required pointer is NULL";
    case DDT_ERR_DIMS: return "unsupported sizes";
    case DDT_ERR_WORKSPACE: return "workspace too small";
    case DDT_ERR_ALIGN: return "a device pointer is misaligned";
    case DDT_ERR_LAUNCH: return "a kernel launch or CUDA runtime call failed";
    case DDT_ERR_DEVICE: return "the current device is not an sm_103 GPU";
    case DDT_ERR_ALIAS: return "kv_compact destinations overlap each other or a live source row";
    default: return "unknown status";
  }
}
