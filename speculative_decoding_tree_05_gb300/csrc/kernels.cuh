// kernels.cuh -- launch parameters shared by the host launcher and the kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace ddt {

constexpr int kDqk = 576;       // q/k width: 512 latent + 64 rope
constexpr int kDv = 512;        // v width: latent part of the same row
constexpr int kRowBytes = kDqk * 2;
constexpr int kChunks = kRowBytes / 16;   // 72 x 16-byte chunks per latent row
constexpr int kMaxNodes = 128;

constexpr int32_t kStatusBadSlot = 1;
constexpr int32_t kStatusBadParent = 2;
constexpr int32_t kStatusBadPrefix = 4;
constexpr int32_t kStatusTimeout = 8;
constexpr int32_t kStatusBadTreeLen = 16;

// Split-KV prefix pass: one CTA pair per (request, 128-row tile, key split).
struct PrefixParams {
  CUtensorMap tmap_rows;     // kv_pool as [N rows][576 cols] bf16, box 64 cols x 1 row, 128-byte swizzle
  CUtensorMap tmap_block;    // same tensor, box 64 cols x 64 rows, 128-byte swizzle
  CUtensorMap tmap_rope;     // same tensor, box 32 cols x 64 rows, 64-byte swizzle
  const uint16_t* q;         // bf16 [B, T, H, 576]
  const uint16_t* kv;        // bf16 [N, 576]
  const int32_t* slot_idx;   // [B, slot_stride]
  const int32_t* prefix_len; // [B], or null: every request has max_prefix_len keys
  int64_t pool_slots;
  int32_t slot_stride;
  int32_t sparse;            // slot tables are index lists: -1 entries are "no key" (no status bit)
  int32_t rows;              // T * H rows per request (the row stride of q)
  int32_t heads;             // H
  int32_t nodes;             // T
  const int32_t* tree_len;   // [B] active nodes per request, or null: all T active
  int32_t row_tiles;         // ceil(rows / 128)
  int32_t chunk0;            // keys of split 0 (groups == 0; see split_begin)
  int32_t chunk;             // keys of every later split
  int32_t max_splits;        // split slots per request in the workspace
  int32_t batch;             // B
  int32_t groups;            // > 0: key-range groups (schedule.cuh; batch <= 64), grid (2 row_tiles, groups)
  int32_t max_prefix_len;
  float scale_log2;          // sm_scale * log2(e)
  int32_t block_loads;       // tmap_block and tmap_rope are valid (pool has >= 64 rows)
  float* o_part;             // fp32 [B, max_splits, row_tiles*128, 512]
  float* lse_part;           // fp32 [B, max_splits, row_tiles*128], natural log
  int32_t* status;           // status word; test builds count lazy O rescales in status[1], 20-bit reruns in status[2]
#ifdef DDT_TEST_HOOKS
  int32_t test_drop_step;    // test builds: producers load nothing for this step of every unit (-1: none)
#endif
};

// Tree tail + merge: one CTA per (request, node, head group).
struct TailParams {
  const uint16_t* q;
  const uint16_t* kv;
  const int32_t* prefix_len;    // [B], or null: every request has max_prefix_len keys
  int32_t no_tail;              // no tree part: the rows are merged from the prefix partials alone
  const int32_t* tree_parent;   // [B, T]
  const int32_t* tree_slot_idx; // [B, T]
  int64_t pool_slots;
  int32_t nodes;                // T
  int32_t heads;                // H
  const int32_t* tree_len;      // [B] active nodes per request, or null: all T active
  int32_t heads_per_cta;
  int32_t row_tiles;
  int32_t chunk0;               // keys of split 0 (groups == 0)
  int32_t chunk;                // keys of every later split
  int32_t max_splits;
  int32_t batch;                // B
  int32_t groups;               // > 0: the prefix pass ran key-range groups: request b has its pieces' partials
  int32_t max_prefix_len;
  float scale_log2;
  const float* o_part;
  const float* lse_part;
  float* out;                   // fp32 [B, T, H, 512]
  float* lse;                   // fp32 [B, T, H]
  int32_t* status;
};

// Fused verify: one persistent launch of CTA pairs that loop over the units
// (request, key split, 128-row tile) of the prefix pass; the pair completing the
// last split of a (request, row tile) merges that tile (tree tail + log-sum-exp).
struct FusedParams {
  PrefixParams pre;             // the prefix pass of every unit (o_part, lse_part, status inside)
  const int32_t* tree_parent;   // [B, T]
  const int32_t* tree_slot_idx; // [B, T]
  float* out;                   // fp32 [B, T, H, 512]
  float* lse;                   // fp32 [B, T, H]
  int32_t* arrivals;            // [B, row_tiles] splits finished per (request, row tile); zero at launch
  int32_t units;                // B * splits * row_tiles
  int32_t splits;               // key-split slots per request (>= 1)
};

struct CompactParams {
  const uint16_t* src;
  uint16_t* dst;
  const int32_t* slot_idx;
  const int32_t* prefix_len;
  const int64_t* dst_start;
  int32_t* slot_idx_out;
  int64_t pool_slots;
  int32_t slot_stride;
  int32_t max_prefix_len;
  int32_t* status;
};

// Prefix kernel geometry: a pair of CTAs per 128-row tile, 64 keys per step.
constexpr int kTileRows = 128;            // query rows per CTA pair (tcgen05 M)
constexpr int kKeysPerTile = 64;          // keys per pipeline step
constexpr int kMinChunk = 256;            // shortest key split the planner makes
constexpr int kUnitOverheadSteps = 6;     // fixed cost of one prefix unit, in 64-key steps (measured)
constexpr int kMaxGroupBatch = 64;        // key-range groups take batches up to this size (one warp's table)

// Fixed-length key splits of a request's prefix: split 0 holds keys
// [0, chunk0), split s >= 1 keys [chunk0 + (s-1) chunk, +chunk), the last one
// cut at the request's length L.  (chunk0 == chunk: equal splits; a longer
// first split lets the row tiles' first units run on most pairs while the
// remaining pairs work through the short splits.)
__host__ __device__ inline int split_begin(int s, int chunk0, int chunk) {
  return s == 0 ? 0 : chunk0 + (s - 1) * chunk;
}
__host__ __device__ inline int split_end(int s, int chunk0, int chunk, int L) {
  const int64_t e = s == 0 ? chunk0 : chunk0 + int64_t(s) * chunk;
  return e < L ? static_cast<int>(e) : L;
}
// number of splits that hold keys of a request with L keys
__host__ __device__ inline int split_count(int L, int chunk0, int chunk) {
  return L <= 0 ? 0 : (L <= chunk0 ? 1 : 1 + (L - chunk0 + chunk - 1) / chunk);
}

// Per-device set-up (shared-memory opt-in), called once per device before launches.
cudaError_t configure_prefix();
cudaError_t configure_tail_merge();

// grid (2 row_tiles, splits, batch), or (2 row_tiles, groups) when p.groups > 0
cudaError_t launch_prefix(const PrefixParams& p, int batch, int splits, cudaStream_t stream);
// pairs: CTA pairs of the persistent grid (at most the clusters that fit at once)
cudaError_t launch_fused(const FusedParams& p, int pairs, cudaStream_t stream);
int fused_max_pairs();  // co-resident CTA pairs of the fused kernel on the current device (0: unknown)
cudaError_t launch_tail_merge(const TailParams& p, int batch, cudaStream_t stream);
cudaError_t launch_kv_compact(const CompactParams& p, int batch, cudaStream_t stream);

#ifdef DDT_TEST_HOOKS
// Test builds: the step whose stage loads the producers skip (-1: none), set by
// ddtree_test_set_drop_step and copied into every prefix launch.
extern int32_t g_test_drop_step;
#endif

}  // namespace ddt
