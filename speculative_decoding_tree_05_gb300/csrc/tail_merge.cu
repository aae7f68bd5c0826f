// tail_merge.cu -- tree-tail attention under the ancestor mask, then the
// log-sum-exp merge of every partial result of a row.
//
// Among the tree nodes a draft node sees only its ancestors and itself ("The Art
// of Systematic Investigation", section "Input Knowledge Required to Understand
// This Message", item 1).  That part is tiny (at most T keys per row), so it runs
// on the CUDA cores next to the merge instead of in the tensor-core pass
// ("The Architecture Detective: Uncovering FlashMLA's Potential for Blackwell
// DDTree Verification", section "The Message in Full": a small custom kernel for
// the masked tree tail, merged with the prefix result through the softmax
// state; "The Anatomy of a Kernel Investigation", section "The Reasoning
// Process: A Deep Dive", phase 2).
//
// One CTA = (request b, node t, group of up to 8 heads).  The CTA loads the
// request's parent and slot arrays into shared memory, thread 0 walks the
// parent chain of t there (validating each link), the CTA stages the visible
// tree rows in shared memory, then each warp takes one head row:
//   tail:  s_u = scale * q.k_u for the visible u, online softmax, o_t = sum p_u v_u
//   merge: lse = log2-sum-exp over {tail, prefix splits}, out = weighted sum of
//          the normalised partial outputs; lse is reported in natural log.
// Launched as a programmatic dependent of the prefix pass: everything before
// the merge step runs while the prefix pass finishes.
#include <cuda_runtime.h>
#include <math_constants.h>
#include "kernels.cuh"
#include "merge_row.cuh"
#include "ptx.cuh"
#include "schedule.cuh"

namespace ddt {
namespace {

constexpr int kTailThreads = 256;

__global__ void __launch_bounds__(kTailThreads) tail_merge_kernel(TailParams p) {
  extern __shared__ __align__(16) uint8_t rows_sh[];  // visible tree rows, 1152 B each
  __shared__ int par_sh[kMaxNodes];
  __shared__ int tslot_sh[kMaxNodes];
  __shared__ int vis_slot_sh[kMaxNodes];
  __shared__ int n_vis_sh;

  const int t = blockIdx.x;
  const int b = blockIdx.z;
  const int T = p.nodes;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // ragged trees: nodes t >= tree_len[b] are inactive (out = 0, lse = -inf);
  // their parent and slot entries are never read
  if (p.tree_len != nullptr) {
    int tl = __ldg(p.tree_len + b);
    if (tl < 0 || tl > T) {
      if (t == 0 && blockIdx.y == 0 && tid == 0) atomicOr(p.status, kStatusBadTreeLen);
      tl = tl < 0 ? 0 : T;
    }
    if (t >= tl) {
      const int h = blockIdx.y * p.heads_per_cta + warp;
      if (warp >= p.heads_per_cta || h >= p.heads) return;
      write_inactive_row(p.out, p.lse, (static_cast<int64_t>(b) * T + t) * p.heads + h, lane);
      return;
    }
  }

  // the request's parent and slot arrays, loaded in parallel, then one walk in smem
  for (int i = tid; i < T && !p.no_tail; i += kTailThreads) {
    par_sh[i] = __ldg(p.tree_parent + static_cast<int64_t>(b) * T + i);
    tslot_sh[i] = __ldg(p.tree_slot_idx + static_cast<int64_t>(b) * T + i);
  }
  __syncthreads();
  if (tid == 0 && p.no_tail) n_vis_sh = 0;
  if (tid == 0 && !p.no_tail) {
    int32_t st = 0;
    n_vis_sh = ancestor_slots(t, T, p.pool_slots, [&](int u) { return par_sh[u]; }, [&](int u) { return tslot_sh[u]; },
                              vis_slot_sh, &st);
    if (st && blockIdx.y == 0) atomicOr(p.status, st);
  }
  __syncthreads();
  const int n_vis = n_vis_sh;
  for (int i = tid; i < n_vis * kChunks; i += kTailThreads) {
    const int v = i / kChunks, c = i - v * kChunks;
    const uint4* src = reinterpret_cast<const uint4*>(p.kv + static_cast<int64_t>(vis_slot_sh[v]) * kDqk) + c;
    reinterpret_cast<uint4*>(rows_sh + v * kRowBytes)[c] = __ldg(src);
  }
  __syncthreads();

  // the prefix partials of request b: its key splits, or with key-range groups
  // the groups its steps span (pieces 0.. in the request's split slots)
  int splits;
  if (p.groups > 0) {
    const StepTable st = step_table(p.prefix_len, p.max_prefix_len, p.batch, lane);
    splits = group_pieces(st.off(b), st.steps(b), st.total, p.groups);
  } else {
    int L = p.prefix_len != nullptr ? __ldg(p.prefix_len + b) : p.max_prefix_len;
    L = L < 0 ? 0 : (L > p.max_prefix_len ? p.max_prefix_len : L);
    splits = split_count(L, p.chunk0, p.chunk);
  }
  const int h = blockIdx.y * p.heads_per_cta + warp;
  if (warp >= p.heads_per_cta || h >= p.heads) return;

  const int r = t * p.heads + h;                                   // row within the request
  const int64_t grow = static_cast<int64_t>(b) * T * p.heads + r;  // global row
  const int64_t pstride = static_cast<int64_t>(p.row_tiles) * kTileRows;
  const MergeRowArgs a{p.q, p.scale_log2, p.o_part, p.lse_part, pstride, p.out, p.lse};
  // everything before the merge is independent of the prefix pass, which may
  // still be running (programmatic dependent launch)
  merge_row<true>(a, grow, static_cast<int64_t>(b) * p.max_splits * pstride + r, splits, n_vis,
                  [&](int v) { return reinterpret_cast<const uint32_t*>(rows_sh + v * kRowBytes); }, lane);
}

}  // namespace

cudaError_t configure_tail_merge() {
  return cudaFuncSetAttribute(tail_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxNodes * kRowBytes);
}

cudaError_t launch_tail_merge(const TailParams& p, int batch, cudaStream_t stream) {
  const int smem = p.nodes * kRowBytes;
  // programmatic dependent launch: the prologue and tree tail overlap the end of the prefix pass
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(p.nodes, (p.heads + p.heads_per_cta - 1) / p.heads_per_cta, batch);
  cfg.blockDim = dim3(kTailThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tail_merge_kernel, p);
}

}  // namespace ddt
