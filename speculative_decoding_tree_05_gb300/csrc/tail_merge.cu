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
#include "ptx.cuh"

namespace ddt {
namespace {

constexpr int kTailThreads = 256;
constexpr int kTailWarps = kTailThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

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
      const int64_t grow = (static_cast<int64_t>(b) * T + t) * p.heads + h;
      float4* dst = reinterpret_cast<float4*>(p.out + grow * kDv);
#pragma unroll
      for (int j = 0; j < 4; ++j) dst[lane + 32 * j] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (lane == 0) p.lse[grow] = -CUDART_INF_F;
      return;
    }
  }

  // the request's parent and slot arrays, loaded in parallel, then one walk in smem
  for (int i = tid; i < T; i += kTailThreads) {
    par_sh[i] = __ldg(p.tree_parent + static_cast<int64_t>(b) * T + i);
    tslot_sh[i] = __ldg(p.tree_slot_idx + static_cast<int64_t>(b) * T + i);
  }
  __syncthreads();
  if (tid == 0) {
    int n = 0, u = t;
    int32_t st = 0;
    for (int guard = 0; u >= 0 && guard < T; ++guard) {
      const int32_t slot = tslot_sh[u];
      if (slot >= 0 && static_cast<int64_t>(slot) < p.pool_slots)
        vis_slot_sh[n++] = slot;
      else
        st |= kStatusBadSlot;
      const int pu = par_sh[u];
      const bool ok = (u == 0) ? (pu == -1) : (pu >= 0 && pu < u);
      if (!ok) {
        st |= kStatusBadParent;
        break;
      }
      u = pu;
    }
    n_vis_sh = n;
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

  int L = __ldg(p.prefix_len + b);
  L = L < 0 ? 0 : (L > p.max_prefix_len ? p.max_prefix_len : L);
  const int splits = (L + p.chunk - 1) / p.chunk;
  const int h = blockIdx.y * p.heads_per_cta + warp;
  if (warp >= p.heads_per_cta || h >= p.heads) return;

  const int r = t * p.heads + h;                                   // row within the request
  const int64_t grow = static_cast<int64_t>(b) * T * p.heads + r;  // global row
  const int64_t pstride = static_cast<int64_t>(p.row_tiles) * kTileRows;
  const int64_t pbase = static_cast<int64_t>(b) * p.max_splits * pstride + r;

  // q: lane holds dims {64 i + 2 lane, +1}, i = 0..8
  uint32_t qv[9];
  const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.q + grow * kDqk);
#pragma unroll
  for (int i = 0; i < 9; ++i) qv[i] = __ldg(qrow + 32 * i + lane);

  // tail: online softmax over the visible tree rows, log2 domain
  float m = -CUDART_INF_F, l = 0.f, o[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j] = 0.f;
  for (int v = 0; v < n_vis; ++v) {
    const uint32_t* krow = reinterpret_cast<const uint32_t*>(rows_sh + v * kRowBytes);
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      const uint32_t kk = krow[32 * i + lane];
      acc = fmaf(bf16_lo(qv[i]), bf16_lo(kk), acc);
      acc = fmaf(bf16_hi(qv[i]), bf16_hi(kk), acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    const float s = acc * p.scale_log2;
    const float mn = fmaxf(m, s);
    const float alpha = fast_exp2(m - mn);
    const float pv = fast_exp2(s - mn);
    l = l * alpha + pv;
    m = mn;
    // v dims of this lane: 4 lane + 128 j + {0..3}, j = 0..3
    const uint2* vrow = reinterpret_cast<const uint2*>(rows_sh + v * kRowBytes);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint2 w = vrow[lane + 32 * j];
      o[4 * j + 0] = fmaf(o[4 * j + 0], alpha, pv * bf16_lo(w.x));
      o[4 * j + 1] = fmaf(o[4 * j + 1], alpha, pv * bf16_hi(w.x));
      o[4 * j + 2] = fmaf(o[4 * j + 2], alpha, pv * bf16_lo(w.y));
      o[4 * j + 3] = fmaf(o[4 * j + 3], alpha, pv * bf16_hi(w.y));
    }
  }

  // Everything above is independent of the prefix pass, which may still be
  // running (programmatic dependent launch); the partials are read only now,
  // through L2 (ld.global.cg), since another SM wrote them.
  grid_dep_wait();
  // prefix split lse values, one per lane (up to 64 here, the rest in the loops)
  float lse_l[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int s = lane + 32 * k;
    lse_l[k] = s < splits ? __ldcg(p.lse_part + pbase + s * pstride) * kLog2e : -CUDART_INF_F;
  }

  // merge: weights 2^(lse_part - max) over the tail and every split
  const float lse2_t = (l > 0.f) ? m + log2f(l) : -CUDART_INF_F;
  float mx = fmaxf(lse_l[0], lse_l[1]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  for (int s = 64; s < splits; ++s) mx = fmaxf(mx, __ldcg(p.lse_part + pbase + s * pstride) * kLog2e);
  mx = fmaxf(mx, lse2_t);

  float acc[16];
  float wsum = 0.f;
  if (mx == -CUDART_INF_F) {
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.f;
  } else {
    const float wt = (l > 0.f) ? fast_exp2(lse2_t - mx) : 0.f;
    const float wt_l = (l > 0.f) ? wt / l : 0.f;
    wsum = wt;
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = o[j] * wt_l;
    const float wl0 = fast_exp2(lse_l[0] - mx), wl1 = fast_exp2(lse_l[1] - mx);
    int s = 0;
    // four splits per round so their loads are in flight together
    for (; s + 4 <= splits; s += 4) {
      float4 x[4][4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4* op = reinterpret_cast<const float4*>(p.o_part + (pbase + (s + u) * pstride) * kDv);
#pragma unroll
        for (int j = 0; j < 4; ++j) x[u][j] = __ldcg(op + lane + 32 * j);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int su = s + u;
        float ws = __shfl_sync(0xffffffffu, (su & 32) ? wl1 : wl0, su & 31);
        if (su >= 64) ws = fast_exp2(__ldcg(p.lse_part + pbase + su * pstride) * kLog2e - mx);
        wsum += ws;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[4 * j + 0] = fmaf(ws, x[u][j].x, acc[4 * j + 0]);
          acc[4 * j + 1] = fmaf(ws, x[u][j].y, acc[4 * j + 1]);
          acc[4 * j + 2] = fmaf(ws, x[u][j].z, acc[4 * j + 2]);
          acc[4 * j + 3] = fmaf(ws, x[u][j].w, acc[4 * j + 3]);
        }
      }
    }
    for (; s < splits; ++s) {
      const float4* op = reinterpret_cast<const float4*>(p.o_part + (pbase + s * pstride) * kDv);
      float ws = __shfl_sync(0xffffffffu, (s & 32) ? wl1 : wl0, s & 31);
      if (s >= 64) ws = fast_exp2(__ldcg(p.lse_part + pbase + s * pstride) * kLog2e - mx);
      wsum += ws;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 x = __ldcg(op + lane + 32 * j);
        acc[4 * j + 0] = fmaf(ws, x.x, acc[4 * j + 0]);
        acc[4 * j + 1] = fmaf(ws, x.y, acc[4 * j + 1]);
        acc[4 * j + 2] = fmaf(ws, x.z, acc[4 * j + 2]);
        acc[4 * j + 3] = fmaf(ws, x.w, acc[4 * j + 3]);
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  float4* dst = reinterpret_cast<float4*>(p.out + grow * kDv);
#pragma unroll
  for (int j = 0; j < 4; ++j)
    dst[lane + 32 * j] = make_float4(acc[4 * j] * inv, acc[4 * j + 1] * inv, acc[4 * j + 2] * inv, acc[4 * j + 3] * inv);
  if (lane == 0) p.lse[grow] = wsum > 0.f ? (mx + log2f(wsum)) * kLn2 : -CUDART_INF_F;
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
