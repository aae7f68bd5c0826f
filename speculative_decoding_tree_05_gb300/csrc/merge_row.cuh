// merge_row.cuh -- one output row: the tree tail (ancestors and self) and the
// log-sum-exp merge of the tail with the prefix key splits.
//
// Among the tree nodes a draft node sees only its ancestors and itself ("The Art
// of Systematic Investigation", section "Input Knowledge Required to Understand
// This Message", item 1); the prefix part arrives as one normalised partial
// (o, lse) per key split, merged through their log-sum-exp ("The Architecture
// Detective: Uncovering FlashMLA's Potential for Blackwell DDTree Verification",
// section "The Message in Full"; "The Anatomy of a Kernel Investigation",
// section "Input Knowledge Required", item 4).
//
// Shared by the tail/merge kernel (one CTA per node, rows staged in shared
// memory) and the fused verify kernel (rows read from the pool), with the same
// arithmetic in the same order, so both give the same bits.
#pragma once
#include <cuda_runtime.h>
#include <math_constants.h>
#include "kernels.cuh"
#include "ptx.cuh"

namespace ddt {

constexpr float kMergeLog2e = 1.4426950408889634f;
constexpr float kMergeLn2 = 0.69314718055994531f;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Node t's visible tree rows: t, its parent, ..., the root, as slots in vis[]
// (at most T).  A link that is not an earlier node (parent[0] != -1 or
// parent[u] not in [0, u)) ends the walk (the node keeps what it has) and sets
// kStatusBadParent; a slot outside the pool leaves that key out and sets
// kStatusBadSlot.  Returns the number of slots; *st gets the status bits.
template <class ParentFn, class SlotFn>
__device__ __forceinline__ int ancestor_slots(int t, int T, int64_t pool_slots, ParentFn parent, SlotFn slot_of,
                                              int* vis, int32_t* st) {
  int n = 0, u = t;
  int32_t bits = 0;
  for (int guard = 0; u >= 0 && guard < T; ++guard) {
    const int32_t slot = slot_of(u);
    if (slot >= 0 && static_cast<int64_t>(slot) < pool_slots)
      vis[n++] = slot;
    else
      bits |= kStatusBadSlot;
    const int pu = parent(u);
    const bool ok = (u == 0) ? (pu == -1) : (pu >= 0 && pu < u);
    if (!ok) {
      bits |= kStatusBadParent;
      break;
    }
    u = pu;
  }
  *st = bits;
  return n;
}

struct MergeRowArgs {
  const uint16_t* q;      // bf16 [rows, 576]
  float scale_log2;       // sm_scale * log2(e)
  const float* o_part;    // fp32 partials [.., splits, pstride rows, 512]
  const float* lse_part;  // fp32 [.., splits, pstride rows], natural log
  int64_t pstride;        // rows between consecutive splits of one request
  float* out;             // fp32 [rows, 512]
  float* lse;             // fp32 [rows], natural log
};

// One warp computes global row `grow`: its tail over the n_vis visible tree
// rows krow(v) (288 32-bit words each: the 576 bf16 dims), then the merge with
// `splits` prefix partials at pbase + s * pstride.  kWaitForPartials: call
// griddepcontrol.wait before the partials are read (the tail/merge kernel runs
// as a programmatic dependent of the prefix pass).
template <bool kWaitForPartials, class KRowFn>
__device__ __forceinline__ void merge_row(const MergeRowArgs& a, int64_t grow, int64_t pbase, int splits, int n_vis,
                                          KRowFn krow, int lane) {
  // q: lane holds dims {64 i + 2 lane, +1}, i = 0..8
  uint32_t qv[9];
  const uint32_t* qrow = reinterpret_cast<const uint32_t*>(a.q + grow * kDqk);
#pragma unroll
  for (int i = 0; i < 9; ++i) qv[i] = __ldg(qrow + 32 * i + lane);

  // tail: online softmax over the visible tree rows, log2 domain
  float m = -CUDART_INF_F, l = 0.f, o[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j] = 0.f;
  for (int v = 0; v < n_vis; ++v) {
    const uint32_t* kr = krow(v);
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      const uint32_t kk = kr[32 * i + lane];
      acc = fmaf(bf16_lo(qv[i]), bf16_lo(kk), acc);
      acc = fmaf(bf16_hi(qv[i]), bf16_hi(kk), acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    const float s = acc * a.scale_log2;
    const float mn = fmaxf(m, s);
    const float alpha = fast_exp2(m - mn);
    const float pv = fast_exp2(s - mn);
    l = l * alpha + pv;
    m = mn;
    // v dims of this lane: 4 lane + 128 j + {0..3}, j = 0..3
    const uint2* vrow = reinterpret_cast<const uint2*>(kr);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint2 w = vrow[lane + 32 * j];
      o[4 * j + 0] = fmaf(o[4 * j + 0], alpha, pv * bf16_lo(w.x));
      o[4 * j + 1] = fmaf(o[4 * j + 1], alpha, pv * bf16_hi(w.x));
      o[4 * j + 2] = fmaf(o[4 * j + 2], alpha, pv * bf16_lo(w.y));
      o[4 * j + 3] = fmaf(o[4 * j + 3], alpha, pv * bf16_hi(w.y));
    }
  }

  // The partials were written by other SMs: read them only now, through L2 (ld.global.cg).
  if (kWaitForPartials) grid_dep_wait();
  // prefix split lse values, one per lane (up to 64 here, the rest in the loops)
  float lse_l[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int s = lane + 32 * k;
    lse_l[k] = s < splits ? __ldcg(a.lse_part + pbase + s * a.pstride) * kMergeLog2e : -CUDART_INF_F;
  }

  // merge: weights 2^(lse_part - max) over the tail and every split
  const float lse2_t = (l > 0.f) ? m + log2f(l) : -CUDART_INF_F;
  float mx = fmaxf(lse_l[0], lse_l[1]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  for (int s = 64; s < splits; ++s) mx = fmaxf(mx, __ldcg(a.lse_part + pbase + s * a.pstride) * kMergeLog2e);
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
        const float4* op = reinterpret_cast<const float4*>(a.o_part + (pbase + (s + u) * a.pstride) * kDv);
#pragma unroll
        for (int j = 0; j < 4; ++j) x[u][j] = __ldcg(op + lane + 32 * j);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int su = s + u;
        float ws = __shfl_sync(0xffffffffu, (su & 32) ? wl1 : wl0, su & 31);
        if (su >= 64) ws = fast_exp2(__ldcg(a.lse_part + pbase + su * a.pstride) * kMergeLog2e - mx);
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
      const float4* op = reinterpret_cast<const float4*>(a.o_part + (pbase + s * a.pstride) * kDv);
      float ws = __shfl_sync(0xffffffffu, (s & 32) ? wl1 : wl0, s & 31);
      if (s >= 64) ws = fast_exp2(__ldcg(a.lse_part + pbase + s * a.pstride) * kMergeLog2e - mx);
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
  float4* dst = reinterpret_cast<float4*>(a.out + grow * kDv);
#pragma unroll
  for (int j = 0; j < 4; ++j)
    dst[lane + 32 * j] = make_float4(acc[4 * j] * inv, acc[4 * j + 1] * inv, acc[4 * j + 2] * inv, acc[4 * j + 3] * inv);
  if (lane == 0) a.lse[grow] = wsum > 0.f ? (mx + log2f(wsum)) * kMergeLn2 : -CUDART_INF_F;
}

// Row of an inactive node (ragged trees): out = 0, lse = -inf.
__device__ __forceinline__ void write_inactive_row(float* out, float* lse, int64_t grow, int lane) {
  float4* dst = reinterpret_cast<float4*>(out + grow * kDv);
#pragma unroll
  for (int j = 0; j < 4; ++j) dst[lane + 32 * j] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (lane == 0) lse[grow] = -CUDART_INF_F;
}

}  // namespace ddt
