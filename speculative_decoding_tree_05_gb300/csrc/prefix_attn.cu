// prefix_attn.cu -- split-KV prefix attention on the tcgen05 tensor cores.
//
// Every tree node of a request attends to the whole shared prefix with no mask
// ("The Architecture Detective: Uncovering FlashMLA's Potential for Blackwell
// DDTree Verification", sections "The Message in Full" and "The Discovery:
// FlashMLA's Hidden Capabilities": all q_len tree queries see all L prefix keys,
// causal=False).  So all T*H (node, head) rows of a request form the M dimension
// of one contraction and each gathered latent row is used by all of them.  The
// prefix is cut into key splits whose partial (o, lse) are merged afterwards
// ("The Anatomy of a Kernel Investigation", section "Input Knowledge Required",
// item 4: split-KV with an online-softmax merge).
//
// One CTA = (request b, 128-row tile, v half, key split).  Per 32-key step:
//   gather   32 slot rows (1152 B each) -> smem, cp.async 16 B with zero fill,
//            double-buffered against the compute of the previous step
//   S        = Q . K^T          tcgen05.mma M=128 N=32 K=576, fp32 in TMEM
//   softmax  one thread per row: running max / sum in the log2 domain,
//            P = exp2(s - m) as bf16 into smem, O rescaled in TMEM when m moves
//   O       += P . V_half       tcgen05.mma M=128 N=256 K=32 (V = the first 512
//            dims of the same smem rows, read MN-major)
// Epilogue: o = O / l and lse = ln(sum) for the split, to the workspace.
//
// Shared-memory layouts (all 128-byte-swizzled canonical K-major atoms of
// 8 rows x 128 B unless noted):
//   Q   [9 dim blocks][128 rows][64 dims]        block stride 16384 B
//   K   [9 dim blocks][32 keys][64 dims] x 2     block stride  4096 B
//   P   [128 rows][32 keys], 64-byte swizzle     8 rows x 64 B atoms
// TMEM: O half at columns [0, 256), S at [256, 288).
#include <cuda_runtime.h>
#include <math_constants.h>
#include "kernels.cuh"
#include "ptx.cuh"

namespace ddt {
namespace {

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 0;
constexpr uint32_t kSCol = 256;
constexpr uint32_t kIdescS = idesc_bf16_f32(kTileRows, kKeysPerTile, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(kTileRows, 256, false, true);

__device__ __forceinline__ uint32_t swz128(int row, int chunk) { return row * 128 + ((chunk ^ (row & 7)) << 4); }

// Gather keys [kbase, kbase+32) of request b into a K tile buffer.  Keys past
// kend or with a slot outside the pool are zero-filled (and masked later).
__device__ __forceinline__ void gather_k_tile(const PrefixParams& p, int b, int kbase, int kend, uint32_t kbuf,
                                              int tid) {
  const int32_t* slots = p.slot_idx + static_cast<int64_t>(b) * p.slot_stride;
#pragma unroll 2
  for (int i = tid; i < kKeysPerTile * kChunks; i += kPrefixThreads) {
    int n = i / kChunks, c = i - n * kChunks;
    int key = kbase + n;
    const uint16_t* src = p.kv;
    uint32_t bytes = 0;
    if (key < kend) {
      int32_t slot = __ldg(slots + key);
      if (slot >= 0 && static_cast<int64_t>(slot) < p.pool_slots) {
        src = p.kv + static_cast<int64_t>(slot) * kDqk + c * 8;
        bytes = 16;
      } else if (c == 0) {
        atomicOr(p.status, kStatusBadSlot);
      }
    }
    uint32_t dst = kbuf + (c >> 3) * (kKeysPerTile * 128) + swz128(n, c & 7);
    cp_async16(dst, src, bytes);
  }
}

__global__ void __launch_bounds__(kPrefixThreads, 1) prefix_attn_kernel(PrefixParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_s, bar_o;
  __shared__ uint32_t tmem_base_sh;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int split = blockIdx.x;
  const int row_tile = blockIdx.y >> 1;
  const int half = blockIdx.y & 1;
  const int b = blockIdx.z;

  int L = __ldg(p.prefix_len + b);
  if (L < 0 || L > p.max_prefix_len) {
    if (tid == 0 && split == 0 && blockIdx.y == 0) atomicOr(p.status, kStatusBadPrefix);
    L = L < 0 ? 0 : p.max_prefix_len;
  }
  const int kbegin = split * p.chunk;
  if (kbegin >= L) return;  // this request has fewer splits; the merge reads only ceil(L/chunk)
  const int kend = min(L, kbegin + p.chunk);
  const int ntiles = (kend - kbegin + kKeysPerTile - 1) / kKeysPerTile;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t q_s = smem_u32(smem);
  const uint32_t k_s[2] = {q_s + kQBytes, q_s + kQBytes + kKTileBytes};
  const uint32_t p_s = q_s + kQBytes + 2 * kKTileBytes;
  uint8_t* p_gen = smem + kQBytes + 2 * kKTileBytes;

  if (tid == 0) {
    mbar_init(&bar_s, 1);
    mbar_init(&bar_o, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }

  // Q tile: rows [row_tile*128, +128) of request b, zero rows past T*H.
  {
    const int64_t row0 = static_cast<int64_t>(b) * p.rows + row_tile * kTileRows;
    for (int i = tid; i < kTileRows * kChunks; i += kPrefixThreads) {
      int r = i / kChunks, c = i - r * kChunks;
      bool ok = row_tile * kTileRows + r < p.rows;
      const uint16_t* src = ok ? p.q + (row0 + r) * kDqk + c * 8 : p.q;
      cp_async16(q_s + (c >> 3) * (kTileRows * 128) + swz128(r, c & 7), src, ok ? 16u : 0u);
    }
  }
  gather_k_tile(p, b, kbegin, kend, k_s[0], tid);
  cp_async_commit();

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;

  float m_run = -CUDART_INF_F, l_run = 0.f;
  int failed = 0;
  const int32_t* slots = p.slot_idx + static_cast<int64_t>(b) * p.slot_stride;

  for (int kt = 0; kt < ntiles; ++kt) {
    const int kbase = kbegin + kt * kKeysPerTile;
    const uint32_t kb = k_s[kt & 1];
    if (kt + 1 < ntiles) {
      gather_k_tile(p, b, kbase + kKeysPerTile, kend, k_s[(kt + 1) & 1], tid);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    fence_proxy_async_smem();
    __syncthreads();

    // S = Q . K^T over 576 dims (36 k-steps of 16)
    if (tid == 0) {
      tc_fence_after();
#pragma unroll 4
      for (int ks = 0; ks < kDqk / 16; ++ks) {
        uint64_t ad = smem_desc(q_s + (ks >> 2) * (kTileRows * 128) + (ks & 3) * 32, 16, 1024, kSwizzle128B);
        uint64_t bd = smem_desc(kb + (ks >> 2) * (kKeysPerTile * 128) + (ks & 3) * 32, 16, 1024, kSwizzle128B);
        mma_ss(tmem + kSCol, ad, bd, kIdescS, ks > 0);
      }
      mma_commit(&bar_s);
    }
    // key mask of this step: lane n checks key kbase+n (past the split end or a bad slot)
    uint32_t masked;
    {
      int key = kbase + (tid & 31);
      bool bad = key >= kend;
      if (!bad) {
        int32_t slot = __ldg(slots + key);
        bad = slot < 0 || static_cast<int64_t>(slot) >= p.pool_slots;
      }
      masked = __ballot_sync(0xffffffffu, bad);
    }
    if (!mbar_wait(&bar_s, kt & 1)) failed = 1;
    tc_fence_after();

    float s[32];
    tmem_ld32(tmem + lane_off + kSCol, s);
    float mx = m_run;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      s[j] = ((masked >> j) & 1u) ? -CUDART_INF_F : s[j] * p.scale_log2;
      mx = fmaxf(mx, s[j]);
    }
    const float alpha = (mx == -CUDART_INF_F) ? 1.f : fast_exp2(m_run - mx);
    const float msub = (mx == -CUDART_INF_F) ? 0.f : mx;
    float sum = 0.f;
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float p0 = fast_exp2(s[2 * j] - msub), p1 = fast_exp2(s[2 * j + 1] - msub);
      sum += p0 + p1;
      pk[j] = pack_bf16x2(p0, p1);
    }
    l_run = l_run * alpha + sum;
    m_run = mx;

    // rescale this row of O when the running max moved (O holds earlier steps)
    if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
      for (int c = 0; c < 256; c += 32) {
        float o[32];
        tmem_ld32(tmem + lane_off + kOCol + c, o);
        uint32_t ob[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) ob[j] = __float_as_uint(o[j] * alpha);
        tmem_st32(tmem + lane_off + kOCol + c, ob);
      }
    }
    // P row -> smem, 64-byte swizzle: chunk c of row r at r*64 + (c ^ ((r>>1)&3))*16
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4 v = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      *reinterpret_cast<uint4*>(p_gen + tid * 64 + ((c ^ ((tid >> 1) & 3)) << 4)) = v;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    failed = __syncthreads_or(failed);
    if (failed) break;

    // O += P . V_half (V = dims [256*half, 256*half+256) of the same rows, MN-major)
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < kKeysPerTile / 16; ++ks) {
        uint64_t ad = smem_desc(p_s + ks * 32, 16, 512, kSwizzle64B);
        uint64_t bd = smem_desc(kb + (4 * half) * (kKeysPerTile * 128) + ks * 16 * 128, kKeysPerTile * 128, 1024,
                                kSwizzle128B);
        mma_ss(tmem + kOCol, ad, bd, kIdescPV, (kt > 0 || ks > 0) ? 1u : 0u);
      }
      mma_commit(&bar_o);
    }
    if (!mbar_wait(&bar_o, kt & 1)) failed = 1;
    tc_fence_after();
    failed = __syncthreads_or(failed);
    if (failed) break;
  }

  if (failed) {
    if (tid == 0) atomicOr(p.status, kStatusTimeout);
    cp_async_wait<0>();
  } else {
    // epilogue: o = O / l, lse = (m + log2 l) * ln 2
    const int r = tid;
    const int grow = row_tile * kTileRows + r;
    const int64_t prow = (static_cast<int64_t>(b) * p.max_splits + split) * (p.row_tiles * kTileRows) + grow;
    const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll 1
    for (int c = 0; c < 256; c += 32) {
      float o[32];
      tmem_ld32(tmem + lane_off + kOCol + c, o);
      if (grow < p.rows) {
        float4* dst = reinterpret_cast<float4*>(p.o_part + prow * kDv + half * 256 + c);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          dst[j] = make_float4(o[4 * j] * inv_l, o[4 * j + 1] * inv_l, o[4 * j + 2] * inv_l, o[4 * j + 3] * inv_l);
      }
    }
    if (half == 0 && grow < p.rows)
      p.lse_part[prow] = l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -CUDART_INF_F;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t configure_prefix() {
  return cudaFuncSetAttribute(prefix_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrefixSmem);
}

cudaError_t launch_prefix(const PrefixParams& p, int batch, int splits, cudaStream_t stream) {
  dim3 grid(splits, p.row_tiles * 2, batch);
  prefix_attn_kernel<<<grid, kPrefixThreads, kPrefixSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ddt
