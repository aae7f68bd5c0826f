// prefix_pair.cu -- split-KV prefix attention on a CTA pair (cluster of 2).
//
// All T*H (node, head) rows of a request attend to every prefix key with no
// mask ("The Architecture Detective: Uncovering FlashMLA's Potential for
// Blackwell DDTree Verification", sections "The Message in Full" and "The
// Discovery: FlashMLA's Hidden Capabilities"), so a 128-row tile of those rows
// is the M side of one tensor-core contraction against gathered latent rows;
// the key range is split and the splits merged later by their log-sum-exp
// ("The Anatomy of a Kernel Investigation", section "Input Knowledge Required",
// item 4).
//
// Why a pair: a 128-row fp32 accumulator of the 512-wide V output fills all
// 512 TMEM columns of an SM, leaving none for scores.  So the two CTAs of a
// cluster share one 128-row tile and split the dimensions:
//   CTA r owns latent dims [256r, 256r+256) and rope dims [512+32r, 512+32r+32)
//   (288 of the 576 q.k dims) and the v dims [256r, 256r+256).
// Each CTA computes a partial score S_r = Q_r . K_r^T over its 288 dims,
// the pair swaps partials through distributed shared memory (st.async into the
// peer's buffer, completion counted on the peer's mbarrier), both add them in
// the same order (so both hold bit-identical scores and make identical softmax
// decisions), and each accumulates O_r += P . V_r for its own 256 v dims.
// Every gathered row is read once per pair and every MMA is useful work.
//
// Per CTA (256 threads):
//   warp 0      TMEM allocation; lane 0 issues every tcgen05.mma
//   warps 1-3   producers: gather the CTA's 576-byte half of 32 slot rows per
//               step with 16-byte cp.async (swizzled on the fly) into an
//               8-stage ring; the step's 32 slot indices are fetched one step
//               ahead and passed between lanes by shuffle; each producer thread
//               signals the stage with cp.async.mbarrier.arrive.noinc, so no
//               producer ever waits for its own copies; rows of keys past the
//               split end or outside the pool are zero-filled
//   warps 4-7   softmax: one query row per thread (= its TMEM lane); Q_r is
//               staged into TMEM first; online softmax in the log2 domain with
//               lazy rescaling (O is rescaled only when the running max grows
//               by more than 2^8); P (bf16) is written back over its S buffer
//               and consumed from TMEM by the P.V MMA; epilogue o = O/l.
// TMEM columns: O_r [0,256), S buffers 3 x 32 at [256,352), Q_r [352,496).
// Shared memory per stage: 4 latent blocks [32 keys][64 dims] (128-byte
// swizzle, 4096 B each) + 1 rope block [32 keys][32 dims] (64-byte swizzle).
// The latent blocks are the K operand of S (K-major) and, read MN-major, the
// V operand of P.V.
#include <cuda_runtime.h>
#include <math_constants.h>
#include "kernels.cuh"
#include "ptx.cuh"

namespace ddt {
namespace {

constexpr int kThreads = 256;
constexpr int kNk = 32;                                  // keys per step
constexpr int kStages = 8;
constexpr int kLatBlock = kNk * 128;                     // 4096
constexpr int kStageBytes = 4 * kLatBlock + kNk * 64;    // 18432
constexpr int kProducers = 96;
constexpr int kXBytes = kTileRows * kNk * 4;             // 16384: one fp32 partial-score tile
constexpr int kXBufs = 4;                                // exchange buffers (tile t uses t % 4)
constexpr int kSmem = kStages * kStageBytes + kXBufs * kXBytes + 1024;
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 352, kTmemCols = 512;
constexpr uint32_t kIdescS = idesc_bf16_f32(kTileRows, kNk, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(kTileRows, 256, false, true);
constexpr float kRescaleThreshold = 8.f;                 // log2 units
constexpr float kLn2 = 0.69314718055994531f;

struct Shared {
  uint64_t k_full[kStages];   // producers -> MMA: stage loaded
  uint64_t k_empty[kStages];  // MMA -> producers: stage consumed (after P.V)
  uint64_t s_full[3];         // MMA -> softmax: partial scores in TMEM
  uint64_t p_ready[3];        // softmax -> MMA: P in TMEM, O rescaled
  uint64_t x_full[kXBufs];    // peer -> softmax: peer's partial scores of tile t arrived (buffer t % 4)
  uint64_t pv_done[3];        // MMA -> softmax: P.V of step i completes phase i/3 of pv_done[i%3]
  uint64_t q_ready;           // softmax -> MMA: Q_r staged in TMEM
  uint32_t tmem_base;
  int abort;
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    prefix_pair_kernel(const __grid_constant__ PrefixParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared sh;
  volatile int* abort = &sh.abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int split = blockIdx.x >> 1;
  const int row_tile = blockIdx.y;
  const int b = blockIdx.z;

  int L = __ldg(p.prefix_len + b);
  if (L < 0 || L > p.max_prefix_len) {
    if (tid == 0 && rank == 0 && split == 0 && row_tile == 0) atomicOr(p.status, kStatusBadPrefix);
    L = L < 0 ? 0 : p.max_prefix_len;
  }
  const int kbegin = split * p.chunk;
  if (kbegin >= L) return;  // both CTAs of the pair leave together
  const int kend = min(L, kbegin + p.chunk);
  const int ntiles = (kend - kbegin + kNk - 1) / kNk;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t stage0 = smem_u32(smem);
  uint8_t* xbuf = smem + kStages * kStageBytes;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sh.k_full[i], kProducers);
      mbar_init(&sh.k_empty[i], 1);
    }
    for (int i = 0; i < 3; ++i) {
      mbar_init(&sh.s_full[i], 1);
      mbar_init(&sh.p_ready[i], 128);
    }
    for (int i = 0; i < kXBufs; ++i) mbar_init(&sh.x_full[i], 1);
    for (int i = 0; i < 3; ++i) mbar_init(&sh.pv_done[i], 1);
    mbar_init(&sh.q_ready, 128);
    sh.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&sh.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      if (!mbar_wait_abortable(&sh.q_ready, 0, abort)) ok = false;
      tc_fence_after();
      for (int j = 0; ok && j < ntiles + 2; ++j) {
        if (j < ntiles) {
          const int st = j % kStages;
          if (!mbar_wait_abortable(&sh.k_full[st], (j / kStages) & 1, abort)) { ok = false; break; }
          // the stage was written by cp.async (generic proxy): order it before the
          // tensor core's async-proxy reads
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t base = stage0 + st * kStageBytes;
          const uint32_t sb = tmem + kColS + (j % 3) * kNk;
#pragma unroll
          for (int ks = 0; ks < 16; ++ks) {
            uint64_t bd = smem_desc(base + (ks >> 2) * kLatBlock + (ks & 3) * 32, 16, 1024, kSwizzle128B);
            mma_ts(sb, tmem + kColQ + ks * 8, bd, kIdescS, ks > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int ks = 0; ks < 2; ++ks) {
            uint64_t bd = smem_desc(base + 4 * kLatBlock + ks * 32, 16, 512, kSwizzle64B);
            mma_ts(sb, tmem + kColQ + (16 + ks) * 8, bd, kIdescS, 1u);
          }
          mma_commit(&sh.s_full[j % 3]);
        }
        const int i = j - 2;
        if (i >= 0) {
          if (!mbar_wait_abortable(&sh.p_ready[i % 3], (i / 3) & 1, abort)) { ok = false; break; }
          tc_fence_after();
          const uint32_t base = stage0 + (i % kStages) * kStageBytes;
          const uint32_t pb = tmem + kColS + (i % 3) * kNk;
#pragma unroll
          for (int ks = 0; ks < kNk / 16; ++ks) {
            uint64_t bd = smem_desc(base + ks * 16 * 128, kLatBlock, 1024, kSwizzle128B);
            mma_ts(tmem + kColO, pb + ks * 8, bd, kIdescPV, (i > 0 || ks > 0) ? 1u : 0u);
          }
          mma_commit(&sh.k_empty[i % kStages]);
          mma_commit(&sh.pv_done[i % 3]);
        }
      }
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------------------------ producers
    const int ptid = tid - 32;
    const int32_t* slots = p.slot_idx + static_cast<int64_t>(b) * p.slot_stride;
    const uint16_t* kv = p.kv;
    // lane l holds the slot of key l of a step (fetched one step ahead)
    auto fetch = [&](int j) -> int {
      const int key = kbegin + j * kNk + lane;
      return key < kend ? __ldg(slots + key) : -1;
    };
    int slot_cur = fetch(0);
    for (int j = 0; j < ntiles; ++j) {
      const int slot_next = (j + 1 < ntiles) ? fetch(j + 1) : -1;
      const int st = j % kStages;
      // warp-uniform wait: the lane shuffles below need every lane
      const bool waited = j < kStages || mbar_wait_abortable(&sh.k_empty[st], ((j / kStages) - 1) & 1, abort);
      if (!__all_sync(0xffffffffu, waited)) {
        ok = false;
        break;
      }
      const int kbase = kbegin + j * kNk;
      if (warp == 1 && rank == 0) {
        const bool bad = kbase + lane < kend && (slot_cur < 0 || static_cast<int64_t>(slot_cur) >= p.pool_slots);
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.status, kStatusBadSlot);
      }
      const uint32_t base = stage0 + st * kStageBytes;
#pragma unroll
      for (int k = 0; k < kNk * 36 / kProducers; ++k) {
        const int i = ptid + k * kProducers;
        const int n = i / 36, c = i - n * 36;
        const int slot = __shfl_sync(0xffffffffu, slot_cur, n);
        const bool valid = slot >= 0 && static_cast<int64_t>(slot) < p.pool_slots;
        const int off = (c < 32) ? 256 * static_cast<int>(rank) + 8 * c : 512 + 32 * static_cast<int>(rank) + 8 * (c - 32);
        const uint16_t* src = valid ? kv + static_cast<int64_t>(slot) * kDqk + off : kv;
        const uint32_t dst = (c < 32) ? base + (c >> 3) * kLatBlock + n * 128 + (((c & 7) ^ (n & 7)) << 4)
                                      : base + 4 * kLatBlock + n * 64 + (((c - 32) ^ ((n >> 1) & 3)) << 4);
        cp_async16(dst, src, valid ? 16u : 0u);
      }
      cp_async_arrive_noinc(&sh.k_full[st]);
      slot_cur = slot_next;
    }
    cp_async_wait<0>();
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    const int r = tid - 128;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int grow = row_tile * kTileRows + r;
    const bool row_valid = grow < p.rows;

    // Q_r -> TMEM: latent dims [256 rank, +256) then rope dims [512 + 32 rank, +32)
    {
      const uint4* qsrc = reinterpret_cast<const uint4*>(p.q + (static_cast<int64_t>(b) * p.rows + grow) * kDqk);
      const uint4 zero = make_uint4(0, 0, 0, 0);
#pragma unroll 1
      for (int c0 = 0; c0 < 32; c0 += 8) {
        uint32_t v[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 x = row_valid ? __ldg(qsrc + 32 * rank + c0 + c) : zero;
          v[4 * c] = x.x, v[4 * c + 1] = x.y, v[4 * c + 2] = x.z, v[4 * c + 3] = x.w;
        }
        tmem_st32(tmem + lane_off + kColQ + c0 * 4, v);
      }
      uint32_t v[16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 x = row_valid ? __ldg(qsrc + 64 + 4 * rank + c) : zero;
        v[4 * c] = x.x, v[4 * c + 1] = x.y, v[4 * c + 2] = x.z, v[4 * c + 3] = x.w;
      }
      tmem_st16(tmem + lane_off + kColQ + 128, v);
      tc_fence_before();
      mbar_arrive(&sh.q_ready);
    }

    const uint32_t peer = rank ^ 1u;
    uint32_t x_remote[kXBufs], xbar_remote[kXBufs];
#pragma unroll
    for (int i = 0; i < kXBufs; ++i) {
      x_remote[i] = mapa_shared(smem_u32(xbuf + i * kXBytes), peer);
      xbar_remote[i] = mapa_shared(smem_u32(&sh.x_full[i]), peer);
    }
    const int32_t* slots = p.slot_idx + static_cast<int64_t>(b) * p.slot_stride;
    const uint32_t rsw = static_cast<uint32_t>(r & 7);
    float m_used = -CUDART_INF_F, l = 0.f;
    auto fetch_slot = [&](int j) -> int {
      const int key = kbegin + j * kNk + lane;
      return key < kend ? __ldg(slots + key) : 0;
    };
    int slot_pf[2] = {fetch_slot(0), fetch_slot(1)};

    // Score exchange, software-pipelined by one step: the partial scores of
    // step j+1 are loaded from TMEM and sent to the peer before step j is
    // finished, so the DSMEM transfer overlaps the softmax of step j.  Step t
    // uses exchange buffer t % 4; the peer writes step t only after it has
    // received our step t-2, which we send after finishing step t-4, the last
    // reader of that buffer.
    float own[32], own_next[32];
    auto load_and_send = [&](int t, float (&dst)[32]) -> bool {
      if (r == 0) mbar_arrive_expect_tx(&sh.x_full[t % kXBufs], kXBytes);
      if (!__all_sync(0xffffffffu, mbar_wait_abortable(&sh.s_full[t % 3], (t / 3) & 1, abort))) return false;
      tc_fence_after();
      tmem_ld32(tmem + lane_off + kColS + (t % 3) * kNk, dst);
      const uint32_t xr = x_remote[t % kXBufs] + r * 128, br = xbar_remote[t % kXBufs];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = make_uint4(__float_as_uint(dst[4 * c]), __float_as_uint(dst[4 * c + 1]),
                                   __float_as_uint(dst[4 * c + 2]), __float_as_uint(dst[4 * c + 3]));
        st_async_v4(xr + ((c ^ rsw) << 4), v, br);
      }
      return true;
    };
    if (!load_and_send(0, own)) ok = false;

    for (int j = 0; ok && j < ntiles; ++j) {
      const int sb = j % 3;
      const int kbase = kbegin + j * kNk;
      if (j + 1 < ntiles && !load_and_send(j + 1, own_next)) { ok = false; break; }
      // key mask of this step (past the split end or a slot outside the pool); the
      // slot of this lane's key was fetched two steps ago
      const int slot_j = slot_pf[0];
      slot_pf[0] = slot_pf[1];
      slot_pf[1] = fetch_slot(j + 2);
      const uint32_t masked = __ballot_sync(
          0xffffffffu, kbase + lane >= kend || slot_j < 0 || static_cast<int64_t>(slot_j) >= p.pool_slots);
      if (!__all_sync(0xffffffffu, mbar_wait_abortable(&sh.x_full[j % kXBufs], (j / kXBufs) & 1, abort, true))) {
        ok = false;
        break;
      }
      const uint8_t* xb = xbuf + (j % kXBufs) * kXBytes + r * 128;
      float sc[32];
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float4 v = *reinterpret_cast<const float4*>(xb + ((c ^ rsw) << 4));
        const float pv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int k = 4 * c + e;
          const float x = (own[k] + pv[e]) * p.scale_log2;
          sc[k] = ((masked >> k) & 1u) ? -CUDART_INF_F : x;
          mx = fmaxf(mx, sc[k]);
        }
      }
      const bool need = mx > m_used + kRescaleThreshold;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mx : m_used;
        const float alpha = need ? fast_exp2(m_used - m_new) : 1.f;
        if (j > 0) {
          // O must hold every earlier step: wait for P.V of step j-1 (MMAs complete in order)
          if (!__all_sync(0xffffffffu, mbar_wait_abortable(&sh.pv_done[(j - 1) % 3], ((j - 1) / 3) & 1, abort))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 256; c += 32) {
            float o[32];
            tmem_ld32(tmem + lane_off + kColO + c, o);
            uint32_t ob[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) ob[e] = __float_as_uint(o[e] * alpha);
            tmem_st32(tmem + lane_off + kColO + c, ob);
          }
        }
        l *= alpha;
        m_used = m_new;
      }
      const float msub = (m_used == -CUDART_INF_F) ? 0.f : m_used;
      float sum = 0.f;
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float p0 = fast_exp2(sc[2 * e] - msub), p1 = fast_exp2(sc[2 * e + 1] - msub);
        sum += p0 + p1;
        pk[e] = pack_bf16x2(p0, p1);
      }
      l += sum;
      tmem_st16(tmem + lane_off + kColS + sb * kNk, pk);
      tc_fence_before();
      mbar_arrive(&sh.p_ready[sb]);
#pragma unroll
      for (int k = 0; k < 32; ++k) own[k] = own_next[k];
    }

    // epilogue: wait for the last P.V, then o = O / l and lse = (m + log2 l) ln 2
    if (ok && !mbar_wait_abortable(&sh.pv_done[(ntiles - 1) % 3], ((ntiles - 1) / 3) & 1, abort)) ok = false;
    tc_fence_after();
    if (__all_sync(0xffffffffu, ok)) {
      const int64_t prow = (static_cast<int64_t>(b) * p.max_splits + split) * (p.row_tiles * kTileRows) + grow;
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int c = 0; c < 256; c += 32) {
        float o[32];
        tmem_ld32(tmem + lane_off + kColO + c, o);
        if (row_valid) {
          float4* dst = reinterpret_cast<float4*>(p.o_part + prow * kDv + 256 * rank + c);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(o[4 * e] * inv_l, o[4 * e + 1] * inv_l, o[4 * e + 2] * inv_l, o[4 * e + 3] * inv_l);
        }
      }
      if (rank == 0 && row_valid)
        p.lse_part[prow] = l > 0.f ? (m_used + log2f(l)) * kLn2 : -CUDART_INF_F;
    }
  }

  if (!ok) {
    *abort = 1;
    atomicOr(p.status, kStatusTimeout);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still write into its shared memory
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

int prefix_pair_smem_bytes() { return kSmem; }

cudaError_t configure_prefix() {
  return cudaFuncSetAttribute(prefix_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
}

cudaError_t launch_prefix(const PrefixParams& p, int batch, int splits, cudaStream_t stream) {
  dim3 grid(2 * splits, p.row_tiles, batch);
  prefix_pair_kernel<<<grid, kThreads, kSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ddt
