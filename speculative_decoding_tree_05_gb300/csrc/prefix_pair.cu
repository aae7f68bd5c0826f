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
// Each CTA computes a partial score over its 288 dims; the pair swaps the
// partials through distributed shared memory (st.async into the peer's buffer,
// completion counted on the peer's mbarrier) and each CTA accumulates
// O_r += P . V_r for its own 256 v dims.  Every gathered row is read once per
// pair and no MMA work is duplicated.
//
// Partial-score exchange format: per row and 64-key step, block floating point
// -- one power-of-two exponent e with every |x| < 2^e and 64 int16 mantissas
// round(x * 2^(14-e)), x being the partial score in log2 units.  That is half
// the bytes of fp32 (the exchange is bound by DSMEM bandwidth) with an error of
// at most 2^-15 * 2^e, i.e. 2^-14 of the row's largest partial in the step.
// Both CTAs decode both halves the same way and add them in the same order, so
// they hold bit-identical scores and make identical softmax decisions.
//
// Per CTA (256 threads):
//   warp 0      TMEM allocation; lane 0 issues every tcgen05.mma.  A
//               tcgen05.mma costs about 45 issue cycles whatever its shape, so
//               each MMA is at least M=128 x N=64 (scores) or N=256 (P.V).
//   warps 1-3   producers: gather the CTA's 576-byte half of 64 slot rows per
//               step with 16-byte cp.async (swizzled on the fly) into a 4-stage
//               ring; slot indices are fetched one step ahead and passed
//               between lanes by shuffle; each producer thread signals the
//               stage with cp.async.mbarrier.arrive.noinc; rows of keys past
//               the split end or outside the pool are zero-filled
//   warps 4-7   softmax: one query row per thread (= its TMEM lane).  Q_r's
//               256 latent dims are staged in TMEM and its 32 rope dims in
//               shared memory; online softmax in the log2 domain with lazy
//               rescaling (O is rescaled only when the running max grows by
//               more than 8); P (bf16) is written over its S buffer and read
//               from TMEM by the P.V MMA; epilogue o = O / l.
// TMEM columns: O_r [0,256), S buffers 2 x 64 at [256,384), Q_r latent [384,512).
// Shared memory per stage: 4 latent blocks [64 keys][64 dims] (128-byte
// swizzle, 8 KB each) + 1 rope block [64 keys][32 dims] (64-byte swizzle).
// The latent blocks are the K operand of S (K-major) and, read MN-major, the
// V operand of P.V.
#include <cuda_runtime.h>
#include <math_constants.h>
#include "kernels.cuh"
#include "ptx.cuh"

namespace ddt {
namespace {

constexpr int kThreads = 256;
constexpr int kNk = kKeysPerTile;                        // 64 keys per step
constexpr int kStages = 4;
constexpr int kLatBlock = kNk * 128;                     // 8192
constexpr int kRopeBlock = kNk * 64;                     // 4096
constexpr int kStageBytes = 4 * kLatBlock + kRopeBlock;  // 36864
constexpr int kProducers = 96;
constexpr int kXBytes = kTileRows * kNk * 2;             // 16384: int16 mantissas of one step
constexpr int kEBytes = kTileRows * 4;                   // 512: one exponent per row
constexpr int kQRopeBytes = kTileRows * 64;              // 8192: Q_r rope dims, 64-byte swizzle
constexpr int kSmemStages = kStages * kStageBytes;
constexpr int kSmem = kSmemStages + 2 * kXBytes + 2 * kEBytes + kQRopeBytes + 1024;
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 384, kTmemCols = 512;
constexpr uint32_t kIdescS = idesc_bf16_f32(kTileRows, kNk, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(kTileRows, 256, false, true);
constexpr float kRescaleThreshold = 8.f;                 // log2 units
constexpr float kLn2 = 0.69314718055994531f;
static_assert(kNk == 64, "the step layout assumes 64 keys");

struct Shared {
  uint64_t k_full[kStages];   // producers -> MMA: stage loaded
  uint64_t k_empty[kStages];  // MMA -> producers: stage consumed (after P.V)
  uint64_t s_full[2];         // MMA -> softmax: partial scores of step t in S buffer t % 2
  uint64_t p_ready[2];        // softmax -> MMA: P of step t in S buffer t % 2, O rescaled
  uint64_t x_full[2];         // peer -> softmax: peer's partial scores of step t in buffer t % 2
  uint64_t pv_done[2];        // MMA -> softmax: P.V of step t completes phase t/2 of pv_done[t%2]
  uint64_t q_ready;           // softmax -> MMA: Q_r staged
  uint32_t tmem_base;
  int abort;
};

// Power-of-two exponent e with |x| < 2^e for every |x| <= amax (amax finite, >= 0).
__device__ __forceinline__ int block_exponent(float amax) {
  const int biased = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu);
  const int e = biased == 0 ? -126 : biased - 126;  // amax < 2^(biased-126)
  return max(-100, min(100, e));
}
__device__ __forceinline__ float pow2i(int k) { return __uint_as_float(static_cast<uint32_t>(127 + k) << 23); }

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) prefix_pair_kernel(PrefixParams p) {
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
  uint8_t* xbuf = smem + kSmemStages;                          // [2][128 rows][128 B]
  uint8_t* ebuf = xbuf + 2 * kXBytes;                          // [2][128 rows] int32
  uint8_t* qrope = ebuf + 2 * kEBytes;                         // [128 rows][64 B], 64-byte swizzle
  const uint32_t qrope_s = smem_u32(qrope);

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sh.k_full[i], kProducers);
      mbar_init(&sh.k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.s_full[i], 1);
      mbar_init(&sh.p_ready[i], 128);
      mbar_init(&sh.x_full[i], 1);
      mbar_init(&sh.pv_done[i], 1);
    }
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
    // Tensor-core order: S_0, S_1, PV_0, S_2, PV_1, ...  S_{j+1} reuses the S
    // buffer of step j-1, whose P was read by PV_{j-1}, issued just before.
    if (lane == 0) {
      if (!mbar_wait_abortable(&sh.q_ready, 0, abort)) ok = false;
      fence_proxy_async_smem();  // Q rope dims were stored to shared memory by the softmax threads
      tc_fence_after();
      auto issue_s = [&](int t) -> bool {
        const int st = t % kStages;
        if (!mbar_wait_abortable(&sh.k_full[st], (t / kStages) & 1, abort)) return false;
        // the stage was written by cp.async (generic proxy): order it before the
        // tensor core's async-proxy reads
        fence_proxy_async_smem();
        tc_fence_after();
        const uint32_t base = stage0 + st * kStageBytes;
        const uint32_t sb = tmem + kColS + (t % 2) * kNk;
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
          const uint64_t bd = smem_desc(base + (ks >> 2) * kLatBlock + (ks & 3) * 32, 16, 1024, kSwizzle128B);
          mma_ts(sb, tmem + kColQ + ks * 8, bd, kIdescS, ks > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          const uint64_t ad = smem_desc(qrope_s + ks * 32, 16, 512, kSwizzle64B);
          const uint64_t bd = smem_desc(base + 4 * kLatBlock + ks * 32, 16, 512, kSwizzle64B);
          mma_ss(sb, ad, bd, kIdescS, 1u);
        }
        mma_commit(&sh.s_full[t % 2]);
        return true;
      };
      if (ok && !issue_s(0)) ok = false;
      for (int j = 0; ok && j < ntiles; ++j) {
        if (j + 1 < ntiles && !issue_s(j + 1)) { ok = false; break; }
        if (!mbar_wait_abortable(&sh.p_ready[j % 2], (j / 2) & 1, abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t base = stage0 + (j % kStages) * kStageBytes;
        const uint32_t pb = tmem + kColS + (j % 2) * kNk;
#pragma unroll
        for (int ks = 0; ks < kNk / 16; ++ks) {
          const uint64_t bd = smem_desc(base + ks * 16 * 128, kLatBlock, 1024, kSwizzle128B);
          mma_ts(tmem + kColO, pb + ks * 8, bd, kIdescPV, (j > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(&sh.k_empty[j % kStages]);
        mma_commit(&sh.pv_done[j % 2]);
      }
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------------------------ producers
    const int ptid = tid - 32;
    const int32_t* slots = p.slot_idx + static_cast<int64_t>(b) * p.slot_stride;
    const uint16_t* kv = p.kv;
    // lane l holds the slots of keys l and l+32 of a step (fetched one step ahead)
    auto fetch = [&](int j, int e) -> int {
      const int key = kbegin + j * kNk + lane + 32 * e;
      return key < kend ? __ldg(slots + key) : -1;
    };
    int cur0 = fetch(0, 0), cur1 = fetch(0, 1);
    for (int j = 0; j < ntiles; ++j) {
      const int nxt0 = (j + 1 < ntiles) ? fetch(j + 1, 0) : -1;
      const int nxt1 = (j + 1 < ntiles) ? fetch(j + 1, 1) : -1;
      const int st = j % kStages;
      // warp-uniform wait: the lane shuffles below need every lane
      const bool waited = j < kStages || mbar_wait_abortable(&sh.k_empty[st], ((j / kStages) - 1) & 1, abort);
      if (!__all_sync(0xffffffffu, waited)) {
        ok = false;
        break;
      }
      const int kbase = kbegin + j * kNk;
      if (warp == 1 && rank == 0) {
        const bool bad0 = kbase + lane < kend && (cur0 < 0 || static_cast<int64_t>(cur0) >= p.pool_slots);
        const bool bad1 = kbase + lane + 32 < kend && (cur1 < 0 || static_cast<int64_t>(cur1) >= p.pool_slots);
        if (__any_sync(0xffffffffu, bad0 || bad1) && lane == 0) atomicOr(p.status, kStatusBadSlot);
      }
      const uint32_t base = stage0 + st * kStageBytes;
#pragma unroll 4
      for (int k = 0; k < kNk * 36 / kProducers; ++k) {
        const int i = ptid + k * kProducers;
        const int n = i / 36, c = i - n * 36;
        const int s0 = __shfl_sync(0xffffffffu, cur0, n & 31);
        const int s1 = __shfl_sync(0xffffffffu, cur1, n & 31);
        const int slot = n < 32 ? s0 : s1;
        const bool valid = slot >= 0 && static_cast<int64_t>(slot) < p.pool_slots;
        const int off = (c < 32) ? 256 * static_cast<int>(rank) + 8 * c : 512 + 32 * static_cast<int>(rank) + 8 * (c - 32);
        const uint16_t* src = valid ? kv + static_cast<int64_t>(slot) * kDqk + off : kv;
        const uint32_t dst = (c < 32) ? base + (c >> 3) * kLatBlock + n * 128 + (((c & 7) ^ (n & 7)) << 4)
                                      : base + 4 * kLatBlock + n * 64 + (((c - 32) ^ ((n >> 1) & 3)) << 4);
        cp_async16(dst, src, valid ? 16u : 0u);
      }
      cp_async_arrive_noinc(&sh.k_full[st]);
      cur0 = nxt0;
      cur1 = nxt1;
    }
    cp_async_wait<0>();
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    const int r = tid - 128;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int grow = row_tile * kTileRows + r;
    const bool row_valid = grow < p.rows;

    // Q_r: latent dims [256 rank, +256) -> TMEM, rope dims [512 + 32 rank, +32) -> smem
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
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 x = row_valid ? __ldg(qsrc + 64 + 4 * rank + c) : zero;
        *reinterpret_cast<uint4*>(qrope + r * 64 + ((c ^ ((r >> 1) & 3)) << 4)) = x;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&sh.q_ready);
    }

    const uint32_t peer = rank ^ 1u;
    uint32_t x_remote[2], e_remote[2], xbar_remote[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      x_remote[i] = mapa_shared(smem_u32(xbuf + i * kXBytes), peer);
      e_remote[i] = mapa_shared(smem_u32(ebuf + i * kEBytes), peer);
      xbar_remote[i] = mapa_shared(smem_u32(&sh.x_full[i]), peer);
    }
    const int32_t* slots = p.slot_idx + static_cast<int64_t>(b) * p.slot_stride;
    const uint32_t rsw = static_cast<uint32_t>(r & 7);
    float m_used = -CUDART_INF_F, l = 0.f;
    auto fetch_slot = [&](int j, int e) -> int {
      const int key = kbegin + j * kNk + lane + 32 * e;
      return key < kend ? __ldg(slots + key) : 0;
    };
    // slots of this lane's two keys, fetched one step ahead
    int sl0 = fetch_slot(0, 0), sl1 = fetch_slot(0, 1);

    // Step t uses exchange buffer t % 2.  The peer writes step t only after it
    // has received our step t-1, which we send after finishing step t-2, the
    // last reader of that buffer.
    for (int j = 0; ok && j < ntiles; ++j) {
      const int sb = j % 2;
      const int kbase = kbegin + j * kNk;
      const int cur0 = sl0, cur1 = sl1;
      if (j + 1 < ntiles) {
        sl0 = fetch_slot(j + 1, 0);
        sl1 = fetch_slot(j + 1, 1);
      }
      if (r == 0) mbar_arrive_expect_tx(&sh.x_full[sb], kXBytes + kEBytes);
      if (!__all_sync(0xffffffffu, mbar_wait_abortable(&sh.s_full[sb], (j / 2) & 1, abort))) { ok = false; break; }
      tc_fence_after();
      float x[64];
      {
        float t0[32], t1[32];
        tmem_ld32(tmem + lane_off + kColS + sb * kNk, t0);
        tmem_ld32(tmem + lane_off + kColS + sb * kNk + 32, t1);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          x[k] = t0[k] * p.scale_log2;
          x[32 + k] = t1[k] * p.scale_log2;
        }
      }
      // encode own partial (block floating point), send it, and decode it again
      float amax = 0.f;
#pragma unroll
      for (int k = 0; k < 64; ++k) amax = fmaxf(amax, fabsf(x[k]));
      const int e = block_exponent(amax);
      const float enc = pow2i(14 - e), dec = pow2i(e - 14);
      {
        const uint32_t xr = x_remote[sb] + r * 128, br = xbar_remote[sb];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int k = 8 * c + 2 * h;
            const int q0 = __float2int_rn(x[k] * enc), q1 = __float2int_rn(x[k + 1] * enc);
            w[h] = (static_cast<uint32_t>(q0) & 0xffffu) | (static_cast<uint32_t>(q1) << 16);
            x[k] = static_cast<float>(q0) * dec;
            x[k + 1] = static_cast<float>(q1) * dec;
          }
          st_async_v4(xr + ((c ^ rsw) << 4), make_uint4(w[0], w[1], w[2], w[3]), br);
        }
        st_async_b32(e_remote[sb] + r * 4, static_cast<uint32_t>(e), br);
      }
      // key mask of this step (past the split end or a slot outside the pool)
      const uint32_t masked0 = __ballot_sync(
          0xffffffffu, kbase + lane >= kend || cur0 < 0 || static_cast<int64_t>(cur0) >= p.pool_slots);
      const uint32_t masked1 = __ballot_sync(
          0xffffffffu, kbase + lane + 32 >= kend || cur1 < 0 || static_cast<int64_t>(cur1) >= p.pool_slots);
      if (!__all_sync(0xffffffffu, mbar_wait_abortable(&sh.x_full[sb], (j / 2) & 1, abort, true))) {
        ok = false;
        break;
      }
      // add the peer's partial: s = own + peer (fp32 addition commutes, so both CTAs agree)
      float mx = -CUDART_INF_F;
      {
        const uint8_t* xb = xbuf + sb * kXBytes + r * 128;
        const int pe = *reinterpret_cast<const int*>(ebuf + sb * kEBytes + r * 4);
        const float pdec = pow2i(pe - 14);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(xb + ((c ^ rsw) << 4));
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int k = 8 * c + 2 * h;
            const float a = static_cast<float>(static_cast<int>(static_cast<int16_t>(w[h] & 0xffffu))) * pdec;
            const float bb = static_cast<float>(static_cast<int>(w[h]) >> 16) * pdec;
            const uint32_t mk = k < 32 ? masked0 : masked1;
            x[k] = ((mk >> (k & 31)) & 1u) ? -CUDART_INF_F : x[k] + a;
            x[k + 1] = ((mk >> ((k + 1) & 31)) & 1u) ? -CUDART_INF_F : x[k + 1] + bb;
            mx = fmaxf(mx, fmaxf(x[k], x[k + 1]));
          }
        }
      }
      const bool need = mx > m_used + kRescaleThreshold;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mx : m_used;
        const float alpha = need ? fast_exp2(m_used - m_new) : 1.f;
        if (j > 0) {
          // O must hold every earlier step: wait for P.V of step j-1 (MMAs complete in order)
          if (!__all_sync(0xffffffffu, mbar_wait_abortable(&sh.pv_done[(j - 1) % 2], ((j - 1) / 2) & 1, abort))) {
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
            for (int k = 0; k < 32; ++k) ob[k] = __float_as_uint(o[k] * alpha);
            tmem_st32(tmem + lane_off + kColO + c, ob);
          }
        }
        l *= alpha;
        m_used = m_new;
      }
      const float msub = (m_used == -CUDART_INF_F) ? 0.f : m_used;
      float sum = 0.f;
      uint32_t pk[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float p0 = fast_exp2(x[2 * k] - msub), p1 = fast_exp2(x[2 * k + 1] - msub);
        sum += p0 + p1;
        pk[k] = pack_bf16x2(p0, p1);
      }
      l += sum;
      tmem_st32(tmem + lane_off + kColS + sb * kNk, pk);
      tc_fence_before();
      mbar_arrive(&sh.p_ready[sb]);
    }

    // epilogue: wait for the last P.V, then o = O / l and lse = (m + log2 l) ln 2
    if (ok && !mbar_wait_abortable(&sh.pv_done[(ntiles - 1) % 2], ((ntiles - 1) / 2) & 1, abort)) ok = false;
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
          for (int k = 0; k < 8; ++k)
            dst[k] = make_float4(o[4 * k] * inv_l, o[4 * k + 1] * inv_l, o[4 * k + 2] * inv_l, o[4 * k + 3] * inv_l);
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

cudaError_t configure_prefix() {
  return cudaFuncSetAttribute(prefix_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
}

cudaError_t launch_prefix(const PrefixParams& p, int batch, int splits, cudaStream_t stream) {
  dim3 grid(2 * splits, p.row_tiles, batch);
  prefix_pair_kernel<<<grid, kThreads, kSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ddt
