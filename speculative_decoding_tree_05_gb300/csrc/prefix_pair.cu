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
// Each CTA has one exchange buffer; step t is signalled on barrier pair t % 2
// (one per softmax set).  Before writing step t the sender waits until the
// receiver has read step t-1 out of it (a barrier in the sender that the
// receiver's warps arrive on remotely).  A step is read out well before the
// other set's next step is ready to send, so one buffer costs no waiting.
//
// Partial-score exchange format: per row and 64-key step, block floating point
// -- one power-of-two exponent e with every |x| < 2^e and 64 mantissas, x being
// the partial score in log2 units.  Every unit first runs with 16-bit mantissas
// round(x * 2^(14-e)) + 2^15 (2 bytes per score, the DSMEM budget the step
// period affords): error <= 2^(e-15), i.e. <= 2^-11 log2 units (3.4e-4 nats)
// while e <= 4, which N(0,1) data at sm_scale 1/sqrt(192) never leaves.  If
// any row of either CTA had e > 4 in any step, the pair computes the unit again
// with 20-bit mantissas round(x * 2^(18-e)) + 2^19 (the low 16 bits plus a
// packed 4-bit nibble, 2.5 bytes per score): error <= 2^(e-19), under 7e-4 nats
// for partial scores below 2^9 log2 units (355 nats).  So the log-sum-exp stays
// within 1e-3 of the exact one even for a dominant key (16-bit mantissas alone
// exceed 1e-3 nats once partial scores reach 32 log2 units).  The two widths
// are separate instantiations of the unit: the normal pass carries no code of
// the wide one, which would cost its issue-bound softmax about a tenth.
// Rounding to an integer and packing use the float adder: x * 2^(k-e) + M with
// M = 1.5 * 2^23 + 2^(k+1) is an integer-valued float whose low k+2 bits are
// the biased mantissa and whose high bits are fixed, so no int/float conversion
// instruction is needed either way.  Each CTA
// adds the peer's decoded partial to its own unrounded one, so the two CTAs'
// scores differ by that rounding alone; each CTA keeps its own running max and
// row sum and normalises its own half of O by them, so neither half depends on
// the other CTA's softmax decisions (rank 0's log-sum-exp serves both halves in
// the split merge, off by the same rounding).
//
// Per CTA (384 threads):
//   warp 0      TMEM allocation; lane 0 issues the score MMAs S(t) into S
//               buffer t % 2 once the stage is loaded and S(t-2) has been read
//               out of that buffer, so the next scores are queued while the
//               softmax reads the last ones.  A tcgen05.mma costs about 45
//               issue cycles whatever its shape, so each MMA is at least
//               M=128 x N=64 (scores) or N=256 (P.V); the pipe takes the next
//               MMA only about as fast as it runs one, so P.V is issued by the
//               softmax set that wrote its P.
//   warps 1-3   producers: load the CTA's dims of 64 slot rows per step into a
//               5-stage ring, the step's slot indices fetched four steps ahead.
//               A step whose 64 slots are consecutive (a compacted pool) is 5
//               tiled TMA boxes of 64 rows.  A scattered step uses TMA
//               tile::gather4 for latent blocks 0-2 (16 lanes of each producer
//               warp, one block per warp) and, at the same time, 16-byte
//               cp.async from all 96 threads for latent block 3 and the rope
//               dims: one SM's TMA unit and load/store path each gather
//               scattered 128-byte row pieces at only ~14-19 B/clk, so both
//               run at once.  A step with a key past the split end or a slot
//               outside the pool is all cp.async with zero fill (its rows are
//               masked and must not carry non-finite values into P.V).
//   warps 4-7   softmax set 0 (even steps), warps 8-11 softmax set 1 (odd
//               steps): one query row per thread (= its TMEM lane), so two
//               steps are in flight at once.  The sets hand each other the
//               running max of every row (step t waits for step t-1's); each
//               set keeps its own row sums against the max it last used and
//               the two are combined at the end.  O is rescaled in TMEM only
//               when the running max grows by more than 8 (lazily).  Set s
//               reads S buffer s, frees it as soon as S is in registers, and
//               writes P (bf16) into the one P buffer once P.V(t-1) is done.
// TMEM columns: O_r [0,256), S buffers 2 x 64 at [256,384), P [384,416),
// Q_r latent dims 0..191 [416,512); dims 192..255 of Q_r are read from shared
// memory (16 KB, 128-byte swizzle), as are its rope dims.
// Shared memory per stage: 4 latent blocks [64 keys][64 dims] (128-byte
// swizzle, 8 KB each) + the CTA's rope block [64 keys][32 dims] (64-byte
// swizzle, 4 KB).  The stage's lifetime runs from its load through S, the
// softmax with its exchange, and P.V, so the ring is as deep as fits.
// The latent blocks are the K operand of S (K-major) and, read MN-major, the
// V operand of P.V.
#include <cuda_runtime.h>
#include <math_constants.h>
#include "kernels.cuh"
#include "schedule.cuh"
#include "merge_row.cuh"
#include "ptx.cuh"

namespace ddt {
namespace {

constexpr int kThreads = 384;
constexpr int kNk = kKeysPerTile;                        // 64 keys per step
constexpr int kStages = 5;
constexpr int kLatBlock = kNk * 128;                     // 8192
constexpr int kRopeBlock = kNk * 64;                     // 4096
constexpr int kStageBytes = 4 * kLatBlock + kRopeBlock;  // 36864
constexpr int kProducers = 96;
constexpr int kSlotLookahead = 4;                        // producers fetch slot indices this many steps ahead
constexpr int kGatherBlocks = 3;                         // latent blocks fetched by gather4 on scattered steps
constexpr int kXSets = 2;                                // exchange barrier pairs (step t uses t % 2)
constexpr int kXChunk = kTileRows * 16;                  // one 16-byte chunk of every row of the tile
constexpr int kXLoChunks = kNk * 2 / 16;                 // 8: low 16 bits of the 64 mantissas
constexpr int kXNibChunks = kNk / 2 / 16;                // 2: their top 4 bits, two per byte
constexpr int kXLoBytes = kXLoChunks * kXChunk;         // 16384: 16-bit mantissas of one step
constexpr int kXBytes = (kXLoChunks + kXNibChunks) * kXChunk;  // 20480: 20-bit mantissas of one step
constexpr int kEBytes = kTileRows * 4;                   // 512: one exponent per row
constexpr int kQRopeBytes = kTileRows * 64;              // 8192: Q_r rope dims, 64-byte swizzle
constexpr int kQLatSmemBytes = kTileRows * 128;          // 16384: Q_r latent dims 192..255, 128-byte swizzle
constexpr int kOffQLat = kStages * kStageBytes;          // 1024-byte aligned (128-byte swizzle atoms)
constexpr int kOffX = kOffQLat + kQLatSmemBytes;         // one exchange buffer: a step is read out before the next is sent
constexpr int kOffE = kOffX + kXBytes;
constexpr int kOffQRope = kOffE + kEBytes;               // 512-byte aligned (64-byte swizzle atoms)
static_assert(kOffQLat % 1024 == 0 && kOffQRope % 512 == 0, "swizzled operands need aligned bases");
constexpr int kOffHand = kOffQRope + kQRopeBytes;        // [2][128] running max handed between sets
// [2 sets][2 (l, m)][128] final row state: written after the last exchange has
// been read out, so it shares the exchange buffer
constexpr int kOffFin = kOffX;
static_assert(2 * 2 * kTileRows * 4 <= kXBytes, "the final row state fits in the exchange buffer");
constexpr int kSmem = kOffHand + 2 * kTileRows * 4 + 1024;
constexpr uint32_t kColO = 0, kColS = 256, kColP = 384, kColQ = 416, kTmemCols = 512;
constexpr int kQTmemKSteps = 12;                         // Q_r latent dims 0..191 from TMEM, 192..255 from smem
constexpr uint32_t kIdescS = idesc_bf16_f32(kTileRows, kNk, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(kTileRows, 256, false, true);
constexpr float kRescaleThreshold = 8.f;                 // log2 units
constexpr float kLn2 = 0.69314718055994531f;
constexpr int kXFracBits = 18;                           // 20-bit mantissa = round(x * 2^(18-e)) + 2^19
constexpr float kMagic = 13107200.0f;                    // 1.5 * 2^23 + 2^19
constexpr int kXFracBits16 = 14;                         // 16-bit mantissa = round(x * 2^(14-e)) + 2^15
constexpr float kMagic16 = 12615680.0f;                  // 1.5 * 2^23 + 2^15
constexpr uint32_t kMagicHi16 = 0x4B400000u;             // top half of every 16-bit-encoded float
constexpr int kX16MaxExp = 4;                            // 16-bit mantissas suffice while every e is <= 4
constexpr int kSoftmaxBarrier = 1;                       // named barrier of the 256 softmax threads
static_assert(kNk == 64, "the step layout assumes 64 keys");

struct Shared {
  uint64_t k_full[kStages];   // producers -> MMA: stage loaded
  uint64_t k_empty[kStages];  // MMA -> producers and softmax: P.V of step t done, its stage free
                              // (phase t / kStages of k_empty[t % kStages])
  uint64_t s_full[2];         // MMA -> softmax set t%2: partial scores of step t in the S buffer
  uint64_t s_free[2];         // softmax set t%2 -> MMA: S of step t loaded into registers
  uint64_t p_ready[2];        // softmax set t%2 -> its P.V issuer: P of step t in the P buffer, O rescaled
  uint64_t x_full[kXSets];    // peer -> softmax set t%2: peer's partial scores of step t in the exchange buffer
  uint64_t x_free[kXSets];    // peer's set t%2 -> sender: step t read out of the peer's exchange buffer
  uint64_t m_ready[2];        // softmax set -> other set: running max after step t in hand[t % 2]
  uint64_t q_ready;           // softmax -> MMA: Q_r staged
  uint64_t mma_drain;         // the three MMA-issuing threads: every MMA issued has completed
  volatile int pv_next;       // the step whose P.V is issued next (P.V goes in step order)
  uint32_t tmem_base;
  int abort;
  int last_arrival;           // fused kernel: this pair finished the last split of its (request, row tile)
  int unit[2];                // fused kernel: the units the pair claimed, by claim parity
  int need_wide;              // 16-bit pass: a partial of this CTA needed more than 16-bit mantissas
  int peer_need_wide;         // the peer CTA's flag word (stored remotely at the end of the 16-bit pass)
};

// Power-of-two exponent e with |x| < 2^e for every |x| <= amax (amax finite, >= 0).
__device__ __forceinline__ int block_exponent(float amax) {
  const int biased = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu);
  const int e = biased == 0 ? -126 : biased - 126;  // amax < 2^(biased-126)
  return max(-100, min(100, e));
}
__device__ __forceinline__ float pow2i(int k) { return __uint_as_float(static_cast<uint32_t>(127 + k) << 23); }

// Barriers of a CTA, set up once per launch: their phases then run on across
// the passes and units a CTA computes (step g of the CTA uses stage g % 5, S
// buffer and softmax set g % 2, ...), so an arrival that lands late -- a
// tensor-core commit or a remote arrive of the previous pass -- still counts in
// the phase it belongs to.  The first run_unit's set-up barriers publish them
// to the peer before any remote access.
__device__ __forceinline__ void init_barriers(Shared& sh) {
  for (int i = 0; i < kStages; ++i) {
    mbar_init(&sh.k_full[i], kProducers + 1);  // every producer thread + one (TMA) arrival
    mbar_init(&sh.k_empty[i], 1);
  }
  for (int i = 0; i < 2; ++i) {
    mbar_init(&sh.s_full[i], 1);
    mbar_init(&sh.s_free[i], 128);
    mbar_init(&sh.p_ready[i], 128);
    mbar_init(&sh.m_ready[i], 128);
  }
  for (int i = 0; i < kXSets; ++i) {
    mbar_init(&sh.x_full[i], 1);
    mbar_init(&sh.x_free[i], 4);  // the 4 warps of the peer's set
  }
  mbar_init(&sh.q_ready, 256);
  mbar_init(&sh.mma_drain, 3);  // one commit from each MMA-issuing thread, per pass
  sh.pv_next = 0;
  sh.abort = 0;
  fence_mbar_init();
}

constexpr int kUnitWide = 1;     // run_unit result: a partial of the 16-bit pass needed wider mantissas
constexpr int kUnitAborted = 2;  // run_unit result: a CTA of the pair gave up on a wait

// One pass over one unit = one CTA pair on one (request, 128-row tile, key
// split), as the CTA's steps G .. G + ntiles - 1 and its pass number `pass`.
// kWide selects the exchange width: false = 16-bit mantissas (the normal pass),
// true = 20-bit (a rerun of the same unit, separately compiled so that the
// normal pass carries none of its code).  Returns the pair's kUnit* flags (the
// same in both CTAs): after kUnitAborted the CTA's barriers are in an unknown
// state and it must not run another pass.
template <bool kWide>
__device__ __forceinline__ int run_unit(const PrefixParams& p, Shared& sh, uint8_t* smem_raw, int row_tile,
                                        int split, int b, int kbegin, int kend, int rows_b, int G, int pass) {
  volatile int* abort = &sh.abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int ntiles = (kend - kbegin + kNk - 1) / kNk;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t stage0 = smem_u32(smem);
  uint8_t* qrope = smem + kOffQRope;
  const uint32_t qrope_s = smem_u32(qrope);

  if (tid == 0) {
    sh.need_wide = 0;
    sh.peer_need_wide = 0;
  }
  // Global reads that need no set-up are issued before the CTA's barrier, so
  // their latency overlaps it: the producers' slot indices of the first steps
  // (lane l holds the slots of keys l and l+32 of a step; -1 past the split
  // end) and the softmax threads' query row.
  const int32_t* slots = p.slot_idx + static_cast<int64_t>(b) * p.slot_stride;
  auto fetch = [&](int j, int e) -> int {
    const int key = kbegin + j * kNk + lane + 32 * e;
    return key < kend ? __ldg(slots + key) : -1;
  };
  const bool producer = warp >= 1 && warp < 4;
  int pf[2 * kSlotLookahead];
#pragma unroll
  for (int i = 0; i < 2 * kSlotLookahead; ++i) pf[i] = producer ? fetch(i >> 1, i & 1) : -1;
  const int qrow = (warp & 3) * 32 + lane;
  const bool q_valid = warp >= 4 && row_tile * kTileRows + qrow < rows_b;
  const uint4* qsrc = reinterpret_cast<const uint4*>(p.q + (static_cast<int64_t>(b) * p.rows + row_tile * kTileRows + qrow) * kDqk);
  uint4 qv[16 + 4];
#pragma unroll
  for (int c = 0; c < 16; ++c)
    qv[c] = q_valid ? __ldg(qsrc + 32 * rank + 16 * ((warp - 4) >> 2) + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int c = 0; c < 4; ++c) qv[16 + c] = q_valid && warp < 8 ? __ldg(qsrc + 64 + 4 * rank + c) : make_uint4(0, 0, 0, 0);
  tc_fence_before();
  __syncthreads();  // this CTA's barriers initialised (first pass), its TMEM allocated and the last pass done
  // The peer addresses this CTA's barriers only after its own cluster_wait,
  // which follows this arrive: threads that touch the peer wait before their
  // first remote access, the others before the final cluster barrier.
  cluster_arrive();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  bool ok = true;
  int issued = G;  // producers: the CTA step after the last one this warp has issued loads for

  if (warp == 0) {
    // ------------------------------------------------------------------ S issuer
    // The tensor pipe takes the next MMA only about as fast as it runs one, so a
    // thread that also issued P.V could not react to a ready stage while inside
    // a P.V group: this thread issues only S, sleeping on the barrier it needs;
    // each softmax set issues the P.V of its own steps.
    if (lane == 0) {
      if (!mbar_wait_abortable(&sh.q_ready, pass & 1, abort, false, __LINE__)) ok = false;
      fence_proxy_async_smem();  // Q rope dims were stored to shared memory by the softmax threads
      tc_fence_after();
      // operand descriptors of stage 0, built once; a stage or k-step is an offset
      const uint64_t d_lat = smem_desc(stage0, 16, 1024, kSwizzle128B);             // K of S: K-major
      const uint64_t d_rope = smem_desc(stage0 + 4 * kLatBlock, 16, 512, kSwizzle64B);
      const uint64_t d_qrope = smem_desc(qrope_s, 16, 512, kSwizzle64B);
      const uint64_t d_qlat = smem_desc(stage0 + kOffQLat, 16, 1024, kSwizzle128B);
      for (int ns = G; ok && ns < G + ntiles; ++ns) {
        // stage loaded, and S(ns-2) read out of S buffer ns % 2
        if (!mbar_wait_abortable(&sh.k_full[ns % kStages], (ns / kStages) & 1, abort, false, __LINE__) ||
            (ns > 1 && !mbar_wait_abortable(&sh.s_free[ns % 2], ((ns - 2) / 2) & 1, abort, false, __LINE__))) {
          ok = false;
          break;
        }
        // the stage may have been written by cp.async (generic proxy): order it
        // before the tensor core's async-proxy reads
        fence_proxy_async_smem();
        tc_fence_after();
        const uint32_t so = (ns % kStages) * kStageBytes;
        const uint64_t dl = desc_advance(d_lat, so), dr = desc_advance(d_rope, so);
        const uint32_t sd = tmem + kColS + (ns % 2) * kNk;
#pragma unroll
        for (int ks = 0; ks < kQTmemKSteps; ++ks)
          mma_ts(sd, tmem + kColQ + ks * 8, desc_advance(dl, (ks >> 2) * kLatBlock + (ks & 3) * 32), kIdescS,
                 ks > 0 ? 1u : 0u);
#pragma unroll
        for (int ks = kQTmemKSteps; ks < 16; ++ks)
          mma_ss(sd, desc_advance(d_qlat, (ks - kQTmemKSteps) * 32),
                 desc_advance(dl, (ks >> 2) * kLatBlock + (ks & 3) * 32), kIdescS, 1u);
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
          mma_ss(sd, desc_advance(d_qrope, ks * 32), desc_advance(dr, ks * 32), kIdescS, 1u);
        mma_commit(&sh.s_full[ns % 2]);
      }
      // nothing of this thread's may still be running when TMEM is released (also after a timeout)
      mma_commit(&sh.mma_drain);
      mbar_wait(&sh.mma_drain, pass & 1);
    }
    __syncwarp();
    cluster_wait();
  } else if (warp < 4) {
    // ------------------------------------------------------------------ producers
    const int ptid = tid - 32;
    const uint16_t* kv = p.kv;
    const int rk = static_cast<int>(rank);
    auto in_pool = [&](int s_) { return s_ >= 0 && static_cast<int64_t>(s_) < p.pool_slots; };
    // 16-byte chunk c of the CTA's 36 per row -> (source column, smem offset in the stage):
    // c < 32 latent block c/8 (128-byte swizzle), c >= 32 the rope block (64-byte swizzle)
    auto chunk_dst = [&](int n, int c) -> uint32_t {
      return c < 32 ? (c >> 3) * kLatBlock + n * 128 + (((c & 7) ^ (n & 7)) << 4)
                    : 4 * kLatBlock + n * 64 + (((c - 32) ^ ((n >> 1) & 3)) << 4);
    };
    auto chunk_col = [&](int c) -> int { return c < 32 ? 256 * rk + 8 * c : 512 + 32 * rk + 8 * (c - 32); };
    // slot indices are fetched kSlotLookahead steps ahead: under a gather-heavy
    // load their latency exceeds a step
    for (int j = 0; j < ntiles; ++j) {
      const int g = G + j;  // the CTA's step
      const int cur0 = pf[0], cur1 = pf[1];
#pragma unroll
      for (int i = 0; i + 2 < 2 * kSlotLookahead; ++i) pf[i] = pf[i + 2];
      pf[2 * kSlotLookahead - 2] = fetch(j + kSlotLookahead, 0);
      pf[2 * kSlotLookahead - 1] = fetch(j + kSlotLookahead, 1);
      const int st = g % kStages;
#ifdef DDT_TEST_HOOKS
      // test builds: a stage that is never loaded, so the waits for it run out
      if (j == p.test_drop_step) continue;
#endif
      // warp-uniform wait: the lane shuffles below need every lane
      const bool waited = g < kStages || mbar_wait_abortable(&sh.k_empty[st], ((g / kStages) - 1) & 1, abort, false, __LINE__);
      if (!__all_sync(0xffffffffu, waited)) {
        ok = false;
        break;
      }
      const int kbase = kbegin + j * kNk;
      const bool v0 = kbase + lane < kend && in_pool(cur0), v1 = kbase + lane + 32 < kend && in_pool(cur1);
      if (warp == 1 && rank == 0) {
        // (index lists: a -1 entry is no key, not a bad slot)
        const bool bad0 = kbase + lane < kend && !in_pool(cur0) && !(p.sparse && cur0 == -1);
        const bool bad1 = kbase + lane + 32 < kend && !in_pool(cur1) && !(p.sparse && cur1 == -1);
        if (__any_sync(0xffffffffu, bad0 || bad1) && lane == 0) atomicOr(p.status, kStatusBadSlot);
      }
      const bool all_valid = __all_sync(0xffffffffu, v0 && v1);
      const int first = __shfl_sync(0xffffffffu, cur0, 0);
      const bool contiguous =
          p.block_loads && all_valid && __all_sync(0xffffffffu, cur0 == first + lane && cur1 == first + 32 + lane);
      const uint32_t base = stage0 + st * kStageBytes;
      if (contiguous) {
        // 64 consecutive rows: five 64-row boxes (the latent blocks and the rope block)
        if (warp == 1 && lane == 0) {
          mbar_arrive_expect_tx(&sh.k_full[st], kStageBytes);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            tma_load_2d(base + c * kLatBlock, &p.tmap_block, 256 * rk + 64 * c, first, &sh.k_full[st]);
          tma_load_2d(base + 4 * kLatBlock, &p.tmap_rope, 512 + 32 * rk, first, &sh.k_full[st]);
        }
      } else if (all_valid) {
        // gather4 for latent blocks 0..2 (producer warp w takes block w-1) ...
        if (warp == 1 && lane == 0) mbar_arrive_expect_tx(&sh.k_full[st], kGatherBlocks * kLatBlock);
        int r[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int n = 4 * (lane & 15) + e;
          const int s0 = __shfl_sync(0xffffffffu, cur0, n & 31), s1 = __shfl_sync(0xffffffffu, cur1, n & 31);
          r[e] = n < 32 ? s0 : s1;
        }
        if (lane < 16) {
          const int blk = warp - 1;
          tma_gather4(base + blk * kLatBlock + lane * 512, &p.tmap_rows, 256 * rk + 64 * blk, r[0], r[1], r[2], r[3],
                      &sh.k_full[st]);
        }
        // ... and cp.async for latent block 3 (chunks 24..31) and the rope chunks (32..35)
#pragma unroll 4
        for (int k = 0; k < kNk * 12 / kProducers; ++k) {
          const int i = ptid + k * kProducers;
          const int n = i / 12, c = 24 + i % 12;
          const int s0 = __shfl_sync(0xffffffffu, cur0, n & 31), s1 = __shfl_sync(0xffffffffu, cur1, n & 31);
          const int slot = n < 32 ? s0 : s1;
          cp_async16(base + chunk_dst(n, c), kv + static_cast<int64_t>(slot) * kDqk + chunk_col(c), 16u);
        }
      } else {
        // a masked key in the step: everything by cp.async, zero-filled where masked
        if (warp == 1 && lane == 0) mbar_arrive(&sh.k_full[st]);
#pragma unroll 4
        for (int k = 0; k < kNk * 36 / kProducers; ++k) {
          const int i = ptid + k * kProducers;
          const int n = i / 36, c = i - n * 36;
          const int s0 = __shfl_sync(0xffffffffu, cur0, n & 31), s1 = __shfl_sync(0xffffffffu, cur1, n & 31);
          const int slot = n < 32 ? s0 : s1;
          const bool valid = kbase + n < kend && in_pool(slot);
          const uint16_t* src = valid ? kv + static_cast<int64_t>(slot) * kDqk + chunk_col(c) : kv;
          cp_async16(base + chunk_dst(n, c), src, valid ? 16u : 0u);
        }
      }
      cp_async_arrive_noinc(&sh.k_full[st]);
      issued = g + 1;
    }
    cp_async_wait<0>();
    cluster_wait();
  } else {
    // ------------------------------------------------------------------ softmax sets + epilogue
    const int set = (warp - 4) >> 2;                   // 0: even steps, 1: odd steps
    const int r = (warp & 3) * 32 + lane;              // row of the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int grow = row_tile * kTileRows + r;
    const bool row_valid = grow < rows_b;
    float* hand = reinterpret_cast<float*>(smem + kOffHand);   // [2][128]
    float* fin = reinterpret_cast<float*>(smem + kOffFin);     // [2 sets][2][128]

    // Q_r (read into registers before the CTA barrier): set s holds latent dims
    // [256 rank + 128 s, +128); dims 0..191 of the CTA's 256 go to TMEM, dims
    // 192..255 (the second half of set 1's) to shared memory, 128-byte swizzle;
    // rope dims [512 + 32 rank, +32) -> shared memory, 64-byte swizzle
    {
#pragma unroll
      for (int c0 = 0; c0 < 16; c0 += 8) {
        if (set == 1 && c0 == 8) {
          uint8_t* ql = smem + kOffQLat + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(ql + ((c ^ (r & 7)) << 4)) = qv[8 + c];
        } else {
          uint32_t v[32];
#pragma unroll
          for (int c = 0; c < 8; ++c)
            v[4 * c] = qv[c0 + c].x, v[4 * c + 1] = qv[c0 + c].y, v[4 * c + 2] = qv[c0 + c].z, v[4 * c + 3] = qv[c0 + c].w;
          tmem_st32(tmem + lane_off + kColQ + 64 * set + c0 * 4, v);
        }
      }
      if (set == 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(qrope + r * 64 + ((c ^ ((r >> 1) & 3)) << 4)) = qv[16 + c];
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&sh.q_ready);
    }
    cluster_wait();  // the peer's barriers exist before the first exchange

    const uint32_t peer = rank ^ 1u;
    const uint32_t x_remote = mapa_shared(stage0 + kOffX, peer);
    const uint32_t e_remote = mapa_shared(stage0 + kOffE, peer);
    uint32_t xbar_remote[kXSets], xfree_remote[kXSets];
#pragma unroll
    for (int i = 0; i < kXSets; ++i) {
      xbar_remote[i] = mapa_shared(smem_u32(&sh.x_full[i]), peer);
      xfree_remote[i] = mapa_shared(smem_u32(&sh.x_free[i]), peer);
    }
    bool need_wide = false;  // 16-bit pass: a row's partial of some step had e > kX16MaxExp
    const bool lead = (warp & 3) == 0 && lane == 0;    // row 0 of this set; issues the set's P.V
    const uint64_t d_v = smem_desc(stage0, kLatBlock, 1024, kSwizzle128B);  // V of P.V: MN-major
    float m_used = -CUDART_INF_F;                      // running max after the last step seen
    float m_ref = -CUDART_INF_F, l = 0.f;              // this set's row sum, relative to m_ref
    auto fetch_slot = [&](int j, int e) -> int {
      const int key = kbegin + j * kNk + lane + 32 * e;
      return key < kend ? __ldg(slots + key) : 0;
    };
    // set s takes the CTA steps g with g % 2 == s; j = g - G is the step within the unit
    const int j0 = (set ^ G) & 1;
    int sl0 = fetch_slot(j0, 0), sl1 = fetch_slot(j0, 1);

    // Step g uses exchange barriers g % 2 (this set's) in both CTAs.
    for (int j = j0; ok && j < ntiles; j += 2) {
      const int g = G + j;
      const int sb = g % 2;
      const int xb_i = g % kXSets;                      // this set's exchange barriers
      const int kbase = kbegin + j * kNk;
      const int cur0 = sl0, cur1 = sl1;
      if (j + 2 < ntiles) {
        sl0 = fetch_slot(j + 2, 0);
        sl1 = fetch_slot(j + 2, 1);
      }
      if (lead) mbar_arrive_expect_tx(&sh.x_full[xb_i], (kWide ? kXBytes : kXLoBytes) + kEBytes);
      if (!__all_sync(0xffffffffu, mbar_wait_abortable(&sh.s_full[sb], (g / 2) & 1, abort, false, __LINE__))) { ok = false; break; }
      tc_fence_after();
      float x[64];
      tmem_ld32(tmem + lane_off + kColS + sb * kNk, *reinterpret_cast<float(*)[32]>(&x[0]));
      tmem_ld32(tmem + lane_off + kColS + sb * kNk + 32, *reinterpret_cast<float(*)[32]>(&x[32]));
      tc_fence_before();
      mbar_arrive(&sh.s_free[sb]);  // S buffer sb may take the scores of step j+2
      // encode own partial (block floating point) and send it; the own partial stays unrounded
      float am[4] = {0.f, 0.f, 0.f, 0.f};  // independent chains: a 64-long max chain is latency-bound
#pragma unroll
      for (int k = 0; k < 64; k += 2) am[(k >> 1) & 3] = fmax3(am[(k >> 1) & 3], fabsf(x[k]), fabsf(x[k + 1]));
      const float amax = fmaxf(fmaxf(am[0], am[1]), fmaxf(am[2], am[3]));
      const float sl2 = p.scale_log2;
      const int e = block_exponent(amax * sl2);
      if (!kWide) need_wide |= e > kX16MaxExp;
      const float enc = sl2 * pow2i((kWide ? kXFracBits : kXFracBits16) - e);
      const float magic = kWide ? kMagic : kMagic16;
      const uint64_t enc2 = f32x2(enc, enc), magic2 = f32x2(magic, magic);
      // the peer must have read step j-1 (the other set's) out of the buffer before it is overwritten
      if (g >= 1 && !__all_sync(0xffffffffu,
                                mbar_wait_abortable(&sh.x_free[xb_i ^ 1], ((g - 1) / 2) & 1, abort, true, __LINE__))) {
        ok = false;
        break;
      }
      {
        // chunk-major buffer [10 chunks][128 rows][16 B]: a warp's store of one chunk is 512 contiguous
        // bytes.  Chunk c < 8 holds the low 16 bits of mantissas 8c..8c+7; for 20-bit mantissas chunk
        // 8 + c/4, word c%4, holds their top nibbles (byte i: mantissa 8c+i in the low nibble, 8c+i+4
        // in the high one).
        const uint32_t xr = x_remote + r * 16, br = xbar_remote[xb_i];
        uint32_t nib[4];
#pragma unroll
        for (int c = 0; c < kXLoChunks; ++c) {
          uint32_t tb[8], w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int k = 8 * c + 2 * q;
            float t0, t1;
            f32x2_split(fma_x2(f32x2(x[k], x[k + 1]), enc2, magic2), t0, t1);
            tb[2 * q] = __float_as_uint(t0);
            tb[2 * q + 1] = __float_as_uint(t1);
            w[q] = __byte_perm(tb[2 * q], tb[2 * q + 1], 0x5410);
          }
          st_async_v4(xr + c * kXChunk, make_uint4(w[0], w[1], w[2], w[3]), br);
          if (kWide) {
            // bits 16..19 sit in byte 2 of each encoded float (as 0x40 | nibble)
            const uint32_t lo4 = __byte_perm(__byte_perm(tb[0], tb[1], 0x0062), __byte_perm(tb[2], tb[3], 0x6200), 0x7610);
            const uint32_t hi4 = __byte_perm(__byte_perm(tb[4], tb[5], 0x0062), __byte_perm(tb[6], tb[7], 0x6200), 0x7610);
            nib[c & 3] = (lo4 & 0x0F0F0F0Fu) | ((hi4 << 4) & 0xF0F0F0F0u);
            if ((c & 3) == 3)
              st_async_v4(xr + (kXLoChunks + (c >> 2)) * kXChunk, make_uint4(nib[0], nib[1], nib[2], nib[3]), br);
          }
        }
        st_async_b32(e_remote + r * 4, static_cast<uint32_t>(e), br);
      }
      // key mask of this step (past the split end or a slot outside the pool)
      const uint32_t masked0 = __ballot_sync(
          0xffffffffu, kbase + lane >= kend || cur0 < 0 || static_cast<int64_t>(cur0) >= p.pool_slots);
      const uint32_t masked1 = __ballot_sync(
          0xffffffffu, kbase + lane + 32 >= kend || cur1 < 0 || static_cast<int64_t>(cur1) >= p.pool_slots);
      if (!__all_sync(0xffffffffu, mbar_wait_abortable(&sh.x_full[xb_i], (g / kXSets) & 1, abort, true, __LINE__))) {
        ok = false;
        break;
      }
      // s = own * scale_log2 + peer (log2 units)
      float mx = -CUDART_INF_F;
      {
        const uint8_t* xbp = smem + kOffX + r * 16;
        const int pe = *reinterpret_cast<const int*>(smem + kOffE + r * 4);
        // the low 16 bits, as (lo - bias) * 2^(e-f): f = 14, bias 2^15 (16-bit) or f = 18, bias 2^19 (20-bit)
        const float pdec = pow2i(pe - (kWide ? kXFracBits : kXFracBits16)), pm = -(kWide ? kMagic : kMagic16) * pdec;
        const uint64_t pdec2 = f32x2(pdec, pdec), pm2 = f32x2(pm, pm), sl22 = f32x2(sl2, sl2);
#pragma unroll
        for (int c = 0; c < kXLoChunks; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(xbp + c * kXChunk);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int k = 8 * c + 2 * q;
            const uint64_t peer = fma_x2(f32x2(__uint_as_float(__byte_perm(w[q], kMagicHi16, 0x7610)),
                                               __uint_as_float(__byte_perm(w[q], kMagicHi16, 0x7632))),
                                         pdec2, pm2);
            f32x2_split(fma_x2(f32x2(x[k], x[k + 1]), sl22, peer), x[k], x[k + 1]);
          }
        }
        if (kWide) {
          // 20-bit mantissas: add nibble * 2^16 * 2^(e-18)
          const float cs = pow2i(pe - 2), cb = -12582912.0f * cs;  // nibble n as float bits 0x4B4000nn = 1.5 * 2^23 + n
          const uint64_t cs2 = f32x2(cs, cs), cb2 = f32x2(cb, cb);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 nv = *reinterpret_cast<const uint4*>(xbp + (kXLoChunks + h) * kXChunk);
            const uint32_t nw[4] = {nv.x, nv.y, nv.z, nv.w};
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              const int c = 4 * h + cc;
              const uint32_t lo = nw[cc] & 0x0F0F0F0Fu, hi = (nw[cc] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
              for (int i = 0; i < 4; i += 2) {
                // mantissas 8c+i, 8c+i+1 (low nibbles) and 8c+i+4, 8c+i+5 (high nibbles)
                const uint64_t nl = f32x2(__uint_as_float(__byte_perm(lo, 0x4B400000u, 0x7640 + i)),
                                          __uint_as_float(__byte_perm(lo, 0x4B400000u, 0x7641 + i)));
                const uint64_t nh = f32x2(__uint_as_float(__byte_perm(hi, 0x4B400000u, 0x7640 + i)),
                                          __uint_as_float(__byte_perm(hi, 0x4B400000u, 0x7641 + i)));
                const int k = 8 * c + i;
                f32x2_split(add_x2(f32x2(x[k], x[k + 1]), fma_x2(nl, cs2, cb2)), x[k], x[k + 1]);
                f32x2_split(add_x2(f32x2(x[k + 4], x[k + 5]), fma_x2(nh, cs2, cb2)), x[k + 4], x[k + 5]);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_relaxed(xfree_remote[xb_i]);  // this warp's rows of the buffer are read
        if ((masked0 | masked1) != 0u) {
#pragma unroll
          for (int k = 0; k < 64; ++k)
            if (((k < 32 ? masked0 : masked1) >> (k & 31)) & 1u) x[k] = -CUDART_INF_F;
        }
        float mq[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
        for (int k = 0; k < 64; k += 2) mq[(k >> 1) & 3] = fmax3(mq[(k >> 1) & 3], x[k], x[k + 1]);
        mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
      }
      // running max after step g-1 comes from the other set (the wait also keeps that set
      // from overwriting the handoff slot early; a unit's first step starts from -inf)
      if (g > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait_abortable(&sh.m_ready[(g - 1) % 2], ((g - 1) / 2) & 1, abort, false, __LINE__))) {
          ok = false;
          break;
        }
        if (j > 0) m_used = hand[((g - 1) % 2) * kTileRows + r];
      }
      const float m_prev = m_used;
      if (mx > m_used + kRescaleThreshold) m_used = mx;
      hand[sb * kTileRows + r] = m_used;
      mbar_arrive(&sh.m_ready[sb]);
      const float alpha = (m_used == m_prev) ? 1.f : fast_exp2(m_prev - m_used);  // 0 on the first growth
      if (__any_sync(0xffffffffu, alpha != 1.f) && j > 0) {
#ifdef DDT_TEST_HOOKS
        if (lane == 0) atomicAdd(p.status + 1, 1);  // test builds count the lazy O rescales
#endif
        // O must hold every earlier step: wait for P.V of step g-1 (MMAs complete in order)
        if (!__all_sync(0xffffffffu,
                        mbar_wait_abortable(&sh.k_empty[(g - 1) % kStages], ((g - 1) / kStages) & 1, abort, false, __LINE__))) {
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
      if (m_used != m_ref) {
        if (l > 0.f) l *= fast_exp2(m_ref - m_used);
        m_ref = m_used;
      }
      const float msub = (m_used == -CUDART_INF_F) ? 0.f : m_used;
      uint64_t sq[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
      const uint64_t msub2 = f32x2(msub, msub);
      uint32_t pk[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        float d0, d1;
        f32x2_split(sub_x2(f32x2(x[2 * k], x[2 * k + 1]), msub2), d0, d1);
        const float p0 = fast_exp2(d0), p1 = fast_exp2(d1);
        sq[k & 1] = add_x2(sq[k & 1], f32x2(p0, p1));
        pk[k] = pack_bf16x2(p0, p1);
      }
      float s0, s1, s2, s3;
      f32x2_split(sq[0], s0, s1);
      f32x2_split(sq[1], s2, s3);
      l += (s0 + s1) + (s2 + s3);
      // the P buffer was last read by P.V of step g-1
      if (g >= 1) {
        if (!__all_sync(0xffffffffu,
                        mbar_wait_abortable(&sh.k_empty[(g - 1) % kStages], ((g - 1) / kStages) & 1, abort, false, __LINE__))) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      tmem_st32(tmem + lane_off + kColP, pk);
      tc_fence_before();
      mbar_arrive(&sh.p_ready[sb]);
      // P.V(j), issued by the set's first thread once every row of P(j) is in
      // TMEM and, to keep P.V in step order (the lazy rescale of O relies on
      // it), once the other set has issued P.V(j-1).  One commit per group:
      // k_empty[stage] also tells everyone that P.V(j) is done.
      bool pv_ok = true;
      if (lead) {
        pv_ok = mbar_wait_abortable(&sh.p_ready[sb], (g / 2) & 1, abort, false, __LINE__);
        for (uint32_t spin = 0; pv_ok && sh.pv_next != g; ++spin) {
          if (spin > 4 * DDT_WAIT_LIMIT) {
#ifdef DDT_TEST_HOOKS
            atomicCAS(&g_timeout_site, 0u, static_cast<unsigned>(__LINE__));
#endif
            pv_ok = false;
          }
          if ((spin & 255) == 255 && *abort) pv_ok = false;
        }
        if (pv_ok) {
          tc_fence_after();
          const uint64_t dv = desc_advance(d_v, (g % kStages) * kStageBytes);
          const uint32_t pb = tmem + kColP;
#pragma unroll
          for (int ks = 0; ks < kNk / 16; ++ks)
            mma_ts(tmem + kColO, pb + ks * 8, desc_advance(dv, ks * 16 * 128), kIdescPV, (j > 0 || ks > 0) ? 1u : 0u);
          mma_commit(&sh.k_empty[g % kStages]);
          sh.pv_next = g + 1;
        }
      }
      if (!__all_sync(0xffffffffu, pv_ok)) {
        ok = false;
        break;
      }
    }

    if (!kWide && __any_sync(0xffffffffu, need_wide) && lane == 0) sh.need_wide = 1;
    // epilogue: combine both sets' row sums, wait for the last P.V, then
    // o = O / l (set s writes O columns [128 s, 128 s + 128)) and lse.
    // The row state shares the exchange buffer: write it only once both sets
    // are past their last exchange (the other set may still be receiving one).
    if (bar_red_or(kSoftmaxBarrier, 256, !ok)) ok = false;
    fin[(set * 2 + 0) * kTileRows + r] = l;
    fin[(set * 2 + 1) * kTileRows + r] = m_ref;
    bar_sync(kSoftmaxBarrier, 256);
    const float l_o = fin[((set ^ 1) * 2 + 0) * kTileRows + r], m_o = fin[((set ^ 1) * 2 + 1) * kTileRows + r];
    const float m_fin = fmaxf(m_ref, m_o);
    const float lrow = (l > 0.f ? l * fast_exp2(m_ref - m_fin) : 0.f) + (l_o > 0.f ? l_o * fast_exp2(m_o - m_fin) : 0.f);
    if (ok && !mbar_wait_abortable(&sh.k_empty[(G + ntiles - 1) % kStages], ((G + ntiles - 1) / kStages) & 1, abort, false, __LINE__))
      ok = false;
    tc_fence_after();
    if (__all_sync(0xffffffffu, ok)) {
      const int64_t prow = (static_cast<int64_t>(b) * p.max_splits + split) * (p.row_tiles * kTileRows) + grow;
      const float inv_l = lrow > 0.f ? 1.f / lrow : 0.f;
      // A thread holds one row, so storing straight from registers would touch
      // 32 rows (32 lines) per store instruction.  Each warp instead stages a
      // 32-row x 32-column chunk in the stage ring (idle now: every P.V is done)
      // and stores it back as 4 row segments of 128 bytes per instruction.
      uint8_t* stage_w = smem + (warp - 4) * (kTileRows / 4 * 32 * 4);  // 4 KB per softmax warp
      const int row0 = row_tile * kTileRows + (warp & 3) * 32;          // first row of this warp
      const int64_t prow0 = prow - lane;
#pragma unroll 1
      for (int c = 0; c < 128; c += 32) {
        float o[32];
        tmem_ld32(tmem + lane_off + kColO + 128 * set + c, o);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          *reinterpret_cast<float4*>(stage_w + lane * 128 + ((k ^ (lane & 7)) << 4)) =
              make_float4(o[4 * k] * inv_l, o[4 * k + 1] * inv_l, o[4 * k + 2] * inv_l, o[4 * k + 3] * inv_l);
        __syncwarp();
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int rr = 4 * it + (lane >> 3), u = lane & 7;  // row of the warp, 16-byte unit of the chunk
          const float4 v = *reinterpret_cast<const float4*>(stage_w + rr * 128 + ((u ^ (rr & 7)) << 4));
          if (row0 + rr < rows_b)
            *reinterpret_cast<float4*>(p.o_part + (prow0 + rr) * kDv + 256 * rank + 128 * set + c + 4 * u) = v;
        }
        __syncwarp();
      }
      if (rank == 0 && set == 0 && row_valid)
        p.lse_part[prow] = lrow > 0.f ? (m_fin + log2f(lrow)) * kLn2 : -CUDART_INF_F;
    }
  }

  if (warp >= 4 && (warp & 3) == 0 && lane == 0) {
    // the P.V MMAs this thread issued: all complete before TMEM is released (also after a timeout)
    mma_commit(&sh.mma_drain);
    mbar_wait(&sh.mma_drain, pass & 1);
  }
  if (!ok) {
    *abort = 1;
    atomicOr(p.status, kStatusTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (*abort && warp >= 1 && warp < 4 && lane == 0) {
    // after a timeout, bulk copies of unconsumed stages may still be landing:
    // wait for them (bounded) before the shared memory is released
    for (int t = max(G, issued - kStages); t < issued; ++t) mbar_wait(&sh.k_full[t % kStages], (t / kStages) & 1);
  }
  // The pair decides together what comes next: each CTA sends the peer its flag
  // word (kUnitWide: a partial of the 16-bit pass needed more than 16 bits;
  // kUnitAborted: this CTA gave up on a wait).  The unit is rerun with 20-bit
  // mantissas only if some partial needed it and neither CTA aborted; after an
  // abort neither CTA runs another pass (its barriers' phases are unknown).
  if (tid == 0)
    st_shared_cluster_b32(mapa_shared(smem_u32(&sh.peer_need_wide), rank ^ 1u),
                          (kWide ? 0 : sh.need_wide) | (*abort ? kUnitAborted : 0));
  cluster_sync();  // no CTA leaves (or starts another pass) while its peer may still write into its shared memory
  const int flags = (kWide ? 0 : sh.need_wide) | (*abort ? kUnitAborted : 0) | sh.peer_need_wide;
  __syncthreads();  // every thread has read the flags before the next pass resets them
  return flags;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) prefix_pair_kernel(const __grid_constant__ PrefixParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared sh;
  const int tid = threadIdx.x;
  const uint32_t rank = cluster_ctarank();
  // the merge kernel may be scheduled once every CTA of this grid has started:
  // it then occupies only SMs freed by finished CTAs and waits for this grid
  // to complete before it reads the partials
  grid_dep_launch();
  // x: the pair of a 128-row tile, y: the key split.  CTAs are dispatched in
  // x-fastest order, so the pairs of one wave share one or two key ranges:
  // their rows stay in L2 instead of every wave re-reading the whole prefix
  // from HBM.
  const int row_tile = blockIdx.x >> 1;
  const int split = blockIdx.y;
  const int b = blockIdx.z;

  int L = p.prefix_len != nullptr ? __ldg(p.prefix_len + b) : p.max_prefix_len;
  if (L < 0 || L > p.max_prefix_len) {
    if (tid == 0 && rank == 0 && split == 0 && row_tile == 0) atomicOr(p.status, kStatusBadPrefix);
    L = L < 0 ? 0 : p.max_prefix_len;
  }
  const int kbegin = split_begin(split, p.chunk0, p.chunk);
  if (kbegin >= L) return;  // both CTAs of the pair leave together
  // ragged trees: only the rows of the request's first tree_len[b] nodes are computed
  int rows_b = p.rows;
  if (p.tree_len != nullptr) {
    const int tl = __ldg(p.tree_len + b);
    rows_b = (tl < 0 ? 0 : (tl > p.nodes ? p.nodes : tl)) * p.heads;  // out-of-range values: the merge reports them
  }
  if (row_tile * kTileRows >= rows_b) return;  // a tile of inactive rows: both CTAs leave together
  const int kend = split_end(split, p.chunk0, p.chunk, L);
  // 16-bit exchange first; the rare unit whose partial scores are too large for
  // it (both CTAs get the same answer) is computed again with 20-bit mantissas
  // and its partial result overwritten
  // TMEM is allocated once for both passes (after relinquishing the allocation
  // permit a CTA may not allocate again); each pass's MMAs have drained before
  // it returns.
  const int warp = tid >> 5;
  if (warp == 0) {
    tmem_alloc(&sh.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) init_barriers(sh);
  if (run_unit<false>(p, sh, smem_raw, row_tile, split, b, kbegin, kend, rows_b, 0, 0) == kUnitWide) {
#ifdef DDT_TEST_HOOKS
    if (tid == 0 && rank == 0) atomicAdd(p.status + 2, 1);  // test builds count the 20-bit reruns
#endif
    run_unit<true>(p, sh, smem_raw, row_tile, split, b, kbegin, kend, rows_b, (kend - kbegin + kNk - 1) / kNk, 1);
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(sh.tmem_base, kTmemCols);
  }
}

// The prefix pass by key-range groups (schedule.cuh): the pair (row tile
// blockIdx.x / 2, group blockIdx.y) computes its row tile over the group's
// steps, one unit per request that they touch, back to back on the same
// barriers (their phases run on: the CTA's steps G and passes count across
// units).  A unit's partial goes to its piece's split slot of the request.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) prefix_group_kernel(const __grid_constant__ PrefixParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  grid_dep_launch();  // as in prefix_pair_kernel
  const int row_tile = blockIdx.x >> 1;
  if (warp == 0) {
    tmem_alloc(&sh.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) init_barriers(sh);
  int G = 0, pass = 0;
  for (int idx = 0;; ++idx) {
    // the step table is rebuilt for each unit (two loads and a few shuffles per
    // warp) instead of being held in registers across the unit
    int b, kbegin, kend, piece;
    {
      const StepTable st = step_table(p.prefix_len, p.max_prefix_len, p.batch, lane);
      if (idx == 0 && st.bad && blockIdx.y == 0 && row_tile == 0 && rank == 0 && tid == 0)
        atomicOr(p.status, kStatusBadPrefix);
      if (!nth_group_unit(
              blockIdx.y, p.groups, st.total, p.batch, idx, [&](int r) { return st.off(r); },
              [&](int r) { return st.steps(r); }, [&](int r) { return st.keys(r); }, &b, &kbegin, &kend, &piece))
        break;
    }
    int rows_b = p.rows;
    if (p.tree_len != nullptr) {
      const int tl = __ldg(p.tree_len + b);
      rows_b = (tl < 0 ? 0 : (tl > p.nodes ? p.nodes : tl)) * p.heads;  // out-of-range values: the merge reports them
    }
    if (row_tile * kTileRows >= rows_b) continue;  // inactive rows: both CTAs skip the unit
    const int ntiles = (kend - kbegin + kNk - 1) / kNk;
    int flags = run_unit<false>(p, sh, smem_raw, row_tile, piece, b, kbegin, kend, rows_b, G, pass);
    G += ntiles;
    ++pass;
    if (flags == kUnitWide) {
#ifdef DDT_TEST_HOOKS
      if (tid == 0 && rank == 0) atomicAdd(p.status + 2, 1);  // test builds count the 20-bit reruns
#endif
      flags = run_unit<true>(p, sh, smem_raw, row_tile, piece, b, kbegin, kend, rows_b, G, pass);
      G += ntiles;
      ++pass;
    }
    if (flags & kUnitAborted) break;  // both CTAs of the pair stop (the status word says TIMEOUT)
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(sh.tmem_base, kTmemCols);
  }
}

// Fused kernel: merge the rows of one (request, row tile): the tree tail of
// each row and the log-sum-exp merge with the request's nsplit prefix partials.
// Rank r of the pair takes rows [64 r, 64 r + 64) of the tile, a warp every
// 12th of them; rows of inactive nodes (ragged trees) get out = 0, lse = -inf.
// The stage ring is idle between units: it holds the request's parent and slot
// arrays, all its tree rows (T x 1152 B) and, per node of this CTA's rows, the
// list of its visible tree nodes, so a row's tail reads shared memory only.
__device__ __noinline__ void merge_tile(const FusedParams& f, uint8_t* smem, int b, int tile, int nsplit,
                                        int rows_b) {
  const PrefixParams& p = f.pre;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int T = p.nodes, H = p.heads;
  const int tile_rows = min(kTileRows, T * H - tile * kTileRows);
  const int i_beg = static_cast<int>(rank) * 64, i_end = min(i_beg + 64, tile_rows);
  if (i_beg >= i_end) return;
  const int r_beg = tile * kTileRows + i_beg, r_end = tile * kTileRows + i_end;  // rows of the request
  const int n_beg = r_beg / H, n_cnt = (r_end - 1) / H - n_beg + 1;              // their nodes (<= 64)
  uint8_t* rows_sh = smem;                                                       // [T][1152]
  int* par_sh = reinterpret_cast<int*>(smem + kMaxNodes * kRowBytes);            // [T]
  int* tslot_sh = par_sh + kMaxNodes;                                            // [T]
  int* nvis_sh = tslot_sh + kMaxNodes;                                           // [n_cnt]
  int* vis_sh = nvis_sh + 64;                                                    // [n_cnt][T] node lists
  static_assert(kMaxNodes * kRowBytes + (3 * kMaxNodes + 64 + 64 * kMaxNodes) * 4 <= kStages * kStageBytes,
                "the merge's staging fits in the stage ring");
  const int32_t* par = f.tree_parent + static_cast<int64_t>(b) * T;
  const int32_t* tslot = f.tree_slot_idx + static_cast<int64_t>(b) * T;
  for (int u = tid; u < T; u += kThreads) {
    par_sh[u] = __ldg(par + u);
    tslot_sh[u] = __ldg(tslot + u);
  }
  __syncthreads();
  // the request's tree rows (rows of out-of-pool slots are never read: the walk leaves them out)
  for (int i = tid; i < T * kChunks; i += kThreads) {
    const int u = i / kChunks, c = i - u * kChunks;
    const int32_t slot = tslot_sh[u];
    if (slot >= 0 && static_cast<int64_t>(slot) < p.pool_slots)
      reinterpret_cast<uint4*>(rows_sh + u * kRowBytes)[c] =
          __ldg(reinterpret_cast<const uint4*>(p.kv + static_cast<int64_t>(slot) * kDqk) + c);
  }
  // one thread per node: its visible nodes (itself, its parent, ..., the root)
  if (tid < n_cnt) {
    const int t = n_beg + tid;
    int32_t st = 0;
    int* list = vis_sh + tid * kMaxNodes;
    int n = 0, u = t;
    for (int guard = 0; u >= 0 && guard < T; ++guard) {
      const int32_t slot = tslot_sh[u];
      if (slot >= 0 && static_cast<int64_t>(slot) < p.pool_slots)
        list[n++] = u;
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
    nvis_sh[tid] = n;
    if (st && t * H < rows_b) atomicOr(p.status, st);
  }
  __syncthreads();
  const int64_t pstride = static_cast<int64_t>(p.row_tiles) * kTileRows;
  const MergeRowArgs a{p.q, p.scale_log2, p.o_part, p.lse_part, pstride, f.out, f.lse};
  for (int r = r_beg + warp; r < r_end; r += kThreads / 32) {
    const int t = r / H;
    const int64_t grow = static_cast<int64_t>(b) * T * H + r;
    if (r >= rows_b) {
      write_inactive_row(f.out, f.lse, grow, lane);
      continue;
    }
    const int* list = vis_sh + (t - n_beg) * kMaxNodes;
    merge_row<false>(a, grow, static_cast<int64_t>(b) * p.max_splits * pstride + r, nsplit, nvis_sh[t - n_beg],
                     [&](int v) { return reinterpret_cast<const uint32_t*>(rows_sh + list[v] * kRowBytes); }, lane);
  }
}

// One launch per verify call.  A persistent grid of CTA pairs claims the units
// (request b, key split, 128-row tile), tile fastest, from a counter, so pairs
// whose units end early (or are empty: splits past a shorter prefix) take more.
// A unit is one run_unit (the 16-bit pass, rerun with 20-bit
// mantissas where needed) writing its normalised partial; then rank 0 counts
// the split in the workspace (release: fence, then atomic add) and the pair
// that completes a (request, row tile) merges its rows (acquire: fence before
// the reads, which go through L2).  Nothing waits on another pair, so no unit
// order or residency can stall the grid.  A tile with no prefix keys (empty
// prefix) or no active row (ragged trees) is merged, or zeroed, by its split-0
// unit.  The merge reads the splits in order, so results do not depend on which
// pair merges, and are the same bits as the two-kernel path's.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) verify_fused_kernel(const __grid_constant__ FusedParams f) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared sh;
  const PrefixParams& p = f.pre;
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (warp == 0) {
    tmem_alloc(&sh.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) init_barriers(sh);
  int G = 0, pass = 0;  // the CTA's steps and passes so far (barrier phases run on across units)
  for (int it = 0;; ++it) {
    // Rank 0 claims the next unit for the pair (a counter in the status words,
    // zero at launch) and hands it to rank 1 through its shared memory.  Claims
    // alternate between two slots: a slot is rewritten two claims later, past a
    // cluster barrier that every thread reaches only after reading it.
    if (rank == 0 && tid == 0) {
      const int claimed = atomicAdd(p.status + 3, 1);
      sh.unit[it & 1] = claimed;
      st_shared_cluster_b32(mapa_shared(smem_u32(&sh.unit[it & 1]), 1u), claimed);
    }
    cluster_sync();
    const int u = sh.unit[it & 1];
    if (u >= f.units) break;
    // units in request, key split, row tile order (tile fastest): the pairs at work at one time
    // share one or two key ranges, whose rows stay in L2
    const int tile = u % p.row_tiles;
    const int split = (u / p.row_tiles) % f.splits;
    const int b = u / (p.row_tiles * f.splits);
    const bool first = split == 0 && tile == 0 && rank == 0 && tid == 0;  // reports the request's status bits
    int L = p.prefix_len != nullptr ? __ldg(p.prefix_len + b) : p.max_prefix_len;
    if (L < 0 || L > p.max_prefix_len) {
      if (first) atomicOr(p.status, kStatusBadPrefix);
      L = L < 0 ? 0 : p.max_prefix_len;
    }
    int rows_b = p.rows;
    if (p.tree_len != nullptr) {
      int tl = __ldg(p.tree_len + b);
      if (tl < 0 || tl > p.nodes) {
        if (first) atomicOr(p.status, kStatusBadTreeLen);
        tl = tl < 0 ? 0 : p.nodes;
      }
      rows_b = tl * p.heads;
    }
    const int nsplit = split_count(L, p.chunk0, p.chunk);
    if (tile * kTileRows >= rows_b || nsplit == 0) {
      if (split == 0) merge_tile(f, smem, b, tile, 0, rows_b);  // tree tail only, or inactive rows
      __syncthreads();
      continue;
    }
    if (split >= nsplit) continue;
    const int kbegin = split_begin(split, p.chunk0, p.chunk), kend = split_end(split, p.chunk0, p.chunk, L);
    const int ntiles = (kend - kbegin + kNk - 1) / kNk;
    int flags = run_unit<false>(p, sh, smem_raw, tile, split, b, kbegin, kend, rows_b, G, pass);
    G += ntiles;
    ++pass;
    if (flags == kUnitWide) {
#ifdef DDT_TEST_HOOKS
      if (tid == 0 && rank == 0) atomicAdd(p.status + 2, 1);  // test builds count the 20-bit reruns
#endif
      flags = run_unit<true>(p, sh, smem_raw, tile, split, b, kbegin, kend, rows_b, G, pass);
      G += ntiles;
      ++pass;
    }
    if (flags & kUnitAborted) break;  // both CTAs of the pair stop (the status word says TIMEOUT)
    // both CTAs' partials are written (run_unit ended with a cluster barrier)
    if (rank == 0 && tid == 0) {
      __threadfence();
      const int last = atomicAdd(f.arrivals + static_cast<int64_t>(b) * p.row_tiles + tile, 1) == nsplit - 1;
      sh.last_arrival = last;
      st_shared_cluster_b32(mapa_shared(smem_u32(&sh.last_arrival), 1u), last);
    }
    cluster_sync();
    if (sh.last_arrival) {
      __threadfence();
      merge_tile(f, smem, b, tile, nsplit, rows_b);
    }
    __syncthreads();  // every thread has read last_arrival and left the ring before the next unit
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(sh.tmem_base, kTmemCols);
  }
}

}  // namespace

namespace {
int g_fused_pairs[64];  // co-resident pairs per device, found once by configure_prefix
}

cudaError_t configure_prefix() {
  cudaError_t e = cudaFuncSetAttribute(prefix_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(prefix_group_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(verify_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem)) != cudaSuccess)
    return e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, verify_fused_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();  // clear it: the planner then falls back to the SM count
    n = 0;
  }
  if (dev >= 0 && dev < 64) g_fused_pairs[dev] = n;
  return cudaSuccess;
}

int fused_max_pairs() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  return g_fused_pairs[dev];
}

cudaError_t launch_fused(const FusedParams& p, int pairs, cudaStream_t stream) {
  verify_fused_kernel<<<dim3(2 * pairs), kThreads, kSmem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_prefix(const PrefixParams& p, int batch, int splits, cudaStream_t stream) {
  if (p.groups > 0) {
    prefix_group_kernel<<<dim3(2 * p.row_tiles, p.groups, 1), kThreads, kSmem, stream>>>(p);
  } else {
    prefix_pair_kernel<<<dim3(2 * p.row_tiles, splits, batch), kThreads, kSmem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace ddt

#ifdef DDT_TEST_HOOKS
// Test builds only (not part of the public header).
extern "C" __attribute__((visibility("default"))) unsigned ddtree_test_timeout_site() {
  unsigned v = 0;
  return cudaMemcpyFromSymbol(&v, ddt::g_timeout_site, sizeof v) == cudaSuccess ? v : 0xFFFFFFFFu;
}
extern "C" __attribute__((visibility("default"))) void ddtree_test_clear_timeout_site() {
  const unsigned z = 0;
  cudaMemcpyToSymbol(ddt::g_timeout_site, &z, sizeof z);
}
extern "C" __attribute__((visibility("default"))) int ddtree_test_fused_pairs() { return ddt::fused_max_pairs(); }
#endif
