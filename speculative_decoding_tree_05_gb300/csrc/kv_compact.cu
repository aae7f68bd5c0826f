// kv_compact.cu -- defragment each request's prefix rows into consecutive slots.
//
// With page_size=1 slots, a churned free list hands a long request scattered
// slots ("The Architecture Detective: Uncovering FlashMLA's Potential for
// Blackwell DDTree Verification", section "Defragmentation: Separating Signal
// from Noise").  This pass copies request b's prefix rows to
// dst_start[b] + j and rewrites the slot table, so later verify steps read
// contiguous memory.  A plain bit-exact copy in 16-byte chunks (72 per 1152-byte
// row, consecutive threads on consecutive chunks of a row); the chunk-0 thread
// also writes the new slot index.
#include <cuda_runtime.h>
#include "kernels.cuh"

namespace ddt {
namespace {

constexpr int kCompactThreads = 256;
constexpr int kChunksPerThread = 4;  // independent 16-byte copies in flight per thread
constexpr int kCompactBlocksPerSm = 8;

// Grid-stride over the (row, chunk) pairs of request blockIdx.y; each pass a
// thread loads 4 chunks 256 apart before storing any, so 4 loads are in flight.
__global__ void __launch_bounds__(kCompactThreads) kv_compact_kernel(CompactParams p) {
  const int b = blockIdx.y;
  int L = __ldg(p.prefix_len + b);
  if (L < 0 || L > p.max_prefix_len) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.status, kStatusBadPrefix);
    L = L < 0 ? 0 : p.max_prefix_len;
  }
  const int64_t total = static_cast<int64_t>(L) * kChunks;
  const int64_t dst0 = __ldg(p.dst_start + b);
  const int32_t* slots = p.slot_idx + static_cast<int64_t>(b) * p.slot_stride;
  const int64_t span = static_cast<int64_t>(gridDim.x) * kCompactThreads * kChunksPerThread;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * kCompactThreads * kChunksPerThread + threadIdx.x;
       base < total; base += span) {
    uint4 v[kChunksPerThread];
    int64_t to[kChunksPerThread];
    bool live[kChunksPerThread];
#pragma unroll
    for (int u = 0; u < kChunksPerThread; ++u) {
      const int64_t idx = base + u * kCompactThreads;
      const int64_t j = idx / kChunks;
      const int c = static_cast<int>(idx - j * kChunks);
      live[u] = false;
      to[u] = -1;
      if (idx >= total) continue;
      const int64_t from = __ldg(slots + j);
      const int64_t dst = dst0 + j;
      if (from < 0 || from >= p.pool_slots || dst < 0 || dst >= p.pool_slots) {
        if (c == 0) atomicOr(p.status, kStatusBadSlot);
        continue;
      }
      v[u] = __ldg(reinterpret_cast<const uint4*>(p.src + from * kDqk) + c);
      to[u] = dst * kDqk * 2 + c * 16;  // byte offset of the chunk in dst
      live[u] = true;
      if (c == 0) p.slot_idx_out[static_cast<int64_t>(b) * p.slot_stride + j] = static_cast<int32_t>(dst);
    }
#pragma unroll
    for (int u = 0; u < kChunksPerThread; ++u)
      if (live[u]) *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.dst) + to[u]) = v[u];
  }
}

}  // namespace

cudaError_t launch_kv_compact(const CompactParams& p, int batch, cudaStream_t stream) {
  const int64_t work = static_cast<int64_t>(p.max_prefix_len) * kChunks;
  if (batch == 0 || work == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorUnknown;
  // enough blocks over all requests to fill the GPU, none idle for the longest request
  const int64_t per_block = static_cast<int64_t>(kCompactThreads) * kChunksPerThread;
  const int64_t need = (work + per_block - 1) / per_block;
  const int64_t fill = (static_cast<int64_t>(sms) * kCompactBlocksPerSm + batch - 1) / batch;
  dim3 grid(static_cast<unsigned>(need < fill ? need : fill), batch);
  kv_compact_kernel<<<grid, kCompactThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ddt
