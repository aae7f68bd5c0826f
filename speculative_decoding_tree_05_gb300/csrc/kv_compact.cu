// kv_compact.cu -- defragment each request's prefix rows into consecutive slots.
//
// With page_size=1 slots, a churned free list hands a long request scattered
// slots ("The Architecture Detective: Uncovering FlashMLA's Potential for
// Blackwell DDTree Verification", section "Defragmentation: Separating Signal
// from Noise").  This pass copies request b's prefix rows to
// dst_start[b] + j and rewrites the slot table, so later verify steps read
// contiguous memory.  A plain bit-exact copy: one thread per 16-byte chunk of a
// 1152-byte row, the chunk-0 thread also writes the new slot index.
#include <cuda_runtime.h>
#include "kernels.cuh"

namespace ddt {
namespace {

constexpr int kCompactThreads = 256;

__global__ void __launch_bounds__(kCompactThreads) kv_compact_kernel(CompactParams p) {
  const int b = blockIdx.y;
  int L = __ldg(p.prefix_len + b);
  if (L < 0 || L > p.max_prefix_len) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.status, kStatusBadPrefix);
    L = L < 0 ? 0 : p.max_prefix_len;
  }
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * kCompactThreads + threadIdx.x;
  const int64_t j = idx / kChunks;
  const int c = static_cast<int>(idx - j * kChunks);
  if (j >= L) return;
  const int64_t from = __ldg(p.slot_idx + static_cast<int64_t>(b) * p.slot_stride + j);
  const int64_t to = __ldg(p.dst_start + b) + j;
  if (from < 0 || from >= p.pool_slots || to < 0 || to >= p.pool_slots) {
    if (c == 0) atomicOr(p.status, kStatusBadSlot);
    return;
  }
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p.src + from * kDqk) + c);
  reinterpret_cast<uint4*>(p.dst + to * kDqk)[c] = v;
  if (c == 0) p.slot_idx_out[static_cast<int64_t>(b) * p.slot_stride + j] = static_cast<int32_t>(to);
}

}  // namespace

cudaError_t launch_kv_compact(const CompactParams& p, int batch, cudaStream_t stream) {
  const int64_t work = static_cast<int64_t>(p.max_prefix_len) * kChunks;
  if (batch == 0 || work == 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>((work + kCompactThreads - 1) / kCompactThreads), batch);
  kv_compact_kernel<<<grid, kCompactThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ddt
