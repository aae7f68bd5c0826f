// static_scratch.cu -- verify attention for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run verify
// attention: code inside a custom allocator or memory-pool callback, plugins
// that are handed fixed buffers by a host framework and may not grow its
// footprint, or launch paths that must not take the allocator's locks.  For
// them this file keeps the per-call scratch (the status word and the key-split
// partial results) in a fixed device array that is part of the library image,
// so the call itself allocates nothing.
//
// The array is kStaticScratchBytes (32 MiB).  Every GPU that loads the library
// holds it until the process exits.  Sizes whose scratch would not fit are
// rejected with DDT_ERR_WORKSPACE before anything is enqueued.
#include <cuda_runtime.h>
#include <mutex>
#include "../../include/ddtree.h"

namespace ddt {
int verify_precheck(const ddt_dims* dims, size_t* workspace_bytes);  // api.cu
namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;
constexpr int kMaxScratchDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch on each device.  In host code the array's
// name is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress, taken once per device with that device current.
void* g_scratch_ptr[kMaxScratchDevices];
cudaError_t g_scratch_err[kMaxScratchDevices];
std::once_flag g_scratch_once[kMaxScratchDevices];

int static_scratch(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) return DDT_ERR_DEVICE;
  std::call_once(g_scratch_once[dev], [dev] {
    void* p = nullptr;
    g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_static_scratch);
    g_scratch_ptr[dev] = p;
  });
  if (g_scratch_err[dev] != cudaSuccess || g_scratch_ptr[dev] == nullptr) return DDT_ERR_LAUNCH;
  *ptr = g_scratch_ptr[dev];
  return DDT_OK;
}

}  // namespace
}  // namespace ddt

extern "C" int ddtree_verify_attn_static_scratch(const void* q, const void* kv_pool, const int32_t* slot_idx,
                                                 const int32_t* prefix_len, const int32_t* tree_parent,
                                                 const int32_t* tree_slot_idx, float sm_scale, float* out,
                                                 float* lse, const ddt_dims* dims, ddt_stream_t stream) {
  size_t need = 0;
  int rc = ddt::verify_precheck(dims, &need);  // the size and device checks of ddtree_verify_attn, same codes
  if (rc != DDT_OK) return rc;
  if (dims->batch == 0) return DDT_OK;
  if (need > ddt::kStaticScratchBytes) return DDT_ERR_WORKSPACE;
  void* scratch = nullptr;
  rc = ddt::static_scratch(&scratch);
  if (rc != DDT_OK) return rc;
  return ddtree_verify_attn(q, kv_pool, slot_idx, prefix_len, tree_parent, tree_slot_idx, sm_scale, out, lse, dims,
                            scratch, ddt::kStaticScratchBytes, stream);
}
