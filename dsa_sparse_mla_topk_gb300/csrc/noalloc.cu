// dsa_sparse_mla_fwd_noalloc: the tensor-core attention call for callers
// that cannot hand the library a scratch buffer.
//
// Some callers are not allowed to allocate device memory when they run the
// attention step: a serving loop that reserves all device memory at start-up
// and forbids later allocations (cudaMalloc can synchronise the device and
// stall every other stream), or a host application that calls this library
// from a plug-in interface that offers no allocator.  This entry point keeps
// its scratch -- the resolved (slot, scale) of every selected position -- in a
// fixed array of device memory that is part of the library image, so the
// call itself allocates nothing.
//
// Limits and sharing:
//  * The array holds kNoallocScratchBytes (24 MiB).  A call needs
//    dsa_sparse_mla_workspace_size() bytes of it -- 8 bytes per selected
//    entry, e.g. 16 MiB for 1024 query tokens at top-k 2048; calls that need
//    more are rejected with
//    DSA_ERR_WORKSPACE_TOO_SMALL before anything is launched.
//  * Every GPU that loads the library holds its own copy of the array until
//    the process exits.
//  * All calls share the array.  Two calls whose work overlaps on the GPU
//    (different streams without ordering between them, or different host
//    threads) race on it and may produce wrong results; serialise them.
//  * Nothing in the array needs clearing: every call rewrites the entries it
//    uses before reading them.
//  * The device address of the array is looked up once per device, with that
//    device current, on the first call made while it is the current device.
//    Make that first call before starting any stream capture on the device.
//  * That address is kept for the life of the process.  A device reset
//    (cudaDeviceReset, or a reset of the primary context) reloads the library
//    image and moves the array, so this entry point must not be used after
//    one.
#include <cuda_runtime.h>

#include <mutex>

#include "dsa.h"
#include "internal.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(24) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once
// per device); nullptr if the lookup failed.
void* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" DSA_API dsa_status dsa_sparse_mla_fwd_noalloc(
    const void* q, const uint8_t* kv, const float* kv_scale, int64_t num_pages, const int32_t* block_table,
    int32_t num_req, int32_t bt_stride, const int32_t* q_req, const int32_t* idx, int32_t num_q, int32_t num_heads,
    int32_t d_latent, int32_t d_rope, int32_t page_size, int32_t k, float softmax_scale, int32_t num_splits,
    void* out, float* lse, float* o_part, float* lse_part, int32_t* dev_status, void* stream) {
  if (num_q < 0 || k <= 0) return DSA_ERR_INVALID_ARG;
  if (num_heads != 64 || d_latent != 512 || d_rope != 64) return DSA_ERR_UNSUPPORTED_SHAPE;
  if (num_q == 0) return DSA_OK;
  const size_t need = dsa_sparse_mla_workspace_size(num_q, num_heads, d_latent, d_rope, k);
  if (need > kNoallocScratchBytes) return DSA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = scratch_on_current_device();
  if (!scratch) return DSA_ERR_CUDA;
  // Everything else (argument checks, the resolve and attention kernels) is
  // the regular entry point, pointed at the fixed array.
  return dsa_sparse_mla_fwd(q, kv, kv_scale, num_pages, block_table, num_req, bt_stride, q_req, idx, num_q, num_heads,
                            d_latent, d_rope, page_size, k, softmax_scale, num_splits, out, lse, o_part, lse_part,
                            scratch, kNoallocScratchBytes, dev_status, stream);
}
