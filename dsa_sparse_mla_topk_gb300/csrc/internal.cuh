// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa.h"

namespace dsa {

// Kernel launchers (each returns the launch's cudaError_t).
cudaError_t launch_topk(const float* scores, int64_t ld, const int32_t* q_pos, int32_t num_q, int32_t k,
                        int32_t* idx, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        cudaStream_t stream);
// Workspace bytes the sliced top-k of rows longer than 65,536 positions uses
// (0 when it does not apply).
size_t topk_workspace_bytes(int32_t num_q, int64_t ld, int32_t k);
// CTAs per top-k row (a thread-block cluster) for this launch.
int topk_cluster_size(int32_t num_q, int64_t ld, int num_sms);

// The page lookup of the attention call folded into the top-k's write: for
// every selected position its cache slot and dequantisation scale, as the
// attention kernel reads them (slot -1 and scale 0 for padding and for bad
// entries, which are reported as the attention call reports them).
struct TopkResolve {
  int2* res;  // [num_q, k]: (slot, scale bits)
  const int32_t* block_table;
  const int32_t* q_req;
  const float* kv_scale;
  int64_t num_pages;
  int32_t num_req, bt_stride, page_size;
};
// Top-k of rows of at most 65,536 positions (ld <= 65,536) that also writes
// rv.res; idx is written as launch_topk writes it.
cudaError_t launch_topk_resolve(const float* scores, int64_t ld, const int32_t* q_pos, int32_t num_q, int32_t k,
                                int32_t* idx, const TopkResolve& rv, int32_t* dev_status, cudaStream_t stream);

// SM count of the current device (cached per device).
int device_sm_count();

struct MlaArgs {
  const void* q;
  const uint8_t* kv;
  const float* kv_scale;
  int64_t num_pages;
  const int32_t* block_table;
  int32_t num_req;
  int32_t bt_stride;
  const int32_t* q_req;
  const int32_t* idx;
  int32_t num_q, heads, d_latent, d_rope, page_size, k;
  float softmax_scale;
  int32_t num_splits;
  void* out;
  float* lse;
  float* o_part;
  float* lse_part;
  int32_t* dev_status;
};

cudaError_t launch_mla_simt(const MlaArgs& a, cudaStream_t stream);

// Tensor-core (tcgen05) version for (heads, d_latent, d_rope) = (64, 512, 64).
// It first resolves every selected position into (slot, scale) in
// `workspace` (mla_tc_workspace_bytes), then runs the attention kernel.
bool mla_tc_supported(const MlaArgs& a);
size_t mla_tc_workspace_bytes(int32_t num_q, int32_t k);
cudaError_t launch_mla_tc(const MlaArgs& a, void* workspace, cudaStream_t stream);
// The attention kernel alone, over entries launch_topk_resolve has just
// written into `workspace` on the same stream (a programmatic dependent of
// that top-k launch).
cudaError_t launch_mla_tc_resolved(const MlaArgs& a, void* workspace, cudaStream_t stream);
// Fused decode path: top-k of each token's scores row, then attention over
// it, one CTA per token (one KV split; rows of at most 65,536 positions; k at
// most mla_tc_fused_max_k()); `workspace` as for launch_mla_tc.
int mla_tc_fused_max_k();
cudaError_t launch_mla_tc_fused(const MlaArgs& a, const float* scores, int64_t ld, const int32_t* q_pos, int32_t* idx,
                                void* workspace, cudaStream_t stream);

// KV cache write: FP8 E4M3 per-token quantisation + paged scatter (rows of up
// to kv_write_max_d() values, a multiple of 16).
int kv_write_max_d();
cudaError_t launch_kv_write(const void* rows, int32_t n, int32_t d, const int32_t* req, const int32_t* pos,
                            const int32_t* block_table, int32_t num_req, int32_t bt_stride, int32_t page_size,
                            int64_t num_pages, uint8_t* kv, float* kv_scale, int32_t* status, cudaStream_t stream);

cudaError_t launch_combine(const float* o_part, const float* lse_part, int32_t num_splits, int32_t num_q,
                           int32_t heads, int32_t d_v, void* out, float* lse, cudaStream_t stream);

// Report a data-dependent error without trapping.
__device__ __forceinline__ void report(int32_t* status, uint32_t bit) {
  if (status) atomicOr(reinterpret_cast<unsigned int*>(status), bit);
}

}  // namespace dsa
