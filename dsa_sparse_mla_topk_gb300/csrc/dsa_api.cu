// C ABI of the library: argument checks, planning helpers and launches.
#include <cuda_runtime.h>
#include <math.h>

#include "dsa.h"
#include "internal.cuh"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_shape(int32_t h, int32_t dl, int32_t dr) {
  return (h == 16 && dl == 64 && dr == 16) || (h == 64 && dl == 512 && dr == 64);
}

dsa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA; }

// The 64-head shape runs on the tensor cores, the 16-head shape on the CUDA
// cores; nothing else changes that choice.
bool use_tensor_cores(int32_t h, int32_t dl, int32_t dr) { return h == 64 && dl == 512 && dr == 64; }

}  // namespace

namespace dsa {
int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  if (dev < 64) cached[dev] = n;
  return n;
}
}  // namespace dsa

extern "C" {

const char* dsa_status_string(int32_t status) {
  switch (status) {
    case DSA_OK: return "ok";
    case DSA_ERR_INVALID_ARG: return "invalid argument";
    case DSA_ERR_UNSUPPORTED_SHAPE: return "unsupported (heads, d_latent, d_rope)";
    case DSA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case DSA_ERR_CUDA: return "CUDA error";
    case DSA_ERR_OUT_OF_PAGES: return "page pool exhausted";
    default: return "unknown status";
  }
}

int32_t dsa_version(void) { return 100; }

int32_t dsa_kv_tile_count(int32_t width, int32_t tile) {
  if (width < 0 || tile <= 0) return -1;
  return (int32_t)(((int64_t)width + tile - 1) / tile);
}

int32_t dsa_kv_tile_size(int32_t num_heads, int32_t d_latent, int32_t d_rope) {
  if (!supported_shape(num_heads, d_latent, d_rope)) return -1;
  return num_heads == 64 ? 64 : 32;  // tensor-core kernel: 64-row tiles; CUDA-core kernel: 32
}

int32_t dsa_pick_num_splits(int32_t num_q, int32_t num_heads, int32_t d_latent, int32_t d_rope, int32_t k,
                            int32_t num_sms) {
  const int32_t tile = dsa_kv_tile_size(num_heads, d_latent, d_rope);
  if (tile <= 0 || num_q <= 0 || k <= 0) return 1;
  if (num_sms <= 0) num_sms = dsa::device_sm_count();
  // query tokens alone fill the GPU: no split (no partials, no combine)
  if (num_q >= num_sms) return 1;
  // One CTA per SM (shared memory bound); a launch takes ceil(CTAs / SMs)
  // waves of ceil(tiles / S) tiles each, plus a fixed per-CTA cost (start-up,
  // pipeline fill, epilogue: about four 64-row tiles on the tensor-core
  // kernel, two 32-row tiles on the CUDA-core one) and one tile more for the
  // Combine when split.
  const int32_t ntiles = dsa_kv_tile_count(k, tile);
  const int64_t fixed = tile == 64 ? 4 : 2;
  int32_t best = 1;
  int64_t best_cost = -1;
  for (int32_t s = 1; s <= 64 && s <= ntiles; ++s) {
    const int64_t waves = ((int64_t)num_q * s + num_sms - 1) / num_sms;
    const int64_t per = (ntiles + s - 1) / s;
    const int64_t cost = waves * (per + fixed) + (s > 1 ? 1 : 0);
    if (best_cost < 0 || cost < best_cost) best = s, best_cost = cost;
  }
  return best;
}

size_t dsa_sparse_mla_workspace_size(int32_t num_q, int32_t num_heads, int32_t d_latent, int32_t d_rope,
                                     int32_t k) {
  if (num_q <= 0 || k <= 0 || !use_tensor_cores(num_heads, d_latent, d_rope)) return 0;
  return dsa::mla_tc_workspace_bytes(num_q, k);
}

size_t dsa_topk_workspace_size(int32_t num_q, int64_t ld_scores, int32_t k) {
  return dsa::topk_workspace_bytes(num_q, ld_scores, k);
}

dsa_status dsa_topk_select(const float* scores, int64_t ld_scores, const int32_t* q_pos, int32_t num_q,
                           int32_t k, int32_t* idx, void* workspace, size_t workspace_bytes,
                           int32_t* dev_status, void* stream) {
  if (num_q < 0 || k <= 0 || ld_scores <= 0) return DSA_ERR_INVALID_ARG;
  if (num_q == 0) return DSA_OK;
  if (!scores || !q_pos || !idx) return DSA_ERR_INVALID_ARG;
  // the workspace is optional: none selects the in-place path; a partial one is an error
  const size_t need = dsa_topk_workspace_size(num_q, ld_scores, k);
  if (workspace_bytes > 0 && workspace_bytes < need) return DSA_ERR_WORKSPACE_TOO_SMALL;
  if (workspace_bytes > 0 && !workspace) return DSA_ERR_INVALID_ARG;
  return from_cuda(dsa::launch_topk(scores, ld_scores, q_pos, num_q, k, idx, workspace, workspace_bytes,
                                    dev_status, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// Argument checks shared by the attention entry points; fills `a` when they pass.
dsa_status check_mla_args(const void* q, const uint8_t* kv, const float* kv_scale, int64_t num_pages,
                          const int32_t* block_table, int32_t num_req, int32_t bt_stride, const int32_t* q_req,
                          const int32_t* idx, int32_t num_q, int32_t num_heads, int32_t d_latent, int32_t d_rope,
                          int32_t page_size, int32_t k, float softmax_scale, int32_t num_splits, void* out,
                          float* lse, float* o_part, float* lse_part, size_t ws_need, void* workspace,
                          size_t workspace_bytes, int32_t* dev_status, dsa::MlaArgs* a) {
  if (num_q < 0 || k <= 0 || page_size <= 0 || num_pages <= 0 || num_req <= 0 || bt_stride <= 0)
    return DSA_ERR_INVALID_ARG;
  if (num_splits < 1 || num_splits > 64 || !isfinite(softmax_scale)) return DSA_ERR_INVALID_ARG;
  if (!supported_shape(num_heads, d_latent, d_rope)) return DSA_ERR_UNSUPPORTED_SHAPE;
  if (num_pages > (int64_t)INT32_MAX / page_size) return DSA_ERR_UNSUPPORTED_SHAPE;
  if (num_q == 0) return DSA_OK;
  if (workspace_bytes < ws_need) return DSA_ERR_WORKSPACE_TOO_SMALL;
  if (ws_need > 0 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 7u))) return DSA_ERR_INVALID_ARG;
  if (!q || !kv || !kv_scale || !block_table || !q_req || !idx) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv)) return DSA_ERR_INVALID_ARG;
  if (num_splits == 1) {
    if (!out || !aligned16(out)) return DSA_ERR_INVALID_ARG;
  } else {
    if (!o_part || !lse_part || !aligned16(o_part)) return DSA_ERR_INVALID_ARG;
  }
  a->q = q;
  a->kv = kv;
  a->kv_scale = kv_scale;
  a->num_pages = num_pages;
  a->block_table = block_table;
  a->num_req = num_req;
  a->bt_stride = bt_stride;
  a->q_req = q_req;
  a->idx = idx;
  a->num_q = num_q;
  a->heads = num_heads;
  a->d_latent = d_latent;
  a->d_rope = d_rope;
  a->page_size = page_size;
  a->k = k;
  a->softmax_scale = softmax_scale;
  a->num_splits = num_splits;
  a->out = out;
  a->lse = lse;
  a->o_part = o_part;
  a->lse_part = lse_part;
  a->dev_status = dev_status;
  return DSA_OK;
}

}  // namespace

extern "C" {

dsa_status dsa_sparse_mla_fwd(const void* q, const uint8_t* kv, const float* kv_scale, int64_t num_pages,
                              const int32_t* block_table, int32_t num_req, int32_t bt_stride,
                              const int32_t* q_req, const int32_t* idx, int32_t num_q, int32_t num_heads,
                              int32_t d_latent, int32_t d_rope, int32_t page_size, int32_t k,
                              float softmax_scale, int32_t num_splits, void* out, float* lse, float* o_part,
                              float* lse_part, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                              void* stream) {
  dsa::MlaArgs a;
  const size_t ws_need = dsa_sparse_mla_workspace_size(num_q, num_heads, d_latent, d_rope, k);
  const dsa_status st = check_mla_args(q, kv, kv_scale, num_pages, block_table, num_req, bt_stride, q_req, idx,
                                       num_q, num_heads, d_latent, d_rope, page_size, k, softmax_scale, num_splits,
                                       out, lse, o_part, lse_part, ws_need, workspace, workspace_bytes, dev_status,
                                       &a);
  if (st != DSA_OK || num_q == 0) return st;
  if (use_tensor_cores(num_heads, d_latent, d_rope))
    return from_cuda(dsa::launch_mla_tc(a, workspace, static_cast<cudaStream_t>(stream)));
  return from_cuda(dsa::launch_mla_simt(a, static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_sparse_mla_topk_fwd(const float* scores, int64_t ld_scores, const int32_t* q_pos, int32_t k,
                                   int32_t* idx, const void* q, const uint8_t* kv, const float* kv_scale,
                                   int64_t num_pages, const int32_t* block_table, int32_t num_req, int32_t bt_stride,
                                   const int32_t* q_req, int32_t num_q, int32_t num_heads, int32_t d_latent,
                                   int32_t d_rope, int32_t page_size, float softmax_scale, void* out, float* lse,
                                   void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (ld_scores <= 0 || k <= 0 || num_q < 0) return DSA_ERR_INVALID_ARG;
  if (!use_tensor_cores(num_heads, d_latent, d_rope)) return DSA_ERR_UNSUPPORTED_SHAPE;
  if (ld_scores > 65536 || k > dsa::mla_tc_fused_max_k()) return DSA_ERR_UNSUPPORTED_SHAPE;
  if (num_q == 0) return DSA_OK;
  if (!scores || !q_pos || !idx) return DSA_ERR_INVALID_ARG;
  dsa::MlaArgs a;
  const size_t ws_need = dsa_sparse_mla_workspace_size(num_q, num_heads, d_latent, d_rope, k);
  const dsa_status st = check_mla_args(q, kv, kv_scale, num_pages, block_table, num_req, bt_stride, q_req, idx,
                                       num_q, num_heads, d_latent, d_rope, page_size, k, softmax_scale, 1, out, lse,
                                       nullptr, nullptr, ws_need, workspace, workspace_bytes, dev_status, &a);
  if (st != DSA_OK) return st;
  return from_cuda(dsa::launch_mla_tc_fused(a, scores, ld_scores, q_pos, idx, workspace,
                                            static_cast<cudaStream_t>(stream)));
}

int32_t dsa_sparse_mla_topk_max_k(void) { return dsa::mla_tc_fused_max_k(); }

dsa_status dsa_topk_sparse_mla_fwd(const float* scores, int64_t ld_scores, const int32_t* q_pos, int32_t k,
                                   int32_t* idx, const void* q, const uint8_t* kv, const float* kv_scale,
                                   int64_t num_pages, const int32_t* block_table, int32_t num_req, int32_t bt_stride,
                                   const int32_t* q_req, int32_t num_q, int32_t num_heads, int32_t d_latent,
                                   int32_t d_rope, int32_t page_size, float softmax_scale, int32_t num_splits,
                                   void* out, float* lse, float* o_part, float* lse_part, void* workspace,
                                   size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (ld_scores <= 0 || k <= 0 || num_q < 0) return DSA_ERR_INVALID_ARG;
  if (!use_tensor_cores(num_heads, d_latent, d_rope) || ld_scores > 65536) return DSA_ERR_UNSUPPORTED_SHAPE;
  if (num_q == 0) return DSA_OK;
  if (!scores || !q_pos || !idx) return DSA_ERR_INVALID_ARG;
  dsa::MlaArgs a;
  const size_t ws_need = dsa_sparse_mla_workspace_size(num_q, num_heads, d_latent, d_rope, k);
  const dsa_status st = check_mla_args(q, kv, kv_scale, num_pages, block_table, num_req, bt_stride, q_req, idx,
                                       num_q, num_heads, d_latent, d_rope, page_size, k, softmax_scale, num_splits,
                                       out, lse, o_part, lse_part, ws_need, workspace, workspace_bytes, dev_status,
                                       &a);
  if (st != DSA_OK) return st;
  const dsa::TopkResolve rv{static_cast<int2*>(workspace), block_table, q_req, kv_scale, num_pages, num_req,
                            bt_stride, page_size};
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = dsa::launch_topk_resolve(scores, ld_scores, q_pos, num_q, k, idx, rv, dev_status, s);
  if (e != cudaSuccess) return from_cuda(e);
  return from_cuda(dsa::launch_mla_tc_resolved(a, workspace, s));
}

// Test hook, not part of include/dsa.h: the fp32 CUDA-core kernel on any
// supported shape, so that tests can cross-check it against the tensor-core
// kernel on the 64-head shape.  Same arguments as dsa_sparse_mla_fwd minus
// the workspace (the CUDA-core kernel needs none).
DSA_API dsa_status dsa_test_sparse_mla_fwd_cuda_cores(const void* q, const uint8_t* kv, const float* kv_scale,
                                                      int64_t num_pages, const int32_t* block_table, int32_t num_req,
                                                      int32_t bt_stride, const int32_t* q_req, const int32_t* idx,
                                                      int32_t num_q, int32_t num_heads, int32_t d_latent,
                                                      int32_t d_rope, int32_t page_size, int32_t k,
                                                      float softmax_scale, int32_t num_splits, void* out, float* lse,
                                                      float* o_part, float* lse_part, int32_t* dev_status,
                                                      void* stream) {
  dsa::MlaArgs a;
  const dsa_status st = check_mla_args(q, kv, kv_scale, num_pages, block_table, num_req, bt_stride, q_req, idx,
                                       num_q, num_heads, d_latent, d_rope, page_size, k, softmax_scale, num_splits,
                                       out, lse, o_part, lse_part, 0, nullptr, 0, dev_status, &a);
  if (st != DSA_OK || num_q == 0) return st;
  return from_cuda(dsa::launch_mla_simt(a, static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_combine(const float* o_part, const float* lse_part, int32_t num_splits, int32_t num_q,
                       int32_t num_heads, int32_t d_v, void* out, float* lse, void* stream) {
  if (num_q < 0 || num_splits < 1 || num_splits > 64 || num_heads < 1 || num_heads > 64 || d_v <= 0 ||
      d_v % 4 != 0)
    return DSA_ERR_INVALID_ARG;
  if (num_q == 0) return DSA_OK;
  if (!o_part || !lse_part || !out || !aligned16(o_part) || !aligned16(out)) return DSA_ERR_INVALID_ARG;
  return from_cuda(dsa::launch_combine(o_part, lse_part, num_splits, num_q, num_heads, d_v, out, lse,
                                       static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

dsa_status dsa_kv_write(const void* rows, int32_t n, int32_t d_qk, const int32_t* req, const int32_t* pos,
                        const int32_t* block_table, int32_t num_req, int32_t bt_stride, int32_t page_size,
                        int64_t num_pages, uint8_t* kv, float* kv_scale, int32_t* dev_status, void* stream) {
  if (n < 0 || d_qk < 16 || d_qk % 16 != 0 || d_qk > dsa::kv_write_max_d() || page_size <= 0 || num_pages <= 0 ||
      num_req <= 0 || bt_stride <= 0)
    return DSA_ERR_INVALID_ARG;
  if (num_pages > (int64_t)INT32_MAX / page_size) return DSA_ERR_UNSUPPORTED_SHAPE;
  if (n == 0) return DSA_OK;
  if (!rows || !req || !pos || !block_table || !kv || !kv_scale) return DSA_ERR_INVALID_ARG;
  if (!aligned16(rows) || !aligned16(kv)) return DSA_ERR_INVALID_ARG;
  return from_cuda(dsa::launch_kv_write(rows, n, d_qk, req, pos, block_table, num_req, bt_stride, page_size,
                                        num_pages, kv, kv_scale, dev_status, static_cast<cudaStream_t>(stream)));
}
