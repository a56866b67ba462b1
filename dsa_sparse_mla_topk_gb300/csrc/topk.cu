// Causal top-k selection over fp32 indexer scores (radix select).
//
// "Accelerating GLM-5.3-Flash on H200", section 3 "Larger KV tiles for DSA
// Partial": the indexer's scores pick the KV positions the Partial step
// attends to.  This kernel makes the pick exact and deterministic: positions
// are ranked by (score descending, position ascending), -0.0 == +0.0, and
// the chosen ones are written in ascending position order, -1 padded.
//
// Method: every fp32 score maps to an order-preserving 32-bit key.  A radix
// select over the key's digits (11, 11, 10 bits) finds the exact key T of the
// k-th largest visible score and how many of the entries equal to T must be
// taken.  One more ordered pass then writes every position whose key beats T
// and the lowest-positioned entries equal to T, using block-wide prefix sums
// so that output order is ascending position order.
#include <cuda_runtime.h>

#include "internal.cuh"

namespace dsa {
namespace {

constexpr int kTopkThreads = 1024;
constexpr int kBins = 2048;

__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0.0 ranks equal to +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum of one value per thread over the whole block; *total
// receives the block sum.  `warp_buf` holds NT/32 words of shared memory.
template <int NT>
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* total, uint32_t* warp_buf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_buf[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < NT / 32 ? warp_buf[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < NT / 32) warp_buf[lane] = w;
  }
  __syncthreads();
  const uint32_t before = warp > 0 ? warp_buf[warp - 1] : 0u;
  *total = warp_buf[NT / 32 - 1];
  __syncthreads();
  return before + x - v;
}

__global__ void __launch_bounds__(kTopkThreads) topk_radix_kernel(const float* __restrict__ scores, int64_t ld,
                                                                  const int32_t* __restrict__ q_pos, int32_t k,
                                                                  int32_t* __restrict__ idx, int32_t* status) {
  constexpr int NT = kTopkThreads;
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t warp_buf[NT / 32];
  __shared__ uint32_t sel_bin, sel_above, sel_count;

  const int64_t row = blockIdx.x;
  const int tid = threadIdx.x;
  int32_t* out = idx + row * (int64_t)k;
  const int64_t p = q_pos[row];
  if (p < 0 || p >= ld) {
    if (tid == 0) report(status, DSA_DEV_BAD_QPOS);
    for (int j = tid; j < k; j += NT) out[j] = -1;
    return;
  }
  const int64_t vis = p + 1;
  if (vis <= k) {  // everything visible is selected
    for (int j = tid; j < k; j += NT) out[j] = j < vis ? j : -1;
    return;
  }
  const float* s = scores + row * ld;
  const bool vec = ((reinterpret_cast<uintptr_t>(s) & 15u) == 0);
  const int64_t vis4 = vec ? (vis & ~int64_t(3)) : 0;

  // ---- radix select: find the key prefix of the k-th largest score ----
  uint32_t prefix = 0, mask = 0;
  uint32_t krem = (uint32_t)k;
  const int shifts[3] = {21, 10, 0};
  const uint32_t digit_mask[3] = {0x7ffu, 0x7ffu, 0x3ffu};
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = shifts[pass];
    const uint32_t dm = digit_mask[pass];
    for (int b = tid; b < kBins; b += NT) hist[b] = 0;
    __syncthreads();
    for (int64_t j = int64_t(tid) * 4; j < vis4; j += int64_t(NT) * 4) {
      const float4 v = *reinterpret_cast<const float4*>(s + j);
      const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint32_t key = score_key(e[t]);
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> sh) & dm], 1u);
      }
    }
    for (int64_t j = vis4 + tid; j < vis; j += NT) {
      const uint32_t key = score_key(s[j]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> sh) & dm], 1u);
    }
    __syncthreads();
    // bins in descending order: thread t owns bins kBins-1-2t and kBins-2-2t
    const int b0 = kBins - 1 - 2 * tid, b1 = b0 - 1;
    const uint32_t c0 = hist[b0], c1 = hist[b1];
    uint32_t total;
    uint32_t above = block_exclusive_scan<NT>(c0 + c1, &total, warp_buf);
    if (above < krem && krem <= above + c0) {
      sel_bin = b0, sel_above = above, sel_count = c0;
    }
    above += c0;
    if (above < krem && krem <= above + c1) {
      sel_bin = b1, sel_above = above, sel_count = c1;
    }
    __syncthreads();
    prefix |= sel_bin << sh;
    mask |= dm << sh;
    krem -= sel_above;
    const bool whole_bin = (sel_count == krem);
    __syncthreads();  // everyone has read sel_* before the next pass rewrites them
    if (whole_bin) break;  // every entry of the bin is taken: no need to refine further
  }

  // ---- ordered compaction: keys above the prefix, then the first krem ties ----
  uint32_t ties_before = 0, written = 0;
  for (int64_t base = 0; base < vis && written < (uint32_t)k; base += int64_t(NT) * 4) {
    const int64_t j0 = base + int64_t(tid) * 4;
    float e[4];
    if (vec && j0 + 3 < vis) {
      const float4 v = *reinterpret_cast<const float4*>(s + j0);
      e[0] = v.x, e[1] = v.y, e[2] = v.z, e[3] = v.w;
    } else {
#pragma unroll
      for (int t = 0; t < 4; ++t) e[t] = (j0 + t < vis) ? s[j0 + t] : 0.f;
    }
    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if (j0 + t < vis) {
        const uint32_t mk = score_key(e[t]) & mask;
        gt |= (mk > prefix) << t;
        eq |= (mk == prefix) << t;
      }
    }
    uint32_t eq_total;
    uint32_t rank = ties_before + block_exclusive_scan<NT>(__popc(eq), &eq_total, warp_buf);
    uint32_t take = gt;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if ((eq >> t) & 1u) {
        if (rank < krem) take |= 1u << t;
        ++rank;
      }
    }
    uint32_t take_total;
    uint32_t o = written + block_exclusive_scan<NT>(__popc(take), &take_total, warp_buf);
#pragma unroll
    for (int t = 0; t < 4; ++t)
      if ((take >> t) & 1u) out[o++] = (int32_t)(j0 + t);
    ties_before += eq_total;
    written += take_total;
  }
}

}  // namespace

cudaError_t launch_topk_radix(const float* scores, int64_t ld, const int32_t* q_pos, int32_t num_q, int32_t k,
                              int32_t* idx, int32_t* dev_status, cudaStream_t stream) {
  if (num_q == 0) return cudaSuccess;
  topk_radix_kernel<<<num_q, kTopkThreads, 0, stream>>>(scores, ld, q_pos, k, idx, dev_status);
  return cudaGetLastError();
}

}  // namespace dsa
