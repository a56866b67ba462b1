// Combine: exact log-sum-exp merge of split-KV partial results.
//
// "Accelerating GLM-5.3-Flash on H200", section 3 "Larger KV tiles for DSA
// Partial": splitting the KV range of a query token adds intermediate writes
// and a Combine step.  Each split s holds O_s (already normalised by its own
// softmax sum) and lse_s; the merged result is
//   lse = ln sum_s exp(lse_s),   O = sum_s exp(lse_s - lse) O_s.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "internal.cuh"

namespace dsa {
namespace {

constexpr int kCombineThreads = 256;
constexpr int kMaxSplits = 64;
constexpr int kMaxHeads = 64;

// One CTA per query token: first the per-(split, head) weights, then the
// weighted sum over d_v with 16-byte loads.
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part, int S, int num_q, int H,
                   int dv, __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  __shared__ float w[kMaxSplits * kMaxHeads];
  const int i = blockIdx.x;
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    float m = -INFINITY;
    for (int s = 0; s < S; ++s) m = fmaxf(m, lse_part[((int64_t)s * num_q + i) * H + h]);
    float l = -INFINITY;
    if (m != -INFINITY) {
      float sum = 0.f;
      for (int s = 0; s < S; ++s) sum += expf(lse_part[((int64_t)s * num_q + i) * H + h] - m);
      l = m + logf(sum);
    }
    for (int s = 0; s < S; ++s) {
      const float ls = lse_part[((int64_t)s * num_q + i) * H + h];
      w[s * H + h] = (l == -INFINITY || ls == -INFINITY) ? 0.f : expf(ls - l);
    }
    if (lse) lse[(int64_t)i * H + h] = l;
  }
  __syncthreads();
  const int n4 = H * dv / 4;
  const int64_t stride_s = (int64_t)num_q * H * dv;
  const float* base = o_part + (int64_t)i * H * dv;
  for (int e = threadIdx.x; e < n4; e += blockDim.x) {
    const int h = (e * 4) / dv;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < S; ++s) {
      const float ws = w[s * H + h];
      if (ws == 0.f) continue;
      const float4 v = reinterpret_cast<const float4*>(base + s * stride_s)[e];
      acc.x = fmaf(ws, v.x, acc.x);
      acc.y = fmaf(ws, v.y, acc.y);
      acc.z = fmaf(ws, v.z, acc.z);
      acc.w = fmaf(ws, v.w, acc.w);
    }
    __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(out + (int64_t)i * H * dv) + 2 * e;
    o[0] = __floats2bfloat162_rn(acc.x, acc.y);
    o[1] = __floats2bfloat162_rn(acc.z, acc.w);
  }
}

}  // namespace

cudaError_t launch_combine(const float* o_part, const float* lse_part, int32_t num_splits, int32_t num_q,
                           int32_t heads, int32_t d_v, void* out, float* lse, cudaStream_t stream) {
  if (num_q == 0) return cudaSuccess;
  if (num_splits > kMaxSplits || heads > kMaxHeads) return cudaErrorInvalidValue;
  combine_kernel<<<num_q, kCombineThreads, 0, stream>>>(o_part, lse_part, num_splits, num_q, heads, d_v,
                                                        static_cast<__nv_bfloat16*>(out), lse);
  return cudaGetLastError();
}

}  // namespace dsa
