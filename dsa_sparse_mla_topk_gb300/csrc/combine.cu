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
constexpr int kMaxChunk = 4 * kCombineThreads;  // floats of one query's H x d_v block per CTA
constexpr int kMaxSplits = 64;
constexpr int kMaxChunkHeads = 32;

// Floats per CTA for rows of d_v floats: a chunk of c floats touches at most
// c / d_v + 2 heads, which must fit the kMaxChunkHeads weight columns.
int chunk_floats(int dv) {
  const int c = (kMaxChunkHeads - 2) * dv;
  return c < kMaxChunk ? (c & ~3) : kMaxChunk;
}

// CTA (i, c): floats [c chunk, (c + 1) chunk) of query i's H x d_v result.
// First the per-(split, head) weights of the heads that chunk touches, then
// one float4 per thread, all splits' loads in flight together.
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part, int S, int num_q, int H,
                   int dv, int chunk, __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  __shared__ float w[kMaxSplits * kMaxChunkHeads];
  const int i = blockIdx.x;
  const int64_t e0 = (int64_t)blockIdx.y * chunk;
  const int64_t n = (int64_t)H * dv;
  const int h0 = (int)(e0 / dv);
  const int h1 = (int)(min(e0 + chunk, n) - 1) / dv;
  for (int t = threadIdx.x; t <= h1 - h0; t += blockDim.x) {
    const int h = h0 + t;
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
      w[s * kMaxChunkHeads + t] = (l == -INFINITY || ls == -INFINITY) ? 0.f : expf(ls - l);
    }
    // the CTA holding the head's first element writes its lse
    if (lse && (int64_t)h * dv >= e0) lse[(int64_t)i * H + h] = l;
  }
  __syncthreads();
  const int64_t e = e0 / 4 + threadIdx.x;  // float4 index within the query
  if (4 * (int)threadIdx.x >= chunk || e * 4 >= n) return;
  const int t = (int)(e * 4 / dv) - h0;
  const int64_t stride_s = (int64_t)num_q * H * dv / 4;
  const float4* base = reinterpret_cast<const float4*>(o_part + (int64_t)i * H * dv) + e;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  int s = 0;
  for (; s + 8 <= S; s += 8) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = __ldg(base + (s + u) * stride_s);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float ws = w[(s + u) * kMaxChunkHeads + t];
      acc.x = fmaf(ws, v[u].x, acc.x);
      acc.y = fmaf(ws, v[u].y, acc.y);
      acc.z = fmaf(ws, v[u].z, acc.z);
      acc.w = fmaf(ws, v[u].w, acc.w);
    }
  }
  for (; s < S; ++s) {
    const float4 v = __ldg(base + s * stride_s);
    const float ws = w[s * kMaxChunkHeads + t];
    acc.x = fmaf(ws, v.x, acc.x);
    acc.y = fmaf(ws, v.y, acc.y);
    acc.z = fmaf(ws, v.z, acc.z);
    acc.w = fmaf(ws, v.w, acc.w);
  }
  __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(out + (int64_t)i * H * dv) + 2 * e;
  o[0] = __floats2bfloat162_rn(acc.x, acc.y);
  o[1] = __floats2bfloat162_rn(acc.z, acc.w);
}

}  // namespace

cudaError_t launch_combine(const float* o_part, const float* lse_part, int32_t num_splits, int32_t num_q,
                           int32_t heads, int32_t d_v, void* out, float* lse, cudaStream_t stream) {
  if (num_q == 0) return cudaSuccess;
  if (num_splits > kMaxSplits || d_v <= 0 || d_v % 4 != 0) return cudaErrorInvalidValue;
  const int chunk = chunk_floats(d_v);
  const int64_t n = (int64_t)heads * d_v;
  const dim3 grid(num_q, (unsigned)((n + chunk - 1) / chunk));
  combine_kernel<<<grid, kCombineThreads, 0, stream>>>(o_part, lse_part, num_splits, num_q, heads, d_v, chunk,
                                                       static_cast<__nv_bfloat16*>(out), lse);
  return cudaGetLastError();
}

}  // namespace dsa
