// KV cache write path: quantise new latent+rope rows to FP8 E4M3 with one
// fp32 scale per token and store them through the block table.
//
// "Accelerating GLM-5.3-Flash on H200", section 2 "KV-only decode
// RadixCache": KV rows live in a paged pool whose pages a block table maps
// per request (shared prefix pages appear in several requests' tables).
// SGLang cookbook page for GLM-5.3-Flash, "Keep the KV and DSA backends
// paired": the KV cache is FP8 E4M3.  Per token: amax = max |x|, scale =
// amax / 448 (448 = the largest finite E4M3 value) and byte_j =
// E4M3(x_j / scale) rounded to nearest even and saturated; an all-zero row
// stores scale 0 and zero bytes.  Both divisions round as IEEE fp32 division.
//
// One warp per row: 16-byte loads of 8 bf16 values, a warp max, then 8-byte
// stores of the 8 codes.
// HBM-bound: d·2 bytes read + d + 4 bytes written per row.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "internal.cuh"

namespace dsa {
namespace {

constexpr int KVW_WARPS = 8;
constexpr int KVW_MAX_CHUNKS = 8;  // per lane: rows of up to 32 * 8 * 8 = 2048 values

// two floats -> two E4M3 codes (round to nearest even, saturating), x0 in the low byte
__device__ __forceinline__ uint32_t e4m3x2(float x0, float x1) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(x1), "f"(x0));
  return r;
}

// The larger of two bf16 pairs, element by element (a NaN loses to a number).
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Two-wide fp32 arithmetic, each lane rounded as its scalar .rn form.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// CH: 16-byte chunks each lane holds per row (rows of up to 32 * 8 * CH
// values); each warp takes KVW_RPW rows, all of their loads in flight before
// the first row is quantised (one row per warp measured fastest: more rows
// per warp cost registers and occupancy).
constexpr int KVW_RPW = 1;

template <int CH>
__global__ void __launch_bounds__(KVW_WARPS * 32)
    kv_write_kernel(const uint4* __restrict__ rows, int32_t n, int32_t d, const int32_t* __restrict__ req,
                    const int32_t* __restrict__ pos, const int32_t* __restrict__ block_table, int32_t num_req,
                    int32_t bt_stride, int32_t page_size, int64_t num_pages, uint8_t* __restrict__ kv,
                    float* __restrict__ kv_scale, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t i0 = ((int64_t)blockIdx.x * KVW_WARPS + (threadIdx.x >> 5)) * KVW_RPW;
  const int nch = d / 8;  // 16-byte chunks of 8 bf16
  uint4 v[KVW_RPW][CH];
#pragma unroll
  for (int q = 0; q < KVW_RPW; ++q) {
#pragma unroll
    for (int u = 0; u < CH; ++u) {
      const int c = lane + 32 * u;
      if (i0 + q < n && c < nch) v[q][u] = __ldg(rows + (i0 + q) * nch + c);
    }
  }
#pragma unroll
  for (int q = 0; q < KVW_RPW; ++q) {
    const int64_t i = i0 + q;
    if (i >= n) break;
    const int32_t r = req[i], p = pos[i];
    if (r < 0 || r >= num_req) {
      if (lane == 0) report(status, DSA_DEV_BAD_PAGE);
      continue;
    }
    if (p < 0 || p / page_size >= bt_stride) {
      if (lane == 0) report(status, DSA_DEV_BAD_INDEX);
      continue;
    }
    const int32_t page = block_table[(int64_t)r * bt_stride + p / page_size];
    if (page < 0 || page >= num_pages) {
      if (lane == 0) report(status, DSA_DEV_BAD_PAGE);
      continue;
    }
    const int64_t slot = (int64_t)page * page_size + p % page_size;
    // max |x| over the lane's bf16 pairs, in bf16 (exact): the sign bits
    // cleared, then an element-wise max
    uint32_t m2 = 0u;
#pragma unroll
    for (int u = 0; u < CH; ++u) {
      if (lane + 32 * u < nch) {
        const uint32_t w[4] = {v[q][u].x, v[q][u].y, v[q][u].z, v[q][u].w};
#pragma unroll
        for (int t = 0; t < 4; ++t) m2 = bf16x2_max(m2, w[t] & 0x7fff7fffu);
      }
    }
    float amax = fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xffff0000u));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = __fdiv_rn(amax, 448.0f);
    if (lane == 0) kv_scale[slot] = scale;
    // x / scale rounded as IEEE fp32 division: the reciprocal r = RN(1/scale)
    // once, then per value q0 = RN(x r) and Markstein's FMA correction
    // q = RN(q0 + r RN(x - q0 scale)), with x's sign kept on zero.  For
    // 2^-90 <= scale < inf this gives the IEEE quotient's E4M3 code for every
    // bf16 x with |x| <= amax (checked exhaustively against the division on
    // the GPU); other rows (tiny or non-finite maxima) divide.
    // (Computed for a bf16 pair at a time with two-wide fp32 operations.)
    const bool fast = scale >= 0x1p-90f && scale <= 3.4028235e38f;
    const float rcp = __frcp_rn(scale);
    const uint64_t rcp2 = f32x2(rcp, rcp), nscale2 = f32x2(-scale, -scale);
    auto quot2 = [&](uint32_t w) -> uint32_t {  // the E4M3 codes of the pair's two quotients
      const float x0 = __uint_as_float(w << 16), x1 = __uint_as_float(w & 0xffff0000u);
      if (!fast) return e4m3x2(__fdiv_rn(x0, scale), __fdiv_rn(x1, scale));
      const uint64_t x = f32x2(x0, x1);
      const uint64_t q0 = mul_f32x2(x, rcp2);
      const uint64_t qc = fma_f32x2(fma_f32x2(q0, nscale2, x), rcp2, q0);
      const uint32_t c0 = (uint32_t)qc | (__float_as_uint(x0) & 0x80000000u);
      const uint32_t c1 = (uint32_t)(qc >> 32) | (__float_as_uint(x1) & 0x80000000u);
      return e4m3x2(__uint_as_float(c0), __uint_as_float(c1));
    };
    uint2* dst = reinterpret_cast<uint2*>(kv + slot * d);
#pragma unroll
    for (int u = 0; u < CH; ++u) {
      const int c = lane + 32 * u;
      if (c < nch) {
        const uint32_t w[4] = {v[q][u].x, v[q][u].y, v[q][u].z, v[q][u].w};
        uint32_t b[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
          b[t] = scale > 0.f ? quot2(w[t]) : 0u;
        dst[c] = make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
      }
    }
  }
}

}  // namespace

int kv_write_max_d() { return 32 * 8 * KVW_MAX_CHUNKS; }

cudaError_t launch_kv_write(const void* rows, int32_t n, int32_t d, const int32_t* req, const int32_t* pos,
                            const int32_t* block_table, int32_t num_req, int32_t bt_stride, int32_t page_size,
                            int64_t num_pages, uint8_t* kv, float* kv_scale, int32_t* status, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int64_t rows_per_cta = (int64_t)KVW_WARPS * KVW_RPW;
  const unsigned grid = (unsigned)((n + rows_per_cta - 1) / rows_per_cta);
  const int ch = (d / 8 + 31) / 32;  // chunks per lane
  auto kern = ch <= 1 ? kv_write_kernel<1> : ch <= 3 ? kv_write_kernel<3> : kv_write_kernel<KVW_MAX_CHUNKS>;
  kern<<<grid, KVW_WARPS * 32, 0, stream>>>(static_cast<const uint4*>(rows), n, d, req, pos, block_table, num_req,
                                            bt_stride, page_size, num_pages, kv, kv_scale, status);
  return cudaGetLastError();
}

}  // namespace dsa
