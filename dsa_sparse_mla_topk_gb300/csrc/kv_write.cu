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
    float amax = 0.f;
#pragma unroll
    for (int u = 0; u < CH; ++u) {
      if (lane + 32 * u < nch) {
        const uint32_t w[4] = {v[q][u].x, v[q][u].y, v[q][u].z, v[q][u].w};
#pragma unroll
        for (int t = 0; t < 4; ++t)
          amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[t] << 16)), fabsf(__uint_as_float(w[t] & 0xffff0000u))));
      }
    }
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
    const bool fast = scale >= 0x1p-90f && scale <= 3.4028235e38f;
    const float rcp = __frcp_rn(scale);
    auto quot = [&](float x) {
      if (!fast) return __fdiv_rn(x, scale);
      const float q0 = __fmul_rn(x, rcp);
      const float qc = __fmaf_rn(__fmaf_rn(-q0, scale, x), rcp, q0);
      return __int_as_float(__float_as_int(qc) | (__float_as_int(x) & 0x80000000));
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
          b[t] = scale > 0.f ? e4m3x2(quot(__uint_as_float(w[t] << 16)), quot(__uint_as_float(w[t] & 0xffff0000u)))
                             : 0u;
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
