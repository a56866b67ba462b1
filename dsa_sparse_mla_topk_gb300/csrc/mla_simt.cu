// Sparse MLA attention over gathered FP8 rows, CUDA-core version.
//
// "Accelerating GLM-5.3-Flash on H200", section 3 "Larger KV tiles for DSA
// Partial": for each query token the Partial step loads the selected KV
// positions and computes QK^T, an online softmax and the weighted value sum,
// one KV tile at a time; with KV splits each split writes a partial result
// that a Combine step merges.  "GLM-5.3 Optimizations, Part 2"
// ("Interpretation"): one latent KV row serves all heads of the token, so a
// CTA owns one (query token, split) and every gathered row is used by all
// heads.
//
// This version runs in fp32 on the CUDA cores.  It is the simple, general
// path (both supported head shapes) that the tensor-core kernel is checked
// and measured against.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math.h>

#include "internal.cuh"

namespace dsa {
namespace {

constexpr int kSimtThreads = 256;
constexpr int kSimtTile = 32;

__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

template <int H, int DL, int DR>
struct SimtCfg {
  static constexpr int NT = kSimtThreads;
  static constexpr int T = kSimtTile;
  static constexpr int DQK = DL + DR;
  static constexpr int QSTRIDE = DQK + 8;  // bf16 elements per Q row in smem (bank spread)
  static constexpr int KSTRIDE = DQK + 1;  // floats per K row in smem
  static constexpr int TPH = NT / H;       // threads per head in the score phase
  static constexpr int JPT = T / TPH;      // rows per thread in the score phase
  static constexpr int DPT = (DL >= NT) ? DL / NT : 1;  // value dims per thread
  static constexpr int DGROUPS = DL / DPT;
  static constexpr int HGROUPS = NT / DGROUPS;
  static constexpr int HPT = H / HGROUPS;  // heads per thread in the PV phase
  static_assert(NT % H == 0 && T % TPH == 0, "score phase mapping");
  static_assert(DL % DPT == 0 && NT % DGROUPS == 0 && H % HGROUPS == 0, "PV phase mapping");
  static_assert(DQK % 16 == 0, "rows are moved in 16-byte chunks");
  static constexpr size_t smem_bytes = sizeof(__nv_bfloat16) * H * QSTRIDE + sizeof(float) * T * KSTRIDE +
                                       sizeof(float) * H * T + sizeof(float) * 3 * H + sizeof(int64_t) * T;
};

template <int H, int DL, int DR>
__global__ void __launch_bounds__(kSimtThreads) mla_simt_kernel(MlaArgs a) {
  using C = SimtCfg<H, DL, DR>;
  constexpr int NT = C::NT, T = C::T, DQK = C::DQK;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  float* ks = reinterpret_cast<float*>(qs + H * C::QSTRIDE);
  float* ps = ks + T * C::KSTRIDE;   // [H][T] scores, then probabilities
  float* alpha_s = ps + H * T;       // [H] rescale factor of this tile
  float* m_s = alpha_s + H;          // [H] final running max
  float* l_s = m_s + H;              // [H] final running sum
  int64_t* slot_s = reinterpret_cast<int64_t*>(l_s + H);  // [T], -1 = no row

  const int tid = threadIdx.x;
  const int i = blockIdx.x;  // query token
  const int split = blockIdx.y;
  const int S = gridDim.y;

  // Q of this token -> smem (bf16, padded rows)
  {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) + (int64_t)i * H * DQK);
    constexpr int CH = DQK / 8;  // 16-byte chunks per row
    for (int c = tid; c < H * CH; c += NT) {
      const int h = c / CH, cc = c % CH;
      *reinterpret_cast<uint4*>(qs + h * C::QSTRIDE + cc * 8) = src[c];
    }
  }
  const int r = a.q_req[i];
  const bool req_ok = (r >= 0 && r < a.num_req);
  if (!req_ok && tid == 0) report(a.dev_status, DSA_DEV_BAD_PAGE);

  const int ntiles = (a.k + T - 1) / T;
  const int t_begin = (int)((int64_t)ntiles * split / S);
  const int t_end = (int)((int64_t)ntiles * (split + 1) / S);

  // score-phase mapping: head hs, rows js + TPH * m
  const int hs = tid / C::TPH, js = tid % C::TPH;
  float m_run = -INFINITY, l_run = 0.f;  // replicated over the TPH threads of head hs
  // PV-phase mapping: dims dv0..dv0+DPT-1, heads hv0..hv0+HPT-1
  const int dv0 = (tid % C::DGROUPS) * C::DPT;
  const int hv0 = (tid / C::DGROUPS) * C::HPT;
  float acc[C::HPT][C::DPT];
#pragma unroll
  for (int h = 0; h < C::HPT; ++h)
#pragma unroll
    for (int d = 0; d < C::DPT; ++d) acc[h][d] = 0.f;

  const int32_t* row_idx = a.idx + (int64_t)i * a.k;
  for (int tile = t_begin; tile < t_end; ++tile) {
    __syncthreads();  // previous tile fully consumed
    if (tid < T) {
      const int e = tile * T + tid;
      int64_t slot = -1;
      if (e < a.k && req_ok) {
        const int32_t pos = row_idx[e];
        if (pos < -1) {
          report(a.dev_status, DSA_DEV_BAD_INDEX);
        } else if (pos >= 0) {
          const int32_t pg = pos / a.page_size;
          if (pg >= a.bt_stride) {
            report(a.dev_status, DSA_DEV_BAD_INDEX);
          } else {
            const int32_t page = a.block_table[(int64_t)r * a.bt_stride + pg];
            if (page < 0 || page >= a.num_pages)
              report(a.dev_status, DSA_DEV_BAD_PAGE);
            else
              slot = (int64_t)page * a.page_size + pos % a.page_size;
          }
        }
      }
      slot_s[tid] = slot;
    }
    __syncthreads();
    // gather + dequantise the tile's rows (16-byte loads)
    {
      constexpr int CH = DQK / 16;
      for (int c = tid; c < T * CH; c += NT) {
        const int j = c / CH, cc = c % CH;
        const int64_t slot = slot_s[j];
        float* dst = ks + j * C::KSTRIDE + cc * 16;
        if (slot >= 0) {
          const uint4 raw = *reinterpret_cast<const uint4*>(a.kv + slot * DQK + cc * 16);
          const float sc = a.kv_scale[slot];
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const float2 lo = e4m3x2_to_float2((uint16_t)(w[q4] & 0xffffu));
            const float2 hi = e4m3x2_to_float2((uint16_t)(w[q4] >> 16));
            dst[q4 * 4 + 0] = lo.x * sc;
            dst[q4 * 4 + 1] = lo.y * sc;
            dst[q4 * 4 + 2] = hi.x * sc;
            dst[q4 * 4 + 3] = hi.y * sc;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) dst[e] = 0.f;
        }
      }
    }
    __syncthreads();
    // scores z = scale * q . x for head hs and rows js + TPH*m
    float z[C::JPT];
#pragma unroll
    for (int m = 0; m < C::JPT; ++m) z[m] = 0.f;
    {
      const __nv_bfloat162* qrow = reinterpret_cast<const __nv_bfloat162*>(qs + hs * C::QSTRIDE);
      for (int d2 = 0; d2 < DQK / 2; ++d2) {
        const float2 qv = __bfloat1622float2(qrow[d2]);
#pragma unroll
        for (int m = 0; m < C::JPT; ++m) {
          const float* kr = ks + (js + C::TPH * m) * C::KSTRIDE + 2 * d2;
          z[m] = fmaf(qv.x, kr[0], z[m]);
          z[m] = fmaf(qv.y, kr[1], z[m]);
        }
      }
    }
    float tmax = -INFINITY;
#pragma unroll
    for (int m = 0; m < C::JPT; ++m) {
      const bool valid = slot_s[js + C::TPH * m] >= 0;
      z[m] = valid ? z[m] * a.softmax_scale : -INFINITY;
      tmax = fmaxf(tmax, z[m]);
    }
#pragma unroll
    for (int o = 1; o < C::TPH; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
    const float m_new = fmaxf(m_run, tmax);
    // all rows so far invalid: keep everything at zero
    const float alpha = (m_new == -INFINITY) ? 1.f : __expf(m_run - m_new);
    float psum = 0.f;
#pragma unroll
    for (int m = 0; m < C::JPT; ++m) {
      const float pj = (z[m] == -INFINITY) ? 0.f : __expf(z[m] - m_new);
      ps[hs * T + js + C::TPH * m] = pj;
      psum += pj;
    }
#pragma unroll
    for (int o = 1; o < C::TPH; o <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
    l_run = l_run * alpha + psum;
    m_run = m_new;
    if (js == 0) alpha_s[hs] = alpha;
    __syncthreads();
    // O = alpha * O + P V
#pragma unroll
    for (int h = 0; h < C::HPT; ++h) {
      const float al = alpha_s[hv0 + h];
#pragma unroll
      for (int d = 0; d < C::DPT; ++d) acc[h][d] *= al;
    }
    for (int j = 0; j < T; ++j) {
      float v[C::DPT];
#pragma unroll
      for (int d = 0; d < C::DPT; ++d) v[d] = ks[j * C::KSTRIDE + dv0 + d];
#pragma unroll
      for (int h = 0; h < C::HPT; ++h) {
        const float pj = ps[(hv0 + h) * T + j];
#pragma unroll
        for (int d = 0; d < C::DPT; ++d) acc[h][d] = fmaf(pj, v[d], acc[h][d]);
      }
    }
  }
  if (js == 0) {
    m_s[hs] = m_run;
    l_s[hs] = l_run;
  }
  __syncthreads();
  // epilogue: normalise, write bf16 output or fp32 partial
#pragma unroll
  for (int h = 0; h < C::HPT; ++h) {
    const int hh = hv0 + h;
    const float l = l_s[hh];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int64_t o_off = ((int64_t)i * H + hh) * DL + dv0;
    if (S == 1) {
      __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + o_off;
#pragma unroll
      for (int d = 0; d < C::DPT; ++d) o[d] = __float2bfloat16_rn(acc[h][d] * inv);
    } else {
      float* o = a.o_part + (int64_t)split * a.num_q * H * DL + o_off;
#pragma unroll
      for (int d = 0; d < C::DPT; ++d) o[d] = acc[h][d] * inv;
    }
    if (dv0 == 0) {
      const float lse = l > 0.f ? m_s[hh] + logf(l) : -INFINITY;
      if (S == 1) {
        if (a.lse) a.lse[(int64_t)i * H + hh] = lse;
      } else {
        a.lse_part[((int64_t)split * a.num_q + i) * H + hh] = lse;
      }
    }
  }
}

template <int H, int DL, int DR>
cudaError_t launch_simt_shape(const MlaArgs& a, cudaStream_t stream) {
  using C = SimtCfg<H, DL, DR>;
  auto kern = mla_simt_kernel<H, DL, DR>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::smem_bytes);
  if (e != cudaSuccess) return e;
  dim3 grid(a.num_q, a.num_splits);
  kern<<<grid, C::NT, C::smem_bytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mla_simt(const MlaArgs& a, cudaStream_t stream) {
  if (a.num_q == 0) return cudaSuccess;
  if (a.heads == 16 && a.d_latent == 64 && a.d_rope == 16) return launch_simt_shape<16, 64, 16>(a, stream);
  if (a.heads == 64 && a.d_latent == 512 && a.d_rope == 64) return launch_simt_shape<64, 512, 64>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace dsa
