// Sparse MLA attention on the Blackwell tensor cores (tcgen05 + TMEM).
//
// "Accelerating GLM-5.3-Flash on H200", section 3 "Larger KV tiles for DSA
// Partial": the Partial step loads the KV positions the indexer selected and
// computes Q K^T, an online softmax and the weighted value sum, one KV tile at
// a time (Figure 4: the last tile is padded virtually, the index tensor is
// left alone); a KV split writes a partial result for the Combine step.
// "GLM-5.3 Optimizations, Part 2" ("Interpretation"): every latent KV row is
// shared by all 64 heads of a query token.
//
// GB300 design (one CTA = one query token x one KV split, 512 threads):
//  * Each KV tile is 64 selected rows, and two tiles are resident (double
//    buffering): while one is multiplied the next is gathered.  Rows are
//    gathered through the block table from the FP8 E4M3 cache, converted
//    exactly to fp16 (one cvt per two values; E4M3 is a subset of fp16) and
//    stored ONCE in shared memory in the 128-byte-swizzled K-major layout.
//    That single copy is the A operand of  S^T = K Q^T  (M = 64 rows, N = 64
//    heads, K = 576) and, read MN-major, of  O^T = V^T P^T  (M = 4 x 128
//    latent dims, N = 64 heads, K = 64 rows).  Heads sit on N: one gathered
//    row serves every head.
//  * Accumulators live in tensor memory: S^T per buffer, O^T in 4 x 64
//    columns.
//  * The per-token dequantisation scale s_j is applied in fp32 where it is
//    exact to do so: to the logits of row j, and folded into P before its
//    fp16 rounding (P'_hj = p_hj s_j 2^E), so V stays raw FP8-valued fp16.
//    2^E is a per-query power of two chosen from the largest selected scale
//    so that P' can never overflow fp16; O is multiplied back by 2^-E.
//    Q is converted from bf16 to fp16 once per CTA.
//  * Online softmax in the log2 domain with lazy rescaling: the running max
//    of a head is only raised (and O, l rescaled) when a tile's max exceeds
//    it by more than 2^8 (so p <= 256); otherwise the stale max is kept,
//    which is exact because O and l always share the same reference.
//  * A small resolve kernel first turns every selected position into its
//    (slot, scale) pair, fully in parallel, into caller-provided scratch.
//  * Warp roles (16 warps): 8 gather warps hold the next tile's FP8 rows in
//    registers (the whole tile is in flight while the current one is
//    multiplied; 8 lanes read one 128-byte row segment, so a warp load
//    touches only 4 cache lines), then convert and store them 128 columns at
//    a time as the previous tile's PV MMAs release the space; 8 softmax
//    warps (2 per TMEM lane quadrant, 32 heads each) turn S into P and
//    finally write O / l; the first softmax warp also allocates TMEM and
//    issues every MMA from one lane.  All hand-offs are mbarriers; every
//    wait is bounded in time and reports DSA_DEV_TIMEOUT instead of hanging.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace dsa {
namespace {

using namespace sm100;

constexpr int H = 64, DL = 512, DR = 64, DQK = DL + DR;
constexpr int T = 64;                  // KV rows per tile (two tiles are resident: double buffering)
constexpr int NKA = DQK / 64;          // 64-column slices ("katoms") per row: 9
constexpr int KATOM_BYTES = T * 128;   // one slice of a KV tile: 64 rows x 128 B
constexpr int TILE_BYTES = NKA * KATOM_BYTES;
constexpr int QATOM_BYTES = H * 128;   // one slice of Q: 64 heads x 128 B
constexpr int NTHREADS = 512;          // 16 warps
constexpr int NGATHER = 8;             // gather/convert warps 0..7; warp 0 also issues Q K^T
constexpr int GATHER_THREADS = NGATHER * 32;
constexpr int SOFTMAX_WARP0 = NGATHER; // softmax warps 8..15; warp 8 also issues P V
constexpr int SOFTMAX_WARPS = 8;
// per gather thread and tile: 2 chunks of each 128-column pair of slices + 1 rope chunk
constexpr int PAIR_CHUNKS = T * 8 / GATHER_THREADS;   // 2
constexpr int ROPE_CHUNKS = T * 4 / GATHER_THREADS;   // 1
static_assert(PAIR_CHUNKS * GATHER_THREADS == T * 8 && ROPE_CHUNKS * GATHER_THREADS == T * 4, "even split of a tile");
constexpr float RESCALE_LOG2 = 8.0f;   // a slow-path tile raises a head's reference max only past 2^8
constexpr float EXCEED_LOG2 = 8.0f;    // fast path while no logit exceeds its reference by 2^8 (p <= 256)
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// TMEM columns.  S^T of a tile is an M = 64 accumulator: row r of the tile
// lives in lane 32 (r / 16) + r % 16, columns = heads.  Each of the two tile
// buffers has its own S^T, accumulated in 2 independent partial sums over
// disjoint parts of the contraction (consecutive MMAs never share an
// accumulator); the softmax adds the parts.  O^T (M = 128) uses all lanes.
constexpr uint32_t TM_S = 0;     // S^T of buffer b, part p at TM_S + 64 (2 b + p)
constexpr uint32_t TM_O = 256;   // O^T chunk c at TM_O + 64 c
constexpr uint32_t TM_COLS = 512;

// shared memory map (offsets from a 1024-byte aligned base)
constexpr int OFF_KV = 0;                                  // 2 tile buffers
constexpr int OFF_Q = OFF_KV + 2 * TILE_BYTES;             // 147456
constexpr int OFF_RED = OFF_Q + NKA * QATOM_BYTES;         // 221184
constexpr int OFF_MUSE = OFF_RED + 4 * H * 4;
constexpr int OFF_ALPHA = OFF_MUSE + H * 4;
constexpr int OFF_FLAG = OFF_ALPHA + H * 4;
constexpr int OFF_BAR = OFF_FLAG + 128;
// barrier indices
constexpr int B_KV = 0;                 // [2] the tile in buffer b is in smem
constexpr int B_QFULL = B_KV + 2;       // Q is in smem
constexpr int B_SFULL = B_QFULL + 1;    // [2] S^T of the tile in buffer b is in TMEM
constexpr int B_PFULL = B_SFULL + 2;    // P of the current tile is in smem (and O rescaled)
constexpr int B_BFREE = B_PFULL + 1;    // [2] P V of the tile in buffer b is done: buffer free
constexpr int B_OFULL = B_BFREE + 2;    // all P V MMAs done
constexpr int B_SYNCA = B_OFULL + 1;    // softmax-group sync points
constexpr int B_SYNCB = B_SYNCA + 1;
constexpr int B_SYNCC = B_SYNCB + 1;
constexpr int B_FINQ = B_SYNCC + 1;     // the Q K^T issuer's MMAs are done
constexpr int B_FINP = B_FINQ + 1;      // the P V issuer's MMAs are done
constexpr int NBAR = B_FINP + 1;
constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
constexpr int SMEM_USED = OFF_TMEM + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint4 ldg_nc(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// 16 E4M3 bytes -> 16 fp16 (exact) as two 16-byte chunks, one cvt per pair
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)two));
  return h2;
}
__device__ __forceinline__ void convert16(const uint4& v, uint4& lo, uint4& hi) {
  lo.x = e4m3x2_to_f16x2(v.x & 0xffffu);
  lo.y = e4m3x2_to_f16x2(v.x >> 16);
  lo.z = e4m3x2_to_f16x2(v.y & 0xffffu);
  lo.w = e4m3x2_to_f16x2(v.y >> 16);
  hi.x = e4m3x2_to_f16x2(v.z & 0xffffu);
  hi.y = e4m3x2_to_f16x2(v.z >> 16);
  hi.z = e4m3x2_to_f16x2(v.w & 0xffffu);
  hi.w = e4m3x2_to_f16x2(v.w >> 16);
}

// 8 bf16 -> 8 fp16 (exact for |x| >= 2^-14; smaller values round to fp16's
// subnormal grid, 2^-24)
__device__ __forceinline__ uint4 bf16x8_to_f16x8(const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float lo = __uint_as_float(w[t] << 16), hi = __uint_as_float(w[t] & 0xffff0000u);
    const __half2 h = __floats2half2_rn(lo, hi);
    o[t] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Offset of 16-byte chunk `c` (0..7) of row `r` inside a 128-byte swizzled slice.
__device__ __forceinline__ uint32_t sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// Per-warp transpose-reduction: v[32] per lane (32 heads) -> lane l returns
// the reduction over the warp's 32 rows of head l.
template <bool IS_MAX>
__device__ __forceinline__ float warp_transpose_reduce(const float (&v)[32], int lane) {
  float a16[16];
  {
    const bool up = lane & 16;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float send = up ? v[i] : v[i + 16];
      const float keep = up ? v[i + 16] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, 16);
      a16[i] = IS_MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  float a8[8];
  {
    const bool up = lane & 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float send = up ? a16[i] : a16[i + 8];
      const float keep = up ? a16[i + 8] : a16[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, 8);
      a8[i] = IS_MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  float a4[4];
  {
    const bool up = lane & 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float send = up ? a8[i] : a8[i + 4];
      const float keep = up ? a8[i + 4] : a8[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, 4);
      a4[i] = IS_MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  float a2[2];
  {
    const bool up = lane & 2;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float send = up ? a4[i] : a4[i + 2];
      const float keep = up ? a4[i + 2] : a4[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, 2);
      a2[i] = IS_MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  const bool up = lane & 1;
  const float send = up ? a2[0] : a2[1];
  const float keep = up ? a2[1] : a2[0];
  const float got = __shfl_xor_sync(0xffffffffu, send, 1);
  return IS_MAX ? fmaxf(keep, got) : keep + got;
}

// Resolve every selected position into (slot, dequantisation scale) once,
// fully in parallel, so that the attention kernel's gathers depend on one
// contiguous load instead of a chain of three: idx -> block table -> scale.
// Invalid or padding entries get slot -1; bad inputs are reported.  It also
// records the largest scale each query selects (for the fp16 range of P).
__global__ void __launch_bounds__(256) resolve_kernel(const MlaArgs a, int2* __restrict__ res,
                                                      unsigned int* __restrict__ max_scale_bits) {
  // block (x, y): entries [256 x, 256 x + 256) of query y
  const int64_t i = blockIdx.y;
  const int j = blockIdx.x * 256 + threadIdx.x;
  float smax = 0.f;
  if (j < a.k) {
    const int64_t e = i * a.k + j;
    const int32_t pos = a.idx[e];
    int32_t slot = -1;
    float sc = 0.f;
    if (pos < -1) {
      report(a.dev_status, DSA_DEV_BAD_INDEX);
    } else if (pos >= 0) {
      const int32_t r = a.q_req[i];
      const int32_t pg = pos / a.page_size;
      if (r < 0 || r >= a.num_req) {
        report(a.dev_status, DSA_DEV_BAD_PAGE);
      } else if (pg >= a.bt_stride) {
        report(a.dev_status, DSA_DEV_BAD_INDEX);
      } else {
        const int32_t page = a.block_table[(int64_t)r * a.bt_stride + pg];
        if (page < 0 || page >= a.num_pages) {
          report(a.dev_status, DSA_DEV_BAD_PAGE);
        } else {
          slot = page * a.page_size + pos % a.page_size;
          sc = a.kv_scale[slot];
          smax = sc;
        }
      }
    }
    res[e] = make_int2(slot, __float_as_int(sc));
  }
  // the block's largest scale, then one atomic per block; scales are
  // non-negative, so their bit patterns order like the values
  __shared__ float wmax[8];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = smax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = wmax[0];
    for (int w = 1; w < 8; ++w) m = fmaxf(m, wmax[w]);
    if (m > 0.f) atomicMax(max_scale_bits + i, __float_as_uint(m));
  }
}

__global__ void __launch_bounds__(NTHREADS, 1) mla_tc_kernel(const MlaArgs a, const int2* __restrict__ res,
                                                             const unsigned int* __restrict__ max_scale_bits) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* kv_s = smem + OFF_KV;
  unsigned char* q_s = smem + OFF_Q;
  float* red_s = reinterpret_cast<float*>(smem + OFF_RED);
  float* muse_s = reinterpret_cast<float*>(smem + OFF_MUSE);
  float* alpha_s = reinterpret_cast<float*>(smem + OFF_ALPHA);
  int* vote_s = reinterpret_cast<int*>(smem + OFF_FLAG);  // [2][8] per-tile votes (double buffered)
  int* resc_s = vote_s + 16;                                // [2] rescale needed, per head half
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_TMEM);
  auto bar = [&](int b) { return smem_u32(bars + b); };
  // a bounded wait whose outcome is the same for every lane of the warp
  auto wait_warp = [&](int b, uint32_t parity) { return __all_sync(0xffffffffu, mbar_wait(bar(b), parity)); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i = blockIdx.x;        // query token
  const int split = blockIdx.y;
  const int S = gridDim.y;
  const int ntiles = (a.k + T - 1) / T;
  const int t_begin = (int)((int64_t)ntiles * split / S);
  const int t_end = (int)((int64_t)ntiles * (split + 1) / S);
  const int ntl = t_end - t_begin;
  const int2* row_res = res + (int64_t)i * a.k;

  if (ntl == 0) {  // an empty split: O = 0, lse = -inf
    for (int e = tid; e < H * DL; e += NTHREADS) {
      if (S == 1)
        static_cast<__nv_bfloat16*>(a.out)[(int64_t)i * H * DL + e] = __float2bfloat16_rn(0.f);
      else
        a.o_part[((int64_t)split * a.num_q + i) * H * DL + e] = 0.f;
    }
    for (int h = tid; h < H; h += NTHREADS) {
      if (S == 1) {
        if (a.lse) a.lse[(int64_t)i * H + h] = -INFINITY;
      } else {
        a.lse_part[((int64_t)split * a.num_q + i) * H + h] = -INFINITY;
      }
    }
    return;
  }

  // ---------------- setup ----------------
  if (warp == SOFTMAX_WARP0) {
    tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_KV + b), NGATHER);
      mbar_init(bar(B_SFULL + b), 1);
      mbar_init(bar(B_BFREE + b), 1);
    }
    mbar_init(bar(B_QFULL), NGATHER);
    mbar_init(bar(B_PFULL), SOFTMAX_WARPS);
    mbar_init(bar(B_OFULL), 1);
    mbar_init(bar(B_SYNCA), SOFTMAX_WARPS);
    mbar_init(bar(B_SYNCB), SOFTMAX_WARPS);
    mbar_init(bar(B_SYNCC), SOFTMAX_WARPS);
    mbar_init(bar(B_FINQ), 1);
    mbar_init(bar(B_FINP), 1);
    fence_mbarrier_init();
  }
  if (tid < H) {
    muse_s[tid] = -INFINITY;
    alpha_s[tid] = 1.f;
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t kv_base = smem_u32(kv_s), q_base = smem_u32(q_s);
  bool ok = true;

  if (warp >= SOFTMAX_WARP0) {
    // ---------------- softmax warps (warp 8 also issues the P V MMAs) ----------------
    const int q4 = warp & 3;                        // TMEM lane quadrant
    const int half = (warp - SOFTMAX_WARP0) >> 2;  // heads [32 half, 32 half + 32)
    const int sw = warp - SOFTMAX_WARP0;            // softmax warp 0..7
    const bool issuer = (warp == SOFTMAX_WARP0);
    const bool row_lane = lane < 16;                // lanes 16..31 hold no row of an M = 64 accumulator
    const int j = 16 * q4 + (lane & 15);            // KV row of the tile held by this lane
    const uint32_t t_lane = tmem + ((uint32_t)(32 * q4) << 16);
    const float qk_scale = a.softmax_scale * LOG2E;
    // P' = p s_j 2^E with p <= 256: pick E so that 256 * max_j s_j * 2^E <= 2^15
    int p_exp = 0;
    {
      const float smax = __uint_as_float(max_scale_bits[i]);
      if (smax > 0.f) {
        int e2;
        frexpf(smax, &e2);  // smax < 2^e2
        p_exp = 7 - e2;
      }
    }
    const float p_scale = ldexpf(1.f, p_exp);
    constexpr uint32_t ID_PV = idesc_f16_f32(128, 64, 1, 1, 0);

    // O^T += V^T P^T for the tile in buffer b: the 4 independent 128-dim
    // chunks are issued round robin so that consecutive MMAs never share an
    // accumulator
    auto issue_pv = [&](int lt, int b) {
      const uint64_t a0 = smem_desc_sw128(kv_base + b * TILE_BYTES, KATOM_BYTES, 1024);
      const uint64_t b0 = smem_desc_sw128(kv_base + b * TILE_BYTES + 8 * KATOM_BYTES, KATOM_BYTES, 1024);
#pragma unroll
      for (int kk = 0; kk < T / 16; ++kk) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          mma_f16_ss_warp(tmem + TM_O + 64 * c, a0 + ((2 * c * KATOM_BYTES + kk * 2048) >> 4), b0 + ((kk * 2048) >> 4),
                          ID_PV, (lt > 0 || kk > 0) ? 1u : 0u);
        }
      }
      mma_commit_warp(bar(B_BFREE + b));
    };

    float l_part[32];
#pragma unroll
    for (int h = 0; h < 32; ++h) l_part[h] = 0.f;
    uint32_t ph_a = 0, ph_b = 0, ph_c = 0;  // completed phases of the group barriers
    auto group_sync = [&](int bb, uint32_t& ph) {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(bb));
      const bool done = wait_warp(bb, ph & 1);
      ++ph;
      return done;
    };
    // (slot, scale) of this thread's row, one tile ahead
    auto row_info = [&](int lt) -> int2 {
      const int e = (t_begin + lt) * T + j;
      return (row_lane && e < a.k) ? __ldg(row_res + e) : make_int2(-1, 0);
    };
    int2 info = row_info(0);
    for (int lt = 0; lt < ntl && ok; ++lt) {
      const int b = lt & 1;
      const int2 info_next = lt + 1 < ntl ? row_info(lt + 1) : make_int2(-1, 0);
      if (!wait_warp(B_SFULL + b, (lt >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const bool valid = info.x >= 0;
      const float sc = __int_as_float(info.y);
      const float cj = sc * qk_scale;
      // logits of row j in the log2 domain (invalid rows and idle lanes: -inf)
      auto load_z = [&](float (&z)[32]) {
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          float v0[16], v1[16];
          tmem_ld16(t_lane + TM_S + 64 * (2 * b) + half * 32 + 16 * g, v0);
          tmem_ld16(t_lane + TM_S + 64 * (2 * b + 1) + half * 32 + 16 * g, v1);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 16; ++h) z[16 * g + h] = valid ? (v0[h] + v1[h]) * cj : -INFINITY;
        }
      };
      float z[32];
      load_z(z);
      // Fast path: probabilities are taken against the heads' current
      // reference maxima; that stays exact as long as no logit exceeds its
      // reference by more than 2^EXCEED (p <= 256, no fp16 overflow).  One
      // vote of the 8 warps decides; only then is the tile maximum reduced.
      bool bad = false;
      {
        const float4* mu4 = reinterpret_cast<const float4*>(muse_s + half * 32);
#pragma unroll
        for (int h4 = 0; h4 < 8; ++h4) {
          const float4 m = mu4[h4];
          bad |= z[4 * h4] > m.x + EXCEED_LOG2;
          bad |= z[4 * h4 + 1] > m.y + EXCEED_LOG2;
          bad |= z[4 * h4 + 2] > m.z + EXCEED_LOG2;
          bad |= z[4 * h4 + 3] > m.w + EXCEED_LOG2;
        }
        bad &= valid;
      }
      const unsigned bv = __ballot_sync(0xffffffffu, bad);
      if (lane == 0) vote_s[(lt & 1) * SOFTMAX_WARPS + sw] = bv != 0u;
      if (!group_sync(B_SYNCA, ph_a)) {
        ok = false;
        break;
      }
      int anybad = 0;
#pragma unroll
      for (int w = 0; w < SOFTMAX_WARPS; ++w) anybad |= vote_s[(lt & 1) * SOFTMAX_WARPS + w];
      if (anybad) {  // uniform over the 8 warps
        red_s[q4 * H + half * 32 + lane] = warp_transpose_reduce<true>(z, lane);
        if (!group_sync(B_SYNCB, ph_b)) {
          ok = false;
          break;
        }
        if (q4 == 0) {  // warps 8 and 12 own 32 heads each
          const int hh = half * 32 + lane;
          const float mt = fmaxf(fmaxf(red_s[hh], red_s[H + hh]), fmaxf(red_s[2 * H + hh], red_s[3 * H + hh]));
          const float mo = muse_s[hh];
          float alpha = 1.f;
          if (mt > mo + RESCALE_LOG2) {
            alpha = (mo == -INFINITY) ? 0.f : ex2(mo - mt);
            muse_s[hh] = mt;
          }
          alpha_s[hh] = alpha;
          const unsigned need = __ballot_sync(0xffffffffu, lt > 0 && alpha != 1.f);
          if (lane == 0) resc_s[half] = need != 0u;
        }
        if (!group_sync(B_SYNCC, ph_c)) {
          ok = false;
          break;
        }
        if (resc_s[half]) {
          // O must hold every P V issued so far: the previous tile's
          if (!wait_warp(B_BFREE + (b ^ 1), ((lt - 1) >> 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const float* al = alpha_s + half * 32;
#pragma unroll
          for (int h = 0; h < 32; ++h) l_part[h] *= al[h];
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              float o[16];
              const uint32_t addr = t_lane + TM_O + 64 * c + half * 32 + 16 * g;
              tmem_ld16(addr, o);
              tmem_wait_ld();
#pragma unroll
              for (int h = 0; h < 16; ++h) o[h] *= al[16 * g + h];
              tmem_st16(addr, o);
            }
          }
          tmem_wait_st();
        }
        load_z(z);  // S is still in TMEM: reload rather than keep z live across the rescale
      }
      // probabilities, folded with the row's dequantisation scale and the
      // query's power of two, as fp16 P (row j of the rope slice of buffer b)
      uint32_t pk[16];
      const float sp = sc * p_scale;
      const float4* mu4 = reinterpret_cast<const float4*>(muse_s + half * 32);
#pragma unroll
      for (int h4 = 0; h4 < 8; ++h4) {
        const float4 m = mu4[h4];
        const float mm[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int h = 4 * h4 + 2 * t;
          const float p0 = valid ? ex2(z[h] - mm[2 * t]) : 0.f;
          const float p1 = valid ? ex2(z[h + 1] - mm[2 * t + 1]) : 0.f;
          l_part[h] += p0;
          l_part[h + 1] += p1;
          const __half2 hp = __floats2half2_rn(p0 * sp, p1 * sp);
          pk[h / 2] = *reinterpret_cast<const uint32_t*>(&hp);
        }
      }
      if (row_lane) {
        unsigned char* p_row = kv_s + b * TILE_BYTES + 8 * KATOM_BYTES;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          *reinterpret_cast<uint4*>(p_row + sw128(j, half * 4 + cc)) =
              make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL));
      if (issuer) {
        ok = wait_warp(B_PFULL, lt & 1);
        if (ok) {
          tc_fence_after_sync();
          issue_pv(lt, b);
        }
      }
      info = info_next;
    }
    if (issuer) {
      __syncwarp();
      mma_commit_warp(bar(B_OFULL));
      mma_commit_warp(bar(B_FINP));
    }
    // ---------------- epilogue: normalise and write ----------------
    if (ok && !wait_warp(B_OFULL, 0)) ok = false;
    if (ok) {
      tc_fence_after_sync();
      red_s[q4 * H + half * 32 + lane] = warp_transpose_reduce<false>(l_part, lane);
      ok = group_sync(B_SYNCB, ph_b);
    }
    if (ok) {
      if (q4 == 0) {
        const int hh = half * 32 + lane;
        const float l = red_s[hh] + red_s[H + hh] + red_s[2 * H + hh] + red_s[3 * H + hh];
        const float m = muse_s[hh];
        alpha_s[hh] = l > 0.f ? ldexpf(1.f / l, -p_exp) : 0.f;
        const float lse = l > 0.f ? (m + log2f(l)) * LN2 : -INFINITY;
        if (S == 1) {
          if (a.lse) a.lse[(int64_t)i * H + hh] = lse;
        } else {
          a.lse_part[((int64_t)split * a.num_q + i) * H + hh] = lse;
        }
      }
      ok = group_sync(B_SYNCC, ph_c);
    }
    if (ok) {
      const float* inv = alpha_s + half * 32;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        const int d = 128 * c + 32 * q4 + lane;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          float o[16];
          tmem_ld16(t_lane + TM_O + 64 * c + half * 32 + 16 * g, o);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 16; ++h) {
            const int hh = half * 32 + 16 * g + h;
            const float val = o[h] * inv[16 * g + h];
            const int64_t off = ((int64_t)i * H + hh) * DL + d;
            if (S == 1)
              static_cast<__nv_bfloat16*>(a.out)[off] = __float2bfloat16_rn(val);
            else
              a.o_part[(int64_t)split * a.num_q * H * DL + off] = val;
          }
        }
      }
    } else {
      report(a.dev_status, DSA_DEV_TIMEOUT);
    }
    // all issued MMAs must be finished before TMEM is released
    if (issuer && lane == 0 && !mbar_wait(bar(B_FINP), 0)) report(a.dev_status, DSA_DEV_TIMEOUT);
    __syncwarp();
  } else {
    // ---------------- gather warps: FP8 rows -> registers -> fp16 swizzled tiles ----------------
    const int gtid = warp * 32 + lane;  // 0..255
    const bool qk_issuer = (warp == 0);
    constexpr uint32_t ID_QK = idesc_f16_f32(64, 64, 0, 0, 0);
    // S^T = K Q^T for the tile in buffer b; the 16-wide steps alternate
    // between the 2 partial accumulators of that buffer
    auto issue_qk = [&](int b) {
      const uint64_t a0 = smem_desc_sw128(kv_base + b * TILE_BYTES, 16, 1024);
      const uint64_t b0 = smem_desc_sw128(q_base, 16, 1024);
#pragma unroll
      for (int ka = 0; ka < NKA; ++ka) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t part = kk & 1;
          mma_f16_ss_warp(tmem + TM_S + 64 * (2 * b + part), a0 + ((ka * KATOM_BYTES + kk * 32) >> 4),
                          b0 + ((ka * QATOM_BYTES + kk * 32) >> 4), ID_QK, (ka > 0 || kk > 1) ? 1u : 0u);
        }
      }
      mma_commit_warp(bar(B_SFULL + b));
    };
    // rows of the tile this thread gathers: 2 for the slice pairs, 1 for the rope slice
    int pr_row[PAIR_CHUNKS], rp_row[ROPE_CHUNKS];
#pragma unroll
    for (int u = 0; u < PAIR_CHUNKS; ++u) pr_row[u] = (gtid + GATHER_THREADS * u) >> 3;
#pragma unroll
    for (int u = 0; u < ROPE_CHUNKS; ++u) rp_row[u] = (gtid + GATHER_THREADS * u) >> 2;
    // Q of this token -> swizzled K-major slices (fp16)
    {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) + (int64_t)i * H * DQK);
      constexpr int CH = DQK / 8;
      uint4 qv[H * CH / GATHER_THREADS];
#pragma unroll
      for (int u = 0; u < H * CH / GATHER_THREADS; ++u) qv[u] = __ldg(src + gtid + GATHER_THREADS * u);
#pragma unroll
      for (int u = 0; u < H * CH / GATHER_THREADS; ++u) {
        const int e = gtid + GATHER_THREADS * u;
        const int h = e / CH, cc = e % CH;
        *reinterpret_cast<uint4*>(q_s + (cc >> 3) * QATOM_BYTES + sw128(h, cc & 7)) = bf16x8_to_f16x8(qv[u]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_QFULL));
    }
    // Two tiles' rows held in registers (stage s holds the tile for buffer s):
    // for each pair c of 64-column slices 2 chunks of 16 bytes (8 lanes per
    // 128-byte row segment), and 1 chunk of the rope slice.
    uint4 pr[2][4][PAIR_CHUNKS];
    uint4 rp[2][ROPE_CHUNKS];
    auto load_tile = [&](int lt, uint4 (&prs)[4][PAIR_CHUNKS], uint4 (&rps)[ROPE_CHUNKS]) {
      const int base = (t_begin + lt) * T;
      int ps[PAIR_CHUNKS], rs[ROPE_CHUNKS];
#pragma unroll
      for (int u = 0; u < PAIR_CHUNKS; ++u) ps[u] = base + pr_row[u] < a.k ? __ldg(&row_res[base + pr_row[u]].x) : -1;
#pragma unroll
      for (int u = 0; u < ROPE_CHUNKS; ++u) rs[u] = base + rp_row[u] < a.k ? __ldg(&row_res[base + rp_row[u]].x) : -1;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int u = 0; u < PAIR_CHUNKS; ++u) {
          const int c8 = (gtid + GATHER_THREADS * u) & 7;
          prs[c][u] = make_uint4(0u, 0u, 0u, 0u);
          if (ps[u] >= 0) prs[c][u] = ldg_nc(a.kv + (int64_t)ps[u] * DQK + c * 128 + c8 * 16);
        }
      }
#pragma unroll
      for (int u = 0; u < ROPE_CHUNKS; ++u) {
        const int c16 = (gtid + GATHER_THREADS * u) & 3;
        rps[u] = make_uint4(0u, 0u, 0u, 0u);
        if (rs[u] >= 0) rps[u] = ldg_nc(a.kv + (int64_t)rs[u] * DQK + DL + c16 * 16);
      }
    };
    auto store_tile = [&](int b, const uint4 (&prs)[4][PAIR_CHUNKS], const uint4 (&rps)[ROPE_CHUNKS]) {
      unsigned char* tile = kv_s + b * TILE_BYTES;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int u = 0; u < PAIR_CHUNKS; ++u) {
          const int e = gtid + GATHER_THREADS * u;
          const int row = e >> 3, c8 = e & 7;
          const int slice = 2 * c + (c8 >> 2), c16 = c8 & 3;
          uint4 lo, hi;
          convert16(prs[c][u], lo, hi);
          unsigned char* dst = tile + slice * KATOM_BYTES;
          // Each quarter warp (8 lanes: one row, two slices) must hit 8
          // distinct 16-byte bank groups: lanes of the second slice store
          // their odd chunk first.
          const bool odd_first = c8 & 4;
          *reinterpret_cast<uint4*>(dst + sw128(row, 2 * c16 + (odd_first ? 1 : 0))) = odd_first ? hi : lo;
          *reinterpret_cast<uint4*>(dst + sw128(row, 2 * c16 + (odd_first ? 0 : 1))) = odd_first ? lo : hi;
        }
      }
#pragma unroll
      for (int u = 0; u < ROPE_CHUNKS; ++u) {
        const int e = gtid + GATHER_THREADS * u;
        const int row = e >> 2, c16 = e & 3;
        uint4 lo, hi;
        convert16(rps[u], lo, hi);
        unsigned char* dst = tile + 8 * KATOM_BYTES;
        *reinterpret_cast<uint4*>(dst + sw128(row, 2 * c16)) = lo;
        *reinterpret_cast<uint4*>(dst + sw128(row, 2 * c16 + 1)) = hi;
      }
    };
    // one step of the pipeline for the tile lt held in stage `st`
    auto step = [&](int lt, uint4 (&prs)[4][PAIR_CHUNKS], uint4 (&rps)[ROPE_CHUNKS]) {
      const int b = lt & 1;
      // the buffer is free once P V of the tile two back is done
      if (lt >= 2 && !wait_warp(B_BFREE + b, ((lt - 2) >> 1) & 1)) ok = false;
      if (ok) store_tile(b, prs, rps);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_KV + b));
      if (qk_issuer && ok) {
        ok = (lt > 0 || wait_warp(B_QFULL, 0)) && wait_warp(B_KV + b, (lt >> 1) & 1);
        if (ok) {
          tc_fence_after_sync();
          issue_qk(b);
        }
      }
      if (ok && lt + 2 < ntl) load_tile(lt + 2, prs, rps);  // two tiles ahead
    };
    load_tile(0, pr[0], rp[0]);
    if (ntl > 1) load_tile(1, pr[1], rp[1]);
    for (int lt = 0; lt < ntl && ok; lt += 2) {
      step(lt, pr[0], rp[0]);
      if (lt + 1 < ntl && ok) step(lt + 1, pr[1], rp[1]);
    }
    if (qk_issuer) {
      __syncwarp();
      mma_commit_warp(bar(B_FINQ));
      if (!mbar_wait(bar(B_FINQ), 0) && lane == 0) report(a.dev_status, DSA_DEV_TIMEOUT);
    }
    if (!ok) report(a.dev_status, DSA_DEV_TIMEOUT);
  }

  // ---------------- teardown ----------------
  tc_fence_before_sync();
  __syncthreads();
  if (warp == SOFTMAX_WARP0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, TM_COLS);
  }
}

}  // namespace

bool mla_tc_supported(const MlaArgs& a) { return a.heads == H && a.d_latent == DL && a.d_rope == DR; }

size_t mla_tc_workspace_bytes(int32_t num_q, int32_t k) {
  // resolved (slot, scale) per entry, then the largest scale per query
  return sizeof(int2) * (size_t)num_q * (size_t)k + sizeof(int2) * (((size_t)num_q + 1) / 2);
}

cudaError_t launch_mla_tc(const MlaArgs& a, void* workspace, cudaStream_t stream) {
  if (a.num_q == 0) return cudaSuccess;
  int2* res = static_cast<int2*>(workspace);
  unsigned int* max_bits = reinterpret_cast<unsigned int*>(res + (size_t)a.num_q * a.k);
  cudaError_t e = cudaMemsetAsync(max_bits, 0, sizeof(unsigned int) * (size_t)a.num_q, stream);
  if (e != cudaSuccess) return e;
  const dim3 rgrid((a.k + 255) / 256, a.num_q);
  resolve_kernel<<<rgrid, 256, 0, stream>>>(a, res, max_bits);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(mla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(a.num_q, a.num_splits);
  mla_tc_kernel<<<grid, NTHREADS, SMEM_BYTES, stream>>>(a, res, max_bits);
  return cudaGetLastError();
}

}  // namespace dsa
