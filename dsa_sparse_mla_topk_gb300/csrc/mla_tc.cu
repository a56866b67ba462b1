// Sparse MLA attention on the Blackwell tensor cores (tcgen05 + TMEM + TMA).
//
// "Accelerating GLM-5.3-Flash on H200", section 3 "Larger KV tiles for DSA
// Partial": the Partial step loads the KV positions the indexer selected and
// computes Q K^T, an online softmax and the weighted value sum, one KV tile at
// a time (Figure 4: the last tile is padded virtually, the index tensor is
// left alone); a KV split writes a partial result for the Combine step.
// "GLM-5.3 Optimizations, Part 2" ("Interpretation"): every latent KV row is
// shared by all 64 heads of a query token.
//
// GB300 design (one CTA = one query token x one KV split, 16 warps):
//  * KV tiles of 64 selected rows stay FP8 E4M3 from HBM to the tensor cores.
//    Seven TMA warps gather the rows straight from the paged cache into
//    shared memory with tile::gather4 (four arbitrary rows per copy; 128-byte
//    swizzle for the 512 latent columns, 64-byte swizzle for the 64 rope
//    columns; rows past the selection read as zeros); five tiles are in
//    flight and no thread touches KV bytes.
//  * One MMA warp issues kind::f8f6f4 MMAs:
//        S    = [Q_hi ; Q_lo] K^T          M = 128 (64 heads hi, 64 lo), N = 64 rows, K = 576
//        O^T += V^T P_hi^T + V^T P_lo^T    M = 4 x 128 latent dims, N = 64 heads, K = 64 rows
//    The latent part of Q is the A operand straight from tensor memory (the
//    MMA then reads only the 2 KB K slice from shared memory per step and
//    runs at the tensor pipe's full rate); its rope part and K come from
//    shared memory.  V^T is the same shared-memory tile read MN-major.  Every
//    gathered row serves all 64 heads.
//  * Q (bf16) and P (fp32) are carried as sums of two E4M3 numbers, hi =
//    E4M3(x) and lo = E4M3(x - hi): about 8 significant bits, the precision
//    of bf16.  Q is scaled by a power of two per query token so that its
//    largest element lies in [128, 256); P by a power of two chosen from the
//    largest selected dequantisation scale so that P < 256.  Both are exact
//    and undone in fp32.
//  * The per-token dequantisation scale s_j multiplies the logits of row j
//    and is folded into P before rounding (P'_hj = p_hj s_j 2^E), so V is used
//    as the raw FP8 values.
//  * 8 softmax warps (2 per TMEM lane quadrant) turn S into P.  Lane quadrant
//    q holds heads 16 q .. 16 q + 15: Q_hi rows in its lanes 0-15, Q_lo rows
//    in lanes 16-31, so one shuffle adds the two halves of a logit; each
//    thread then owns one head and 16 rows of a tile.  Online softmax in the
//    log2 domain with lazy rescaling: a head's reference max is raised (and
//    O, l rescaled) only when a logit exceeds it by more than 2^4, so
//    p <= 16 always.
//  * TMEM holds two S buffers (2 x 64 columns), Q's latent A operand (128
//    columns) and O^T (4 x 64 columns); shared memory holds two P buffers.
//    QK^T runs two tiles ahead of P V: QK^T of tile t+2 is issued right after
//    P V of tile t, while the softmax of tile t+1 runs.  All hand-offs
//    between warp roles are mbarriers, and every mbarrier wait is bounded in
//    time and reports DSA_DEV_TIMEOUT instead of hanging; the softmax warps'
//    per-tile vote is a named barrier with an OR reduction, which every
//    softmax warp reaches once per tile whatever happened before.
//  * The epilogue reads O^T from TMEM and stores it, normalised, straight to
//    global memory (bf16 output, or the fp32 partial of a KV split).
//  * A small resolve kernel first turns every selected position into its
//    (slot, scale) pair, fully in parallel, into caller-provided scratch;
//    the attention kernel is its programmatic dependent and overlaps it.
//    On the two-kernel pass the top-k kernel writes those pairs itself and
//    the attention kernel follows it directly.  The single-kernel variant
//    (FUSED) selects its token's top k, resolves it and converts Q in its
//    own prologue instead.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "internal.cuh"
#include "sm100_ptx.cuh"
#include "topk_row.cuh"

namespace dsa {
namespace {

using namespace sm100;

constexpr int H = 64, DL = 512, DR = 64, DQK = DL + DR;
constexpr int T = 64;                            // KV rows per tile
constexpr int NST = 5;                           // KV tiles in flight
constexpr int NLAT = DL / 128;                   // 128-column latent slices per row: 4
constexpr int LAT_BYTES = T * 128;               // one latent slice of a tile (128-byte swizzle)
constexpr int ROPE_OFF = NLAT * LAT_BYTES;       // the rope slice (64-byte swizzle)
constexpr int STAGE_BYTES = ROPE_OFF + T * DR;   // 36 KB per tile
constexpr int QM = 2 * H;                        // A rows of Q K^T: Q_hi and Q_lo of every head
constexpr int QROPE_BYTES = QM * DR;             // Q's rope part in shared memory (64-byte swizzle)
constexpr int P_BYTES = H * T;                   // P_hi (or P_lo) of a tile: [head][row], K-major, 64-byte swizzle
constexpr int NPB = 2;                           // P buffers
constexpr int NTHREADS = 512;
// Warp roles: 0-3 and 5-7 gather (a single CTA's TMA throughput grows with
// the number of warps issuing copies), 4 issues the MMAs, 8-15 run the
// softmax (two per TMEM lane quadrant).
constexpr int WARP_MMA = 4, NTMA = 7;
constexpr int SOFTMAX_WARP0 = 8, SOFTMAX_WARPS = 8;
constexpr int GROUPS = T / 4;                    // gather4 row groups per tile
constexpr float EXCEED_LOG2 = 4.0f;              // p = 2^(z - m) <= 2^4
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// TMEM columns: S of buffer b at TM_S + 64 b (M = 128: lane = Q row, column =
// tile row), Q's latent A operand at TM_Q (128 columns, 4 bytes of K each),
// O^T chunk c at TM_O + 64 c (M = 128: latent dim 128 c + lane, column = head).
// Q row (= lane) of head h: 32 (h / 16) + h % 16 for Q_hi, 16 more for Q_lo.
constexpr uint32_t TM_S = 0, TM_Q = 2 * T, TM_O = 256, TM_COLS = 512;
static_assert(TM_Q + DL / 4 == TM_O, "S, Q and O fill the 512 TMEM columns");
__host__ __device__ constexpr int q_row(int h, int lo) { return 32 * (h >> 4) + (h & 15) + 16 * lo; }

// shared memory map (offsets from a 1024-byte aligned base)
constexpr int OFF_KV = 0;
constexpr int OFF_QR = OFF_KV + NST * STAGE_BYTES;   // Q rope rows (hi and lo)
constexpr int OFF_P = OFF_QR + QROPE_BYTES;          // [buffer][hi, lo]
constexpr int OFF_RED = OFF_P + NPB * 2 * P_BYTES;   // [4][64] floats: reductions
constexpr int OFF_ALPHA = OFF_RED + 4 * H * 4;       // per-head rescale factor, then 1 / l
constexpr int OFF_ROWF = OFF_ALPHA + H * 4;          // [8 warps][2 tiles][32 rows] logit factor
constexpr int OFF_FLAG = OFF_ROWF + SOFTMAX_WARPS * 2 * 32 * 4;  // rescale flags [4], Q exponent, largest scales [8]
constexpr int OFF_BAR = OFF_FLAG + 128;
constexpr int B_KVF = 0;                  // [NST] tile in stage s has landed (TMA transaction bytes)
constexpr int B_KVE = B_KVF + NST;        // [NST] stage s is free (its P V MMAs are done)
constexpr int B_SF = B_KVE + NST;         // [2] S buffer b is complete
constexpr int B_PF = B_SF + 2;            // [2] P buffer b is written (and O rescaled)
constexpr int B_PVD = B_PF + NPB;         // [2] P V of the tile in P buffer b is done (waited on before rescaling O)
constexpr int B_OF = B_PVD + NPB;         // every P V is done
constexpr int B_SYNCB = B_OF + 1;         // softmax-group sync points
constexpr int B_SYNCC = B_SYNCB + 1;
constexpr int B_FIN = B_SYNCC + 1;        // every MMA is done (teardown)
constexpr int B_QREADY = B_FIN + 1;       // Q hi/lo is in shared memory (and the Q staging stages are free)
constexpr int B_QLOAD = B_QREADY + 1;     // raw bf16 Q has landed in the staging stages
constexpr int B_QEXP = B_QLOAD + 1;       // Q's power-of-two scale is in shared memory
constexpr int NBAR = B_QEXP + 1;
constexpr int QSTAGE = NST - 2;           // raw bf16 Q is staged in KV stages NST - 2 and NST - 1
static_assert(2 * STAGE_BYTES == H * DQK * 2, "bf16 Q fills two KV stages");
constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
constexpr int SMEM_USED = OFF_TMEM + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(OFF_QR % 1024 == 0 && OFF_P % 1024 == 0 && STAGE_BYTES % 1024 == 0, "swizzle atoms stay aligned");

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// f16x2 -> hi = E4M3(x) and lo = E4M3(x - hi) as byte pairs (low half ->
// low byte).  x - hi is exact in fp16: hi is x rounded to 4 significant bits.
__device__ __forceinline__ void split_e4m3x2(uint32_t h2, uint32_t& hi, uint32_t& lo) {
  unsigned short a, b;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(a) : "r"(h2));
  uint32_t back;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(back) : "h"(a));
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h2), *reinterpret_cast<const __half2*>(&back));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(b) : "r"(*reinterpret_cast<const uint32_t*>(&r)));
  hi = a;
  lo = b;
}
// Two-wide fp32 arithmetic, each lane rounded as its scalar .rn form.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float x0, float x1) {
  const __half2 h = __floats2half2_rn(x0, x1);  // x0 in the low half
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Resolve every selected position into (slot, dequantisation scale) once,
// fully in parallel, so that the attention kernel's gathers depend on one
// contiguous load instead of a chain of three: idx -> block table -> scale.
// Invalid or padding entries get slot -1; bad inputs are reported.  It is
// itself a programmatic dependent of the previous kernel on the stream
// (normally the top-k, whose indices it reads), and the attention kernel is
// its programmatic dependent: that starts (Q copy and split) while this runs
// and waits for it before reading `res`.
constexpr int RES_THREADS = 256;
// RES_ENT entries per thread: block (x, y) resolves entries
// [256 RES_ENT x, 256 RES_ENT (x + 1)) of query y, thread t the entries
// 256 RES_ENT x + 256 e + t.  Each of the chain's three dependent loads
// (index, block table, scale) is issued for all of a thread's entries before
// the next, so a thread waits for three round trips whatever RES_ENT is.  One
// entry per thread while the call fits in about two waves of threads (the
// most CTAs for the latency chain); eight beyond that, so that a large call
// (verify, prefill) takes about one wave instead of many.
template <int RES_ENT>
__global__ void __launch_bounds__(RES_THREADS) resolve_kernel(const MlaArgs a, int2* __restrict__ res) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t i = blockIdx.y;
  const int j0 = blockIdx.x * RES_THREADS * RES_ENT + threadIdx.x;
  // block 0 of each query also pulls the query's Q (72 KB) into L2 for the
  // attention kernel's bulk copy
  if (blockIdx.x == 0) {
    const char* qb = reinterpret_cast<const char*>(static_cast<const __nv_bfloat16*>(a.q) + i * H * DQK);
    for (int off = threadIdx.x * 128; off < H * DQK * 2; off += RES_THREADS * 128)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(qb + off));
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the indices are complete
  const int32_t r = a.q_req[i];
  const bool req_ok = r >= 0 && r < a.num_req;
  int32_t pos[RES_ENT], page[RES_ENT];
#pragma unroll
  for (int e = 0; e < RES_ENT; ++e) {
    const int j = j0 + RES_THREADS * e;
    pos[e] = j < a.k ? a.idx[i * a.k + j] : -1;
  }
#pragma unroll
  for (int e = 0; e < RES_ENT; ++e) {
    page[e] = -1;
    if (pos[e] >= 0 && req_ok && pos[e] / a.page_size < a.bt_stride)
      page[e] = a.block_table[(int64_t)r * a.bt_stride + pos[e] / a.page_size];
  }
  int32_t slot[RES_ENT];
  float sc[RES_ENT];
#pragma unroll
  for (int e = 0; e < RES_ENT; ++e) {
    slot[e] = -1;
    sc[e] = 0.f;
    if (pos[e] < -1) {
      report(a.dev_status, DSA_DEV_BAD_INDEX);
    } else if (pos[e] >= 0) {
      if (!req_ok) {
        report(a.dev_status, DSA_DEV_BAD_PAGE);
      } else if (pos[e] / a.page_size >= a.bt_stride) {
        report(a.dev_status, DSA_DEV_BAD_INDEX);
      } else if (page[e] < 0 || page[e] >= a.num_pages) {
        report(a.dev_status, DSA_DEV_BAD_PAGE);
      } else {
        slot[e] = page[e] * a.page_size + pos[e] % a.page_size;
        sc[e] = a.kv_scale[slot[e]];
      }
    }
  }
#pragma unroll
  for (int e = 0; e < RES_ENT; ++e) {
    const int j = j0 + RES_THREADS * e;
    if (j < a.k) res[i * a.k + j] = make_int2(slot[e], __float_as_int(sc[e]));
  }
}

// The single-kernel path's top-k inputs (unused by the plain kernel).
struct TopkIn {
  const float* scores;  // fp32 [num_q, ld]
  int64_t ld;
  const int32_t* q_pos;
  int32_t* idx;         // output: int32 [num_q, k]
};

// The fused kernel selects its token's top k in KV stages 0 and 1 (candidate
// keys, histogram, candidate positions, one bitmap) and the P buffers (the
// other bitmap), all idle until the gathers start; the raw bf16 Q lands in
// the last two stages meanwhile.
// The chosen positions overwrite the candidate keys once those are read.
// The resolve step holds four entries per thread: k <= 2048.
constexpr int FUSED_MAX_K = 4 * NTHREADS;
static_assert(FUSED_MAX_K <= RLCAP, "the chosen positions fit where the candidate keys were");
static_assert(sizeof(uint32_t) * (RLCAP + HBINS + RWORDS) + sizeof(uint16_t) * RLCAP == 2 * STAGE_BYTES,
              "the top-k arrays but one bitmap fill KV stages 0 and 1");
static_assert(sizeof(uint32_t) * RWORDS <= NPB * 2 * P_BYTES, "the other bitmap fits in the P buffers");
static_assert(QSTAGE >= 2, "the raw Q stays clear of the top-k arrays");
static_assert(NTHREADS == RNT, "one CTA selects a row");

// FUSED = false: attention over indices a previous top-k call chose, with
// `res` filled by resolve_kernel.  FUSED = true (decode, one KV split): the
// CTA first selects its own token's top k (the same selection the top-k
// kernel makes), writes it to tk.idx and resolves it into `res`, then
// attends to it: no kernel boundary and no wait for other tokens' rows.
template <bool FUSED>
__global__ void __launch_bounds__(NTHREADS, 1)
    mla_tc_kernel(const MlaArgs a, const __grid_constant__ CUtensorMap tmap_lat,
                  const __grid_constant__ CUtensorMap tmap_rope, int2* __restrict__ res, const TopkIn tk) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* qr_s = smem + OFF_QR;
  unsigned char* p_s = smem + OFF_P;
  float* red_s = reinterpret_cast<float*>(smem + OFF_RED);
  float* alpha_s = reinterpret_cast<float*>(smem + OFF_ALPHA);
  int* resc_s = reinterpret_cast<int*>(smem + OFF_FLAG);  // [4] rescale needed, per lane quadrant
  int* qexp_s = resc_s + 4;                                  // Q's power-of-two scale
  float* smax_s = reinterpret_cast<float*>(resc_s + 5);     // [8] softmax warps' largest scales
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
  // the fused kernel writes `res` itself, so it reads it back coherently
  auto ld_res = [&](const int2* p) -> int2 {
    if constexpr (FUSED) return __ldcg(p);
    else return __ldg(p);
  };

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
  if (warp == WARP_MMA) {
    tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar(B_KVF + s), NTMA);
      mbar_init(bar(B_KVE + s), 1);
    }
    for (int b = 0; b < 2; ++b) mbar_init(bar(B_SF + b), 1);
    for (int b = 0; b < NPB; ++b) {
      mbar_init(bar(B_PF + b), SOFTMAX_WARPS);
      mbar_init(bar(B_PVD + b), 1);
    }
    mbar_init(bar(B_OF), 1);
    mbar_init(bar(B_SYNCB), SOFTMAX_WARPS);
    mbar_init(bar(B_SYNCC), SOFTMAX_WARPS);
    mbar_init(bar(B_FIN), 1);
    mbar_init(bar(B_QREADY), NTHREADS / 32);
    mbar_init(bar(B_QLOAD), 1);
    mbar_init(bar(B_QEXP), 1);
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tmap_lat);
    tma_prefetch_map(&tmap_rope);
  }
  if (tid < H) alpha_s[tid] = 1.f;

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  if (tid == 0) {  // raw Q into the staging stages, converted by all but the MMA warp
    mbar_arrive_expect_tx(bar(B_QLOAD), 2 * STAGE_BYTES);
    tma_bulk_load(smem_u32(smem + OFF_KV + QSTAGE * STAGE_BYTES),
                  static_cast<const __nv_bfloat16*>(a.q) + (int64_t)i * H * DQK, 2 * STAGE_BYTES, bar(B_QLOAD));
  }

  const uint32_t kv_base = smem_u32(smem + OFF_KV), qr_base = smem_u32(qr_s), p_base = smem_u32(p_s);
  bool ok = true;

  // Q of this token: bf16 [64 heads][576] (bulk-copied into the two staging
  // KV stages) -> x 2^qexp -> E4M3 hi and lo.  The latent part goes to TMEM
  // (the QK^T A operand: row q_row(h, lo) in that lane, 4 bytes per column),
  // written by the warps of the row's lane quadrant; the rope part goes to
  // shared memory (K-major, 64-byte swizzle).  Two passes: the largest |Q|
  // (q_max_pass: threads qt < nq, sync() their barrier; thread 0 writes the
  // scale), then the split (q_split_pass, all 16 warps, the TMA warps once
  // the copies of tile 0 are out; with `arrive`, every warp arrives on
  // B_QREADY at the end).
  constexpr int CH = DQK / 8;  // 16-byte chunks (8 bf16) per head
  const uint4* qraw = reinterpret_cast<const uint4*>(smem + OFF_KV + QSTAGE * STAGE_BYTES);
  auto bf_lo = [](uint32_t w) { return __uint_as_float(w << 16); };
  auto bf_hi = [](uint32_t w) { return __uint_as_float(w & 0xffff0000u); };
  auto q_max_pass = [&](int qt, int nq, auto sync) {
    if (!wait_warp(B_QLOAD, 0)) ok = false;
    float mx = 0.f;
#pragma unroll 4
    for (int e = qt; e < H * CH; e += nq) {
      const uint4 v = qraw[e];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) mx = fmaxf(mx, fmaxf(fabsf(bf_lo(w[t])), fabsf(bf_hi(w[t]))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) red_s[qt >> 5] = mx;
    sync();
    if (qt == 0) {
      float m = red_s[0];
      for (int w = 1; w < nq / 32; ++w) m = fmaxf(m, red_s[w]);
      int e = 0;
      if (m > 0.f && m <= 3.0e38f) frexpf(m, &e);  // m < 2^e
      *qexp_s = (m > 0.f && m <= 3.0e38f) ? 8 - e : 0;
    }
  };
  auto q_split_pass = [&](int qt, int nq, bool arrive) {
    const float qs = ldexpf(1.f, *qexp_s);
    // hi and lo of 8 elements (one 16-byte chunk of raw Q), as byte quadruples
    auto split8 = [&](const uint4 v, uint2& hv, uint2& lv) {
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        float y0, y1;
        upk2(mul2(pk2(bf_lo(w[t]), bf_hi(w[t])), pk2(qs, qs)), y0, y1);
        split_e4m3x2(f32x2_to_f16x2(y0, y1), hi[t], lo[t]);
      }
      hv = make_uint2(hi[0] | (hi[1] << 16), hi[2] | (hi[3] << 16));
      lv = make_uint2(lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16));
    };
    {
      // latent: lane u of warp w (lane quadrant q4 = w % 4) writes row 32 q4 + u,
      // i.e. Q_hi (u < 16) or Q_lo (u >= 16) of head 16 q4 + u % 16, 32-element
      // column blocks j = w / 4, w / 4 + 4, ...  The two lanes of a head split
      // each block's four 8-element chunks between them and swap halves.
      const int q4 = warp & 3, h = 16 * q4 + (lane & 15), lo = lane >> 4;
      const uint32_t t_q = tmem + ((uint32_t)(32 * q4) << 16) + TM_Q;
      for (int j = warp >> 2; j < DL / 32; j += 4) {
        // this lane splits chunks 2 lo and 2 lo + 1 of the block (loaded in an
        // order that staggers the banks), keeps its half and swaps the other
        const uint4* src = qraw + h * CH + 4 * j + 2 * lo;
        const uint4 ra = src[lane & 1], rb = src[(lane & 1) ^ 1];
        uint2 keep[2], recv[2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          uint2 hv, lv;
          split8((t ^ (lane & 1)) ? rb : ra, hv, lv);
          keep[t] = lo ? lv : hv;
          const uint2 send = lo ? hv : lv;
          recv[t] = make_uint2(__shfl_xor_sync(0xffffffffu, send.x, 16), __shfl_xor_sync(0xffffffffu, send.y, 16));
        }
        const uint2 c0 = lo ? recv[0] : keep[0], c1 = lo ? recv[1] : keep[1];  // chunks 0, 1
        const uint2 c2 = lo ? keep[0] : recv[0], c3 = lo ? keep[1] : recv[1];  // chunks 2, 3
        const uint32_t col[8] = {c0.x, c0.y, c1.x, c1.y, c2.x, c2.y, c3.x, c3.y};
        tmem_st8(t_q + 8 * j, col);
      }
      tmem_wait_st();
    }
    // rope: 8 chunks of 8 elements per head
    for (int e = qt; e < H * (DR / 8); e += nq) {
      const int h = e >> 3, c = e & 7;
      uint2 hv, lv;
      split8(qraw[h * CH + DL / 8 + c], hv, lv);
      const int cc = c >> 1, half = c & 1;  // 16-byte column and its half
      const int rh = q_row(h, 0), rl = q_row(h, 1);
      *reinterpret_cast<uint2*>(qr_s + rh * DR + ((cc ^ ((rh >> 1) & 3)) << 4) + half * 8) = hv;
      *reinterpret_cast<uint2*>(qr_s + rl * DR + ((cc ^ ((rl >> 1) & 3)) << 4) + half * 8) = lv;
    }
    // the raw Q reads and the hi/lo writes are ordered before the TMA
    // warps' next copies into the staging stages and before the MMAs
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncwarp();
    if (arrive && lane == 0) mbar_arrive(bar(B_QREADY));
  };
  auto convert_q_by = [&](int qt, int nq, auto sync, bool arrive) {
    q_max_pass(qt, nq, sync);
    sync();
    q_split_pass(qt, nq, arrive);
  };
  // The plain kernel: the MMA and softmax warps (qt 224 .. 511) take the max
  // pass alone as soon as Q has landed, so that the split can start before
  // the TMA warps, busy with tile 0's copies, join it.
  auto convert_q = [&](int qt) {
    constexpr int NMX = NTHREADS - NTMA * 32;
    if (qt >= NTMA * 32) {
      q_max_pass(qt - NTMA * 32, NMX, [] { named_barrier_sync(4, NMX); });
      if (qt == NTMA * 32) mbar_arrive(bar(B_QEXP));  // after writing the scale
    } else if (!wait_warp(B_QLOAD, 0)) {
      ok = false;
    }
    if (!wait_warp(B_QEXP, 0)) ok = false;
    q_split_pass(qt, NTHREADS, true);
  };

  // TMA warps: a tile's 80 copies (16 row groups of 4 rows x 4 latent slices
  // + 1 rope slice) are numbered group-major, c = 5 g + slice, and dealt out in
  // contiguous runs of 11 or 12: lane l of TMA warp tw issues copy
  // 80 tw / 7 + l (lanes of a warp that share a group load the same slots)
  const int tw = warp < WARP_MMA ? warp : warp - 1;
  constexpr int NCP = (NLAT + 1) * GROUPS;  // copies per tile
  const int cp0 = NCP * tw / NTMA, cp = cp0 + lane;
  const bool has_cp = lane < NCP * (tw + 1) / NTMA - cp0;
  const int g = cp / (NLAT + 1), part = cp % (NLAT + 1);
  // this warp's bytes per tile
  const uint32_t my_bytes = (uint32_t)__popc(__ballot_sync(0xffffffffu, has_cp && part < NLAT)) * 512u +
                            (uint32_t)__popc(__ballot_sync(0xffffffffu, has_cp && part == NLAT)) * 256u;
  // the slots of this lane's row group of tile lt (-1: past k, read as zeros)
  auto tile_rows = [&](int lt) -> int4 {
    int r4[4] = {-1, -1, -1, -1};
    if (has_cp && lt < ntl) {
      const int base = (t_begin + lt) * T + 4 * g;
#pragma unroll
      for (int q = 0; q < 4; ++q) r4[q] = base + q < a.k ? ld_res(&row_res[base + q]).x : -1;
    }
    return make_int4(r4[0], r4[1], r4[2], r4[3]);
  };
  auto gather_tile = [&](int s, int4 rows) {  // a tile's rows into stage s (whole TMA warp)
    if (lane == 0) mbar_arrive_expect_tx(bar(B_KVF + s), my_bytes);
    __syncwarp();
    if (has_cp) {
      const uint32_t dst = kv_base + s * STAGE_BYTES;
      if (part < NLAT)
        tma_gather4(dst + part * LAT_BYTES + g * 512, &tmap_lat, part * 128, rows, bar(B_KVF + s));
      else
        tma_gather4(dst + ROPE_OFF + g * 256, &tmap_rope, DL, rows, bar(B_KVF + s));
    }
  };

  if constexpr (FUSED) {
    // ---------------- this token's top k, then its (slot, scale) pairs and Q ----------------
    uint32_t* tk_small = reinterpret_cast<uint32_t*>(smem + OFF_RED);  // warp_buf[32] sel[4] minmax[2] wcount[16]
    uint32_t* ckey = reinterpret_cast<uint32_t*>(smem + OFF_KV);
    uint32_t* thist = ckey + RLCAP;
    uint16_t* cpos = reinterpret_cast<uint16_t*>(thist + HBINS);
    uint32_t* above_bm = reinterpret_cast<uint32_t*>(cpos + RLCAP);
    uint32_t* equal_bm = reinterpret_cast<uint32_t*>(p_s);
    int32_t* chosen = reinterpret_cast<int32_t*>(ckey);  // [k]: written after the candidates were read
    const int64_t p = tk.q_pos[i];
    const int32_t r = a.q_req[i];  // loaded now, used by the resolve after the selection
    const bool bad = p < 0 || p >= tk.ld;
    const int vis = bad ? 0 : (int)(p + 1);
    if (bad && tid == 0) report(a.dev_status, DSA_DEV_BAD_QPOS);
    // the request's block-table entries for the visible positions into L2,
    // for the resolve after the selection (one warp, one line per lane)
    if (warp == NTHREADS / 32 - 1 && r >= 0 && r < a.num_req && vis > 0) {
      const int64_t nb = 4 * (int64_t)min(a.bt_stride, (vis + a.page_size - 1) / a.page_size);
      const char* row = reinterpret_cast<const char*>(a.block_table + (int64_t)r * a.bt_stride);
      for (int64_t off = lane * 128; off < nb; off += 32 * 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + off));
      if (lane == 0) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + nb - 1));  // an unaligned row's last line
    }
    if (vis > a.k) {
      row_select(tk.scores + (int64_t)i * tk.ld, vis, a.k, [&](uint32_t o, int32_t q) { chosen[o] = q; }, ckey, thist,
                 above_bm, equal_bm, cpos, tk_small, tk_small + 32, tk_small + 36, tk_small + 38);
    } else {
      for (int j = tid; j < a.k; j += NTHREADS) chosen[j] = j < vis ? j : -1;
    }
    __syncthreads();
    // Resolve four entries per thread at a time; the dependent loads (block
    // table, then scale) overlap the two passes of the Q conversion.
    const bool req_ok = r >= 0 && r < a.num_req;
    constexpr int RPT = (FUSED_MAX_K + NTHREADS - 1) / NTHREADS;  // entries per thread at most
    int32_t pos[RPT], page[RPT];
#pragma unroll
    for (int u = 0; u < RPT; ++u) {
      const int j = tid + u * NTHREADS;
      pos[u] = j < a.k ? chosen[j] : -1;
      page[u] = -1;
      if (pos[u] >= 0 && req_ok && pos[u] / a.page_size < a.bt_stride)
        page[u] = __ldcg(&a.block_table[(int64_t)r * a.bt_stride + pos[u] / a.page_size]);
    }
    float sc[RPT];
    int32_t slot[RPT];
    bool issued_scales = false;
    auto issue_scales = [&] {
#pragma unroll
      for (int u = 0; u < RPT; ++u) {
        slot[u] = -1;
        sc[u] = 0.f;
        if (pos[u] >= 0 && req_ok && pos[u] / a.page_size < a.bt_stride && page[u] >= 0 && page[u] < a.num_pages) {
          slot[u] = page[u] * a.page_size + pos[u] % a.page_size;
          sc[u] = __ldcg(&a.kv_scale[slot[u]]);
        }
      }
      issued_scales = true;
    };
    // the Q conversion by all 16 warps, the scales' loads issued between its passes
    convert_q_by(tid, NTHREADS, [&] {
      if (!issued_scales) issue_scales();
      __syncthreads();
    }, false);
#pragma unroll
    for (int u = 0; u < RPT; ++u) {
      const int j = tid + u * NTHREADS;
      if (j >= a.k) continue;
      if (pos[u] >= 0) {
        if (!req_ok) report(a.dev_status, DSA_DEV_BAD_PAGE);
        else if (pos[u] / a.page_size >= a.bt_stride) report(a.dev_status, DSA_DEV_BAD_INDEX);
        else if (slot[u] < 0) report(a.dev_status, DSA_DEV_BAD_PAGE);
      }
      tk.idx[(int64_t)i * a.k + j] = pos[u];
      res[(int64_t)i * a.k + j] = make_int2(slot[u], __float_as_int(sc[u]));
    }
    __syncthreads();  // `res` is complete, Q is converted, the top-k's shared memory is free again
    if (tid == 0) mbar_arrive_count(bar(B_QREADY), NTHREADS / 32);
  }

  if (warp < SOFTMAX_WARP0 && warp != WARP_MMA) {
    // ---------------- TMA warps: gather the selected rows, 4 per copy ----------------
    // (the slots of the tile two ahead are loaded early, so that no L2 round
    // trip sits between a stage's release and its next copies)
    int issued = 0;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the resolve kernel's entries are complete
    int4 rows_cur = tile_rows(0), rows_nxt = tile_rows(1);
    for (int lt = 0; lt < ntl; ++lt) {
      const int s = lt % NST;
      const int4 rows_far = tile_rows(lt + 2);
      if (lt >= NST && !wait_warp(B_KVE + s, ((lt - NST) / NST) & 1)) {
        ok = false;
        break;
      }
      if (lt == QSTAGE && !wait_warp(B_QREADY, 0)) {  // the staging stages hold raw Q until then
        ok = false;
        break;
      }
      gather_tile(s, rows_cur);
      rows_cur = rows_nxt;
      rows_nxt = rows_far;
      issued = lt + 1;
      if (!FUSED && lt == 0) convert_q(tw * 32 + lane);  // join the Q conversion once tile 0's copies are out
    }
    // no copy may land after the CTA is gone: wait for the last ones (normally long complete)
    for (int lt = issued > NST ? issued - NST : 0; lt < issued; ++lt)
      if (!wait_warp(B_KVF + lt % NST, (lt / NST) & 1)) ok = false;
    if (!ok && lane == 0) report(a.dev_status, DSA_DEV_TIMEOUT);
  } else if (warp == WARP_MMA) {
    // ---------------- MMA warp ----------------
    constexpr uint32_t ID_QK = idesc_f16_f32(QM, T, 0, 0, 0);  // kind::f8f6f4: E4M3 x E4M3 -> f32
    constexpr uint32_t ID_PV = idesc_f16_f32(128, H, 1, 0, 0);
    const uint64_t a_rope = smem_desc(qr_base, 16, 512, SWIZZLE_64B);
    auto issue_qk = [&](int lt) {
      const uint32_t stage = kv_base + (lt % NST) * STAGE_BYTES;
      const uint64_t b_lat = smem_desc(stage, 16, 1024, SWIZZLE_128B);
      const uint64_t b_rope = smem_desc(stage + ROPE_OFF, 16, 512, SWIZZLE_64B);
      const uint32_t d = tmem + TM_S + T * (lt & 1);
#pragma unroll
      for (int ka = 0; ka < NLAT; ++ka) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f8_ts_warp(d, tmem + TM_Q + 8 * (4 * ka + kk), b_lat + ((ka * LAT_BYTES + kk * 32) >> 4), ID_QK,
                         (ka | kk) ? 1u : 0u);
      }
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) mma_f8_ss_warp(d, a_rope + ((kk * 32) >> 4), b_rope + ((kk * 32) >> 4), ID_QK, 1u);
      mma_commit_warp(bar(B_SF + (lt & 1)));
    };
    // the 4 independent d-chunks innermost: consecutive MMAs never share an accumulator
    auto issue_pv = [&](int lt) {
      const int s = lt % NST, pb = lt % NPB;
      const uint64_t a0 = smem_desc(kv_base + s * STAGE_BYTES, LAT_BYTES, 1024, SWIZZLE_128B);
      const uint64_t b0 = smem_desc(p_base + pb * 2 * P_BYTES, 16, 512, SWIZZLE_64B);
#pragma unroll
      for (int w = 0; w < 2; ++w) {
#pragma unroll
        for (int kk = 0; kk < T / 32; ++kk) {
#pragma unroll
          for (int c = 0; c < NLAT; ++c)
            mma_f8_ss_warp(tmem + TM_O + 64 * c, a0 + ((c * LAT_BYTES + kk * 32 * 128) >> 4),
                           b0 + ((w * P_BYTES + kk * 32) >> 4), ID_PV, (lt > 0 || w > 0 || kk > 0) ? 1u : 0u);
        }
      }
      mma_commit_warp(bar(B_KVE + s));
      mma_commit_warp(bar(B_PVD + pb));
    };
    auto kv_landed = [&](int lt) { return wait_warp(B_KVF + lt % NST, (lt / NST) & 1); };
    if (!FUSED) convert_q((NTMA + SOFTMAX_WARPS) * 32 + lane);  // threads 480 .. 511
    // QK^T of tiles 0 and 1 fill both S buffers
    ok = wait_warp(B_QREADY, 0);
    for (int lt = 0; lt < 2 && lt < ntl && ok; ++lt) {
      ok = kv_landed(lt);
      if (ok) {
        tc_fence_after_sync();
        issue_qk(lt);
      }
    }
    for (int lt = 0; lt < ntl && ok; ++lt) {
      // P(lt) written: P V(lt) goes first (the softmax of tile lt + 1 is
      // running meanwhile); S buffer lt % 2 has been read, so QK^T(lt + 2)
      // may overwrite it once its tile has landed
      if (!wait_warp(B_PF + lt % NPB, (lt / NPB) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      issue_pv(lt);
      if (lt + 2 < ntl) {
        if (!kv_landed(lt + 2)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        issue_qk(lt + 2);
      }
    }
    __syncwarp();
    mma_commit_warp(bar(B_OF));
    mma_commit_warp(bar(B_FIN));
    if (!wait_warp(B_FIN, 0)) ok = false;  // every MMA done before TMEM is released
    if (!ok && lane == 0) report(a.dev_status, DSA_DEV_TIMEOUT);
  } else if (warp >= SOFTMAX_WARP0) {
    // ---------------- softmax warps ----------------
    const int sw = warp - SOFTMAX_WARP0;            // 0..7
    const int q4 = warp & 3;                        // TMEM lane quadrant: heads [16 q4, 16 q4 + 16)
    const int half = sw >> 2;                       // tile rows [32 half, 32 half + 32); O heads [32 half, +32)
    const int hh = 16 * q4 + (lane & 15);           // this thread's head
    const int up = lane >> 4;                       // 0: this lane holds Q_hi logits, 1: Q_lo
    const int cc = 2 * half + up;                   // after the exchange: tile rows [16 cc, 16 cc + 16)
    const uint32_t t_lane = tmem + ((uint32_t)(32 * q4) << 16);
    if (!FUSED) convert_q(tid - SOFTMAX_WARP0 * 32 + NTMA * 32);  // threads 224 .. 479
    const float qk_scale = a.softmax_scale * LOG2E * ldexpf(1.f, -*qexp_s);
    // P' = p s_j 2^E with p <= 16: pick E so that 16 max_j s_j 2^E < 256,
    // max_j over the entries of this CTA's tiles
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the resolve kernel's entries are complete
    int p_exp = 0;
    {
      float sm = 0.f;
      const int e_end = t_end * T < a.k ? t_end * T : a.k;
      for (int e = t_begin * T + sw * 32 + lane; e < e_end; e += SOFTMAX_WARPS * 32)
        sm = fmaxf(sm, __int_as_float(ld_res(&row_res[e]).y));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sm = fmaxf(sm, __shfl_xor_sync(0xffffffffu, sm, o));
      if (lane == 0) smax_s[sw] = sm;
      named_barrier_sync(2, SOFTMAX_WARPS * 32);
      float smax = smax_s[0];
#pragma unroll
      for (int w = 1; w < SOFTMAX_WARPS; ++w) smax = fmaxf(smax, smax_s[w]);
      if (smax > 0.f) {
        int e2;
        frexpf(smax, &e2);  // smax < 2^e2
        p_exp = 4 - e2;
      }
    }
    const float p_scale = ldexpf(1.f, p_exp);
    // P' = p s_j 2^E = p c_j (2^E / qk_scale), c_j = s_j qk_scale the row's logit factor
    const float p_ratio = p_scale / qk_scale;

    // head hh's reference max (log2 domain) and its share of l; the four
    // threads of a head keep identical copies of the reference
    float m_ref = -INFINITY;
    uint64_t l2 = pk2(0.f, 0.f);  // head hh's share of l, two running sums
    // per tile, this warp's 32 rows' logit factors, double buffered
    float* rowf = reinterpret_cast<float*>(smem + OFF_ROWF) + sw * 2 * 32;
    uint32_t ph_b = 0, ph_c = 0;  // completed phases of the group barriers
    auto group_sync = [&](int bb, uint32_t& ph) {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(bb));
      if (ok && !wait_warp(bb, ph & 1)) ok = false;
      ++ph;
      return ok;
    };
    auto row_info = [&](int lt) -> int2 {  // lane's row: 32 half + lane
      const int e = (t_begin + lt) * T + 32 * half + lane;
      return e < a.k ? ld_res(row_res + e) : make_int2(-1, 0);
    };
    int2 info = row_info(0);
    for (int lt = 0; lt < ntl; ++lt) {  // no early exit: every warp reaches every vote barrier
      const int sb = lt & 1;
      const int2 info_next = lt + 1 < ntl ? row_info(lt + 1) : make_int2(-1, 0);
      // the warp's rows: validity bits (bit r: row 32 half + r) and logit factors
      const unsigned vmask = __ballot_sync(0xffffffffu, info.x >= 0);
      rowf[sb * 32 + lane] = __int_as_float(info.y) * qk_scale;
      __syncwarp();
      float cj[16];  // this thread's rows' factors
      {
        const float4* rf4 = reinterpret_cast<const float4*>(rowf + sb * 32 + 16 * up);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 f = rf4[i];
          cj[4 * i] = f.x;
          cj[4 * i + 1] = f.y;
          cj[4 * i + 2] = f.z;
          cj[4 * i + 3] = f.w;
        }
      }
      if (ok && !wait_warp(B_SF + sb, (lt >> 1) & 1)) ok = false;
      tc_fence_after_sync();
      // logits of head hh, rows 16 cc + c, in the log2 domain (invalid rows: -inf):
      // lane u holds S_hi (u < 16) or S_lo (u >= 16) of the warp's 32 rows;
      // the partner lane u ^ 16 sends the other half of this thread's 16 rows
      float z[16];
      {
        float v[32];
        tmem_ld32(t_lane + TM_S + T * sb + 32 * half, v);
        tmem_wait_ld();
        float got[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) got[c] = __shfl_xor_sync(0xffffffffu, up ? v[c] : v[16 + c], 16);
#pragma unroll
        for (int i = 0; i < 8; ++i) {  // (hi + lo) c_j, two rows at a time
          const uint64_t mine = up ? pk2(v[16 + 2 * i], v[17 + 2 * i]) : pk2(v[2 * i], v[2 * i + 1]);
          upk2(mul2(add2(mine, pk2(got[2 * i], got[2 * i + 1])), pk2(cj[2 * i], cj[2 * i + 1])), z[2 * i], z[2 * i + 1]);
        }
        if (vmask != 0xffffffffu) {  // a tile with rows past the selection (warp-uniform)
          const unsigned my_valid = vmask >> (16 * up);
#pragma unroll
          for (int c = 0; c < 16; ++c)
            if (!((my_valid >> c) & 1u)) z[c] = -INFINITY;
        }
      }
      // Fast path: probabilities are taken against the heads' current
      // reference maxima; that stays exact as long as no logit exceeds its
      // reference by more than 2^EXCEED.  One vote of the 8 warps decides;
      // only then is the tile maximum reduced.
      float tm = z[0];  // this thread's largest logit (-inf when none is valid)
#pragma unroll
      for (int c = 1; c < 16; ++c) tm = fmaxf(tm, z[c]);
      if (named_barrier_or(3, SOFTMAX_WARPS * 32, tm > m_ref + EXCEED_LOG2)) {  // one vote of the 8 warps: uniform
        tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 16));
        if (up == 0) red_s[half * H + hh] = tm;
        group_sync(B_SYNCB, ph_b);
        const float mt = fmaxf(red_s[hh], red_s[H + hh]);
        float alpha = 1.f;
        if (mt > m_ref + EXCEED_LOG2) {
          alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - mt);
          m_ref = mt;
        }
        l2 = mul2(l2, pk2(alpha, alpha));
        if (half == 0 && up == 0) alpha_s[hh] = alpha;
        const unsigned need = __ballot_sync(0xffffffffu, lt > 0 && alpha != 1.f);
        if (half == 0 && lane == 0) resc_s[q4] = need != 0u;
        group_sync(B_SYNCC, ph_c);
        if (resc_s[0] | resc_s[1] | resc_s[2] | resc_s[3]) {
          // O must hold every P V issued so far: the previous tile's
          if (ok && !wait_warp(B_PVD + (lt - 1) % NPB, ((lt - 1) / NPB) & 1)) ok = false;
          tc_fence_after_sync();
          const float* al = alpha_s + 32 * half;
#pragma unroll 1
          for (int c = 0; c < NLAT; ++c) {
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              float o[16];
              const uint32_t addr = t_lane + TM_O + 64 * c + 32 * half + 16 * g;
              tmem_ld16(addr, o);
              tmem_wait_ld();
#pragma unroll
              for (int h = 0; h < 16; ++h) o[h] *= al[16 * g + h];
              tmem_st16(addr, o);
            }
          }
          tmem_wait_st();
        }
      }
      // probabilities, folded with the row's dequantisation scale and the
      // query's power of two, as E4M3 hi + lo (computed before waiting for
      // the P buffer, so that only the stores wait)
      // invalid rows have z = -inf and p = 2^-inf = 0; a head whose reference
      // is still -inf has only such rows
      uint32_t phi[8], plo[8];
      const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
      const uint64_t nm2 = pk2(-m_use, -m_use), ratio2 = pk2(p_ratio, p_ratio);
      // (the row factors are read again rather than kept in registers across the vote)
      const float4* rfp = reinterpret_cast<const float4*>(rowf + sb * 32 + 16 * up);
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        const float4 f = rfp[k4];
        const float cf[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int i = 2 * k4 + t;
          float d0, d1;
          upk2(add2(pk2(z[2 * i], z[2 * i + 1]), nm2), d0, d1);
          const float p0 = ex2(d0), p1 = ex2(d1);
          l2 = add2(l2, pk2(p0, p1));
          float q0, q1;
          upk2(mul2(pk2(p0, p1), mul2(pk2(cf[2 * t], cf[2 * t + 1]), ratio2)), q0, q1);
          split_e4m3x2(f32x2_to_f16x2(q0, q1), phi[i], plo[i]);
        }
      }
      // P buffer lt % 2 was last read by P V(lt - 2), which the MMA warp issued
      // before QK^T(lt): the commit that completed S(lt) tracks every MMA issued
      // before it, so the buffer is free without a wait of its own
      {
        unsigned char* pr = p_s + (lt % NPB) * 2 * P_BYTES + hh * T + ((cc ^ ((hh >> 1) & 3)) << 4);
        *reinterpret_cast<uint4*>(pr) = make_uint4(phi[0] | (phi[1] << 16), phi[2] | (phi[3] << 16),
                                                   phi[4] | (phi[5] << 16), phi[6] | (phi[7] << 16));
        *reinterpret_cast<uint4*>(pr + P_BYTES) = make_uint4(plo[0] | (plo[1] << 16), plo[2] | (plo[3] << 16),
                                                             plo[4] | (plo[5] << 16), plo[6] | (plo[7] << 16));
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PF + lt % NPB));
      info = info_next;
    }
    // ---------------- epilogue: normalise and write ----------------
    if (ok && !wait_warp(B_OF, 0)) ok = false;
    if (ok) {
      tc_fence_after_sync();
      float la, lb;
      upk2(l2, la, lb);
      const float l_part = la + lb;
      const float lw = l_part + __shfl_xor_sync(0xffffffffu, l_part, 16);  // the warp's 32 rows
      if (up == 0) red_s[half * H + hh] = lw;
      ok = group_sync(B_SYNCB, ph_b);
    }
    if (ok) {
      if (half == 0 && up == 0) {
        const float l = red_s[hh] + red_s[H + hh];
        alpha_s[hh] = l > 0.f ? ldexpf(1.f / l, -p_exp) : 0.f;
        const float lse = l > 0.f ? (m_ref + log2f(l)) * LN2 : -INFINITY;
        if (S == 1) {
          if (a.lse) a.lse[(int64_t)i * H + hh] = lse;
        } else {
          a.lse_part[((int64_t)split * a.num_q + i) * H + hh] = lse;
        }
      }
      ok = group_sync(B_SYNCC, ph_c);
    }
    if (ok) {
      // O^T (TMEM) -> registers -> global memory: thread (q4, lane) holds
      // latent dim d = 128 c + 32 q4 + lane of its 32 heads, so a warp's
      // store covers 32 consecutive d of one head.  The per-head factors of
      // each group of 16 heads go to registers first.
      const int h2 = half;
#pragma unroll 1
      for (int g = 0; g < 2; ++g) {
        float inv[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) inv[h] = alpha_s[32 * h2 + 16 * g + h];
        const int64_t hbase = 32 * h2 + 16 * g;
#pragma unroll 1
        for (int c = 0; c < NLAT; ++c) {
          const int d = 128 * c + 32 * q4 + lane;
          float o[16];
          tmem_ld16(t_lane + TM_O + 64 * c + hbase, o);
          tmem_wait_ld();
          if (S == 1) {
            __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(a.out) + ((int64_t)i * H + hbase) * DL + d;
#pragma unroll
            for (int h = 0; h < 16; h += 2) {
              float y0, y1;
              upk2(mul2(pk2(o[h], o[h + 1]), pk2(inv[h], inv[h + 1])), y0, y1);
              ob[h * DL] = __float2bfloat16_rn(y0);
              ob[(h + 1) * DL] = __float2bfloat16_rn(y1);
            }
          } else {
            float* op = a.o_part + (((int64_t)split * a.num_q + i) * H + hbase) * DL + d;
#pragma unroll
            for (int h = 0; h < 16; ++h) op[h * DL] = o[h] * inv[h];
          }
        }
      }
    } else if (lane == 0) {
      report(a.dev_status, DSA_DEV_TIMEOUT);
    }
  }

  // ---------------- teardown ----------------
  tc_fence_before_sync();
  __syncthreads();
  if (warp == WARP_MMA) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, TM_COLS);
  }
}

// cuTensorMapEncodeTiled, looked up once from the driver
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// The KV pool as a 2-D byte tensor [slots][576]; boxes of one row, `box_cols`
// wide from any column, for tile::gather4.
bool make_kv_map(CUtensorMap* map, const MlaArgs& a, uint32_t box_cols, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)DQK, (cuuint64_t)a.num_pages * (cuuint64_t)a.page_size};
  const cuuint64_t strides[1] = {(cuuint64_t)DQK};
  const cuuint32_t box[2] = {box_cols, 1}, elem[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.kv), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool mla_tc_supported(const MlaArgs& a) { return a.heads == H && a.d_latent == DL && a.d_rope == DR; }

size_t mla_tc_workspace_bytes(int32_t num_q, int32_t k) {
  // the resolved (slot, scale) of every selected entry
  return sizeof(int2) * (size_t)num_q * (size_t)k;
}

namespace {
// resolve: launch the resolve kernel first (else `workspace` already holds the
// entries, written by the kernel just before on the stream)
cudaError_t launch_mla_tc_impl(const MlaArgs& a, void* workspace, cudaStream_t stream, bool resolve) {
  if (a.num_q == 0) return cudaSuccess;
  alignas(64) CUtensorMap map_lat, map_rope;
  if (!make_kv_map(&map_lat, a, 128, CU_TENSOR_MAP_SWIZZLE_128B) || !make_kv_map(&map_rope, a, DR, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  int2* res = static_cast<int2*>(workspace);
  // both launches are programmatic dependents of the kernel before them
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t rcfg = {};
  // one entry per thread up to two waves of 2,048 threads per SM, else eight
  const bool wide = (int64_t)a.num_q * a.k > (int64_t)device_sm_count() * 2048 * 2;
  const int ent = wide ? 8 : 1;
  rcfg.gridDim = dim3((a.k + RES_THREADS * ent - 1) / (RES_THREADS * ent), a.num_q);
  rcfg.blockDim = dim3(RES_THREADS);
  rcfg.stream = stream;
  rcfg.attrs = attr;
  rcfg.numAttrs = 1;
  cudaError_t e = cudaSuccess;
  if (resolve) {
    e = wide ? cudaLaunchKernelEx(&rcfg, resolve_kernel<8>, a, res) : cudaLaunchKernelEx(&rcfg, resolve_kernel<1>, a, res);
    if (e != cudaSuccess) return e;
  }
  e = cudaFuncSetAttribute(mla_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the attention CTAs may start while the
  // kernel before them (the resolve kernel, or the top-k that wrote the
  // entries) runs; they wait for it (griddepcontrol.wait) before reading the
  // entries
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.num_q, a.num_splits);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, mla_tc_kernel<false>, a, map_lat, map_rope, res, TopkIn{});
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_mla_tc(const MlaArgs& a, void* workspace, cudaStream_t stream) {
  return launch_mla_tc_impl(a, workspace, stream, true);
}

cudaError_t launch_mla_tc_resolved(const MlaArgs& a, void* workspace, cudaStream_t stream) {
  return launch_mla_tc_impl(a, workspace, stream, false);
}

int mla_tc_fused_max_k() { return FUSED_MAX_K; }

cudaError_t launch_mla_tc_fused(const MlaArgs& a, const float* scores, int64_t ld, const int32_t* q_pos, int32_t* idx,
                                void* workspace, cudaStream_t stream) {
  if (a.num_q == 0) return cudaSuccess;
  if (a.num_splits != 1 || a.k > FUSED_MAX_K || ld > RMAXV) return cudaErrorInvalidValue;
  alignas(64) CUtensorMap map_lat, map_rope;
  if (!make_kv_map(&map_lat, a, 128, CU_TENSOR_MAP_SWIZZLE_128B) || !make_kv_map(&map_rope, a, DR, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(mla_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const TopkIn tk{scores, ld, q_pos, idx};
  mla_tc_kernel<true><<<a.num_q, NTHREADS, SMEM_BYTES, stream>>>(a, map_lat, map_rope, static_cast<int2*>(workspace), tk);
  return cudaGetLastError();
}

}  // namespace dsa
