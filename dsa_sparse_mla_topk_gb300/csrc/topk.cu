// Causal top-k selection over fp32 indexer scores.
//
// "Accelerating GLM-5.3-Flash on H200", section 3 "Larger KV tiles for DSA
// Partial": the indexer's scores pick the KV positions the Partial step
// attends to.  These kernels make the pick exact and deterministic: positions
// are ranked by (score descending, position ascending), -0.0 == +0.0, and
// the chosen ones are written in ascending position order, -1 padded.
//
// Every fp32 score maps to an order-preserving 32-bit key.  Two kernels:
//   topk_row_kernel      rows of up to 65,536 positions, one CTA per row; longer
//                        rows one CTA per 65,536-position slice plus a merge of
//                        the slices' top-k blocks (needs the caller's workspace);
//   topk_cluster_kernel  long rows without a workspace: a thread-block
//                        cluster of C CTAs per row, each owning a contiguous
//                        slice of the visible positions.
// Both follow the same plan: a 1/16 sample places a lower threshold T_lo that,
// with a wide margin, lies below the k-th largest key; one streaming pass
// collects the keys >= T_lo with their positions; an exact radix select over
// those candidates finds the k-th largest key T; the keys above T and the
// lowest-positioned keys equal to T are written.  If the sample misleads
// (fewer than k candidates, or more than fit), the CTA falls back to an exact
// multi-pass radix select over the row in global memory, so the result never
// depends on the score distribution.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include "internal.cuh"

namespace cg = cooperative_groups;

namespace dsa {
namespace {

constexpr int NT = 512;           // threads per CTA (two CTAs fit on an SM)
constexpr int HBINS = 4096;       // histogram bins (12 key bits)
constexpr int MCAP = 6144;        // candidates CTA 0 can hold for the final selection
constexpr int SAMPLE_BLOCK = 128; // the sample takes the first SAMPLE_RUN of every
constexpr int SAMPLE_RUN = 8;     // SAMPLE_BLOCK positions (1/16)

__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0.0 ranks equal to +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum of one value per thread over a block of NTH threads;
// *total gets the block sum.  `warp_buf` holds 32 words of shared memory.
template <int NTH = NT>
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* total, uint32_t* warp_buf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_buf[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < NTH / 32 ? warp_buf[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < NTH / 32) warp_buf[lane] = w;
  }
  __syncthreads();
  const uint32_t before = warp > 0 ? warp_buf[warp - 1] : 0u;
  *total = warp_buf[NTH / 32 - 1];
  __syncthreads();
  return before + x - v;
}

// Among the keys in bins [0, nbins) of `hist` counted from the top, find the
// bin holding the krem-th largest key.  Every thread returns the same
// (bin, count above the bin, count in the bin).
__device__ __forceinline__ void find_bin(const uint32_t* hist, int nbins, uint32_t krem, uint32_t* warp_buf,
                                         uint32_t* sel, uint32_t& bin, uint32_t& above, uint32_t& count) {
  const int per = nbins / NT;  // bins per thread, highest bins to thread 0
  uint32_t c[HBINS / NT];
  for (int t = 0; t < HBINS / NT; ++t) c[t] = 0u;
  uint32_t sum = 0;
  for (int t = 0; t < per; ++t) {
    c[t] = hist[nbins - 1 - (threadIdx.x * per + t)];
    sum += c[t];
  }
  uint32_t total;
  uint32_t acc = block_exclusive_scan(sum, &total, warp_buf);
  for (int t = 0; t < per; ++t) {
    if (acc < krem && krem <= acc + c[t]) {
      sel[0] = nbins - 1 - (threadIdx.x * per + t);
      sel[1] = acc;
      sel[2] = c[t];
    }
    acc += c[t];
  }
  __syncthreads();
  bin = sel[0], above = sel[1], count = sel[2];
  __syncthreads();
}

// Exact selection over n keys with positions (keys/pos in any memory, in
// ascending position order): emit(slot, position) receives the k chosen
// positions in ascending order, slot 0..k-1.
// Radix passes of up to 11 bits run over (key - kmin) from its highest set
// bit down, so the bins spread over the keys' actual range (candidate keys
// share their top bits; fixed digits would pile them into a few bins).
template <bool GLOBAL_ROW, class Emit>
__device__ void select_exact(const float* row_scores, const uint32_t* keys, const int32_t* pos, int64_t n, uint32_t k,
                             Emit emit, uint32_t* hist, uint32_t* warp_buf, uint32_t* sel) {
  auto key_at = [&](int64_t e) -> uint32_t { return GLOBAL_ROW ? score_key(row_scores[e]) : keys[e]; };
  auto pos_at = [&](int64_t e) -> int32_t { return GLOBAL_ROW ? (int32_t)e : pos[e]; };
  uint32_t kmin = 0, top = 32;
  if (!GLOBAL_ROW) {
    uint32_t lo = 0xffffffffu, hi = 0u;
    for (int64_t e = threadIdx.x; e < n; e += NT) {
      const uint32_t key = keys[e];
      lo = min(lo, key);
      hi = max(hi, key);
    }
    for (int o = 16; o > 0; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if ((threadIdx.x & 31) == 0) {
      atomicMin(&sel[2], lo);
      atomicMax(&sel[3], hi);
    }
    __syncthreads();
    kmin = sel[2];
    const uint32_t diff = sel[3] - kmin;
    top = 32 - __clz(diff);  // significant bits of (key - kmin); 0 when all keys are equal
    __syncthreads();
  }
  uint32_t prefix = 0, mask = 0, krem = k;
  while (top > 0) {
    const int sh = top > 11 ? (int)top - 11 : 0;
    const uint32_t dm = (1u << (top - sh)) - 1u;
    for (int b = threadIdx.x; b < 2048; b += NT) hist[b] = 0;
    __syncthreads();
    for (int64_t e = threadIdx.x; e < n; e += NT) {
      const uint32_t u = key_at(e) - kmin;
      if ((u & mask) == prefix) atomicAdd(&hist[(u >> sh) & dm], 1u);
    }
    __syncthreads();
    uint32_t bin, above, count;
    find_bin(hist, 2048, krem, warp_buf, sel, bin, above, count);
    prefix |= bin << sh;
    mask |= dm << sh;
    krem -= above;
    top = sh;
    if (count == krem) break;  // the whole bin is taken
  }
  // ordered output: keys above the prefix, then the first krem equal ones
  uint32_t ties_before = 0, written = 0;
  constexpr int PER = 4;
  for (int64_t base = 0; base < n && written < k; base += (int64_t)NT * PER) {
    const int64_t e0 = base + (int64_t)threadIdx.x * PER;
    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int t = 0; t < PER; ++t) {
      if (e0 + t < n) {
        const uint32_t mk = (key_at(e0 + t) - kmin) & mask;
        gt |= (uint32_t)(mk > prefix) << t;
        eq |= (uint32_t)(mk == prefix) << t;
      }
    }
    uint32_t eq_total;
    uint32_t rank = ties_before + block_exclusive_scan(__popc(eq), &eq_total, warp_buf);
    uint32_t take = gt;
#pragma unroll
    for (int t = 0; t < PER; ++t) {
      if ((eq >> t) & 1u) {
        if (rank < krem) take |= 1u << t;
        ++rank;
      }
    }
    uint32_t take_total;
    uint32_t o = written + block_exclusive_scan(__popc(take), &take_total, warp_buf);
#pragma unroll
    for (int t = 0; t < PER; ++t)
      if (((take >> t) & 1u) && o < k) emit(o++, pos_at(e0 + t));
    ties_before += eq_total;
    written += take_total;
  }
}

template <int C>
struct TopkSmem {
  // candidates one CTA collects; sized so that two CTAs fit on an SM
  static constexpr int LCAP = C == 1 ? MCAP : 3072;
  static constexpr size_t bytes = sizeof(uint32_t) * HBINS + (sizeof(uint32_t) + sizeof(int32_t)) * LCAP +
                                  (C > 1 ? (sizeof(uint32_t) + sizeof(int32_t)) * MCAP : 0);
};

template <int C>
__global__ void __cluster_dims__(C, 1, 1) __launch_bounds__(NT, 2)
    topk_cluster_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ q_pos, int32_t k,
                        int32_t* __restrict__ idx, int32_t* status) {
  constexpr int LCAP = TopkSmem<C>::LCAP;
  extern __shared__ __align__(16) uint32_t smem[];
  uint32_t* hist = smem;
  uint32_t* ckey = hist + HBINS;
  int32_t* cpos = reinterpret_cast<int32_t*>(ckey + LCAP);
  uint32_t* mkey = C > 1 ? reinterpret_cast<uint32_t*>(cpos + LCAP) : ckey;
  int32_t* mpos = C > 1 ? reinterpret_cast<int32_t*>(mkey + MCAP) : cpos;
  __shared__ uint32_t warp_buf[32];
  __shared__ uint32_t sel[4];
  // vars: [0] T_lo (CTA 0), [1] candidate count, [2] overflow, [3] sampled count
  __shared__ uint32_t vars[4];

  // the next kernel on the stream (the attention call's resolve step) may be
  // scheduled now; it waits for this grid's results before reading them
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x / C;
  int32_t* out = idx + row * (int64_t)k;
  const int64_t p = q_pos[row];
  // row-uniform early exits (the same for every CTA of the cluster)
  if (p < 0 || p >= ld) {
    if (rank == 0) {
      if (tid == 0) report(status, DSA_DEV_BAD_QPOS);
      for (int j = tid; j < k; j += NT) out[j] = -1;
    }
    return;
  }
  const int64_t vis = p + 1;
  if (vis <= k) {
    if (rank == 0)
      for (int j = tid; j < k; j += NT) out[j] = j < vis ? j : -1;
    return;
  }
  const float* s = scores + row * ld;
  const bool vec = ((reinterpret_cast<uintptr_t>(s) & 15u) == 0);
  // this CTA's slice [lo, hi), a multiple of 128 positions long
  const int64_t per = ((vis + C - 1) / C + 127) & ~int64_t(127);
  const int64_t lo = (int64_t)rank * per;
  const int64_t hi = lo + per < vis ? lo + per : vis;

  // ---- 1. sampled histogram of the top 12 key bits ----
  for (int b = tid; b < HBINS; b += NT) hist[b] = 0;
  if (tid == 0) vars[1] = vars[2] = 0;
  __syncthreads();
  uint32_t nsampled = 0;
  for (int64_t blk = lo + (int64_t)tid * SAMPLE_BLOCK; blk < hi; blk += (int64_t)NT * SAMPLE_BLOCK) {
    float v[SAMPLE_RUN];  // all loads in flight before the first atomic
#pragma unroll
    for (int t = 0; t < SAMPLE_RUN; ++t) v[t] = blk + t < hi ? __ldg(s + blk + t) : 0.f;
#pragma unroll
    for (int t = 0; t < SAMPLE_RUN; ++t) {
      if (blk + t < hi) {
        atomicAdd(&hist[score_key(v[t]) >> 20], 1u);
        ++nsampled;
      }
    }
  }
  {
    uint32_t tot;
    block_exclusive_scan(nsampled, &tot, warp_buf);
    if (tid == 0) vars[3] = tot;
  }
  cluster.sync();
  if (rank == 0) {
    // sum the cluster's histograms into this CTA's, then place T_lo so that
    // the sample above it exceeds its expected share of the top k by 25% + 16
    for (int r = 1; r < C; ++r) {
      const uint32_t* rh = cluster.map_shared_rank(hist, r);
      uint32_t rv[HBINS / NT];  // all remote reads in flight before the adds
#pragma unroll
      for (int t = 0; t < HBINS / NT; ++t) rv[t] = rh[tid + NT * t];
#pragma unroll
      for (int t = 0; t < HBINS / NT; ++t) hist[tid + NT * t] += rv[t];
    }
    uint32_t ns = vars[3];
    for (int r = 1; r < C; ++r) ns += *cluster.map_shared_rank(&vars[3], r);
    __syncthreads();
    uint32_t t_lo = 0;
    if (vis > MCAP / 2 && ns > 0) {
      // (fp32: fp64 arithmetic in every thread costs microseconds here)
      const float expect = (float)k * (float)ns / (float)vis;
      uint32_t need = (uint32_t)(expect * 1.25f) + 16u;
      if (need > ns) need = ns;
      uint32_t bin, above, count;
      find_bin(hist, HBINS, need > 0 ? need : 1u, warp_buf, sel, bin, above, count);
      t_lo = bin << 20;
    }
    if (tid == 0) vars[0] = t_lo;
  }
  cluster.sync();
  const uint32_t t_lo = *cluster.map_shared_rank(&vars[0], 0);

  // ---- 2. ordered collection of the candidates (key >= T_lo) ----
  // Positions are processed in steps of NT*PER; the loads of two steps are
  // issued before the first is scanned, so two steps are in flight at once.
  constexpr int PER = 16;  // contiguous positions per thread per step
  uint32_t written = 0;
  bool overflow = false;
  auto load_step = [&](int64_t base, float (&v)[PER]) {
    const int64_t e0 = base + (int64_t)tid * PER;
    if (vec && e0 + PER <= hi) {
#pragma unroll
      for (int t = 0; t < PER / 4; ++t) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(s + e0) + t);
        v[4 * t] = f.x, v[4 * t + 1] = f.y, v[4 * t + 2] = f.z, v[4 * t + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int t = 0; t < PER; ++t) v[t] = (e0 + t < hi) ? __ldg(s + e0 + t) : -INFINITY;
    }
  };
  auto scan_step = [&](int64_t base, const float (&v)[PER]) -> bool {
    const int64_t e0 = base + (int64_t)tid * PER;
    uint32_t flags = 0;
#pragma unroll
    for (int t = 0; t < PER; ++t) flags |= (uint32_t)(e0 + t < hi && score_key(v[t]) >= t_lo) << t;
    uint32_t total;
    uint32_t o = written + block_exclusive_scan(__popc(flags), &total, warp_buf);
    if (written + total > (uint32_t)LCAP) return false;
#pragma unroll
    for (int t = 0; t < PER; ++t) {
      if ((flags >> t) & 1u) {
        ckey[o] = score_key(v[t]);
        cpos[o] = (int32_t)(e0 + t);
        ++o;
      }
    }
    written += total;
    return true;
  };
  for (int64_t base = lo; base < hi && !overflow; base += 2 * (int64_t)NT * PER) {
    float va[PER], vb[PER];
    const int64_t base_b = base + (int64_t)NT * PER;
    load_step(base, va);
    if (base_b < hi) load_step(base_b, vb);
    if (!scan_step(base, va)) overflow = true;
    if (!overflow && base_b < hi && !scan_step(base_b, vb)) overflow = true;
  }
  if (tid == 0) {
    vars[1] = written;
    vars[2] = overflow ? 1u : 0u;
  }
  cluster.sync();

  // ---- 3. CTA 0: gather, select exactly, write ----
  bool fallback = false;
  if (rank == 0) {
    uint32_t offs[C];
    uint32_t total = 0;
    for (int r = 0; r < C; ++r) {
      const uint32_t* rv = cluster.map_shared_rank(vars, r);
      offs[r] = total;
      total += rv[1];
      if (rv[2]) fallback = true;
    }
    if (total > (uint32_t)MCAP || total < (uint32_t)k) fallback = true;
    if (!fallback && C > 1) {
      for (int r = 0; r < C; ++r) {
        const uint32_t* rk = cluster.map_shared_rank(ckey, r);
        const int32_t* rp = cluster.map_shared_rank(cpos, r);
        const uint32_t n = *cluster.map_shared_rank(&vars[1], r);
        for (uint32_t e = tid; e < n; e += NT) {
          mkey[offs[r] + e] = rk[e];
          mpos[offs[r] + e] = rp[e];
        }
      }
    }
    __syncthreads();
    if (!fallback) vars[3] = total;
  }
  if (tid == 0) {
    sel[2] = 0xffffffffu;
    sel[3] = 0u;
  }
  cluster.sync();  // the other CTAs' shared memory is no longer read
  if (rank != 0) return;
  if (!fallback) {
    select_exact<false>(nullptr, mkey, mpos, vars[3], (uint32_t)k, [&](uint32_t o, int32_t q) { out[o] = q; },
                        hist, warp_buf, sel);
  } else {
    select_exact<true>(s, nullptr, nullptr, vis, (uint32_t)k, [&](uint32_t o, int32_t q) { out[o] = q; }, hist,
                       warp_buf, sel);
  }
}

// ---------------------------------------------------------------------------
// Rows of up to 65,536 visible positions: one CTA of 512 threads per row,
// two CTAs per SM (80 KB of shared memory each), so that one CTA streams
// while the other selects.
//   0. The loads of a 1/16 sample (the first 8 of every 128 positions) are
//      issued first, then an L2 bulk prefetch of the whole row.
//   1. The sample places a lower 12-bit threshold T_lo as in the cluster
//      kernel.
//   2. One streaming pass screens every score against T_lo with one float
//      compare.  Each warp appends its candidates (score bits, position) to
//      its own segment of a shared-memory list through ballots: no atomics,
//      no block-wide synchronisation.
//   3. The k-th largest candidate key is found exactly by radix passes over
//      (key - min key), up to 11 bits each, from the highest significant bit.
//   4. The keys above it and the keys equal to it are marked in two position
//      bitmaps; one ordered pass over the bitmaps writes the positions above,
//      plus the lowest-positioned equal ones, in ascending order.
// If the sample misleads (fewer than k candidates, or a full segment), the
// CTA falls back to the exact multi-pass radix select over the row in global
// memory, so the result never depends on the score distribution.
constexpr int RNT = 512;                 // threads per CTA
constexpr int RWARPS = RNT / 32;
constexpr int RMAXV = 65536;             // visible positions (positions fit in 16 bits)
constexpr int RWCAP = 512;               // candidates one warp can hold
constexpr int RLCAP = RWARPS * RWCAP;    // 8192
constexpr int RALL = 4096;               // rows this short take every position as a candidate
constexpr int RDEPTH = 8;                // float4 loads in flight per thread
constexpr int RWORDS = RMAXV / 32;       // bitmap words
constexpr size_t RSMEM = sizeof(uint32_t) * (RLCAP + HBINS + 2 * RWORDS) + sizeof(uint16_t) * RLCAP;
static_assert(RNT * SAMPLE_BLOCK == RMAXV, "one sample block per thread must cover a row");

__device__ __forceinline__ void l2_prefetch_bulk(uintptr_t addr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(addr), "r"(bytes) : "memory");
}

// find_bin with three barriers instead of five.  It skips the barriers that
// protect warp_buf and sel from the next call, so consecutive calls must be
// separated by at least one other barrier.
__device__ __forceinline__ void find_bin_fast(const uint32_t* hist, int nbins, uint32_t krem, uint32_t* warp_buf,
                                              uint32_t* sel, uint32_t& bin, uint32_t& above, uint32_t& count) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = nbins / NT;  // bins per thread, highest bins to thread 0
  uint32_t c[HBINS / NT];
  uint32_t sum = 0;
#pragma unroll
  for (int t = 0; t < HBINS / NT; ++t) {
    c[t] = t < per ? hist[nbins - 1 - (threadIdx.x * per + t)] : 0u;
    sum += c[t];
  }
  uint32_t x = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_buf[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < NT / 32 ? warp_buf[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < NT / 32) warp_buf[lane] = w;
  }
  __syncthreads();
  uint32_t acc = (warp > 0 ? warp_buf[warp - 1] : 0u) + x - sum;
#pragma unroll
  for (int t = 0; t < HBINS / NT; ++t) {
    if (t < per && acc < krem && krem <= acc + c[t]) {
      sel[0] = nbins - 1 - (threadIdx.x * per + t);
      sel[1] = acc;
      sel[2] = c[t];
    }
    acc += c[t];
  }
  __syncthreads();
  bin = sel[0], above = sel[1], count = sel[2];
}

// What one CTA of topk_row_kernel does:
//   ROW_PLAIN  the top k of a row of up to RMAXV positions, into idx;
//   ROW_SLICE  the top k of slice blockIdx.x % nslices (RMAXV positions) of a
//              longer row, as (score, position) into a k-entry block of the
//              workspace: ascending positions, then (-NaN, -1) padding, which
//              ranks below every number;
//   ROW_MERGE  the top k of a long row from the union of its slices' blocks.
//              The blocks are in slice order and each is ascending, so union
//              order is position order and ties still go to the lower position.
enum RowMode { ROW_PLAIN = 0, ROW_SLICE = 1, ROW_MERGE = 2 };
constexpr uint32_t PAD_SCORE_BITS = 0xffc00000u;  // -NaN: its key is below every number's

template <int MODE>
__global__ void __launch_bounds__(RNT, 2)
    topk_row_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ q_pos, int32_t k,
                    int32_t* __restrict__ idx, int32_t* status, float* __restrict__ ws_score,
                    int32_t* __restrict__ ws_pos, int nslices) {
  extern __shared__ __align__(16) uint32_t rsm[];
  uint32_t* ckey = rsm;                                              // [RLCAP] candidate scores, then keys
  uint32_t* hist = ckey + RLCAP;                                     // [HBINS]
  uint32_t* above_bm = hist + HBINS;                                 // [RWORDS] keys above the threshold
  uint32_t* equal_bm = above_bm + RWORDS;                            // [RWORDS] keys equal to it
  uint16_t* cpos = reinterpret_cast<uint16_t*>(equal_bm + RWORDS);   // [RLCAP] candidate positions
  __shared__ uint32_t warp_buf[32];
  __shared__ uint32_t sel[4];
  __shared__ uint32_t minmax[2];
  __shared__ uint32_t wcount[RWARPS];

  // the next kernel on the stream may be scheduled now; it waits for this
  // grid's results before reading them
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = MODE == ROW_SLICE ? blockIdx.x / nslices : blockIdx.x;
  const int64_t p = q_pos[row];
  const bool bad = p < 0 || p >= ld;
  int32_t* out = idx + row * (int64_t)k;
  const float* s;  // the scores this CTA selects from
  int vis;         // how many of them
  int64_t wbase = 0;
  int64_t first = 0;  // ROW_SLICE: the slice's first position
  if (MODE == ROW_SLICE) {
    first = (int64_t)(blockIdx.x % nslices) * RMAXV;
    const int64_t len = bad ? 0 : (p + 1 - first < 0 ? 0 : (p + 1 - first < RMAXV ? p + 1 - first : RMAXV));
    s = scores + row * ld + first;
    vis = (int)len;
    wbase = (int64_t)blockIdx.x * k;
    if (vis <= k) {  // the whole slice (maybe empty), then padding
      for (int j = tid; j < k; j += RNT) {
        ws_pos[wbase + j] = j < vis ? (int32_t)(first + j) : -1;
        ws_score[wbase + j] = j < vis ? s[j] : __uint_as_float(PAD_SCORE_BITS);
      }
      return;
    }
  } else {
    if (MODE == ROW_MERGE) asm volatile("griddepcontrol.wait;" ::: "memory");  // the slices' blocks
    if (bad) {
      if (tid == 0) report(status, DSA_DEV_BAD_QPOS);
      for (int j = tid; j < k; j += RNT) out[j] = -1;
      return;
    }
    if (p + 1 <= k) {
      for (int j = tid; j < k; j += RNT) out[j] = j < p + 1 ? j : -1;
      return;
    }
    if (MODE == ROW_MERGE) {
      wbase = row * (int64_t)nslices * k;
      s = ws_score + wbase;
      vis = nslices * k;  // <= RMAXV
    } else {
      s = scores + row * ld;
      vis = (int)(p + 1);  // <= ld <= RMAXV
    }
  }
  // output slot o gets the element at offset q of s
  auto emit = [&](uint32_t o, int32_t q) {
    if (MODE == ROW_PLAIN) {
      out[o] = q;
    } else if (MODE == ROW_SLICE) {
      ws_pos[wbase + o] = (int32_t)(first + q);
      ws_score[wbase + o] = s[q];
    } else {
      out[o] = ws_pos[wbase + q];
    }
  };
  const int head0 = (int)(((16u - (uint32_t)(reinterpret_cast<uintptr_t>(s) & 15u)) & 15u) >> 2);
  const int h0 = head0 < vis ? head0 : vis;  // positions before the first 16-byte boundary
  const int nv4 = (vis - h0) >> 2;           // whole float4s after them
  const float4* s4 = reinterpret_cast<const float4*>(s + h0);
  constexpr int HB = RDEPTH / 2;  // float4s per thread in a half-batch
  auto load = [&](float4 (&v)[HB], int base) {
#pragma unroll
    for (int d = 0; d < HB; ++d) {
      const int f = base + d * RNT + tid;
      v[d] = f < nv4 ? __ldg(s4 + f) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };

  // ---- 0. loads in this order: a 1/16 sample (the first 8 of every 128
  // positions), then the whole row into L2 (eight 16-byte-aligned pieces
  // inside it) ----
  const bool sampled = vis > RALL;
  const int blk = tid * SAMPLE_BLOCK;  // one sample block per thread covers a row
  float sv[SAMPLE_RUN];
#pragma unroll
  for (int t = 0; t < SAMPLE_RUN; ++t) sv[t] = sampled && blk + t < vis ? __ldg(s + blk + t) : 0.f;
  if (tid < 8) {
    const uintptr_t a0 = (reinterpret_cast<uintptr_t>(s) + 15u) & ~uintptr_t(15);
    const uintptr_t a1 = reinterpret_cast<uintptr_t>(s + vis) & ~uintptr_t(15);
    if (a1 > a0) {
      const uintptr_t piece = ((a1 - a0) / 8 + 15u) & ~uintptr_t(15);
      const uintptr_t b0 = a0 + piece * (uintptr_t)tid;
      const uintptr_t b1 = b0 + piece < a1 ? b0 + piece : a1;
      if (b1 > b0) l2_prefetch_bulk(b0, (uint32_t)(b1 - b0));
    }
  }
  for (int b = tid; b < HBINS; b += RNT) hist[b] = 0u;
  for (int b = tid; b < 2 * RWORDS; b += RNT) above_bm[b] = 0u;
  if (tid == 0) minmax[0] = 0xffffffffu, minmax[1] = 0u;
  __syncthreads();

  // ---- 1. the lower threshold from the sample ----
  uint32_t t_lo = 0u;
  if (sampled) {
#pragma unroll
    for (int t = 0; t < SAMPLE_RUN; ++t)
      if (blk + t < vis) atomicAdd(&hist[score_key(sv[t]) >> 20], 1u);
    const uint32_t ns = (uint32_t)(vis / SAMPLE_BLOCK) * SAMPLE_RUN + (uint32_t)min(vis % SAMPLE_BLOCK, SAMPLE_RUN);
    const float expect = (float)k * (float)ns / (float)vis;
    uint32_t need = (uint32_t)(expect * 1.25f) + 16u;
    if (need > ns) need = ns;
    __syncthreads();
    uint32_t bin, above, count;
    find_bin_fast(hist, HBINS, need, warp_buf, sel, bin, above, count);
    t_lo = bin << 20;
    for (int b = tid; b < HBINS; b += RNT) hist[b] = 0u;  // read by now; both radix buffers start cleared
  }

  // ---- 2. one streaming pass; each warp lists its candidates ----
  // The screen is a float compare: for every score that is not a NaN,
  // key(x) >= T_lo exactly when x >= f_lo, f_lo being the number whose key is
  // T_lo (-inf when T_lo lies below the key of -inf; a NaN, which nothing
  // passes, when it lies above the key of +inf).  The list keeps the scores'
  // bits; keys are formed only for the candidates, after the stream.
  const uint32_t lo_bits = t_lo >= 0x80000000u ? (t_lo & 0x7fffffffu) : ~t_lo;
  const float f_lo = t_lo < 0x80000000u && lo_bits > 0xff800000u ? -INFINITY : __uint_as_float(lo_bits);
  uint32_t wcnt = 0;  // the same in every lane of the warp
  uint32_t* wkey = ckey + warp * RWCAP;
  uint16_t* wpos = cpos + warp * RWCAP;
  const uint32_t lanes_below = (1u << lane) - 1u;
  auto push = [&](bool cand, float x, int pos) {
    const uint32_t b = __ballot_sync(0xffffffffu, cand);
    if (b) {
      const uint32_t r = wcnt + __popc(b & lanes_below);
      if (cand && r < (uint32_t)RWCAP) {
        wkey[r] = __float_as_uint(x);
        wpos[r] = (uint16_t)pos;
      }
      wcnt += __popc(b);
    }
  };
  auto screen = [&](const float4 (&v)[HB], int base) {
#pragma unroll
    for (int d = 0; d < HB; ++d) {
      const int f = base + d * RNT + tid;
      const bool ok = f < nv4;
      const int e = h0 + 4 * f;
      push(ok && v[d].x >= f_lo, v[d].x, e);
      push(ok && v[d].y >= f_lo, v[d].y, e + 1);
      push(ok && v[d].z >= f_lo, v[d].z, e + 2);
      push(ok && v[d].w >= f_lo, v[d].w, e + 3);
    }
  };
  // the loads of one half-batch are in flight while the other is screened
  float4 va[HB], vb[HB];
  load(va, 0);
  for (int base = 0; base < nv4; base += 2 * RNT * HB) {
    load(vb, base + RNT * HB);
    screen(va, base);
    load(va, base + 2 * RNT * HB);
    screen(vb, base + RNT * HB);
  }
  if (warp == 0) {  // the unaligned head (lanes 0-2) and tail (lanes 4-6)
    const int nt = vis - h0 - 4 * nv4;
    const int pe = lane < h0 ? lane : (lane >= 4 && lane - 4 < nt ? h0 + 4 * nv4 + lane - 4 : -1);
    const float x = pe >= 0 ? __ldg(s + pe) : 0.f;
    push(pe >= 0 && x >= f_lo, x, pe);
  }
  if (lane == 0) wcount[warp] = wcnt;
  __syncthreads();
  uint32_t total = 0;
  bool full = false;
#pragma unroll
  for (int w = 0; w < RWARPS; ++w) {
    total += wcount[w];
    full |= wcount[w] > (uint32_t)RWCAP;
  }
  if (full || total < (uint32_t)k) {
    // the sample misled: exact selection over the row in global memory
    select_exact<true>(s, nullptr, nullptr, vis, (uint32_t)k, emit, hist, warp_buf, sel);
    return;
  }

  // ---- 3. exact k-th largest key among the candidates ----
  // thread t holds entry t of every warp's segment
  uint32_t have = 0;  // bit w: entry t of segment w exists
#pragma unroll
  for (int w = 0; w < RWARPS; ++w)
    if ((uint32_t)tid < wcount[w]) have |= 1u << w;
  uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll
  for (int w = 0; w < RWARPS; ++w) {
    if ((have >> w) & 1u) {
      const uint32_t key = score_key(__uint_as_float(ckey[w * RWCAP + tid]));
      ckey[w * RWCAP + tid] = key;  // from here on the list holds keys
      lo = min(lo, key);
      hi = max(hi, key);
    }
  }
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  if (lane == 0) {
    atomicMin(&minmax[0], lo);
    atomicMax(&minmax[1], hi);
  }
  __syncthreads();
  // radix state over u = key - kmin: every u with (u & mask) > prefix is
  // taken, and the first krem by position with (u & mask) == prefix
  const uint32_t kmin = minmax[0];
  uint32_t top = 32 - __clz(minmax[1] - kmin);  // significant bits of (key - kmin)
  uint32_t prefix = 0, mask = 0, krem = (uint32_t)k;
  for (int pass = 0; top > 0; ++pass) {
    uint32_t* h = hist + (pass & 1) * 2048;  // each buffer is cleared while the other counts
    const int sh = top > 11 ? (int)top - 11 : 0;
    const uint32_t dm = (1u << (top - sh)) - 1u;
#pragma unroll
    for (int w = 0; w < RWARPS; ++w) {
      if ((have >> w) & 1u) {
        const uint32_t u = ckey[w * RWCAP + tid] - kmin;
        if ((u & mask) == prefix) atomicAdd(&h[(u >> sh) & dm], 1u);
      }
    }
    __syncthreads();
    uint32_t bin, above, count;
    find_bin_fast(h, 2048, krem, warp_buf, sel, bin, above, count);
    for (int b = tid; b < 2048; b += RNT) h[b] = 0u;
    prefix |= bin << sh;
    mask |= dm << sh;
    krem -= above;
    top = sh;
    if (count == krem) break;  // the whole bin is taken
  }

  // ---- 4. mark, then write in position order ----
#pragma unroll
  for (int w = 0; w < RWARPS; ++w) {
    if ((have >> w) & 1u) {
      const uint32_t mk = (ckey[w * RWCAP + tid] - kmin) & mask;
      const uint32_t q = cpos[w * RWCAP + tid];
      if (mk > prefix) atomicOr(&above_bm[q >> 5], 1u << (q & 31));
      else if (mk == prefix) atomicOr(&equal_bm[q >> 5], 1u << (q & 31));
    }
  }
  __syncthreads();
  constexpr int WPT = RWORDS / RNT;  // bitmap words per thread: positions 32*WPT*t onwards
  uint32_t aw[WPT], ew[WPT];
  uint32_t n_above = 0, n_eq = 0;
#pragma unroll
  for (int j = 0; j < WPT; ++j) {
    aw[j] = above_bm[tid * WPT + j];
    ew[j] = equal_bm[tid * WPT + j];
    n_above += __popc(aw[j]);
    n_eq += __popc(ew[j]);
  }
  // one scan of (keys above, equal keys) packed in 16 bits each (both < 65536)
  uint32_t packed_total;
  const uint32_t before = block_exclusive_scan((n_above << 16) | n_eq, &packed_total, warp_buf);
  const uint32_t eq_before = before & 0xffffu;
  uint32_t o = (before >> 16) + min(eq_before, krem);  // output slot of this thread's first position
  uint32_t rank = eq_before;
#pragma unroll
  for (int j = 0; j < WPT; ++j) {
    uint32_t e = ew[j];
    while (e && rank < krem) {
      aw[j] |= e & (~e + 1u);  // the lowest equal key still unclaimed
      e &= e - 1u;
      ++rank;
    }
    uint32_t a = aw[j];
    while (a && o < (uint32_t)k) {
      const int b = __ffs(a) - 1;
      a &= a - 1u;
      emit(o++, (tid * WPT + j) * 32 + b);
    }
  }
}

template <int C>
cudaError_t launch_c(const float* scores, int64_t ld, const int32_t* q_pos, int32_t num_q, int32_t k, int32_t* idx,
                     int32_t* dev_status, cudaStream_t stream) {
  auto kern = topk_cluster_kernel<C>;
  const size_t smem = TopkSmem<C>::bytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)num_q * C, NT, smem, stream>>>(scores, ld, q_pos, k, idx, dev_status);
  return cudaGetLastError();
}

}  // namespace

int topk_cluster_size(int32_t num_q, int64_t ld, int num_sms) {
  // One CTA per row once the rows alone give half the SMs work; otherwise
  // split long rows over a cluster until about one CTA per SM, keeping
  // slices of at least 64K positions.
  int c = 1;
  if ((int64_t)num_q * 2 >= num_sms) return 1;
  while (c < 8 && (int64_t)num_q * c * 2 <= (int64_t)num_sms && ld / (2 * c) >= 65536) c *= 2;
  return c;
}

size_t topk_workspace_bytes(int32_t num_q, int64_t ld, int32_t k) {
  if (num_q <= 0 || k <= 0 || ld <= RMAXV) return 0;
  const int64_t slices = (ld + RMAXV - 1) / RMAXV;
  if (slices * k > RMAXV) return 0;  // the union would not fit one CTA: the cluster kernel runs
  return (size_t)num_q * (size_t)slices * (size_t)k * (sizeof(float) + sizeof(int32_t));
}

cudaError_t launch_topk(const float* scores, int64_t ld, const int32_t* q_pos, int32_t num_q, int32_t k,
                        int32_t* idx, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        cudaStream_t stream) {
  if (num_q == 0) return cudaSuccess;
  if (ld <= RMAXV) {
    cudaError_t e =
        cudaFuncSetAttribute(topk_row_kernel<ROW_PLAIN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)RSMEM);
    if (e != cudaSuccess) return e;
    topk_row_kernel<ROW_PLAIN><<<(unsigned)num_q, RNT, RSMEM, stream>>>(scores, ld, q_pos, k, idx, dev_status,
                                                                        nullptr, nullptr, 1);
    return cudaGetLastError();
  }
  const size_t need = topk_workspace_bytes(num_q, ld, k);
  if (need > 0 && workspace != nullptr && workspace_bytes >= need) {
    // slices of RMAXV positions, then one merge per row (a programmatic
    // dependent launch that waits for the slices' blocks)
    const int slices = (int)((ld + RMAXV - 1) / RMAXV);
    float* ws_score = static_cast<float*>(workspace);
    int32_t* ws_pos = reinterpret_cast<int32_t*>(ws_score + (size_t)num_q * slices * k);
    cudaError_t e =
        cudaFuncSetAttribute(topk_row_kernel<ROW_SLICE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)RSMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(topk_row_kernel<ROW_MERGE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)RSMEM);
    if (e != cudaSuccess) return e;
    topk_row_kernel<ROW_SLICE><<<(unsigned)num_q * slices, RNT, RSMEM, stream>>>(scores, ld, q_pos, k, idx,
                                                                                 dev_status, ws_score, ws_pos,
                                                                                 slices);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)num_q);
    cfg.blockDim = dim3(RNT);
    cfg.dynamicSmemBytes = RSMEM;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, topk_row_kernel<ROW_MERGE>, scores, ld, q_pos, k, idx, dev_status, ws_score,
                           ws_pos, slices);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  const int sms = device_sm_count();
  switch (topk_cluster_size(num_q, ld, sms)) {
    case 8: return launch_c<8>(scores, ld, q_pos, num_q, k, idx, dev_status, stream);
    case 4: return launch_c<4>(scores, ld, q_pos, num_q, k, idx, dev_status, stream);
    case 2: return launch_c<2>(scores, ld, q_pos, num_q, k, idx, dev_status, stream);
    default: return launch_c<1>(scores, ld, q_pos, num_q, k, idx, dev_status, stream);
  }
}

}  // namespace dsa
