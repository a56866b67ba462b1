// Exact causal top-k selection of one row by one CTA of 512 threads: the
// shared part of the standalone top-k kernels (topk.cu) and of the fused
// decode kernel (mla_tc.cu), which selects its own token's positions before
// attending to them.
//
// "Accelerating GLM-5.3-Flash on H200", section 3 "Larger KV tiles for DSA
// Partial": the indexer's scores pick the KV positions the Partial step
// attends to.  Positions are ranked by (score descending, position
// ascending), -0.0 == +0.0, and the chosen ones are written in ascending
// position order.  Every fp32 score maps to an order-preserving 32-bit key.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.cuh"

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


// ---------------------------------------------------------------------------
// Rows of up to 65,536 visible positions: one CTA of 512 threads per row,
// two CTAs per SM (80 KB of shared memory each), so that one CTA streams
// while the other selects.
//   0. The loads of a 1/16 sample (the first 32 of every 512 positions: whole
//      128-byte lines) are issued first, then an L2 bulk prefetch of the row.
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
// The row's sample: the first RS_RUN positions of every RS_BLOCK (1/16),
// whole 128-byte lines, eight positions per thread.
constexpr int RS_BLOCK = 512, RS_RUN = 32;
static_assert((RNT / (RS_RUN / 8)) * RS_BLOCK == RMAXV, "the threads' sample runs cover a row");

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

// Steps 0-4 above for the `vis` scores at `s` (vis <= RMAXV, vis > k): emit(o,
// q) receives output slot o (0..k-1, ascending positions) and the offset q of
// the chosen score within s.  Called by all RNT threads of the CTA; the
// shared-memory arrays are the caller's: ckey[RLCAP], hist[HBINS],
// above_bm[RWORDS], equal_bm[RWORDS], cpos[RLCAP], warp_buf[32], sel[4],
// minmax[2], wcount[RWARPS].
template <class Emit>
__device__ __forceinline__ void row_select(const float* s, int vis, int k, Emit emit, uint32_t* ckey, uint32_t* hist,
                                           uint32_t* above_bm, uint32_t* equal_bm, uint16_t* cpos,
                                           uint32_t* warp_buf, uint32_t* sel, uint32_t* minmax, uint32_t* wcount) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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

  // ---- 0. loads in this order: a 1/16 sample (the first 32 of every 512
  // positions) and the stream's first half-batch; the rest of the row into
  // L2 (16-byte-aligned pieces inside it) follows in step 1 ----
  const bool sampled = vis > RALL;
  constexpr int SPT = 8;  // sampled positions per thread: two float4s
  const int blk = (tid / (RS_RUN / SPT)) * RS_BLOCK + (tid % (RS_RUN / SPT)) * SPT;
  float sv[SPT];
  if (sampled && head0 == 0 && blk + SPT <= vis) {  // 16-byte aligned: two vector loads
    const float4 u0 = __ldg(reinterpret_cast<const float4*>(s + blk));
    const float4 u1 = __ldg(reinterpret_cast<const float4*>(s + blk) + 1);
    sv[0] = u0.x, sv[1] = u0.y, sv[2] = u0.z, sv[3] = u0.w;
    sv[4] = u1.x, sv[5] = u1.y, sv[6] = u1.z, sv[7] = u1.w;
  } else {
#pragma unroll
    for (int t = 0; t < SPT; ++t) sv[t] = sampled && blk + t < vis ? __ldg(s + blk + t) : 0.f;
  }
  // the stream's first half-batch is in flight during the threshold step
  float4 va[HB], vb[HB];
  load(va, 0);
  for (int b = tid; b < HBINS; b += RNT) hist[b] = 0u;
  for (int b = tid; b < RWORDS; b += RNT) {  // the two bitmaps need not be adjacent
    above_bm[b] = 0u;
    equal_bm[b] = 0u;
  }
  if (tid == 0) minmax[0] = 0xffffffffu, minmax[1] = 0u;
  __syncthreads();

  // ---- 1. the lower threshold from the sample ----
  uint32_t t_lo = 0u;
  if (sampled) {
#pragma unroll
    for (int t = 0; t < SPT; ++t)
      if (blk + t < vis) atomicAdd(&hist[score_key(sv[t]) >> 20], 1u);
  }
  // the rest of the row (past the first half-batch) into L2 in 16 pieces,
  // once this thread's sample has landed: issued at kernel start, the 128
  // rows' prefetches held back the samples
  if (tid < 16) {
    const uintptr_t a0 = (reinterpret_cast<uintptr_t>(s4 + min(nv4, RNT * HB)) + 15u) & ~uintptr_t(15);
    const uintptr_t a1 = reinterpret_cast<uintptr_t>(s + vis) & ~uintptr_t(15);
    if (a1 > a0) {
      const uintptr_t piece = ((a1 - a0) / 16 + 15u) & ~uintptr_t(15);
      const uintptr_t b0 = a0 + piece * (uintptr_t)tid;
      const uintptr_t b1 = b0 + piece < a1 ? b0 + piece : a1;
      if (b1 > b0) l2_prefetch_bulk(b0, (uint32_t)(b1 - b0));
    }
  }
  if (sampled) {
    const uint32_t ns = (uint32_t)(vis / RS_BLOCK) * RS_RUN + (uint32_t)min(vis % RS_BLOCK, RS_RUN);
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
  // A float4 per lane at a time: its four ballots first, then every
  // candidate's slot from their counts (component-major within the warp's
  // step; the list's order does not matter), stored without branches.
  auto screen = [&](const float4 (&v)[HB], int base) {
#pragma unroll
    for (int d = 0; d < HB; ++d) {
      const int f = base + d * RNT + tid;
      const bool ok = f < nv4;
      const int e = h0 + 4 * f;
      const float x[4] = {v[d].x, v[d].y, v[d].z, v[d].w};
      bool c[4];
      uint32_t b[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        c[q] = ok && x[q] >= f_lo;
        b[q] = __ballot_sync(0xffffffffu, c[q]);
      }
      uint32_t r = wcnt;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t slot = r + __popc(b[q] & lanes_below);
        if (c[q] && slot < (uint32_t)RWCAP) {
          wkey[slot] = __float_as_uint(x[q]);
          wpos[slot] = (uint16_t)(e + q);
        }
        r += __popc(b[q]);
      }
      wcnt = r;
    }
  };
  // the loads of one half-batch are in flight while the other is screened
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

}  // namespace
}  // namespace dsa
