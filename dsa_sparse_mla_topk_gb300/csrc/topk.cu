// Causal top-k selection over fp32 indexer scores.
//
// "Accelerating GLM-5.3-Flash on H200", section 3 "Larger KV tiles for DSA
// Partial": the indexer's scores pick the KV positions the Partial step
// attends to.  This kernel makes the pick exact and deterministic: positions
// are ranked by (score descending, position ascending), -0.0 == +0.0, and
// the chosen ones are written in ascending position order, -1 padded.
//
// Every fp32 score maps to an order-preserving 32-bit key.  A row is handled
// by a thread-block cluster of C CTAs, each owning a contiguous slice of the
// visible positions:
//   1. each CTA histograms the top 12 key bits of a 1/16 sample of its slice;
//      the histograms are summed over the cluster (distributed shared memory)
//      and give a lower threshold T_lo that, with a wide safety margin, lies
//      below the k-th largest key;
//   2. one streaming pass collects every key >= T_lo with its position, in
//      position order (warp ballots + a scan of warp counts);
//   3. CTA 0 gathers the candidates of the cluster, finds the exact key T of
//      the k-th largest entry by radix select over the candidates, and writes
//      the keys above T plus the lowest-positioned entries equal to T.
// If the sample misleads (fewer than k candidates, or more than fit), CTA 0
// falls back to an exact multi-pass radix select over the whole row in
// global memory, so the result never depends on the score distribution.
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

// Exclusive prefix sum of one value per thread over the block; *total gets
// the block sum.  `warp_buf` holds 32 words of shared memory.
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
    uint32_t w = lane < NT / 32 ? warp_buf[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
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
// ascending position order): writes the k chosen positions ascending.
// Radix passes of up to 11 bits run over (key - kmin) from its highest set
// bit down, so the bins spread over the keys' actual range (candidate keys
// share their top bits; fixed digits would pile them into a few bins).
template <bool GLOBAL_ROW>
__device__ void select_exact(const float* row_scores, const uint32_t* keys, const int32_t* pos, int64_t n, uint32_t k,
                             int32_t* out, uint32_t* hist, uint32_t* warp_buf, uint32_t* sel) {
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
      if (((take >> t) & 1u) && o < k) out[o++] = pos_at(e0 + t);
    ties_before += eq_total;
    written += take_total;
  }
}

template <int C>
struct TopkSmem {
  // candidates one CTA collects; sized so that two 1024-thread CTAs fit on an SM
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
      const double expect = (double)k * (double)ns / (double)vis;
      uint32_t need = (uint32_t)(expect * 1.25) + 16u;
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
    select_exact<false>(nullptr, mkey, mpos, vars[3], (uint32_t)k, out, hist, warp_buf, sel);
  } else {
    select_exact<true>(s, nullptr, nullptr, vis, (uint32_t)k, out, hist, warp_buf, sel);
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

cudaError_t launch_topk(const float* scores, int64_t ld, const int32_t* q_pos, int32_t num_q, int32_t k,
                        int32_t* idx, int32_t* dev_status, cudaStream_t stream) {
  if (num_q == 0) return cudaSuccess;
  const int sms = device_sm_count();
  switch (topk_cluster_size(num_q, ld, sms)) {
    case 8: return launch_c<8>(scores, ld, q_pos, num_q, k, idx, dev_status, stream);
    case 4: return launch_c<4>(scores, ld, q_pos, num_q, k, idx, dev_status, stream);
    case 2: return launch_c<2>(scores, ld, q_pos, num_q, k, idx, dev_status, stream);
    default: return launch_c<1>(scores, ld, q_pos, num_q, k, idx, dev_status, stream);
  }
}

}  // namespace dsa
