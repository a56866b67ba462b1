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
#include "topk_row.cuh"

namespace cg = cooperative_groups;

namespace dsa {
namespace {


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

// ROW_RESOLVE: ROW_PLAIN that also writes each output's (slot, scale) pair.
enum RowMode { ROW_PLAIN = 0, ROW_SLICE = 1, ROW_MERGE = 2, ROW_RESOLVE = 3 };
constexpr uint32_t PAD_SCORE_BITS = 0xffc00000u;  // -NaN: its key is below every number's

template <int MODE>
__global__ void __launch_bounds__(RNT, 2)
    topk_row_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ q_pos, int32_t k,
                    int32_t* __restrict__ idx, int32_t* status, float* __restrict__ ws_score,
                    int32_t* __restrict__ ws_pos, int nslices, const TopkResolve rv) {
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
  const int tid = threadIdx.x;
  const int64_t row = MODE == ROW_SLICE ? blockIdx.x / nslices : blockIdx.x;
  const int64_t p = q_pos[row];
  const int32_t r = MODE == ROW_RESOLVE ? rv.q_req[row] : 0;  // the row's request, for the lookups
  const bool bad = p < 0 || p >= ld;
  int32_t* out = idx + row * (int64_t)k;
  // ROW_RESOLVE: outputs j of the row, at positions pos_of(j) (or -1), go to
  // idx and, looked up in the block table, to rv.res; each of the two
  // dependent loads (page, scale) is issued for four outputs at once
  auto resolve_outputs = [&](auto pos_of) {
    const bool req_ok = r >= 0 && r < rv.num_req;
    int2* res = rv.res + row * (int64_t)k;
    for (int j0 = tid; j0 < k; j0 += 4 * RNT) {
      int32_t pos[4], page[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) pos[e] = j0 + e * RNT < k ? pos_of(j0 + e * RNT) : -1;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        page[e] = -1;
        if (pos[e] >= 0 && req_ok && pos[e] / rv.page_size < rv.bt_stride)
          page[e] = rv.block_table[(int64_t)r * rv.bt_stride + pos[e] / rv.page_size];
      }
      int32_t slot[4];
      float sc[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        slot[e] = -1;
        sc[e] = 0.f;
        if (pos[e] >= 0) {
          if (!req_ok) {
            report(status, DSA_DEV_BAD_PAGE);
          } else if (pos[e] / rv.page_size >= rv.bt_stride) {
            report(status, DSA_DEV_BAD_INDEX);
          } else if (page[e] < 0 || page[e] >= rv.num_pages) {
            report(status, DSA_DEV_BAD_PAGE);
          } else {
            slot[e] = page[e] * rv.page_size + pos[e] % rv.page_size;
            sc[e] = rv.kv_scale[slot[e]];
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {  // the stores after all four scale loads
        const int j = j0 + e * RNT;
        if (j < k) {
          out[j] = pos[e];
          res[j] = make_int2(slot[e], __float_as_int(sc[e]));
        }
      }
    }
  };
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
      if (MODE == ROW_RESOLVE)
        resolve_outputs([](int) { return -1; });
      else
        for (int j = tid; j < k; j += RNT) out[j] = -1;
      return;
    }
    if (MODE == ROW_RESOLVE && (tid >> 5) == RWARPS - 1 && r >= 0 && r < rv.num_req) {
      // the request's block-table entries for the visible positions into L2
      // for the lookups after the selection (one line per lane)
      const int lane = tid & 31;
      const int64_t nb = 4 * (int64_t)min((int64_t)rv.bt_stride, (p + rv.page_size) / rv.page_size);
      const char* btrow = reinterpret_cast<const char*>(rv.block_table + (int64_t)r * rv.bt_stride);
      for (int64_t off = lane * 128; off < nb; off += 32 * 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(btrow + off));
      if (lane == 0) asm volatile("prefetch.global.L2 [%0];" ::"l"(btrow + nb - 1));  // an unaligned row's last line
    }
    if (p + 1 <= k) {
      if (MODE == ROW_RESOLVE)
        resolve_outputs([&](int j) { return j < p + 1 ? j : -1; });
      else
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
  // output slot o gets the element at offset q of s.  With k <= RLCAP the
  // slice and merge kernels keep q in shared memory (where the candidate keys
  // were, read by then) and look the outputs up afterwards, all of a thread's
  // loads at once, instead of one dependent load per output.
  int32_t* chosen = reinterpret_cast<int32_t*>(ckey);
  const bool deferred = MODE != ROW_PLAIN && k <= RLCAP;
  auto emit = [&](uint32_t o, int32_t q) {
    if (MODE == ROW_PLAIN || (MODE == ROW_RESOLVE && !deferred)) {
      out[o] = q;
    } else if (deferred) {
      chosen[o] = q;
    } else if (MODE == ROW_SLICE) {
      ws_pos[wbase + o] = (int32_t)(first + q);
      ws_score[wbase + o] = s[q];
    } else {
      out[o] = ws_pos[wbase + q];
    }
  };
  row_select(s, vis, k, emit, ckey, hist, above_bm, equal_bm, cpos, warp_buf, sel, minmax, wcount);
  if (MODE == ROW_RESOLVE) {
    __syncthreads();
    if (deferred)
      resolve_outputs([&](int j) { return chosen[j]; });
    else
      resolve_outputs([&](int j) { return __ldcg(out + j); });  // this CTA's own stores, before the barrier
  } else if (deferred) {
    __syncthreads();
    if (MODE == ROW_SLICE) {
      for (int j = tid; j < k; j += RNT) {
        const int32_t q = chosen[j];
        ws_pos[wbase + j] = (int32_t)(first + q);
        ws_score[wbase + j] = s[q];
      }
    } else {
      for (int j = tid; j < k; j += RNT) out[j] = ws_pos[wbase + chosen[j]];
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
                                                                        nullptr, nullptr, 1, TopkResolve{});
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
                                                                                 slices, TopkResolve{});
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
                           ws_pos, slices, TopkResolve{});
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

cudaError_t launch_topk_resolve(const float* scores, int64_t ld, const int32_t* q_pos, int32_t num_q, int32_t k,
                                int32_t* idx, const TopkResolve& rv, int32_t* dev_status, cudaStream_t stream) {
  if (num_q == 0) return cudaSuccess;
  if (ld > RMAXV) return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(topk_row_kernel<ROW_RESOLVE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)RSMEM);
  if (e != cudaSuccess) return e;
  topk_row_kernel<ROW_RESOLVE><<<(unsigned)num_q, RNT, RSMEM, stream>>>(scores, ld, q_pos, k, idx, dev_status,
                                                                          nullptr, nullptr, 1, rv);
  return cudaGetLastError();
}

}  // namespace dsa
