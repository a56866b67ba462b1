/*
 * dsa_oracle.c -- fp64 CPU oracle for DSA sparse MLA with top-k selection.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library: it is the plain definition of what the library computes,
 * written out in double precision so that a reader can check it against the
 * sources below by eye.
 *
 * Sources (page titles as published):
 *  - "Accelerating GLM-5.3-Flash on H200: High-Throughput Disaggregated
 *    Serving" (LMSYS blog), section 1 "Architecture and workloads": an
 *    indexer selects historical positions and sparse attention (DSA) runs over
 *    them; section 3 "Larger KV tiles for DSA Partial": the Partial step loads
 *    the selected KV positions and computes Q K^T, softmax and the weighted
 *    value sum, and a Combine step merges KV splits; section 2 "KV-only decode
 *    RadixCache": prefix KV pages are shared between requests.
 *  - "GLM-5.3 Optimizations, Part 2: PCP, DCP, and Hybrid HiSparse on 16
 *    H200s" (vLLM digest), "Interpretation": MLA's latent KV row is shared by
 *    all 64 heads.
 *  - SGLang cookbook page for GLM-5.3-Flash, "Keep the KV and DSA backends
 *    paired": the KV cache is FP8 (E4M3) on Blackwell.
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes): a KV row is latent (d_latent) || rope (d_rope) FP8 e4m3 bytes with
 * one fp32 scale per token; K is the whole row and V is its latent part; top-k
 * orders positions by (score descending, position ascending), treats -0.0 and
 * +0.0 as equal, and emits the chosen positions in ascending order padded with
 * -1; a query token at position p sees positions 0..p (causal).
 *
 * Every function below is pinned by tests/test_oracle_pins.py against things
 * other than itself (library routines on special cases, closed forms,
 * brute force, invariants, hand-written fixtures).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_BAD_QPOS 1
#define ORACLE_BAD_INDEX 2
#define ORACLE_BAD_PAGE 4
#define ORACLE_NOMEM 8

/* ---- number formats --------------------------------------------------- */

/* FP8 E4M3 ("fn" variant): 1 sign bit, 4 exponent bits with bias 7, 3
 * mantissa bits; exponent field 0 encodes subnormals m/8 * 2^-6; the pattern
 * S.1111.111 is NaN and there is no infinity, so the largest finite value is
 * 1.75 * 2^8 = 448. */
double oracle_e4m3_to_double(uint8_t b) {
  int sign = (b >> 7) & 1;
  int e = (b >> 3) & 15;
  int m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* ---- a tiny thread pool over query tokens ----------------------------- */

typedef void (*row_fn)(void* ctx, int64_t row);
typedef struct {
  row_fn fn;
  void* ctx;
  int64_t n;
  int64_t next;
  pthread_mutex_t mu;
} pool_t;

static void* pool_worker(void* arg) {
  pool_t* p = (pool_t*)arg;
  for (;;) {
    pthread_mutex_lock(&p->mu);
    int64_t r = p->next++;
    pthread_mutex_unlock(&p->mu);
    if (r >= p->n) break;
    p->fn(p->ctx, r);
  }
  return NULL;
}

static int oracle_threads(int requested) {
  if (requested > 0) return requested;
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

static void run_rows(row_fn fn, void* ctx, int64_t n, int nthreads) {
  pool_t p;
  p.fn = fn;
  p.ctx = ctx;
  p.n = n;
  p.next = 0;
  pthread_mutex_init(&p.mu, NULL);
  int t = oracle_threads(nthreads);
  if (t > n) t = (int)(n > 0 ? n : 1);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)t);
  int started = 0;
  for (int i = 1; th && i < t; ++i)
    if (pthread_create(&th[started], NULL, pool_worker, &p) == 0) ++started;
  /* the calling thread works too */
  pool_worker(&p);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  free(th);
  pthread_mutex_destroy(&p.mu);
}

/* ---- top-k ------------------------------------------------------------- */

typedef struct {
  double score;
  int32_t pos;
} cand_t;

/* (score descending, position ascending).  Comparing as doubles makes -0.0
 * and +0.0 equal, so such a pair is a tie and goes to the lower position. */
static int cmp_rank(const void* a, const void* b) {
  const cand_t* x = (const cand_t*)a;
  const cand_t* y = (const cand_t*)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
  return (x->pos > y->pos) - (x->pos < y->pos);
}

static int cmp_i32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

typedef struct {
  const float* scores;
  int64_t ld;
  const int32_t* q_pos;
  int32_t k;
  int32_t* idx;
  int status;
  pthread_mutex_t mu;
} topk_ctx;

static void topk_row(void* vctx, int64_t i) {
  topk_ctx* c = (topk_ctx*)vctx;
  int32_t* out = c->idx + i * (int64_t)c->k;
  int64_t p = c->q_pos[i];
  if (p < 0 || p >= c->ld) {
    pthread_mutex_lock(&c->mu);
    c->status |= ORACLE_BAD_QPOS;
    pthread_mutex_unlock(&c->mu);
    for (int32_t j = 0; j < c->k; ++j) out[j] = -1;
    return;
  }
  int64_t vis = p + 1; /* causal: positions 0..p are visible */
  cand_t* cand = (cand_t*)malloc(sizeof(cand_t) * (size_t)vis);
  if (!cand) {
    pthread_mutex_lock(&c->mu);
    c->status |= ORACLE_NOMEM;
    pthread_mutex_unlock(&c->mu);
    return;
  }
  const float* s = c->scores + i * c->ld;
  for (int64_t j = 0; j < vis; ++j) {
    cand[j].score = (double)s[j];
    cand[j].pos = (int32_t)j;
  }
  qsort(cand, (size_t)vis, sizeof(cand_t), cmp_rank);
  int64_t take = vis < c->k ? vis : c->k;
  for (int64_t j = 0; j < take; ++j) out[j] = cand[j].pos;
  qsort(out, (size_t)take, sizeof(int32_t), cmp_i32);
  for (int64_t j = take; j < c->k; ++j) out[j] = -1;
  free(cand);
}

/* idx[num_q, k]: for query row i, the min(k, q_pos[i]+1) visible positions
 * with the largest scores[i, :], ties to the lower position, listed in
 * ascending position order, then -1 padding. */
int oracle_topk(const float* scores, int64_t ld, const int32_t* q_pos, int32_t num_q, int32_t k,
                int32_t* idx, int nthreads) {
  topk_ctx c;
  c.scores = scores;
  c.ld = ld;
  c.q_pos = q_pos;
  c.k = k;
  c.idx = idx;
  c.status = ORACLE_OK;
  pthread_mutex_init(&c.mu, NULL);
  run_rows(topk_row, &c, num_q, nthreads);
  pthread_mutex_destroy(&c.mu);
  return c.status;
}

/* ---- sparse MLA attention ---------------------------------------------- */

typedef struct {
  const uint16_t* q; /* bf16 [num_q, H, d_latent + d_rope] */
  const uint8_t* kv; /* e4m3 [slots, d_latent + d_rope] */
  const float* kv_scale; /* [slots] */
  const int32_t* block_table;
  int64_t bt_stride;
  int64_t num_pages;
  const int32_t* q_req;
  const int32_t* idx;
  int32_t k, H, dl, dr, page;
  int32_t num_splits;
  double softmax_scale;
  double* out; /* [num_q, H, dl] */
  double* lse; /* [num_q, H] */
  double* o_part; /* optional [S, num_q, H, dl] */
  double* lse_part; /* optional [S, num_q, H] */
  int64_t num_q;
  int status;
  pthread_mutex_t mu;
} mla_ctx;

static void set_status(mla_ctx* c, int bit) {
  pthread_mutex_lock(&c->mu);
  c->status |= bit;
  pthread_mutex_unlock(&c->mu);
}

/* Plain softmax attention of one query token (all heads) over n dequantised
 * rows x[n, dqk]: z = scale * q . x, p = exp(z - max z), l = sum p,
 * O = sum p x[:, :dl] / l, lse = max z + ln l.  With n == 0 the result is
 * O = 0 and lse = -inf. */
static void attend(const double* q, const double* x, int64_t n, int32_t H, int32_t dqk, int32_t dl,
                   double scale, double* z, double* O, double* lse) {
  for (int32_t h = 0; h < H; ++h) {
    const double* qh = q + (int64_t)h * dqk;
    double* oh = O + (int64_t)h * dl;
    for (int32_t d = 0; d < dl; ++d) oh[d] = 0.0;
    if (n == 0) {
      lse[h] = -INFINITY;
      continue;
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
      const double* xj = x + j * dqk;
      double acc = 0.0;
      for (int32_t d = 0; d < dqk; ++d) acc += qh[d] * xj[d];
      z[j] = scale * acc;
      if (z[j] > m) m = z[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
      double p = exp(z[j] - m);
      l += p;
      const double* xj = x + j * dqk;
      for (int32_t d = 0; d < dl; ++d) oh[d] += p * xj[d];
    }
    for (int32_t d = 0; d < dl; ++d) oh[d] /= l;
    lse[h] = m + log(l);
  }
}

/* Log-sum-exp merge of S partial results of one query token:
 * lse = ln sum_s exp(lse_s); O = sum_s exp(lse_s - lse) O_s.  Splits with
 * lse_s = -inf hold no rows and are skipped; if all are empty, O = 0 and
 * lse = -inf. */
static void merge(const double* O_s, const double* lse_s, int32_t S, int64_t s_stride_o,
                  int64_t s_stride_l, int32_t H, int32_t dl, double* O, double* lse) {
  for (int32_t h = 0; h < H; ++h) {
    double m = -INFINITY;
    for (int32_t s = 0; s < S; ++s) {
      double v = lse_s[s * s_stride_l + h];
      if (v > m) m = v;
    }
    double* oh = O + (int64_t)h * dl;
    for (int32_t d = 0; d < dl; ++d) oh[d] = 0.0;
    if (m == -INFINITY) {
      lse[h] = -INFINITY;
      continue;
    }
    double sum = 0.0;
    for (int32_t s = 0; s < S; ++s) sum += exp(lse_s[s * s_stride_l + h] - m);
    lse[h] = m + log(sum);
    for (int32_t s = 0; s < S; ++s) {
      double w = exp(lse_s[s * s_stride_l + h] - lse[h]);
      if (w == 0.0) continue;
      const double* os = O_s + s * s_stride_o + (int64_t)h * dl;
      for (int32_t d = 0; d < dl; ++d) oh[d] += w * os[d];
    }
  }
}

static void mla_row(void* vctx, int64_t i) {
  mla_ctx* c = (mla_ctx*)vctx;
  const int32_t H = c->H, dl = c->dl, dqk = c->dl + c->dr, P = c->page;
  const int32_t* row_idx = c->idx + i * (int64_t)c->k;
  const int32_t r = c->q_req[i];

  double* q = (double*)malloc(sizeof(double) * (size_t)H * dqk);
  double* x = (double*)malloc(sizeof(double) * (size_t)c->k * dqk);
  double* z = (double*)malloc(sizeof(double) * (size_t)(c->k > 0 ? c->k : 1));
  int32_t S = c->num_splits > 0 ? c->num_splits : 1;
  double* Os = (double*)malloc(sizeof(double) * (size_t)S * H * dl);
  double* Ls = (double*)malloc(sizeof(double) * (size_t)S * H);
  if (!q || !x || !z || !Os || !Ls) {
    set_status(c, ORACLE_NOMEM);
    free(q), free(x), free(z), free(Os), free(Ls);
    return;
  }
  for (int64_t e = 0; e < (int64_t)H * dqk; ++e) q[e] = oracle_bf16_to_double(c->q[i * (int64_t)H * dqk + e]);

  /* dequantise the selected rows through the block table; -1 entries are
   * padding and carry no row */
  int64_t n = 0;
  for (int32_t j = 0; j < c->k; ++j) {
    int32_t pos = row_idx[j];
    if (pos == -1) continue;
    if (pos < -1 || (int64_t)(pos / P) >= c->bt_stride) {
      set_status(c, ORACLE_BAD_INDEX);
      continue;
    }
    int64_t page = c->block_table[(int64_t)r * c->bt_stride + pos / P];
    if (page < 0 || page >= c->num_pages) {
      set_status(c, ORACLE_BAD_PAGE);
      continue;
    }
    int64_t slot = page * P + pos % P;
    const uint8_t* b = c->kv + slot * dqk;
    double sc = (double)c->kv_scale[slot];
    for (int32_t d = 0; d < dqk; ++d) x[n * dqk + d] = oracle_e4m3_to_double(b[d]) * sc;
    ++n;
  }

  /* S contiguous chunks of the selected list, each attended separately and
   * then merged; with S == 1 this is plain attention over all rows */
  for (int32_t s = 0; s < S; ++s) {
    int64_t lo = n * s / S, hi = n * (s + 1) / S;
    attend(q, x + lo * dqk, hi - lo, H, dqk, dl, c->softmax_scale, z, Os + (int64_t)s * H * dl, Ls + (int64_t)s * H);
    if (c->o_part) memcpy(c->o_part + ((int64_t)s * c->num_q + i) * H * dl, Os + (int64_t)s * H * dl, sizeof(double) * (size_t)H * dl);
    if (c->lse_part) memcpy(c->lse_part + ((int64_t)s * c->num_q + i) * H, Ls + (int64_t)s * H, sizeof(double) * (size_t)H);
  }
  merge(Os, Ls, S, (int64_t)H * dl, H, H, dl, c->out + i * (int64_t)H * dl, c->lse + i * (int64_t)H);
  free(q), free(x), free(z), free(Os), free(Ls);
}

/* out[num_q, H, d_latent], lse[num_q, H] in fp64.  The selected list of each
 * query is cut into num_splits contiguous chunks whose partial results are
 * optionally written to o_part/lse_part and merged (num_splits = 1: no
 * split). */
int oracle_sparse_mla(const uint16_t* q, const uint8_t* kv, const float* kv_scale, int64_t num_pages,
                      const int32_t* block_table, int64_t bt_stride, const int32_t* q_req,
                      const int32_t* idx, int64_t num_q, int32_t k, int32_t H, int32_t d_latent,
                      int32_t d_rope, int32_t page_size, double softmax_scale, int32_t num_splits,
                      double* out, double* lse, double* o_part, double* lse_part, int nthreads) {
  mla_ctx c;
  c.q = q;
  c.kv = kv;
  c.kv_scale = kv_scale;
  c.block_table = block_table;
  c.bt_stride = bt_stride;
  c.num_pages = num_pages;
  c.q_req = q_req;
  c.idx = idx;
  c.k = k;
  c.H = H;
  c.dl = d_latent;
  c.dr = d_rope;
  c.page = page_size;
  c.num_splits = num_splits;
  c.softmax_scale = softmax_scale;
  c.out = out;
  c.lse = lse;
  c.o_part = o_part;
  c.lse_part = lse_part;
  c.num_q = num_q;
  c.status = ORACLE_OK;
  pthread_mutex_init(&c.mu, NULL);
  run_rows(mla_row, &c, num_q, nthreads);
  pthread_mutex_destroy(&c.mu);
  return c.status;
}

/* Merge given partials: o_part[S, num_q, H, dv], lse_part[S, num_q, H] ->
 * out[num_q, H, dv], lse[num_q, H]. */
int oracle_combine(const double* o_part, const double* lse_part, int32_t S, int64_t num_q, int32_t H,
                   int32_t dv, double* out, double* lse) {
  for (int64_t i = 0; i < num_q; ++i)
    merge(o_part + i * (int64_t)H * dv, lse_part + i * (int64_t)H, S, num_q * (int64_t)H * dv, num_q * (int64_t)H, H, dv,
          out + i * (int64_t)H * dv, lse + i * (int64_t)H);
  return ORACLE_OK;
}

/* ---- KV cache write: per-token FP8 quantisation and paged scatter ------ */

/* Nearest FP8 E4M3 code of a finite float, ties to even, magnitudes at or
 * above the largest finite value (448) saturating to it (E4M3 has no
 * infinity).  On the E4M3 grid a normal binade [2^e, 2^(e+1)) has 8 steps of
 * 2^(e-3); below 2^-6 the subnormal step is 2^-9.  Scaling by a power of two
 * and rint() (round half to even in the default rounding mode) are exact in
 * double. */
uint8_t oracle_e4m3_encode(float y) {
  const uint8_t sign = signbit(y) ? 0x80 : 0x00;
  const double a = fabs((double)y);
  if (a >= 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) {
    /* subnormal codes 0..7; rounding up to 8 gives the smallest normal, code 8 */
    const double m = rint(a / ldexp(1.0, -9));
    return sign | (uint8_t)m;
  }
  int e2;
  frexp(a, &e2); /* a = f * 2^e2, f in [0.5, 1): a lies in [2^(e2-1), 2^e2) */
  int e = e2 - 1;
  double m = rint(a / ldexp(1.0, e - 3)); /* 8..16 */
  if (m == 16.0) {
    m = 8.0;
    e += 1;
  }
  /* a < 448 keeps the result at or below 1.75 * 2^8 (code 0x7E) */
  return sign | (uint8_t)(((e + 7) << 3) | ((int)m - 8));
}

/* Store n new KV rows.  Row i (bf16 values x, d of them) belongs to request
 * req[i] at position pos[i]; its slot is block_table[req][pos / P] * P +
 * pos % P (the paged pool of "KV-only decode RadixCache", LMSYS section 2).
 * The row is stored as FP8 E4M3 with one fp32 scale per token (SGLang
 * cookbook, "Keep the KV and DSA backends paired"): amax = max |x|, scale =
 * amax / 448 and byte_j = e4m3(x_j / scale), both divisions in fp32 as the
 * device computes them (the quantised codes are decided in that precision).
 * An all-zero row gets scale 0 and zero bytes.  Rows whose request, position
 * or page is out of range are skipped and flagged (BAD_INDEX for a position
 * outside the block table, BAD_PAGE for a request or page id out of range). */
int oracle_kv_write(const uint16_t* rows, int64_t n, int32_t d, const int32_t* req, const int32_t* pos,
                    const int32_t* block_table, int32_t num_req, int32_t bt_stride, int32_t page_size,
                    int64_t num_pages, uint8_t* kv, float* kv_scale) {
  int status = ORACLE_OK;
  for (int64_t i = 0; i < n; ++i) {
    const int32_t r = req[i], p = pos[i];
    if (r < 0 || r >= num_req) {
      status |= ORACLE_BAD_PAGE;
      continue;
    }
    if (p < 0 || p / page_size >= bt_stride) {
      status |= ORACLE_BAD_INDEX;
      continue;
    }
    const int32_t page = block_table[(int64_t)r * bt_stride + p / page_size];
    if (page < 0 || page >= num_pages) {
      status |= ORACLE_BAD_PAGE;
      continue;
    }
    const int64_t slot = (int64_t)page * page_size + p % page_size;
    const uint16_t* x = rows + i * (int64_t)d;
    float amax = 0.0f;
    for (int32_t j = 0; j < d; ++j) {
      const float v = fabsf((float)oracle_bf16_to_double(x[j]));
      if (v > amax) amax = v;
    }
    const float scale = amax / 448.0f;
    kv_scale[slot] = scale;
    for (int32_t j = 0; j < d; ++j) {
      const float v = (float)oracle_bf16_to_double(x[j]);
      kv[slot * d + j] = scale > 0.0f ? oracle_e4m3_encode(v / scale) : 0;
    }
  }
  return status;
}
