/*
 * Plain fp64 CPU oracle for paged Multi-head Latent Attention (MLA) decode.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * definition that the CUDA path is checked against.  It shares no code,
 * header, table or helper with the CUDA library; only the test-suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it.
 *
 * What it computes (one output row per batch element b, query token i,
 * query head h):
 *
 *   1. Key set J.
 *        dense : J = {0 .. L-1}, L = cache_seqlens[b]; with is_causal the
 *                query token i sits at position L - s_q + i (bottom-right
 *                aligned), so J = {0 .. L - s_q + i}.
 *        sparse: J = the multiset {indices[b,i,k] : 0 <= indices[b,i,k] < L},
 *                in k order; ids outside [0, L) (e.g. -1) are skipped and a
 *                repeated id counts once per occurrence, as a gather does.
 *      ("Why FlashMLA's decode kernel reaches 660 TFLOPS", usage section:
 *       sparse semantics written as kv[indices] gather then softmax.)
 *   2. Token fetch through the block table: page = table[b][j / page_size],
 *      slot = j % page_size.  (Modular design-doc overview, section 4
 *      "PagedAttention": divmod(token, page_size) then a lookup-table read.)
 *        bf16 cache : K_j = the 576 stored bf16 values, exactly.
 *        fp8 cache  : 656-byte row = 512 float8_e4m3 codes, 4 float32
 *                     scales (scale k covers dims [128k, 128k+128)), 64 bf16
 *                     RoPE values.  K_j[d] = bf16_rne(fp32_rn(e4m3 * scale))
 *                     for d < 512; the RoPE dims are copied.
 *      ("Why FlashMLA ...", Design 2: FP8 KV cache, 512 + 16 + 128 = 656
 *       bytes per token, dequantised to bf16 before every MMA.)
 *      V_j = K_j[0:512]  (Modular overview, section 9 "Multi-Head Latent
 *      Attention": MQA form with V = K[:, :, :512]).
 *   3. s_j = sm_scale * sum_d q[d] * K_j[d]          (fp64)
 *   4. two-pass softmax: m = max s_j, Z = sum exp(s_j - m),
 *      out = sum exp(s_j - m) V_j / Z, lse = (m + ln Z) / ln 2, i.e. the
 *      base-2 log-sum-exp log2(sum_j e^{s_j}).
 *   5. empty J: out = 0, lse = -inf.
 *
 * Two helpers expose the split-KV view used by the invariant tests:
 * oracle_mla_partial restricts J to a window [k0, k1) of its natural order,
 * and oracle_lse_merge combines partials (Modular overview, section 6:
 * online softmax rescales partial sums by exp(old_max - new_max)).
 *
 * No blocking, fusion or reordering beyond these definitions.  Built with
 * plain gcc (no fast-math), threaded only over independent output rows.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define D_QK 576
#define D_V 512
#define FP8_ROW_BYTES 656
#define FP8_SCALE_OFFSET 512
#define FP8_ROPE_OFFSET 528

static double bf16_bits_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* float -> bf16 bits, round to nearest even (NaN kept quiet). */
static uint16_t float_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x40);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

/* E4M3 ("fn" variant): sign, 4 exponent bits with bias 7, 3 mantissa bits;
 * exponent field 0 encodes subnormals 2^-6 * m/8; S.1111.111 is NaN; there
 * is no infinity, so the largest finite magnitude is 1.75 * 2^8 = 448. */
double oracle_e4m3_to_double(uint8_t code) {
  int sign = code >> 7;
  int e = (code >> 3) & 0xf;
  int m = code & 0x7;
  double v;
  if (e == 0xf && m == 0x7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

/* Dequantise one 656-byte token row into 576 doubles (bf16 values). */
void oracle_dequant_row(const uint8_t* row, double* k) {
  for (int d = 0; d < D_V; ++d) {
    float scale;
    memcpy(&scale, row + FP8_SCALE_OFFSET + 4 * (d / 128), sizeof scale);
    /* e4m3 has a 4-bit significand and the scale 24 bits: the double
     * product is exact, and the cast to float is the single fp32 rounding. */
    float prod = (float)(oracle_e4m3_to_double(row[d]) * (double)scale);
    k[d] = bf16_bits_to_double(float_to_bf16_rne(prod));
  }
  for (int d = D_V; d < D_QK; ++d) {
    uint16_t h;
    memcpy(&h, row + FP8_ROPE_OFFSET + 2 * (d - D_V), sizeof h);
    k[d] = bf16_bits_to_double(h);
  }
}

/* Per-token-scale FP8 row (MAX kernels summary, MLA section: the scaled
 * decode takes explicit per-token KV scales [num_blocks, ..., page_size, ...]
 * and an FP8 + BF16 layout whose row is 640 bytes): bytes [0, 512) the E4M3
 * codes of dims 0..511, bytes [512, 640) dims 512..575 as bf16; one float32
 * scale per token.  K[d] = bf16_rn(fp32_rn(e4m3 * scale)) for d < 512. */
void oracle_dequant_row_token_scale(const uint8_t* row, float scale, double* k) {
  for (int d = 0; d < D_V; ++d) {
    float prod = (float)(oracle_e4m3_to_double(row[d]) * (double)scale);
    k[d] = bf16_bits_to_double(float_to_bf16_rne(prod));
  }
  for (int d = D_V; d < D_QK; ++d) {
    uint16_t h;
    memcpy(&h, row + D_V + 2 * (d - D_V), sizeof h);
    k[d] = bf16_bits_to_double(h);
  }
}

typedef struct {
  const uint16_t* q;        /* bf16 bits [batch, s_q, h_q, 576] */
  const void* kvcache;      /* bf16 [pages, page_size, 576], uint8 [pages, page_size, 656] (is_fp8 1)
                               or uint8 [pages, page_size, 640] with per-token scales (is_fp8 2) */
  int is_fp8;
  const float* kv_scales;   /* is_fp8 2: float32 [pages, page_size] */
  const int32_t* topk_lengths; /* sparse, optional: int32 [batch, s_q], valid index slots per row */
  int num_pages;
  int page_size;
  const int32_t* block_table;
  int block_table_stride;
  const int32_t* cache_seqlens;
  int batch, s_q, h_q;
  const int32_t* indices;   /* int32 [batch, s_q, topk] or NULL */
  int topk;
  double sm_scale;
  int is_causal;
} oracle_problem;

/* Fetch logical token j of element b as 576 doubles. Returns 0 when the
 * block-table entry is not a valid page. */
static int fetch_token(const oracle_problem* p, int b, int j, double* k) {
  int page = p->block_table[(int64_t)b * p->block_table_stride + j / p->page_size];
  int slot = j % p->page_size;
  if (page < 0 || page >= p->num_pages) return 0;
  int64_t token = (int64_t)page * p->page_size + slot;
  if (p->is_fp8 == 2) {
    oracle_dequant_row_token_scale((const uint8_t*)p->kvcache + token * 640, p->kv_scales[token], k);
  } else if (p->is_fp8) {
    oracle_dequant_row((const uint8_t*)p->kvcache + token * FP8_ROW_BYTES, k);
  } else {
    const uint16_t* row = (const uint16_t*)p->kvcache + token * D_QK;
    for (int d = 0; d < D_QK; ++d) k[d] = bf16_bits_to_double(row[d]);
  }
  return 1;
}

/* Build the key set J of output row (b, i) as logical token ids, in the
 * natural order.  Returns |J|. keys must hold max(seqlen, topk) entries. */
static int64_t key_set(const oracle_problem* p, int b, int i, int32_t* keys) {
  int L = p->cache_seqlens[b];
  int64_t n = 0;
  if (p->indices) {
    const int32_t* idx = p->indices + ((int64_t)b * p->s_q + i) * p->topk;
    /* with topk_lengths, only the first topk_lengths[b, i] slots hold ids (the
       MAX kernels summary names sparse_topk_lengths beside sparse_indices) */
    int n_slots = p->topk;
    if (p->topk_lengths) {
      const int32_t len = p->topk_lengths[(int64_t)b * p->s_q + i];
      n_slots = len < 0 ? 0 : (len < p->topk ? len : p->topk);
    }
    for (int k = 0; k < n_slots; ++k)
      if (idx[k] >= 0 && idx[k] < L) keys[n++] = idx[k];
  } else {
    int last = L - 1;
    if (p->is_causal) last = L - p->s_q + i;
    if (last > L - 1) last = L - 1;
    for (int j = 0; j <= last; ++j) keys[n++] = j;
  }
  return n;
}

/* One output row over the window [k0, k1) of its key set (k1 < 0: to the
 * end).  out[512], lse (base 2).  Returns 0 on a bad page id. */
static int one_row(const oracle_problem* p, int64_t row, int64_t k0, int64_t k1, double* out,
                   double* lse, int32_t* keys, double* s, double* kbuf) {
  int h = (int)(row % p->h_q);
  int i = (int)((row / p->h_q) % p->s_q);
  int b = (int)(row / ((int64_t)p->h_q * p->s_q));
  const uint16_t* q = p->q + row * D_QK;
  int64_t n = key_set(p, b, i, keys);
  (void)h;
  if (k1 < 0 || k1 > n) k1 = n;
  if (k0 < 0) k0 = 0;
  for (int d = 0; d < D_V; ++d) out[d] = 0.0;
  if (k0 >= k1) {
    *lse = -INFINITY;
    return 1;
  }
  /* pass 1: logits */
  for (int64_t t = k0; t < k1; ++t) {
    if (!fetch_token(p, b, keys[t], kbuf)) return 0;
    double acc = 0.0;
    for (int d = 0; d < D_QK; ++d) acc += bf16_bits_to_double(q[d]) * kbuf[d];
    s[t - k0] = p->sm_scale * acc;
  }
  double m = -INFINITY;
  for (int64_t t = 0; t < k1 - k0; ++t)
    if (s[t] > m) m = s[t];
  /* pass 2: weights and weighted sum of V */
  double z = 0.0;
  for (int64_t t = k0; t < k1; ++t) {
    double w = exp(s[t - k0] - m);
    z += w;
    fetch_token(p, b, keys[t], kbuf);
    for (int d = 0; d < D_V; ++d) out[d] += w * kbuf[d];
  }
  for (int d = 0; d < D_V; ++d) out[d] /= z;
  *lse = (m + log(z)) / log(2.0);
  return 1;
}

typedef struct {
  const oracle_problem* p;
  const int64_t* rows;
  int64_t n_rows;
  int64_t k0, k1;
  double* out;
  double* lse;
  int64_t next;      /* shared work counter (guarded by mu) */
  int bad;
  pthread_mutex_t mu;
} oracle_job;

static void* worker(void* arg) {
  oracle_job* job = (oracle_job*)arg;
  const oracle_problem* p = job->p;
  int64_t cap = p->topk > 0 ? p->topk : 0;
  for (int b = 0; b < p->batch; ++b)
    if (p->cache_seqlens[b] > cap) cap = p->cache_seqlens[b];
  if (cap < 1) cap = 1;
  int32_t* keys = (int32_t*)malloc(sizeof(int32_t) * cap);
  double* s = (double*)malloc(sizeof(double) * cap);
  double kbuf[D_QK];
  for (;;) {
    pthread_mutex_lock(&job->mu);
    int64_t r = job->next++;
    pthread_mutex_unlock(&job->mu);
    if (r >= job->n_rows) break;
    int64_t row = job->rows ? job->rows[r] : r;
    if (!one_row(p, row, job->k0, job->k1, job->out + r * D_V, job->lse + r, keys, s, kbuf)) {
      pthread_mutex_lock(&job->mu);
      job->bad = 1;
      pthread_mutex_unlock(&job->mu);
    }
  }
  free(keys);
  free(s);
  return NULL;
}

static int run(const oracle_problem* p, const int64_t* rows, int64_t n_rows, int64_t k0, int64_t k1,
               double* out, double* lse, int n_threads) {
  oracle_job job;
  memset(&job, 0, sizeof job);
  job.p = p;
  job.rows = rows;
  job.n_rows = n_rows;
  job.k0 = k0;
  job.k1 = k1;
  job.out = out;
  job.lse = lse;
  pthread_mutex_init(&job.mu, NULL);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  pthread_t tid[256];
  for (int t = 1; t < n_threads; ++t) pthread_create(&tid[t], NULL, worker, &job);
  worker(&job);
  for (int t = 1; t < n_threads; ++t) pthread_join(tid[t], NULL);
  pthread_mutex_destroy(&job.mu);
  return job.bad ? 1 : 0;
}

static void fill_problem(oracle_problem* p, const uint16_t* q, const void* kvcache, int is_fp8,
                         int num_pages, int page_size, const int32_t* block_table,
                         int block_table_stride, const int32_t* cache_seqlens, int batch, int s_q,
                         int h_q, const int32_t* indices, int topk, double sm_scale, int is_causal,
                         const int32_t* topk_lengths, const float* kv_scales) {
  p->topk_lengths = topk_lengths;
  p->kv_scales = kv_scales;
  p->q = q;
  p->kvcache = kvcache;
  p->is_fp8 = is_fp8;
  p->num_pages = num_pages;
  p->page_size = page_size;
  p->block_table = block_table;
  p->block_table_stride = block_table_stride;
  p->cache_seqlens = cache_seqlens;
  p->batch = batch;
  p->s_q = s_q;
  p->h_q = h_q;
  p->indices = indices;
  p->topk = topk;
  p->sm_scale = sm_scale;
  p->is_causal = is_causal;
}

/* Full decode for the listed flat rows ((b*s_q + i)*h_q + h); rows == NULL
 * means every row in order.  out: [n_rows, 512], lse: [n_rows].
 * Returns 0, or 1 if some block-table entry was not a valid page. */
int oracle_mla_decode(const uint16_t* q, const void* kvcache, int is_fp8, int num_pages,
                      int page_size, const int32_t* block_table, int block_table_stride,
                      const int32_t* cache_seqlens, int batch, int s_q, int h_q,
                      const int32_t* indices, int topk, double sm_scale, int is_causal,
                      const int32_t* topk_lengths, const float* kv_scales,
                      const int64_t* rows, int64_t n_rows, double* out, double* lse,
                      int n_threads) {
  oracle_problem p;
  fill_problem(&p, q, kvcache, is_fp8, num_pages, page_size, block_table, block_table_stride,
               cache_seqlens, batch, s_q, h_q, indices, topk, sm_scale, is_causal, topk_lengths, kv_scales);
  return run(&p, rows, n_rows, 0, -1, out, lse, n_threads);
}

/* Same, restricted to positions [k0, k1) of each row's key set. */
int oracle_mla_partial(const uint16_t* q, const void* kvcache, int is_fp8, int num_pages,
                       int page_size, const int32_t* block_table, int block_table_stride,
                       const int32_t* cache_seqlens, int batch, int s_q, int h_q,
                       const int32_t* indices, int topk, double sm_scale, int is_causal,
                       const int32_t* topk_lengths, const float* kv_scales,
                       const int64_t* rows, int64_t n_rows, int64_t k0, int64_t k1, double* out,
                       double* lse, int n_threads) {
  oracle_problem p;
  fill_problem(&p, q, kvcache, is_fp8, num_pages, page_size, block_table, block_table_stride,
               cache_seqlens, batch, s_q, h_q, indices, topk, sm_scale, is_causal, topk_lengths, kv_scales);
  return run(&p, rows, n_rows, k0, k1, out, lse, n_threads);
}

/* Merge n partial results of one row by their base-2 log-sum-exps:
 * L = log2 sum_i 2^{lse_i}, out = sum_i 2^{lse_i - L} out_i.  Partials with
 * lse = -inf contribute nothing; all empty gives out = 0, lse = -inf. */
void oracle_lse_merge(int n, const double* outs, const double* lses, double* out, double* lse) {
  double mx = -INFINITY;
  for (int i = 0; i < n; ++i)
    if (lses[i] > mx) mx = lses[i];
  for (int d = 0; d < D_V; ++d) out[d] = 0.0;
  if (mx == -INFINITY) {
    *lse = -INFINITY;
    return;
  }
  double sum = 0.0;
  for (int i = 0; i < n; ++i) sum += exp2(lses[i] - mx);
  double L = mx + log2(sum);
  for (int i = 0; i < n; ++i) {
    double w = exp2(lses[i] - L);
    for (int d = 0; d < D_V; ++d) out[d] += w * outs[(int64_t)i * D_V + d];
  }
  *lse = L;
}

/* ------------------------------------------------------------------------
 * FP8 cache write ("Why FlashMLA's decode kernel reaches 660 TFLOPS",
 * Design 2: per token, the 512 NoPE dims are quantised to float8_e4m3 in
 * 1 x 128 tiles with one float32 scale per tile, the 64 RoPE dims stay
 * bf16; the MAX kernels summary, KV-cache store section: new tokens of a
 * ragged batch are written at the end of each sequence through the page
 * lookup table).
 *
 * Reading of the quantiser (the pages name only amax / 448 and E4M3):
 *   amax  = max |x| over the tile's 128 values (exact),
 *   scale = amax / 448 in float32 (round to nearest), 1 if amax == 0,
 *   code  = e4m3 of x / scale (float32 division, round to nearest), rounded
 *           to the nearest E4M3 value, ties to the even code, magnitudes
 *           above 448 saturated to 448 ("satfinite"); NaN -> 0x7F.
 * ------------------------------------------------------------------------ */

/* The 127 non-negative finite E4M3 values, by code 0x00 .. 0x7E (ascending). */
static double e4m3_pos_value(int code) { return oracle_e4m3_to_double((uint8_t)code); }

/* float -> E4M3 code: nearest value, ties to the even code, saturating. */
uint8_t oracle_e4m3_from_float(float q) {
  if (isnan(q)) return 0x7F;
  const uint8_t sign = signbit(q) ? 0x80 : 0x00;
  const double a = fabs((double)q);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  /* largest code lo with value(lo) <= a (binary search over the ascending grid) */
  int lo = 0, hi = 0x7E;
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if (e4m3_pos_value(mid) <= a)
      lo = mid;
    else
      hi = mid - 1;
  }
  if (e4m3_pos_value(lo) == a) return (uint8_t)(sign | lo);
  /* a lies strictly between value(lo) and value(lo + 1) */
  const double d_lo = a - e4m3_pos_value(lo), d_hi = e4m3_pos_value(lo + 1) - a;
  int code;
  if (d_lo < d_hi)
    code = lo;
  else if (d_hi < d_lo)
    code = lo + 1;
  else
    code = (lo % 2 == 0) ? lo : lo + 1; /* tie: the even code */
  return (uint8_t)(sign | code);
}

/* One token: 576 bf16 values (bits) -> one 656-byte cache row. */
void oracle_fp8_quantize_row(const uint16_t* x, uint8_t* row) {
  for (int t = 0; t < 4; ++t) {
    float amax = 0.0f;
    for (int d = 128 * t; d < 128 * t + 128; ++d) {
      float v = (float)bf16_bits_to_double(x[d]);
      if (fabsf(v) > amax) amax = fabsf(v);
    }
    const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int d = 128 * t; d < 128 * t + 128; ++d) {
      const float v = (float)bf16_bits_to_double(x[d]);
      row[d] = oracle_e4m3_from_float(v / scale);
    }
    memcpy(row + FP8_SCALE_OFFSET + 4 * t, &scale, sizeof scale);
  }
  memcpy(row + FP8_ROPE_OFFSET, x + D_V, 2 * (D_QK - D_V));
}

/* Ragged store: token i of element b (row input_row_offsets[b] + i of x)
 * goes to logical position cache_lengths[b] + i of element b, i.e. page
 * block_table[b][pos / page_size], slot pos % page_size.  Tokens whose page
 * entry lies outside the table or the pool are skipped.  Returns the number
 * of skipped tokens. */
int64_t oracle_fp8_cache_store(const uint16_t* x, const int32_t* input_row_offsets,
                               const int32_t* cache_lengths, const int32_t* block_table,
                               int block_table_stride, int batch, int num_pages, int page_size,
                               uint8_t* kvcache) {
  int64_t skipped = 0;
  for (int b = 0; b < batch; ++b) {
    for (int32_t r = input_row_offsets[b]; r < input_row_offsets[b + 1]; ++r) {
      const int64_t pos = (int64_t)cache_lengths[b] + (r - input_row_offsets[b]);
      const int64_t blk = pos / page_size;
      const int32_t page = blk < block_table_stride ? block_table[(int64_t)b * block_table_stride + blk] : -1;
      if (page < 0 || page >= num_pages) {
        ++skipped;
        continue;
      }
      uint8_t* dst = kvcache + ((int64_t)page * page_size + pos % page_size) * FP8_ROW_BYTES;
      oracle_fp8_quantize_row(x + (int64_t)r * D_QK, dst);
    }
  }
  return skipped;
}

/* ------------------------------------------------------------------------
 * Sparse prefill ("Why FlashMLA's decode kernel reaches 660 TFLOPS", usage
 * section: flash_mla_sparse_fwd(q, kv, indices, sm_scale)).  No batch and no
 * paging: the single KV head is squeezed out, so kv is [s_kv, 576] bf16 and
 * indices is [s_q, topk].  For query token i and head h, in the order the
 * article states the computation:
 *   1. gather: the focused rows K_k = kv[indices[i, k]], k = 0 .. topk-1;
 *      ids outside [0, s_kv) are skipped and a repeated id counts once per
 *      occurrence (the reading taken for sparse decode),
 *   2. logits P_k = sm_scale * q[i, h] . K_k                    (fp64),
 *   3. lse = log2 sum_k e^{P_k}, the base-2 log-sum-exp of the natural
 *      logits (the article's base-2 exponentials read with the factor
 *      log2(e) folded into the scale, as for decode),
 *   4. S_k = e^{P_k} / sum_k' e^{P_k'}, out = sum_k S_k K_k[0:512] (V is the
 *      first 512 dims of the gathered row, the MQA form of MLA).
 *   No valid id: out = 0, lse = -inf.
 * ------------------------------------------------------------------------ */
typedef struct {
  const uint16_t* q;
  const uint16_t* kv;
  int64_t s_kv;
  const int32_t* indices;
  int topk;
  int h_q;
  double sm_scale;
  const int64_t* rows;
  int64_t n_rows;
  double* out;
  double* lse;
  int64_t next;
  pthread_mutex_t mu;
} prefill_job;

/* Output row `row` = i * h_q + h.  p: topk logits scratch. */
static void prefill_row(const prefill_job* j, int64_t row, double* out, double* lse, double* p) {
  const int64_t i = row / j->h_q;
  const uint16_t* q = j->q + row * D_QK;
  const int32_t* idx = j->indices + i * j->topk;
  /* steps 1-2: logits of the valid gathered rows */
  double m = -INFINITY;
  for (int k = 0; k < j->topk; ++k) {
    p[k] = -INFINITY;
    if (idx[k] < 0 || idx[k] >= j->s_kv) continue;
    const uint16_t* kr = j->kv + (int64_t)idx[k] * D_QK;
    double acc = 0.0;
    for (int d = 0; d < D_QK; ++d) acc += bf16_bits_to_double(q[d]) * bf16_bits_to_double(kr[d]);
    p[k] = j->sm_scale * acc;
    if (p[k] > m) m = p[k];
  }
  for (int d = 0; d < D_V; ++d) out[d] = 0.0;
  if (m == -INFINITY) {
    *lse = -INFINITY;
    return;
  }
  /* step 3: log-sum-exp */
  double z = 0.0;
  for (int k = 0; k < j->topk; ++k)
    if (p[k] != -INFINITY) z += exp(p[k] - m);
  *lse = (m + log(z)) / log(2.0);
  /* step 4: softmax weights times the value dims of the gathered rows */
  for (int k = 0; k < j->topk; ++k) {
    if (p[k] == -INFINITY) continue;
    const double w = exp(p[k] - m) / z;
    const uint16_t* kr = j->kv + (int64_t)idx[k] * D_QK;
    for (int d = 0; d < D_V; ++d) out[d] += w * bf16_bits_to_double(kr[d]);
  }
}

static void* prefill_worker(void* arg) {
  prefill_job* j = (prefill_job*)arg;
  double* p = (double*)malloc(sizeof(double) * (j->topk > 0 ? j->topk : 1));
  for (;;) {
    pthread_mutex_lock(&j->mu);
    int64_t r = j->next++;
    pthread_mutex_unlock(&j->mu);
    if (r >= j->n_rows) break;
    const int64_t row = j->rows ? j->rows[r] : r;
    prefill_row(j, row, j->out + r * D_V, j->lse + r, p);
  }
  free(p);
  return NULL;
}

/* q [s_q, h_q, 576] bf16 bits, kv [s_kv, 576] bf16 bits, indices [s_q, topk].
 * Computes the listed flat rows (i * h_q + h; rows == NULL: all n_rows rows
 * in order) into out [n_rows, 512] and lse [n_rows]. */
void oracle_sparse_prefill(const uint16_t* q, const uint16_t* kv, int64_t s_kv, const int32_t* indices,
                           int topk, int h_q, double sm_scale, const int64_t* rows, int64_t n_rows,
                           double* out, double* lse, int n_threads) {
  prefill_job j;
  memset(&j, 0, sizeof j);
  j.q = q;
  j.kv = kv;
  j.s_kv = s_kv;
  j.indices = indices;
  j.topk = topk;
  j.h_q = h_q;
  j.sm_scale = sm_scale;
  j.rows = rows;
  j.n_rows = n_rows;
  j.out = out;
  j.lse = lse;
  pthread_mutex_init(&j.mu, NULL);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  pthread_t tid[256];
  for (int t = 1; t < n_threads; ++t) pthread_create(&tid[t], NULL, prefill_worker, &j);
  prefill_worker(&j);
  for (int t = 1; t < n_threads; ++t) pthread_join(tid[t], NULL);
  pthread_mutex_destroy(&j.mu);
}

/* ------------------------------------------------------------------------
 * FP8 top-k indexer (MAX kernels summary, MLA indexing kernels:
 * mla_fp8_index_top_k — FP8 scores of FP8 queries against a quantised,
 * paged key cache with their scales, aggregated over the index heads,
 * masked, reduced to the top-k key ids per query token as int32 with -1 in
 * the unused slots).  The pages give no formula; the readings taken:
 *
 *   query token t (ragged: rows row_offsets[b] .. row_offsets[b+1]-1 belong
 *   to element b, n_b of them, the last n_b tokens of its cache of L_b):
 *   position L_b - n_b + j for its j-th row, so it sees keys
 *   s <= L_b - n_b + j (and s < L_b);
 *   index heads h < h_idx, head dim 128; q codes / k codes are E4M3 with one
 *   float32 scale per (token, head) and per cached key;
 *   score(t, s) = sum_h w[t,h] * f(qs[t,h] * ks[s] * sum_d q[t,h,d] k[s,d])
 *   with f = ReLU when `relu` is set, else the identity (fp64 from the
 *   exactly decoded codes);
 *   top-k: the k visible keys of largest score, in descending score order,
 *   ties to the smaller key id; slots beyond the visible keys hold -1.
 * Key s of element b is row block_table[b][s / page_size] * page_size +
 * s % page_size of the key cache (codes [rows][128], scales [rows]).
 * ------------------------------------------------------------------------ */
#define IDX_DIM 128

typedef struct {
  const uint8_t* q_codes;
  const float* q_scales;
  const float* weights;
  int h_idx;
  const int32_t* row_offsets;
  int batch;
  const uint8_t* k_codes;
  const float* k_scales;
  int num_pages, page_size;
  const int32_t* block_table;
  int block_table_stride;
  const int32_t* cache_seqlens;
  int relu;
} index_problem;

/* Element of query row t (row_offsets is non-decreasing). */
static int index_element(const index_problem* p, int64_t t) {
  int b = 0;
  while (b + 1 < p->batch && p->row_offsets[b + 1] <= t) ++b;
  return b;
}

/* Scores of query row t against keys 0 .. width-1 into sc (-inf where not
 * visible).  Returns the number of visible keys, or -1 on a bad page id. */
static int64_t index_row_scores(const index_problem* p, int64_t t, int64_t width, double* sc) {
  const int b = index_element(p, t);
  const int64_t n_b = p->row_offsets[b + 1] - p->row_offsets[b];
  const int64_t j = t - p->row_offsets[b];
  const int64_t L = p->cache_seqlens[b];
  int64_t last = L - n_b + j;
  if (last > L - 1) last = L - 1;
  double dec[256]; /* the E4M3 values by code */
  for (int c = 0; c < 256; ++c) dec[c] = oracle_e4m3_to_double((uint8_t)c);
  int64_t visible = 0;
  for (int64_t s = 0; s < width; ++s) {
    sc[s] = -INFINITY;
    if (s > last) continue;
    const int64_t blk = s / p->page_size;
    const int32_t page = blk < p->block_table_stride ? p->block_table[(int64_t)b * p->block_table_stride + blk] : -1;
    if (page < 0 || page >= p->num_pages) return -1;
    const int64_t row = (int64_t)page * p->page_size + s % p->page_size;
    const uint8_t* kc = p->k_codes + row * IDX_DIM;
    double acc = 0.0;
    for (int h = 0; h < p->h_idx; ++h) {
      const uint8_t* qc = p->q_codes + (t * p->h_idx + h) * IDX_DIM;
      double dot = 0.0;
      for (int d = 0; d < IDX_DIM; ++d) dot += dec[qc[d]] * dec[kc[d]];
      double v = (double)p->q_scales[t * p->h_idx + h] * (double)p->k_scales[row] * dot;
      if (p->relu && v < 0.0) v = 0.0;
      acc += (double)p->weights[t * p->h_idx + h] * v;
    }
    sc[s] = acc;
    ++visible;
  }
  return visible;
}

/* All scores: out [num_tokens, width] (-inf where not visible).  Returns 0,
 * or 1 on a bad page id. */
int oracle_index_scores(const uint8_t* q_codes, const float* q_scales, const float* weights, int h_idx,
                        const int32_t* row_offsets, int batch, const uint8_t* k_codes, const float* k_scales,
                        int num_pages, int page_size, const int32_t* block_table, int block_table_stride,
                        const int32_t* cache_seqlens, int relu, int64_t width, double* out) {
  index_problem p = {q_codes, q_scales, weights, h_idx, row_offsets, batch, k_codes, k_scales, num_pages,
                     page_size, block_table, block_table_stride, cache_seqlens, relu};
  const int64_t n = row_offsets[batch];
  for (int64_t t = 0; t < n; ++t)
    if (index_row_scores(&p, t, width, out + t * width) < 0) return 1;
  return 0;
}

/* Top-k ids per query row: out [num_tokens, topk].  Selection by repeated
 * scans for the best remaining key (largest score, then smallest id).
 * Returns 0, or 1 on a bad page id. */
int oracle_index_topk(const uint8_t* q_codes, const float* q_scales, const float* weights, int h_idx,
                      const int32_t* row_offsets, int batch, const uint8_t* k_codes, const float* k_scales,
                      int num_pages, int page_size, const int32_t* block_table, int block_table_stride,
                      const int32_t* cache_seqlens, int relu, int topk, int32_t* out) {
  index_problem p = {q_codes, q_scales, weights, h_idx, row_offsets, batch, k_codes, k_scales, num_pages,
                     page_size, block_table, block_table_stride, cache_seqlens, relu};
  const int64_t n = row_offsets[batch];
  int64_t width = 1;
  for (int b = 0; b < batch; ++b)
    if (cache_seqlens[b] > width) width = cache_seqlens[b];
  double* sc = (double*)malloc(sizeof(double) * width);
  char* taken = (char*)malloc(width);
  int bad = 0;
  for (int64_t t = 0; t < n && !bad; ++t) {
    const int64_t visible = index_row_scores(&p, t, width, sc);
    if (visible < 0) {
      bad = 1;
      break;
    }
    memset(taken, 0, width);
    for (int k = 0; k < topk; ++k) {
      int64_t best = -1;
      if (k < visible)
        for (int64_t s = 0; s < width; ++s) {
          if (taken[s] || sc[s] == -INFINITY) continue;
          if (best < 0 || sc[s] > sc[best]) best = s; /* strict: the smaller id wins a tie */
        }
      out[t * topk + k] = (int32_t)best;
      if (best >= 0) taken[best] = 1;
    }
  }
  free(sc);
  free(taken);
  return bad;
}
