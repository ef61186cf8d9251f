/*
 * Paged verify-attention oracle: plain, slow, fp64, CPU only.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may build, load or call this file. It shares no code,
 * header, table or constant with the CUDA library and must never be reached
 * from the product path.
 *
 * What it computes (the definition, written out; no blocking, no fusion):
 *
 *   For sequence b with context length L and query length q, the q verify
 *   tokens are the last q tokens of the context. Query row (token i, q head h)
 *   of that sequence attends to keys t = 0 .. L - q + i of KV head
 *   g = h / (Hq / Hkv):
 *       K[t] = dec(k_cache[pg][g][t % 16][:]) * (FP8 ? k_scale[pg][g][t % 16] : 1)
 *       V[t] = dec(v_cache[pg][g][t % 16][:]) * (FP8 ? v_scale[pg][g][t % 16] : 1)
 *       pg   = block_table[b][t / 16]
 *       z_t  = softmax_scale * sum_d Q[i, h, d] * K[t, d]
 *       out  = sum_t exp(z_t - max z) V[t] / sum_t exp(z_t - max z)
 *
 * Sources, by page and section:
 *   - rows = query length x GQA group, several q heads per KV head:
 *     "fix(attention): keep MTP-5 decode on FlyDSL pa_decode past the gluon
 *     query-length limit", Motivation.
 *   - lengths + block table + per-token FP8 KV scales (trailing singleton
 *     dimension) handed to the decode kernel: same page, Change and Tests.
 *   - 16-token pages, head-major within a page: "[MiniMax-M3.1] P/D from a
 *     PP4 prefill into a TP4 decode (2/2: DSpark)", description ("page-16
 *     views", "head-major per page").
 *   - causal mask inside the drafts, lengths that count the verify tokens,
 *     contiguous GQA groups: readings where the pages are silent (the
 *     repository's design notes list them).
 *   - E4M3: OCP 8-bit floating point format (E4M3: 1 sign, 4 exponent bits
 *     with bias 7, 3 mantissa bits, subnormals, no infinities, S.1111.111 = NaN).
 *
 * Parity pins: brute force on tiny inputs, the decode special case against a
 * library attention routine, the causal-prefix identity, block-table
 * permutation invariance, FP8 equal to attention on dequantised tensors,
 * closed forms, and the E4M3 decoder against a library conversion; the
 * tests under tests/test_oracle.py hold them.
 *
 * Compile-time ORACLE_MUTANT=k plants one known mistake (for the test that
 * shows the pins catch it); it is 0 in every normal build.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

#define ORACLE_PAGE 16

typedef struct {
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t kv_dtype; /* 0 = bf16 bits, 1 = OCP E4M3 bytes */
  int32_t num_pages;
  int32_t block_table_stride;
  int32_t pad_;
  const uint16_t* q;     /* [T][Hq][D] bf16 bits */
  const void* k_cache;   /* [N_pg][Hkv][16][D] */
  const void* v_cache;   /* [N_pg][Hkv][16][D] */
  const float* k_scale;  /* [N_pg][Hkv][16] or NULL */
  const float* v_scale;  /* [N_pg][Hkv][16] or NULL */
  const int32_t* block_table; /* [B][stride] */
  const int32_t* context_lens; /* [B] */
  const int32_t* query_lens;   /* [B] */
  double softmax_scale;
} oracle_problem;

/* bf16 -> fp64: a bf16 value is the top 16 bits of an IEEE binary32. */
double oracle_decode_bf16(uint16_t bits) {
  uint32_t w = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* OCP E4M3 -> fp64, from the format definition. */
double oracle_decode_e4m3(uint8_t byte) {
  int sign = (byte >> 7) & 1;
  int e = (byte >> 3) & 0xF;
  int m = byte & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, 1 - 7); /* subnormal: 2^(1-bias) * 0.m */
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -mag : mag;
}

static double load_kv(const oracle_problem* p, const void* cache, const float* scale,
                      int32_t page, int g, int slot, int d) {
  size_t idx = (((size_t)page * p->num_kv_heads + g) * ORACLE_PAGE + slot) * p->head_dim + d;
  if (p->kv_dtype == 0) return oracle_decode_bf16(((const uint16_t*)cache)[idx]);
  double s = scale[((size_t)page * p->num_kv_heads + g) * ORACLE_PAGE + slot];
#if ORACLE_MUTANT == 4
  s = 1.0; /* planted: scale dropped */
#endif
  return oracle_decode_e4m3(((const uint8_t*)cache)[idx]) * s;
}

/* One query row (token tau, q head h); out has head_dim entries.
 * Returns 0, or -1 when the row does not exist. */
static int row_attention(const oracle_problem* p, int64_t tau, int h, double* out, double* z) {
  int64_t off = 0;
  int b = -1;
  for (int s = 0; s < p->num_seqs; ++s) {
    if (tau < off + p->query_lens[s]) { b = s; break; }
    off += p->query_lens[s];
  }
  if (b < 0 || h < 0 || h >= p->num_q_heads) return -1;
  const int D = p->head_dim;
  const int G = p->num_q_heads / p->num_kv_heads;
  const int64_t i = tau - off;
  const int64_t L = p->context_lens[b];
  const int64_t q = p->query_lens[b];
  int g = h / G;
#if ORACLE_MUTANT == 2
  g = h % p->num_kv_heads; /* planted: interleaved GQA groups */
#endif
  int64_t last = L - q + i; /* last visible key */
#if ORACLE_MUTANT == 1
  last = L - 1; /* planted: no causal mask inside the drafts */
#endif
  const uint16_t* qrow = p->q + ((size_t)tau * p->num_q_heads + h) * D;
  const float* ks = p->k_scale;
  const float* vs = p->v_scale;
#if ORACLE_MUTANT == 5
  ks = p->v_scale; vs = p->k_scale; /* planted: K and V scales swapped */
#endif

  /* pass 1: logits and their maximum */
  double zmax = -INFINITY;
  for (int64_t t = 0; t <= last; ++t) {
    int32_t pg = p->block_table[(size_t)b * p->block_table_stride + t / ORACLE_PAGE];
    int slot = (int)(t % ORACLE_PAGE);
#if ORACLE_MUTANT == 3
    slot = (int)((t + 1) % ORACLE_PAGE); /* planted: slot off by one */
#endif
    double acc = 0.0;
    for (int d = 0; d < D; ++d)
      acc += oracle_decode_bf16(qrow[d]) * load_kv(p, p->k_cache, ks, pg, g, slot, d);
    z[t] = p->softmax_scale * acc;
    if (z[t] > zmax) zmax = z[t];
  }
  /* pass 2: weights and the weighted mean of V */
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  double wsum = 0.0;
  for (int64_t t = 0; t <= last; ++t) {
    int32_t pg = p->block_table[(size_t)b * p->block_table_stride + t / ORACLE_PAGE];
    int slot = (int)(t % ORACLE_PAGE);
    double w = exp(z[t] - zmax);
#if ORACLE_MUTANT == 6
    w = exp(z[t]); /* planted: weights not normalised by the running max; fine
                      numerically for small logits, so it must be caught by
                      a pin with large logits */
    if (z[t] - zmax < -700) w = 0.0;
#endif
    wsum += w;
    for (int d = 0; d < D; ++d) out[d] += w * load_kv(p, p->v_cache, vs, pg, g, slot, d);
  }
  for (int d = 0; d < D; ++d) out[d] /= wsum;
  return 0;
}

typedef struct {
  const oracle_problem* p;
  const int64_t* rows; /* pairs (tau, h) or NULL for all */
  int64_t n_rows;
  double* out;
  int64_t next;
  pthread_mutex_t lock;
  int status;
  int64_t max_ctx;
} oracle_job;

static void* worker(void* arg) {
  oracle_job* job = (oracle_job*)arg;
  double* z = (double*)malloc(sizeof(double) * (size_t)(job->max_ctx + 1));
  if (!z) {
    pthread_mutex_lock(&job->lock);
    job->status = -5;
    pthread_mutex_unlock(&job->lock);
    return NULL;
  }
  for (;;) {
    pthread_mutex_lock(&job->lock);
    int64_t k = job->next++;
    pthread_mutex_unlock(&job->lock);
    if (k >= job->n_rows) break;
    int64_t tau;
    int h;
    if (job->rows) {
      tau = job->rows[2 * k];
      h = (int)job->rows[2 * k + 1];
    } else {
      tau = k / job->p->num_q_heads;
      h = (int)(k % job->p->num_q_heads);
    }
    if (row_attention(job->p, tau, h, job->out + (size_t)k * job->p->head_dim, z) != 0) {
      pthread_mutex_lock(&job->lock);
      job->status = -1;
      pthread_mutex_unlock(&job->lock);
    }
  }
  free(z);
  return NULL;
}

/* Computes the selected rows (pairs (token, q head) in `rows`, or every row
 * [T][Hq] when rows == NULL; n_rows is then T * Hq) into out[n_rows][D].
 * n_threads <= 0 means one thread. Returns 0, -1 on a bad row or argument,
 * -5 when out of host memory. */
int oracle_verify_attention(const oracle_problem* p, const int64_t* rows, int64_t n_rows,
                            double* out, int n_threads) {
  if (!p || !out || n_rows < 0 || p->num_kv_heads <= 0 || p->num_q_heads % p->num_kv_heads)
    return -1;
  oracle_job job;
  memset(&job, 0, sizeof job);
  job.p = p;
  job.rows = rows;
  job.n_rows = n_rows;
  job.out = out;
  job.max_ctx = 1;
  for (int s = 0; s < p->num_seqs; ++s)
    if (p->context_lens[s] > job.max_ctx) job.max_ctx = p->context_lens[s];
  pthread_mutex_init(&job.lock, NULL);
  if (n_threads <= 1) {
    worker(&job);
  } else {
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
    if (!th) return -5;
    for (int k = 0; k < n_threads; ++k) pthread_create(&th[k], NULL, worker, &job);
    for (int k = 0; k < n_threads; ++k) pthread_join(th[k], NULL);
    free(th);
  }
  pthread_mutex_destroy(&job.lock);
  return job.status;
}

/* ---------------------------------------------------------------------------
 * Paged KV write with per-token FP8 quantisation (the step that fills the
 * cache the verify step reads): the new tokens' K/V rows are stored into
 * their slots (slot = page * 16 + offset, from a slot mapping), and a slot of
 * -1 (a padded or dead row) stores nothing ("every store masked by its row's
 * liveness": DeepSeek-V4.1 page, description of the in-place KV writes).
 * FP8: per (token, head), s = amax / 448 (s = 1 when amax = 0) and
 * code = E4M3(x / s), round to nearest even, saturating at +-448. The
 * division and the scale are single-precision IEEE operations: the codes are
 * integers decided by floating point, and the CUDA kernel takes the same
 * decision in the same precision.
 * ------------------------------------------------------------------------- */

/* fp32 -> OCP E4M3, round to nearest (ties to even), saturating to +-448;
 * NaN -> 0x7F. Written from the format: values are (-1)^s 2^(e-7) (1 + m/8)
 * for e = 1..15 (except S.1111.111), subnormals 2^-6 (m/8). */
uint8_t oracle_encode_e4m3(float x) {
  if (x != x) return 0x7F;
  uint8_t sign = (x < 0.0f || (x == 0.0f && 1.0f / x < 0.0f)) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a >= 448.0) return sign | 0x7E;
  /* scale to units of the smallest subnormal step 2^-9 within the binade */
  int e;
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: value = m * 2^-9, m = 0..7 (8 rounds up to the min normal) */
    double m = a / ldexp(1.0, -9);
    double fl = floor(m);
    double frac = m - fl;
    int mi = (int)fl;
    if (frac > 0.5 || (frac == 0.5 && (mi & 1))) mi += 1;
    if (mi >= 8) return sign | 0x08; /* rounds to 2^-6 */
    return sign | (uint8_t)mi;
  }
  frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) -> a in [2^(e-1), 2^e) */
  int ue = e - 1; /* unbiased exponent: a in [2^ue, 2^(ue+1)) */
  double m = (a / ldexp(1.0, ue) - 1.0) * 8.0; /* mantissa in [0, 8) */
  double fl = floor(m);
  double frac = m - fl;
  int mi = (int)fl;
  if (frac > 0.5 || (frac == 0.5 && (mi & 1))) mi += 1;
  if (mi == 8) { mi = 0; ue += 1; }
  int be = ue + 7;
  if (be > 15 || (be == 15 && mi == 7)) return sign | 0x7E; /* above 448 saturates */
  return sign | (uint8_t)((be << 3) | mi);
}

/* Writes n_tokens new rows. k_new/v_new: [n][Hkv][D] bf16 bits; slot: [n]
 * (-1 = skip); caches/scales as in the attention problem. kv_dtype 0 stores
 * the bf16 bits unchanged. Returns 0, or -1 when a slot is out of range (that
 * token is skipped, the others are written). */
int oracle_kv_write(int32_t n_tokens, int32_t num_kv_heads, int32_t head_dim, int32_t kv_dtype,
                    int32_t num_pages, const uint16_t* k_new, const uint16_t* v_new, const int64_t* slot,
                    void* k_cache, void* v_cache, float* k_scale, float* v_scale) {
  int status = 0;
  for (int32_t t = 0; t < n_tokens; ++t) {
    const int64_t sl = slot[t];
    if (sl < 0) continue;
    if (sl >= (int64_t)num_pages * ORACLE_PAGE) { status = -1; continue; }
    const int64_t page = sl / ORACLE_PAGE, off = sl % ORACLE_PAGE;
    for (int g = 0; g < num_kv_heads; ++g) {
      const size_t src = ((size_t)t * num_kv_heads + g) * head_dim;
      const size_t dst = (((size_t)page * num_kv_heads + g) * ORACLE_PAGE + off) * head_dim;
      const size_t sdst = ((size_t)page * num_kv_heads + g) * ORACLE_PAGE + off;
      for (int which = 0; which < 2; ++which) {
        const uint16_t* x = (which ? v_new : k_new) + src;
        void* cache = which ? v_cache : k_cache;
        if (kv_dtype == 0) {
          memcpy((uint16_t*)cache + dst, x, sizeof(uint16_t) * (size_t)head_dim);
          continue;
        }
        float amax = 0.0f;
        for (int d = 0; d < head_dim; ++d) {
          float v = (float)oracle_decode_bf16(x[d]);
          if (fabsf(v) > amax) amax = fabsf(v);
        }
        volatile float s = amax > 0.0f ? amax / 448.0f : 1.0f;
        for (int d = 0; d < head_dim; ++d) {
          volatile float y = (float)oracle_decode_bf16(x[d]) / s;
          ((uint8_t*)cache)[dst + d] = oracle_encode_e4m3(y);
        }
        (which ? v_scale : k_scale)[sdst] = s;
      }
    }
  }
  return status;
}

/* ---------------------------------------------------------------------------
 * Greedy verify verdict (the step after verify attention: the target model's
 * picks at the q_b verify positions decide how many drafts are accepted; the
 * DeepSeek-V4.1 page keeps "ids + verdict" on the device, in the graph).
 * Position i of sequence b was fed token x_i (x_0 the last committed token,
 * x_1 .. x_{q-1} the drafts). The target's pick t_i is the first index of
 * the maximum of logits[i] (a NaN counts as the maximum). The accepted count
 * a is the largest k <= q - 1 with x_{j+1} == t_j for every j < k; the next
 * token is t_a.
 * ------------------------------------------------------------------------- */
int oracle_greedy_verdict(int32_t num_seqs, const int32_t* query_lens, int32_t vocab,
                          const uint16_t* logits, /* [T][vocab] bf16 bits */
                          const int32_t* input_ids, /* [T] */
                          int32_t* target_ids, /* [T] out */
                          int32_t* accepted, int32_t* next_token /* [B] out */) {
  int64_t row = 0;
  for (int b = 0; b < num_seqs; ++b) {
    const int q = query_lens[b];
    if (q < 1) return -1;
    for (int i = 0; i < q; ++i) {
      const uint16_t* lr = logits + (size_t)(row + i) * vocab;
      int best = 0;
      double bv = oracle_decode_bf16(lr[0]);
      for (int v = 1; v < vocab; ++v) {
        if (bv != bv) break; /* a NaN is already the maximum */
        double x = oracle_decode_bf16(lr[v]);
        if (x != x || x > bv) { bv = x; best = v; }
      }
      target_ids[row + i] = best;
    }
    int a = 0;
    while (a < q - 1 && input_ids[row + a + 1] == target_ids[row + a]) ++a;
    accepted[b] = a;
    next_token[b] = target_ids[row + a];
    row += q;
  }
  return 0;
}
