/*
 * Plain CPU oracle for attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, loads or
 * calls this file; only the tests, the package smoke check and the benchmark's
 * CPU-baseline arm do. It shares no code, header, table or helper with the
 * CUDA path.
 *
 * What it computes is the plain definition, written out with no blocking,
 * fusion, splitting or reordering:
 *
 *  1. KV write ("vLLM v1 Deep Dive", Part 3, "Aside - KV cache and prefix
 *     caching", the slot_mapping paragraph; "vLLM: An Exhaustive Technical
 *     Study for Kernel Engineers", section 2.1, "Reaching the kernel"):
 *     every new token t with slot s = slot_mapping[t] >= 0 has its K and V
 *     rows copied, bit for bit, to physical block s / block_size, offset
 *     s % block_size. A negative slot is padding and is skipped.
 *
 *  2. Attention ("vLLM v1 Deep Dive", Part 3, "Step 4c - Mixed batches" and
 *     the block_table paragraph of the same Aside): for each request r the
 *     new tokens are query_start_loc[r] .. query_start_loc[r+1]-1, its total
 *     KV length is seq_lens[r], so ctx = seq_lens[r] - qlen tokens were
 *     cached before this step. The request's logical K/V sequence is gathered
 *     through its block table (logical block p / bs -> physical block id).
 *     Query j (absolute position ctx + j) attends causally to keys
 *     0 .. ctx + j, which covers a decode (qlen 1, all keys) and a prefill
 *     chunk on top of a cached prefix alike. Query head h reads KV head
 *     h / (Hq / Hkv): heads that share a KV head are consecutive
 *     ("vLLM: An Exhaustive Technical Study for Kernel Engineers", 2.4, the
 *     Triton unified attention paragraph on GQA grouping).
 *     Scores s_p = scale * sum_d q[d] k_p[d]; m = max_p s_p;
 *     w_p = exp(s_p - m); o = sum_p w_p v_p / sum_p w_p.
 *     Everything is evaluated in double precision in sequence order.
 *
 *  3. FP8 KV cache ("vLLM: An Exhaustive Technical Study for Kernel Engineers",
 *     2.8, the KV-cache quantization paragraph: --kv-cache-dtype fp8 means
 *     E4M3 with an fp32 per-tensor scale, k_scale for K and v_scale for V).
 *     Writing stores code = E4M3(x / scale), the quotient taken in binary32
 *     (as the GPU takes it) and rounded to the nearest E4M3 value, ties to
 *     even, magnitudes beyond the largest finite value saturating to it.
 *     Reading uses value(code) * scale. E4M3 here is the OCP 8-bit format
 *     the GPU implements: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits,
 *     no infinities, S.1111.111 the only NaN pattern, largest finite 448.
 *     Attention over an FP8 cache is item 2 on the dequantised values.
 *
 * bf16 values are passed as their raw 16-bit patterns; the widening to double
 * is exact (a bf16 is the top half of an IEEE binary32).
 *
 * Build: gcc -O2 -shared -fPIC -pthread pa_oracle.c -o liboracle.so -lm
 * (the package's build step does this; it is a checker, not the product).
 *
 * Mutation hooks: compiling with -DORACLE_MUTANT=n plants a deliberate
 * mistake (used only by the test that shows the oracle's pins catch such
 * mistakes). The default build has none of them.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* error codes (own numbering, independent of the library's) */
#define OR_OK 0
#define OR_BAD_ARG 1
#define OR_BAD_SLOT 2
#define OR_BAD_BLOCK 3
#define OR_BAD_LENGTH 4
#define OR_NO_MEMORY 5

static double widen_bf16(uint16_t bits) {
  /* the bf16 pattern is the upper half of a binary32 */
  uint32_t w = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* ---- E4M3 ---------------------------------------------------------------- */

/* Value of an E4M3 code: (-1)^s * 2^(e-7) * (1 + m/8) for e > 0, and
 * (-1)^s * 2^-6 * (m/8) for e == 0 (subnormals); S.1111.111 is NaN. */
double oracle_e4m3_value(uint8_t c) {
  const int sgn = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
#if ORACLE_MUTANT == 9
  const double mag = e == 0 ? ldexp((double)m, -10) : ldexp((double)(8 + m), e - 11); /* bias 8 */
#else
  const double mag = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
#endif
  return sgn ? -mag : mag;
}

/* Nearest E4M3 code to y (ties to even), saturating at +-448; NaN to NaN. */
uint8_t oracle_e4m3_encode(float y) {
  if (isnan(y)) return signbit(y) ? 0xFF : 0x7F;
  const uint8_t sgn = signbit(y) ? 0x80 : 0x00;
  const double a = fabs((double)y);
  if (a >= 448.0) return sgn | 0x7E;
  /* the spacing of E4M3 values around a: 2^-9 below 2^-6 (subnormals),
   * else 2^(E-3) in the binade [2^E, 2^(E+1)) */
  int e2;
  frexp(a, &e2);
  const int E = e2 - 1;
  const double quantum = E < -6 ? ldexp(1.0, -9) : ldexp(1.0, E - 3);
#if ORACLE_MUTANT == 8
  const double n = floor(a / quantum); /* rounding toward zero */
#else
  const double n = nearbyint(a / quantum); /* round half to even (default mode) */
#endif
  const double q = n * quantum;            /* the chosen E4M3 magnitude */
  if (q == 0.0) return sgn;
  if (q < ldexp(1.0, -6)) return (uint8_t)(sgn | (uint8_t)n); /* subnormal: m = n */
  frexp(q, &e2);
  const int Eq = e2 - 1;
  const int m = (int)(q / ldexp(1.0, Eq - 3)) - 8;
  return (uint8_t)(sgn | (uint8_t)((Eq + 7) << 3) | (uint8_t)m);
}

/* Quantise n bf16 values with one scale: code = E4M3(binary32(x / scale)). */
void oracle_e4m3_quantize(const uint16_t* x, float scale, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) {
    const float xf = (float)widen_bf16(x[i]);
    const float y = xf / scale; /* binary32 division, as on the GPU */
    out[i] = oracle_e4m3_encode(y);
  }
}

int oracle_write_kv(const uint16_t* k, const uint16_t* v, const int64_t* slot_mapping,
                    uint16_t* k_cache, uint16_t* v_cache, int num_tokens, int num_kv_heads,
                    int head_dim, int block_size, int num_blocks) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0)
    return OR_BAD_ARG;
  const int64_t num_slots = (int64_t)num_blocks * block_size;
  /* check every slot first: a bad slot leaves the caches untouched */
  for (int t = 0; t < num_tokens; ++t)
    if (slot_mapping[t] >= num_slots) return OR_BAD_SLOT;
  for (int t = 0; t < num_tokens; ++t) {
    const int64_t s = slot_mapping[t];
    if (s < 0) continue; /* padding token */
    const int64_t blk = s / block_size;
    const int64_t off = s % block_size;
    for (int h = 0; h < num_kv_heads; ++h) {
      /* cache layout: [num_blocks][num_kv_heads][block_size][head_dim] */
      const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * head_dim;
      const int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim;
      for (int d = 0; d < head_dim; ++d) {
        k_cache[dst + d] = k[src + d];
        v_cache[dst + d] = v[src + d];
      }
    }
  }
  return OR_OK;
}

/* KV write into E4M3 caches [num_blocks][num_kv_heads][block_size][head_dim]. */
int oracle_write_kv_fp8(const uint16_t* k, const uint16_t* v, const int64_t* slot_mapping,
                        uint8_t* k_cache, uint8_t* v_cache, float k_scale, float v_scale,
                        int num_tokens, int num_kv_heads, int head_dim, int block_size,
                        int num_blocks) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0 ||
      !(k_scale > 0.0f) || !(v_scale > 0.0f))
    return OR_BAD_ARG;
  const int64_t num_slots = (int64_t)num_blocks * block_size;
  for (int t = 0; t < num_tokens; ++t)
    if (slot_mapping[t] >= num_slots) return OR_BAD_SLOT;
  for (int t = 0; t < num_tokens; ++t) {
    const int64_t s = slot_mapping[t];
    if (s < 0) continue;
    const int64_t blk = s / block_size, off = s % block_size;
    for (int h = 0; h < num_kv_heads; ++h) {
      const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * head_dim;
      const int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim;
      oracle_e4m3_quantize(k + src, k_scale, k_cache + dst, head_dim);
      oracle_e4m3_quantize(v + src, v_scale, v_cache + dst, head_dim);
    }
  }
  return OR_OK;
}

typedef struct {
  const uint16_t* q;
  const void* k_cache;  /* bf16 patterns, or E4M3 codes when kv_fp8 */
  const void* v_cache;
  int kv_fp8;
  double k_scale, v_scale;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* qsl;
  const int32_t* reqs; /* list of requests to evaluate */
  double scale;
  double* out;
  int n_reqs_listed;
  int bt_stride;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  int block_size;
  int num_blocks;
  /* work distribution: item = (listed request index, kv head) */
  int next_item;
  int n_items;
  int status;
  pthread_mutex_t lock;
} oracle_job;

/* One (request, kv head): gather the request's logical K/V rows through the
 * block table, then run every (query token, query head of this group). */
static int run_item(oracle_job* job, int item, double* Kr, double* Vr, double* w) {
  const int r = job->reqs[item / job->num_kv_heads];
  const int kvh = item % job->num_kv_heads;
  const int D = job->head_dim, bs = job->block_size;
  const int Hq = job->num_q_heads, Hkv = job->num_kv_heads;
  const int G = Hq / Hkv;
  const int q0 = job->qsl[r];
  const int qlen = job->qsl[r + 1] - q0;
  const int L = job->seq_lens[r];
  if (qlen < 0 || L < qlen) return OR_BAD_LENGTH;
  const int ctx = L - qlen;

  /* gather: logical position p lives in block table entry p / bs, offset p % bs */
  for (int p = 0; p < L; ++p) {
#if ORACLE_MUTANT == 5
    const int32_t blk = job->block_tables[(int64_t)r * job->bt_stride + (p % bs)];
    const int off = p / bs;
#else
    const int32_t blk = job->block_tables[(int64_t)r * job->bt_stride + p / bs];
    const int off = p % bs;
#endif
    if (blk < 0 || blk >= job->num_blocks) return OR_BAD_BLOCK;
    const int64_t base = (((int64_t)blk * Hkv + kvh) * bs + off) * D;
    for (int d = 0; d < D; ++d) {
      if (job->kv_fp8) {
        Kr[(int64_t)p * D + d] =
            oracle_e4m3_value(((const uint8_t*)job->k_cache)[base + d]) * job->k_scale;
        Vr[(int64_t)p * D + d] =
            oracle_e4m3_value(((const uint8_t*)job->v_cache)[base + d]) * job->v_scale;
      } else {
        Kr[(int64_t)p * D + d] = widen_bf16(((const uint16_t*)job->k_cache)[base + d]);
        Vr[(int64_t)p * D + d] = widen_bf16(((const uint16_t*)job->v_cache)[base + d]);
      }
    }
  }

  for (int j = 0; j < qlen; ++j) {
#if ORACLE_MUTANT == 1
    const int last = ctx + j - 1; /* off-by-one causal limit */
#elif ORACLE_MUTANT == 6
    const int last = L - 1; /* no causal mask inside the chunk */
#else
    const int last = ctx + j; /* keys 0 .. ctx + j are visible */
#endif
    for (int g = 0; g < G; ++g) {
#if ORACLE_MUTANT == 2
      const int h = g * Hkv + kvh; /* wrong GQA head mapping */
#else
      const int h = kvh * G + g; /* consecutive query heads share a KV head */
#endif
      const uint16_t* qrow = job->q + ((int64_t)(q0 + j) * Hq + h) * D;
      double m = -INFINITY;
      for (int p = 0; p <= last; ++p) {
        double s = 0.0;
        for (int d = 0; d < D; ++d) {
#if ORACLE_MUTANT == 3
          s += widen_bf16(qrow[d]) * Kr[(int64_t)p * D + (D - 1 - d)]; /* transposed operand */
#else
          s += widen_bf16(qrow[d]) * Kr[(int64_t)p * D + d];
#endif
        }
#if ORACLE_MUTANT == 4
        w[p] = s; /* scale dropped */
#else
        w[p] = job->scale * s;
#endif
        if (w[p] > m) m = w[p];
      }
      double denom = 0.0;
      for (int p = 0; p <= last; ++p) {
        w[p] = exp(w[p] - m);
        denom += w[p];
      }
      double* orow = job->out + ((int64_t)(q0 + j) * Hq + h) * D;
      for (int d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int p = 0; p <= last; ++p) acc += w[p] * Vr[(int64_t)p * D + d];
#if ORACLE_MUTANT == 7
        orow[d] = acc; /* normaliser dropped */
#else
        orow[d] = acc / denom;
#endif
      }
    }
  }
  return OR_OK;
}

static void* worker(void* arg) {
  oracle_job* job = (oracle_job*)arg;
  /* scratch sized for the longest listed request */
  int maxL = 1;
  for (int i = 0; i < job->n_reqs_listed; ++i) {
    const int L = job->seq_lens[job->reqs[i]];
    if (L > maxL) maxL = L;
  }
  double* Kr = (double*)malloc(sizeof(double) * (size_t)maxL * job->head_dim);
  double* Vr = (double*)malloc(sizeof(double) * (size_t)maxL * job->head_dim);
  double* w = (double*)malloc(sizeof(double) * (size_t)maxL);
  if (!Kr || !Vr || !w) {
    pthread_mutex_lock(&job->lock);
    job->status = OR_NO_MEMORY;
    pthread_mutex_unlock(&job->lock);
    free(Kr); free(Vr); free(w);
    return NULL;
  }
  for (;;) {
    pthread_mutex_lock(&job->lock);
    const int item = job->status == OR_OK ? job->next_item++ : job->n_items;
    pthread_mutex_unlock(&job->lock);
    if (item >= job->n_items) break;
    const int st = run_item(job, item, Kr, Vr, w);
    if (st != OR_OK) {
      pthread_mutex_lock(&job->lock);
      if (job->status == OR_OK) job->status = st;
      pthread_mutex_unlock(&job->lock);
    }
  }
  free(Kr); free(Vr); free(w);
  return NULL;
}

/* out: double [num_tokens][num_q_heads][head_dim]; rows of requests not in the
 * list are left untouched. reqs == NULL evaluates every request. */
static int attention_job(const uint16_t* q, const void* k_cache, const void* v_cache, int kv_fp8,
                         double k_scale, double v_scale, const int32_t* block_tables,
                         int bt_stride, const int32_t* seq_lens, const int32_t* query_start_loc,
                         double scale, double* out, int num_reqs, int num_q_heads,
                         int num_kv_heads, int head_dim, int block_size, int num_blocks,
                         const int32_t* reqs, int n_reqs_listed, int num_threads) {
  if (num_reqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      block_size <= 0 || num_q_heads % num_kv_heads != 0)
    return OR_BAD_ARG;
  int32_t* all = NULL;
  if (reqs == NULL) {
    all = (int32_t*)malloc(sizeof(int32_t) * (size_t)(num_reqs > 0 ? num_reqs : 1));
    if (!all) return OR_NO_MEMORY;
    for (int i = 0; i < num_reqs; ++i) all[i] = i;
    reqs = all;
    n_reqs_listed = num_reqs;
  }
  for (int i = 0; i < n_reqs_listed; ++i)
    if (reqs[i] < 0 || reqs[i] >= num_reqs) { free(all); return OR_BAD_ARG; }

  oracle_job job;
  memset(&job, 0, sizeof job);
  job.q = q; job.k_cache = k_cache; job.v_cache = v_cache;
  job.kv_fp8 = kv_fp8; job.k_scale = k_scale; job.v_scale = v_scale;
  job.block_tables = block_tables; job.seq_lens = seq_lens; job.qsl = query_start_loc;
  job.reqs = reqs; job.n_reqs_listed = n_reqs_listed; job.scale = scale; job.out = out;
  job.bt_stride = bt_stride; job.num_q_heads = num_q_heads; job.num_kv_heads = num_kv_heads;
  job.head_dim = head_dim; job.block_size = block_size; job.num_blocks = num_blocks;
  job.n_items = n_reqs_listed * num_kv_heads;
  job.status = OR_OK;
  pthread_mutex_init(&job.lock, NULL);

  if (num_threads < 1) num_threads = 1;
  if (num_threads > job.n_items) num_threads = job.n_items > 0 ? job.n_items : 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)num_threads);
  int started = 0;
  if (th) {
    for (int i = 1; i < num_threads; ++i)
      if (pthread_create(&th[started], NULL, worker, &job) == 0) ++started;
  }
  worker(&job);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  free(th);
  pthread_mutex_destroy(&job.lock);
  free(all);
  return job.status;
}

int oracle_attention(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                     const int32_t* block_tables, int bt_stride, const int32_t* seq_lens,
                     const int32_t* query_start_loc, double scale, double* out, int num_reqs,
                     int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                     int num_blocks, const int32_t* reqs, int n_reqs_listed, int num_threads) {
  return attention_job(q, k_cache, v_cache, 0, 1.0, 1.0, block_tables, bt_stride, seq_lens,
                       query_start_loc, scale, out, num_reqs, num_q_heads, num_kv_heads, head_dim,
                       block_size, num_blocks, reqs, n_reqs_listed, num_threads);
}

/* Attention over E4M3 caches: keys value(code) * k_scale, values
 * value(code) * v_scale, otherwise as oracle_attention. */
int oracle_attention_fp8(const uint16_t* q, const uint8_t* k_cache, const uint8_t* v_cache,
                         double k_scale, double v_scale, const int32_t* block_tables,
                         int bt_stride, const int32_t* seq_lens, const int32_t* query_start_loc,
                         double scale, double* out, int num_reqs, int num_q_heads,
                         int num_kv_heads, int head_dim, int block_size, int num_blocks,
                         const int32_t* reqs, int n_reqs_listed, int num_threads) {
  if (!(k_scale > 0.0) || !(v_scale > 0.0)) return OR_BAD_ARG;
  return attention_job(q, k_cache, v_cache, 1, k_scale, v_scale, block_tables, bt_stride,
                       seq_lens, query_start_loc, scale, out, num_reqs, num_q_heads, num_kv_heads,
                       head_dim, block_size, num_blocks, reqs, n_reqs_listed, num_threads);
}

int oracle_mutant_id(void) { return ORACLE_MUTANT; }
