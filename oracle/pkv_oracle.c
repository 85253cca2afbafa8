/*
 * pkv_oracle.c -- plain, slow, obviously-correct CPU oracle for paged KV append and
 * paged decode attention.  TEST INFRASTRUCTURE ONLY: it exists so that tests, the
 * smoke check and the benchmark's CPU baseline can check the CUDA path against the
 * definitions written out below.  The product path never links, loads or calls it,
 * and it shares no code, header, table or constant with the CUDA library.
 *
 * Sources (the pages the method is taken from):
 *   [P1]  habr.com/ru/articles/1021832, "KV-Cache ... в рамках одного GPU":
 *         S1 "Prefill и Decode" (append of one new K/V per step),
 *         S2 "KV-Cache: цена памяти" (bytes/token formula, FP8 KV),
 *         S3 "Вспомним FlashAttention" (Attention(Q,K,V) = softmax(QK^T/sqrt(d_k))V,
 *            and the statement that tiling + online softmax give exactly this),
 *         S4 "Вспомним PagedAttention" (16-token blocks, block table, worked example),
 *         S5 "Как vLLM объединяет FlashAttention и PagedAttention" (the
 *            flash_attn_with_kvcache shapes: k_cache [num_physical_blocks, block_size,
 *            num_kv_heads, d_head], block_table [batch, max_num_blocks] int32,
 *            cache_seqlens [batch]).
 *   [P3]  actionbridge.io ... chapter 8 "KV cache management" (flat physical pool,
 *         gather through the block table).
 *   OCP 8-bit Floating Point Specification (OFP8), E4M3 encoding (for the FP8 KV
 *   cache that [P1] S2 mentions via --kv-cache-dtype fp8).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - GQA head map: query head hq reads kv head hq / G, G = Hq / Hkv (contiguous groups).
 *   - slot = physical_block * block_size + offset; a negative slot means "skip".
 *   - FP8 is OCP E4M3 ("fn": bias 7, no infinities, max finite 448, NaN = S.1111.111),
 *     quantised as RNE(float(x) / scale) saturating to +-448; one fp32 scale per
 *     (K or V, kv head), stored as scales[0][h] for K and scales[1][h] for V.
 *   - context_lens[b] counts every cached token of sequence b, including the one
 *     appended in this step; len 0 gives an all-zero output.
 *
 * Arithmetic: fp64 throughout (exact widening of bf16 and of decoded e4m3 times its
 * fp32 scale), libm exp(); no blocking, no online softmax, no reordering.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_KV_BF16 0
#define ORC_KV_E4M3 1

/* ---------------------------------------------------------------- element codecs */

/* bf16 -> fp64: a bf16 is the top 16 bits of an IEEE binary32, so widening is exact. */
double orc_bf16_to_f64(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP E4M3: sign s, exponent field E (4 bits, bias 7), mantissa M (3 bits).
 *   E == 0          : subnormal, value = (-1)^s * 2^-6 * M/8
 *   E == 15, M == 7 : NaN (the format has no infinities)
 *   otherwise       : normal,    value = (-1)^s * 2^(E-7) * (1 + M/8)          */
double orc_e4m3_decode(uint8_t code) {
  int s = code >> 7;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* Round an fp32 value to the nearest E4M3 value, ties to the even code, saturating
 * to the largest finite magnitude (448) for anything larger, NaN -> 0x7F.
 * Written as a search over the 127 finite non-negative codes: the magnitudes grow
 * with the code, so the nearest one (and, on a tie, the one with an even code)
 * is the correctly rounded result.  The sign is carried over unchanged (so -0 stays
 * -0 and tiny negative values round to 0x80). */
uint8_t orc_e4m3_encode(float x) {
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  int best = 0;
  double best_err = a; /* distance to code 0 (value 0) */
  for (int c = 1; c <= 0x7E; ++c) {
    double err = fabs(orc_e4m3_decode((uint8_t)c) - a);
    if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      best_err = err;
    }
  }
  return (uint8_t)(sign | best);
}

/* ---------------------------------------------------------------- pool addressing */

/* Byte offset of element [blk][off][h][i] in a pool laid out as
 * [num_blocks][block_size][num_kv_heads][head_dim] ([P1] S5). */
static size_t pool_index(int64_t blk, int off, int h, int i, int block_size, int hkv, int d) {
  return (((size_t)blk * (size_t)block_size + (size_t)off) * (size_t)hkv + (size_t)h) * (size_t)d +
         (size_t)i;
}

/* Value of one pool element as fp64 (bf16 widened, or e4m3 decoded times its scale). */
static double pool_value(const void* pool, size_t idx, int kv_dtype, double scale) {
  if (kv_dtype == ORC_KV_BF16) return orc_bf16_to_f64(((const uint16_t*)pool)[idx]);
  return orc_e4m3_decode(((const uint8_t*)pool)[idx]) * scale;
}

/* ---------------------------------------------------------------- append (plain indexed copy) */

/* For every new token t with slot_mapping[t] >= 0 and every kv head h, element i:
 *   cache[slot / block_size][slot % block_size][h][i] = enc(x[t][h][i])
 * for x = k into k_cache and x = v into v_cache ([P1] S1 "append", S4 worked example).
 * enc is a bit copy for bf16 and orc_e4m3_encode(float(x) / scale) for E4M3.
 * Returns 0, or -1 if a slot lies outside the pool (nothing is written for it). */
int orc_append(void* k_cache, void* v_cache, int64_t num_blocks, int block_size, int hkv, int d,
               int kv_dtype, const uint16_t* k, const uint16_t* v, const int64_t* slot_mapping,
               int64_t num_tokens, const float* scales) {
  int rc = 0;
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    int64_t blk = slot / block_size;
    int off = (int)(slot % block_size);
    if (blk >= num_blocks) {
      rc = -1;
      continue;
    }
    for (int h = 0; h < hkv; ++h) {
      for (int i = 0; i < d; ++i) {
        size_t src = ((size_t)t * (size_t)hkv + (size_t)h) * (size_t)d + (size_t)i;
        size_t dst = pool_index(blk, off, h, i, block_size, hkv, d);
        if (kv_dtype == ORC_KV_BF16) {
          ((uint16_t*)k_cache)[dst] = k[src];
          ((uint16_t*)v_cache)[dst] = v[src];
        } else {
          float kx = (float)orc_bf16_to_f64(k[src]);
          float vx = (float)orc_bf16_to_f64(v[src]);
          float ks = scales[h], vs = scales[hkv + h];
          float kq = kx / ks; /* one correctly rounded binary32 division */
          float vq = vx / vs;
          ((uint8_t*)k_cache)[dst] = orc_e4m3_encode(kq);
          ((uint8_t*)v_cache)[dst] = orc_e4m3_encode(vq);
        }
      }
    }
  }
  return rc;
}

/* ---------------------------------------------------------------- copy-on-write */

/* Block copy for copy-on-write ([P1] S4 "Copy-on-Write для parallel sampling": a block
 * shared by several sequences is copied before one of them writes into it; the original
 * stays untouched).  For each pair (src, dst): block dst of both pools becomes a byte copy of
 * block src.  Pairs naming a block outside the pool are skipped; returns -1 if any was. */
int orc_copy_blocks(void* k_cache, void* v_cache, int64_t num_blocks, int64_t block_bytes,
                    const int64_t* pairs, int64_t num_pairs) {
  int rc = 0;
  for (int64_t p = 0; p < num_pairs; ++p) {
    int64_t src = pairs[2 * p], dst = pairs[2 * p + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      rc = -1;
      continue;
    }
    if (src == dst) continue;
    memcpy((char*)k_cache + dst * block_bytes, (const char*)k_cache + src * block_bytes, (size_t)block_bytes);
    memcpy((char*)v_cache + dst * block_bytes, (const char*)v_cache + src * block_bytes, (size_t)block_bytes);
  }
  return rc;
}

/* ---------------------------------------------------------------- gather */

/* Contiguous fp64 copy of tokens 0..len-1 of one kv head h of one sequence:
 *   out[t][i] = value(pool[block_table[t / block_size]][t % block_size][h][i])
 * ([P1] S4 block table as a page table; [P3] gather through the block table). */
void orc_gather(const void* pool, int kv_dtype, const float* scales_row, int block_size, int hkv,
                int d, const int32_t* block_table_row, int len, int h, double* out) {
  double sc = scales_row ? (double)scales_row[h] : 1.0;
  for (int t = 0; t < len; ++t) {
    int64_t blk = block_table_row[t / block_size];
    int off = t % block_size;
    for (int i = 0; i < d; ++i)
      out[(size_t)t * (size_t)d + (size_t)i] =
          pool_value(pool, pool_index(blk, off, h, i, block_size, hkv, d), kv_dtype, sc);
  }
}

/* ---------------------------------------------------------------- attention (the definition) */

/* out = softmax(scale * q K^T) V for one query vector over n contiguous keys/values
 * ([P1] S3: Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V; the scale is a parameter).
 * Two passes in fp64: scores, their maximum, weights exp(s - max), weighted sum / sum
 * of weights.  n == 0 gives zeros. */
void orc_attention_one(const double* q, const double* K, const double* V, int n, int d,
                       double scale, double* out) {
  for (int i = 0; i < d; ++i) out[i] = 0.0;
  if (n <= 0) return;
  double* s = (double*)malloc((size_t)n * sizeof(double));
  double mx = -INFINITY;
  for (int t = 0; t < n; ++t) {
    double dot = 0.0;
    for (int i = 0; i < d; ++i) dot += q[i] * K[(size_t)t * (size_t)d + (size_t)i];
    s[t] = scale * dot;
    if (s[t] > mx) mx = s[t];
  }
  double den = 0.0;
  for (int t = 0; t < n; ++t) {
    s[t] = exp(s[t] - mx);
    den += s[t];
  }
  for (int t = 0; t < n; ++t)
    for (int i = 0; i < d; ++i) out[i] += s[t] * V[(size_t)t * (size_t)d + (size_t)i];
  for (int i = 0; i < d; ++i) out[i] /= den;
  free(s);
}

/* ---------------------------------------------------------------- paged decode (gather + definition) */

typedef struct {
  const uint16_t* q; /* [batch][hq][d] bf16 */
  const void* k_cache;
  const void* v_cache;
  int kv_dtype;
  const float* scales; /* [2][hkv] or NULL */
  int block_size, hkv, hq, d;
  const int32_t* block_tables; /* [batch][max_blocks] */
  int max_blocks;
  const int32_t* context_lens; /* [batch] */
  double softmax_scale;
  const int32_t* pairs; /* list of (b, hq) to compute, 2 ints each */
  int64_t num_pairs;
  double* out; /* [num_pairs][d] */
  int nthreads;
  int tid;
} decode_job;

static void* decode_worker(void* arg) {
  decode_job* j = (decode_job*)arg;
  int g = j->hq / j->hkv;
  int cap = 0;
  double *K = NULL, *V = NULL;
  double* qd = (double*)malloc((size_t)j->d * sizeof(double));
  for (int64_t p = j->tid; p < j->num_pairs; p += j->nthreads) {
    int b = j->pairs[2 * p], hq = j->pairs[2 * p + 1];
    int h = hq / g;
    int n = j->context_lens[b];
    if (n > cap) {
      free(K);
      free(V);
      cap = n;
      K = (double*)malloc((size_t)cap * (size_t)j->d * sizeof(double));
      V = (double*)malloc((size_t)cap * (size_t)j->d * sizeof(double));
    }
    const int32_t* row = j->block_tables + (size_t)b * (size_t)j->max_blocks;
    orc_gather(j->k_cache, j->kv_dtype, j->scales, j->block_size, j->hkv, j->d, row, n, h, K);
    orc_gather(j->v_cache, j->kv_dtype, j->scales ? j->scales + j->hkv : NULL, j->block_size,
               j->hkv, j->d, row, n, h, V);
    for (int i = 0; i < j->d; ++i)
      qd[i] = orc_bf16_to_f64(j->q[((size_t)b * (size_t)j->hq + (size_t)hq) * (size_t)j->d + (size_t)i]);
    orc_attention_one(qd, K, V, n, j->d, j->softmax_scale, j->out + (size_t)p * (size_t)j->d);
  }
  free(K);
  free(V);
  free(qd);
  return NULL;
}

/* Decode attention for the listed (b, hq) pairs: gather the sequence's K/V for kv head
 * hq / (hq_total / hkv) through its block table, then apply the definition above.
 * out[p][:] receives the fp64 result for pair p.  Work is spread over nthreads POSIX
 * threads (the arithmetic of each pair is the same for any thread count). */
int orc_decode_pairs(const uint16_t* q, const void* k_cache, const void* v_cache, int kv_dtype,
                     const float* scales, int block_size, int hkv, int hq, int d,
                     const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                     double softmax_scale, const int32_t* pairs, int64_t num_pairs, double* out,
                     int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (hkv <= 0 || hq % hkv != 0) return -1;
  pthread_t* th = (pthread_t*)malloc((size_t)nthreads * sizeof(pthread_t));
  decode_job* jobs = (decode_job*)malloc((size_t)nthreads * sizeof(decode_job));
  for (int t = 0; t < nthreads; ++t) {
    decode_job j = {q,          k_cache,       v_cache,      kv_dtype,   scales, block_size,
                    hkv,        hq,            d,            block_tables, max_blocks,
                    context_lens, softmax_scale, pairs,      num_pairs,  out,    nthreads, t};
    jobs[t] = j;
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, decode_worker, &jobs[t]);
  decode_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(th);
  free(jobs);
  return 0;
}

/* ---------------------------------------------------------------- KV size formula */

/* Bytes of KV cache per token: 2 (K and V) x layers x kv heads x head dim x bytes per
 * element ([P1] S2 formula; the same formula on the gotacat.dev page, section
 * "Почему этот кэш так дорого хранить"). */
int64_t orc_kv_bytes_per_token(int64_t layers, int64_t kv_heads, int64_t head_dim,
                               int64_t bytes_per_elem) {
  return 2 * layers * kv_heads * head_dim * bytes_per_elem;
}
