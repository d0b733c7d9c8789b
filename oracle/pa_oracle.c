/*
 * pa_oracle.c -- float64 CPU oracle for paged grouped-query decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library calls, links or includes
 * this file; only the tests, __graft_entry__.smoke() and the CPU-baseline leg
 * of bench.py use it.  It shares no code, header, table or constant with the
 * CUDA path.
 *
 * What it computes (a plain definition, no blocking or fusion):
 *
 *   For every sequence b and query head h, with kv head j = floor(h / G),
 *   G = H / Hkv:
 *     K_b[t] = k_cache[block_table[b][t / bs], t % bs, j, :]   t < len_b
 *     V_b[t] = v_cache[block_table[b][t / bs], t % bs, j, :]
 *     s_t    = scale * sum_k q[b,h,k] * K_b[t,k]
 *     M      = max_t s_t
 *     w_t    = exp(s_t - M),  L = sum_t w_t
 *     out    = sum_t w_t V_b[t] / L          (len_b == 0  ->  out = 0)
 *
 * Sources, by page and section:
 *   - "Paged Attention Kernel Architecture for BI-V100", section 1 (Problem
 *     Definition): output = softmax(Q K^T / sqrt(d)) V over paged K/V.
 *   - "Paged attention" (Hugging Face Transformers docs), decoding path:
 *     block_table of shape (batch, max_blocks_per_seq) holds physical block
 *     ids, -1 marks an unallocated block, cache_seqlens is the key length.
 *   - "Detailed Design Document -- AHBM GQA Fused Attention", section 5.3
 *     (head_of_group = id // C) and section 4.3 (contiguous [G, ...] group):
 *     query head h reads kv head floor(h / G).
 *   - The two-pass softmax (max, then exp-sum) is the textbook definition;
 *     "v10_triton_paged_gqa", Core Principle, states that the online
 *     recurrence reaches this same context vector.
 *
 * Split-KV pieces (pa_oracle_partial / pa_oracle_combine) follow the compound
 * (max_score, exp_sum, weighted_v) state and its binary combine op of
 * "Paged Attention Kernel Architecture for BI-V100", section 2, Level 1 and
 * Level 3.
 *
 * Several query tokens per sequence (pa_oracle_decode_multi) follow the
 * varlen indexing of the Hugging Face page (cumulative query lengths) with
 * the query tokens taken as the last positions of the key sequence.
 *
 * Cache append (pa_oracle_append) follows the decoding-path example of the
 * Hugging Face page: the new token of a sequence with len cached tokens goes
 * to row len % bs of physical block block_table[b][len / bs].
 *
 * Inputs are raw 16-bit storage (IEEE binary16 or bfloat16 bit patterns);
 * every stored value is widened to double exactly before any arithmetic.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F16 0
#define ORACLE_BF16 1

#define ORACLE_OK 0
#define ORACLE_ERR_SHAPE (-1)
#define ORACLE_ERR_SEQLEN (-2)
#define ORACLE_ERR_BLOCK (-3)
#define ORACLE_ERR_NOMEM (-4)
#define ORACLE_ERR_RANGE (-5)

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  Exact widening to double. */
static double half_bits_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int expo = (h >> 10) & 0x1f;
  int frac = h & 0x3ff;
  double v;
  if (expo == 0) {
    v = ldexp((double)frac, -24); /* subnormal: frac * 2^-14 * 2^-10 */
  } else if (expo == 31) {
    v = frac ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + frac), expo - 25); /* (1.frac) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32 pattern. */
static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double widen(uint16_t bits, int dtype) {
  return dtype == ORACLE_BF16 ? bf16_bits_to_double(bits) : half_bits_to_double(bits);
}

/* Decode a double back to the 16-bit storage of its type is never needed:
 * the oracle only reads stored values and writes float64 results. */

typedef struct {
  int B, H, Hkv, d, bs, maxblk, P, dtype;
} shape_t;

static int check_shape(const shape_t* s) {
  if (s->B < 0 || s->H <= 0 || s->Hkv <= 0 || s->d <= 0 || s->bs <= 0 ||
      s->maxblk < 0 || s->P < 0)
    return ORACLE_ERR_SHAPE;
  if (s->H % s->Hkv != 0) return ORACLE_ERR_SHAPE;
  if (s->dtype != ORACLE_F16 && s->dtype != ORACLE_BF16) return ORACLE_ERR_SHAPE;
  return ORACLE_OK;
}

/* Address of the stored row (token t of sequence b, kv head j) in a
 * [P, bs, Hkv, d] pool, or NULL when the table does not map it. */
static const uint16_t* pool_row(const shape_t* s, const uint16_t* pool,
                                const int32_t* block_table, int b, int t, int j) {
  int logical = t / s->bs;
  int within = t % s->bs;
  int32_t phys = block_table[(int64_t)b * s->maxblk + logical];
  if (phys < 0 || phys >= s->P) return NULL;
  int64_t row = ((int64_t)phys * s->bs + within) * s->Hkv + j;
  return pool + row * s->d;
}

/* Validate sequence b: its length and every table entry it must read. */
static int check_sequence(const shape_t* s, const int32_t* block_table,
                          const int32_t* seqlens, int b) {
  int32_t len = seqlens[b];
  if (len < 0 || (int64_t)len > (int64_t)s->maxblk * s->bs) return ORACLE_ERR_SEQLEN;
  int nblk = (len + s->bs - 1) / s->bs;
  for (int i = 0; i < nblk; ++i) {
    int32_t phys = block_table[(int64_t)b * s->maxblk + i];
    if (phys < 0 || phys >= s->P) return ORACLE_ERR_BLOCK;
  }
  return ORACLE_OK;
}

/* One (b, h) output row by the plain definition, over tokens [t0, t1).
 * Writes the softmax-normalised result into out[d].  scratch holds t1-t0
 * doubles. */
static void attend_one(const shape_t* s, const uint16_t* qrow, const uint16_t* k_cache,
                       const uint16_t* v_cache, const int32_t* block_table, int b, int h,
                       int t0, int t1, double scale, double* scores, double* out) {
  int G = s->H / s->Hkv;
  int j = h / G;
  int n = t1 - t0;
  for (int k = 0; k < s->d; ++k) out[k] = 0.0;
  if (n <= 0) return;
  /* scores s_t = scale * q . K_b[t] */
  for (int t = t0; t < t1; ++t) {
    const uint16_t* krow = pool_row(s, k_cache, block_table, b, t, j);
    double acc = 0.0;
    for (int k = 0; k < s->d; ++k) acc += widen(qrow[k], s->dtype) * widen(krow[k], s->dtype);
    scores[t - t0] = scale * acc;
  }
  /* two-pass softmax */
  double M = -INFINITY;
  for (int i = 0; i < n; ++i)
    if (scores[i] > M) M = scores[i];
  double L = 0.0;
  for (int i = 0; i < n; ++i) {
    scores[i] = exp(scores[i] - M);
    L += scores[i];
  }
  for (int t = t0; t < t1; ++t) {
    const uint16_t* vrow = pool_row(s, v_cache, block_table, b, t, j);
    double w = scores[t - t0];
    for (int k = 0; k < s->d; ++k) out[k] += w * widen(vrow[k], s->dtype);
  }
  for (int k = 0; k < s->d; ++k) out[k] /= L;
}

/*
 * pa_oracle_decode: out[pair, :] for the requested (b, h) pairs.
 *   pairs == NULL or n_pairs < 0  ->  all B*H pairs in (b, h) row-major order,
 *                                      out is [B, H, d].
 *   otherwise pairs holds n_pairs (b, h) int32 pairs; out is [n_pairs, d].
 * Returns ORACLE_OK, or a negative code if a requested sequence has a length
 * outside [0, maxblk*bs] or an unmapped/out-of-range table entry inside its
 * length (the oracle refuses such inputs instead of guessing).
 */
int pa_oracle_decode(int B, int H, int Hkv, int d, int bs, int maxblk, int P, int dtype,
                     const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                     const int32_t* block_table, const int32_t* cache_seqlens, double scale,
                     int n_pairs, const int32_t* pairs, double* out, int n_threads) {
  shape_t s = {B, H, Hkv, d, bs, maxblk, P, dtype};
  int rc = check_shape(&s);
  if (rc) return rc;
  int64_t count = (pairs == NULL || n_pairs < 0) ? (int64_t)B * H : n_pairs;
  /* validate every sequence that is touched before computing anything */
  for (int64_t i = 0; i < count; ++i) {
    int b = pairs ? pairs[2 * i] : (int)(i / H);
    int h = pairs ? pairs[2 * i + 1] : (int)(i % H);
    if (b < 0 || b >= B || h < 0 || h >= H) return ORACLE_ERR_RANGE;
    rc = check_sequence(&s, block_table, cache_seqlens, b);
    if (rc) return rc;
  }
  int maxlen = 0;
  for (int b = 0; b < B; ++b)
    if (cache_seqlens[b] > maxlen) maxlen = cache_seqlens[b];
  int failed = 0;
#ifdef _OPENMP
  if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads)
#endif
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
    if (!scores) {
      failed = 1;
    } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
      for (int64_t i = 0; i < count; ++i) {
        int b = pairs ? pairs[2 * i] : (int)(i / H);
        int h = pairs ? pairs[2 * i + 1] : (int)(i % H);
        attend_one(&s, q + ((int64_t)b * H + h) * d, k_cache, v_cache, block_table, b, h, 0,
                   cache_seqlens[b], scale, scores, out + i * d);
      }
      free(scores);
    }
  }
  (void)n_threads;
  return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/*
 * pa_oracle_decode_multi: several query tokens per sequence over the paged
 * cache (chunked decode).
 *
 * Query rows are packed as in the varlen path of the Hugging Face "Paged
 * attention" page: sequence b owns rows cu_q[b] .. cu_q[b+1]-1 of
 * q [total_q, H, d] (cumulative query lengths, cu_seq_lens_q), so row r
 * belongs to the b with cu_q[b] <= r < cu_q[b+1].  Its keys are the
 * k_len = cache_seqlens[b] tokens of the paged cache (block_table as in
 * pa_oracle_decode), the new tokens already included.  The n_q query tokens
 * are the last n_q positions of the key sequence, so query i (0-based within
 * its sequence) sees
 *   causal != 0:  keys t < clamp(k_len - n_q + i + 1, 0, k_len)
 *   causal == 0:  keys t < k_len
 * and its output is the plain softmax-weighted sum of those V rows; a query
 * that sees no key gets 0 (as an empty sequence does), and so does a row
 * that belongs to no sequence.  out is [total_q, H, d], or [n_pairs, d] for
 * the (row, h) pairs given.
 * Returns ORACLE_ERR_RANGE when cu_q is not non-decreasing within
 * [0, total_q] or a pair is out of range, and the pa_oracle_decode codes for
 * a bad length or table entry of a sequence that owns a requested row.
 */
int pa_oracle_decode_multi(int B, int H, int Hkv, int d, int bs, int maxblk, int P, int dtype,
                           const uint16_t* q, int total_q, const int32_t* cu_q, int causal,
                           const uint16_t* k_cache, const uint16_t* v_cache,
                           const int32_t* block_table, const int32_t* cache_seqlens,
                           double scale, int n_pairs, const int32_t* pairs, double* out,
                           int n_threads) {
  shape_t s = {B, H, Hkv, d, bs, maxblk, P, dtype};
  int rc = check_shape(&s);
  if (rc) return rc;
  if (total_q < 0) return ORACLE_ERR_SHAPE;
  if (B > 0 && (cu_q[0] < 0 || cu_q[B] > total_q)) return ORACLE_ERR_RANGE;
  for (int b = 0; b < B; ++b)
    if (cu_q[b + 1] < cu_q[b]) return ORACLE_ERR_RANGE;
  int64_t count = (pairs == NULL || n_pairs < 0) ? (int64_t)total_q * H : n_pairs;
  int32_t* owner = (int32_t*)malloc(sizeof(int32_t) * (size_t)(count > 0 ? count : 1));
  if (!owner) return ORACLE_ERR_NOMEM;
  /* the sequence of every requested row (-1: none); validate those sequences */
  for (int64_t i = 0; i < count; ++i) {
    int r = pairs ? pairs[2 * i] : (int)(i / H);
    int h = pairs ? pairs[2 * i + 1] : (int)(i % H);
    if (r < 0 || r >= total_q || h < 0 || h >= H) {
      free(owner);
      return ORACLE_ERR_RANGE;
    }
    owner[i] = -1;
    for (int b = 0; b < B; ++b)
      if (cu_q[b] <= r && r < cu_q[b + 1]) owner[i] = b;
    if (owner[i] >= 0) {
      rc = check_sequence(&s, block_table, cache_seqlens, owner[i]);
      if (rc) {
        free(owner);
        return rc;
      }
    }
  }
  int maxlen = 0;
  for (int b = 0; b < B; ++b)
    if (cache_seqlens[b] > maxlen) maxlen = cache_seqlens[b];
  int failed = 0;
#ifdef _OPENMP
  if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads)
#endif
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
    if (!scores) {
      failed = 1;
    } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
      for (int64_t i = 0; i < count; ++i) {
        int r = pairs ? pairs[2 * i] : (int)(i / H);
        int h = pairs ? pairs[2 * i + 1] : (int)(i % H);
        int b = owner[i];
        int visible = 0;
        if (b >= 0) {
          int k_len = cache_seqlens[b];
          int n_q = cu_q[b + 1] - cu_q[b];
          int qi = r - cu_q[b];
          visible = k_len;
          if (causal) {
            int64_t lim = (int64_t)k_len - n_q + qi + 1;
            visible = lim < 0 ? 0 : (lim > k_len ? k_len : (int)lim);
          }
        }
        attend_one(&s, q + ((int64_t)r * H + h) * d, k_cache, v_cache, block_table,
                   b < 0 ? 0 : b, h, 0, visible, scale, scores, out + i * d);
      }
      free(scores);
    }
  }
  (void)n_threads;
  free(owner);
  return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/*
 * pa_oracle_partial: the compound state of one split-KV piece, tokens
 * [t0, t1) of (b, h):
 *   max_score  m = max_t s_t                       (-inf for an empty piece)
 *   exp_sum    l = sum_t exp(s_t - m)               (0 for an empty piece)
 *   weighted_v a = sum_t exp(s_t - m) V_b[t]        (0 for an empty piece)
 * ("Paged Attention Kernel Architecture for BI-V100", section 2, Level 1,
 * compound type.)
 */
int pa_oracle_partial(int B, int H, int Hkv, int d, int bs, int maxblk, int P, int dtype,
                      const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                      const int32_t* block_table, const int32_t* cache_seqlens, double scale,
                      int b, int h, int t0, int t1, double* m_out, double* l_out,
                      double* acc_out) {
  shape_t s = {B, H, Hkv, d, bs, maxblk, P, dtype};
  int rc = check_shape(&s);
  if (rc) return rc;
  if (b < 0 || b >= B || h < 0 || h >= H) return ORACLE_ERR_RANGE;
  rc = check_sequence(&s, block_table, cache_seqlens, b);
  if (rc) return rc;
  if (t0 < 0 || t1 > cache_seqlens[b] || t0 > t1) return ORACLE_ERR_RANGE;
  int n = t1 - t0;
  for (int k = 0; k < d; ++k) acc_out[k] = 0.0;
  if (n == 0) {
    *m_out = -INFINITY;
    *l_out = 0.0;
    return ORACLE_OK;
  }
  int G = H / Hkv;
  int j = h / G;
  const uint16_t* qrow = q + ((int64_t)b * H + h) * d;
  double* scores = (double*)malloc(sizeof(double) * (size_t)n);
  if (!scores) return ORACLE_ERR_NOMEM;
  double m = -INFINITY;
  for (int t = t0; t < t1; ++t) {
    const uint16_t* krow = pool_row(&s, k_cache, block_table, b, t, j);
    double acc = 0.0;
    for (int k = 0; k < d; ++k) acc += widen(qrow[k], dtype) * widen(krow[k], dtype);
    scores[t - t0] = scale * acc;
    if (scores[t - t0] > m) m = scores[t - t0];
  }
  double l = 0.0;
  for (int t = t0; t < t1; ++t) {
    double w = exp(scores[t - t0] - m);
    const uint16_t* vrow = pool_row(&s, v_cache, block_table, b, t, j);
    l += w;
    for (int k = 0; k < d; ++k) acc_out[k] += w * widen(vrow[k], dtype);
  }
  free(scores);
  *m_out = m;
  *l_out = l;
  return ORACLE_OK;
}

/*
 * pa_oracle_combine: fold n compound states left to right with the binary
 * combine op ("Paged Attention Kernel Architecture for BI-V100", section 2,
 * Level 1 binary op; Level 3 cross-partition reduce):
 *   new_max = max(ma, mb)
 *   exp_sum = e^(ma-new_max) la + e^(mb-new_max) lb
 *   weighted_v = e^(ma-new_max) aa + e^(mb-new_max) ab
 * An empty state (m = -inf, l = 0) is the identity.  Writes the folded state.
 */
void pa_oracle_combine(int n, int d, const double* m, const double* l, const double* acc,
                       double* m_out, double* l_out, double* acc_out) {
  double cm = -INFINITY, cl = 0.0;
  for (int k = 0; k < d; ++k) acc_out[k] = 0.0;
  for (int i = 0; i < n; ++i) {
    double mi = m[i];
    if (mi == -INFINITY) continue; /* identity element */
    double nm = cm > mi ? cm : mi;
    double sa = (cm == -INFINITY) ? 0.0 : exp(cm - nm);
    double sb = exp(mi - nm);
    cl = sa * cl + sb * l[i];
    for (int k = 0; k < d; ++k) acc_out[k] = sa * acc_out[k] + sb * acc[(int64_t)i * d + k];
    cm = nm;
  }
  *m_out = cm;
  *l_out = cl;
}

/*
 * pa_oracle_append: write k_new[b, j, :] and v_new[b, j, :] into the slot of
 * the token at position len_b = cache_seqlens[b]: row len_b % bs of physical
 * block block_table[b][len_b / bs], kv head j.  The 16-bit patterns are
 * copied unchanged.  slot_out (nullable) receives (phys, row) per sequence.
 * Returns ORACLE_ERR_SEQLEN if a position has no table column, and
 * ORACLE_ERR_BLOCK if its table entry is unmapped; nothing is written for
 * such a sequence (all other sequences are still written).
 */
int pa_oracle_append(int B, int Hkv, int d, int bs, int maxblk, int P, const uint16_t* k_new,
                     const uint16_t* v_new, uint16_t* k_cache, uint16_t* v_cache,
                     const int32_t* block_table, const int32_t* cache_seqlens,
                     int32_t* slot_out) {
  int rc = ORACLE_OK;
  for (int b = 0; b < B; ++b) {
    int32_t pos = cache_seqlens[b];
    if (slot_out) {
      slot_out[2 * b] = -1;
      slot_out[2 * b + 1] = -1;
    }
    if (pos < 0 || (int64_t)pos >= (int64_t)maxblk * bs) {
      rc = ORACLE_ERR_SEQLEN;
      continue;
    }
    int32_t phys = block_table[(int64_t)b * maxblk + pos / bs];
    int row = pos % bs;
    if (phys < 0 || phys >= P) {
      rc = ORACLE_ERR_BLOCK;
      continue;
    }
    if (slot_out) {
      slot_out[2 * b] = phys;
      slot_out[2 * b + 1] = row;
    }
    for (int j = 0; j < Hkv; ++j) {
      int64_t dst = (((int64_t)phys * bs + row) * Hkv + j) * d;
      int64_t src = ((int64_t)b * Hkv + j) * d;
      memcpy(k_cache + dst, k_new + src, sizeof(uint16_t) * (size_t)d);
      memcpy(v_cache + dst, v_new + src, sizeof(uint16_t) * (size_t)d);
    }
  }
  return rc;
}

/* Exposed so the tests can pin the 16-bit decoders against known patterns. */
double pa_oracle_widen(uint16_t bits, int dtype) { return widen(bits, dtype); }

int pa_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
