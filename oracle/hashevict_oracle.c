/*
 * hashevict_oracle.c — CPU oracle of the HashEvict decode step.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load or call this file.  It is plain, slow and written to
 * be checked by eye against the method's description; it shares no code with
 * the CUDA library.
 *
 * Source: "HashEvict: A Pre-Attention KV Cache Eviction Strategy using
 * Locality-Sensitive Hashing" (arXiv 2412.16187), abstract and the method
 * section's technical framework, steps 1-5:
 *   1. Gaussian projection of the token's key (and of the query) to b dims,
 *   2. binarisation of the projection,
 *   3. Hamming distance between the query's code and each cached key's code,
 *   4. eviction of the cached token most dissimilar to the current query,
 *   5. the current token's key and value replace the evicted token's.
 * Decode attention over the retained cache follows (TTKV page, introduction:
 * every decode step attends the whole cache).
 *
 * Readings taken where the pages are silent:
 *   - projection W[d][j] ~ N(0,1) (Irwin-Hall(12) counter-based draw, below),
 *     shared by the query and the keys; no normalisation;
 *   - the projection sum is fp32, fused multiply-add, d = 0..D-1 in order,
 *     starting from +0; bit j = (sum > 0): exactly +-0 gives 0;
 *   - bit j of the code is bit j of a 64-bit word (LSB first);
 *   - GQA: a KV head's slots are scored by the sum of the Hamming distances to
 *     the codes of the G query heads of its group;
 *   - "most dissimilar" = largest summed distance; ties go to the lowest slot;
 *   - scoring uses only the current step's distances (no accumulation);
 *     the extended stream below also takes the binarisation threshold tau
 *     (bit j = sum > tau; the method's design choices name the threshold; or
 *     one threshold per bit, e.g. the per-bit medians of the filled keys'
 *     projections, orc_median_thresholds) and a
 *     score memory gamma in [0, 1]: every resident slot s keeps a score
 *     A(s) = fmaf(gamma, A(s), d(s)) in fp32 at each scoring step, the largest
 *     A is evicted (ties: lowest slot) and a written slot starts at A = 0;
 *     gamma = 0 gives A = d, the method as described;
 *   - score the resident slots, then overwrite, then attend: the new token is
 *     always resident and attended;
 *   - while the cache holds fewer than `budget` tokens the new token is appended;
 *   - attention: softmax(q.K / sqrt(D)) V in fp64 from the stored values,
 *     no mask, no positional term.
 *
 * Element types: dtype 0 = bf16 (uint16 bit patterns), dtype 1 = fp32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0 /* >0 plants a known mistake (used only by the pin tests) */
#endif

/* ------------------------------------------------------------------------- */
/* Element access                                                             */
/* ------------------------------------------------------------------------- */

static float bf16_value(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static float elem(const void* base, int dtype, size_t i) {
  if (dtype == 1) return ((const float*)base)[i];
  return bf16_value(((const uint16_t*)base)[i]);
}

static size_t elem_bytes(int dtype) { return dtype == 1 ? 4u : 2u; }

/* ------------------------------------------------------------------------- */
/* The projection matrix: a counter-based Gaussian draw from a seed.          */
/* Generator: SplitMix64 finaliser (Steele, Lea, Flood, OOPSLA 2014) over the */
/* counter, Irwin-Hall sum of 12 uniform 16-bit integers for N(0,1).          */
/* W[d][j] (row-major, D rows of b columns), element e = d*b + j:             */
/*   st  = mix(seed ^ 0x48455F50524F4A57)                                     */
/*   u_r = mix(st + 3e + r), r = 0,1,2;  z = (sum of the 12 16-bit lanes      */
/*         - 393210) / 65536;  W = bf16_rne(z) (dtype 0) or z (dtype 1).      */
/* ------------------------------------------------------------------------- */

static uint64_t mix(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static uint16_t round_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  uint32_t lsb = (u >> 16) & 1u;
  u = u + 0x7FFFu + lsb; /* round half to even */
  return (uint16_t)(u >> 16);
}

void orc_projection(uint64_t seed, int32_t D, int32_t bits, int32_t dtype, void* W) {
  uint64_t st = mix(seed ^ 0x48455F50524F4A57ull);
  for (int32_t d = 0; d < D; ++d) {
    for (int32_t j = 0; j < bits; ++j) {
      uint64_t e = (uint64_t)d * (uint64_t)bits + (uint64_t)j;
      int64_t sum = 0;
      for (int r = 0; r < 3; ++r) {
        uint64_t u = mix(st + 3u * e + (uint64_t)r);
        for (int lane = 0; lane < 4; ++lane) sum += (int64_t)((u >> (16 * lane)) & 0xFFFFu);
      }
      float z = (float)(sum - 393210) / 65536.0f;
      if (dtype == 1)
        ((float*)W)[e] = z;
      else
        ((uint16_t*)W)[e] = round_to_bf16(z);
    }
  }
}

/* ------------------------------------------------------------------------- */
/* Steps 1-2: Gaussian projection and binarisation of one vector.             */
/* ------------------------------------------------------------------------- */

/* Bit j of the code: the projection onto column j of W against the threshold
 * of bit j, tauv[j] (one threshold per bit), or tau for every bit when tauv is
 * NULL. */
uint64_t orc_code_thr(const void* x, int32_t dtype, int32_t D, const void* W, int32_t bits,
                      float tau, const float* tauv) {
  uint64_t code = 0;
  for (int32_t j = 0; j < bits; ++j) {
    float acc = 0.0f;
    for (int32_t d = 0; d < D; ++d) {
      float xd = elem(x, dtype, (size_t)d);
      float wdj = elem(W, dtype, (size_t)d * (size_t)bits + (size_t)j);
#if ORACLE_MUTANT == 1 /* planted: projection uses the wrong W index (transpose) */
      wdj = elem(W, dtype, ((size_t)j * (size_t)D + (size_t)d) % ((size_t)D * (size_t)bits));
#endif
      acc = fmaf(xd, wdj, acc);
    }
    float t = tauv ? tauv[j] : tau;
#if ORACLE_MUTANT == 22 /* planted: bit j compared with the threshold of bit j + 1 */
    if (tauv) t = tauv[(j + 1) % bits];
#endif
#if ORACLE_MUTANT == 2 /* planted: threshold >= instead of > */
    if (acc >= t) code |= (uint64_t)1 << j;
#elif ORACLE_MUTANT == 11 /* planted: threshold with the wrong sign */
    if (acc > -t) code |= (uint64_t)1 << j;
#else
    if (acc > t) code |= (uint64_t)1 << j;
#endif
  }
  return code;
}

uint64_t orc_code_tau(const void* x, int32_t dtype, int32_t D, const void* W, int32_t bits,
                      float tau) {
  return orc_code_thr(x, dtype, D, W, bits, tau, NULL);
}

/* The method's sign test: threshold 0. */
uint64_t orc_code(const void* x, int32_t dtype, int32_t D, const void* W, int32_t bits) {
  return orc_code_tau(x, dtype, D, W, bits, 0.0f);
}

void orc_code_many_tau(const void* x, int32_t n, int32_t dtype, int32_t D, const void* W,
                       int32_t bits, float tau, const float* tauv, uint64_t* codes) {
  const char* p = (const char*)x;
  for (int32_t i = 0; i < n; ++i)
    codes[i] = orc_code_thr(p + (size_t)i * (size_t)D * elem_bytes(dtype), dtype, D, W, bits,
                            tau, tauv);
}

void orc_code_many(const void* x, int32_t n, int32_t dtype, int32_t D, const void* W,
                   int32_t bits, uint64_t* codes) {
  orc_code_many_tau(x, n, dtype, D, W, bits, 0.0f, NULL, codes);
}

/* Per-bit median thresholds (the method's "binarisation threshold" design
 * choice, read as one threshold per bit that splits the cached keys in half):
 * tau[j] = the lower median of the projections of the n keys onto column j of
 * W (element (n - 1) / 2, counting from 0, of the ascending projections; the
 * same fp32 fused multiply-add chain as the code), so that for distinct
 * projections exactly floor(n / 2) keys have bit j set.  No keys: tau = 0. */
static int cmp_float(const void* a, const void* b) {
  const float x = *(const float*)a, y = *(const float*)b;
  return (x > y) - (x < y);
}

void orc_median_thresholds(const void* K, int32_t n, int32_t dtype, int32_t D, const void* W,
                           int32_t bits, float* tau) {
  float* s = (float*)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
  for (int32_t j = 0; j < bits; ++j) {
    for (int32_t i = 0; i < n; ++i) {
      float acc = 0.0f;
      for (int32_t d = 0; d < D; ++d)
        acc = fmaf(elem(K, dtype, (size_t)i * (size_t)D + (size_t)d),
                   elem(W, dtype, (size_t)d * (size_t)bits + (size_t)j), acc);
      s[i] = acc;
    }
    qsort(s, (size_t)n, sizeof(float), cmp_float);
#if ORACLE_MUTANT == 21 /* planted: the upper median */
    tau[j] = n > 0 ? s[n / 2] : 0.0f;
#else
    tau[j] = n > 0 ? s[(n - 1) / 2] : 0.0f;
#endif
  }
  free(s);
}

/* ------------------------------------------------------------------------- */
/* Step 3: Hamming distance, summed over the G query codes of a KV group.     */
/* ------------------------------------------------------------------------- */

static int32_t popcount64(uint64_t v) {
  int32_t c = 0;
  while (v) {
    c += (int32_t)(v & 1u);
    v >>= 1;
  }
  return c;
}

int32_t orc_group_distance(const uint64_t* code_q, int32_t G, uint64_t code_slot) {
  int32_t dist = 0;
  for (int32_t g = 0; g < G; ++g) {
#if ORACLE_MUTANT == 3 /* planted: only the first query head of the group scores */
    if (g > 0) break;
#endif
    dist += popcount64(code_q[g] ^ code_slot);
  }
  return dist;
}

/* Step 4: the slot with the largest distance; ties go to the lowest index. */
int32_t orc_most_dissimilar(const int32_t* dist, int32_t n) {
  int32_t best = 0;
  for (int32_t s = 1; s < n; ++s) {
#if ORACLE_MUTANT == 4 /* planted: ties go to the highest index */
    if (dist[s] >= dist[best]) best = s;
#elif ORACLE_MUTANT == 5 /* planted: evicts the most similar slot */
    if (dist[s] < dist[best]) best = s;
#else
    if (dist[s] > dist[best]) best = s;
#endif
  }
  return best;
}

/* Step 4 with score memory: the slot with the largest score; ties go to the
 * lowest index. */
int32_t orc_most_dissimilar_score(const float* score, int32_t n) {
  int32_t best = 0;
  for (int32_t s = 1; s < n; ++s) {
#if ORACLE_MUTANT == 12 /* planted: ties go to the highest index */
    if (score[s] >= score[best]) best = s;
#else
    if (score[s] > score[best]) best = s;
#endif
  }
  return best;
}

/* ------------------------------------------------------------------------- */
/* Decode attention of G query heads over n cached rows, in fp64.             */
/* ------------------------------------------------------------------------- */

void orc_attend(const void* q, const void* K, const void* V, int32_t n, int32_t D, int32_t G,
                int32_t dtype, double* out) {
  double* logit = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double scale = 1.0 / sqrt((double)D);
#if ORACLE_MUTANT == 6 /* planted: scale dropped */
  scale = 1.0;
#endif
  for (int32_t g = 0; g < G; ++g) {
    double m = -INFINITY;
    for (int32_t s = 0; s < n; ++s) {
      double dot = 0.0;
      for (int32_t d = 0; d < D; ++d)
        dot += (double)elem(q, dtype, (size_t)g * D + d) *
               (double)elem(K, dtype, (size_t)s * D + d);
      logit[s] = dot * scale;
      if (logit[s] > m) m = logit[s];
    }
    double den = 0.0;
    for (int32_t s = 0; s < n; ++s) den += exp(logit[s] - m);
    for (int32_t d = 0; d < D; ++d) {
      double num = 0.0;
      for (int32_t s = 0; s < n; ++s) {
#if ORACLE_MUTANT == 7 /* planted: value rows read with the key's index transposed */
        num += exp(logit[s] - m) * (double)elem(V, dtype, ((size_t)d * n + s) % ((size_t)n * D));
#else
        num += exp(logit[s] - m) * (double)elem(V, dtype, (size_t)s * D + d);
#endif
      }
      out[(size_t)g * D + d] = n > 0 ? num / den : 0.0;
    }
  }
  free(logit);
}

/* ------------------------------------------------------------------------- */
/* One (batch, KV head) unit: fill, then the per-token step.                  */
/* State: K[budget][D], V[budget][D] (dtype), codes[budget], *occupancy.      */
/* ------------------------------------------------------------------------- */

void orc_unit_fill_tau(const void* W, int32_t D, int32_t bits, int32_t dtype, int32_t budget,
                       const void* Kin, const void* Vin, int32_t n, float tau,
                       const float* tauv, void* K, void* V, uint64_t* codes,
                       int32_t* occupancy) {
  size_t row = (size_t)D * elem_bytes(dtype);
  (void)budget;
  memcpy(K, Kin, row * (size_t)n);
  memcpy(V, Vin, row * (size_t)n);
  for (int32_t s = 0; s < n; ++s)
    codes[s] = orc_code_thr((const char*)Kin + (size_t)s * row, dtype, D, W, bits, tau, tauv);
  *occupancy = n;
}

void orc_unit_fill(const void* W, int32_t D, int32_t bits, int32_t dtype, int32_t budget,
                   const void* Kin, const void* Vin, int32_t n, void* K, void* V,
                   uint64_t* codes, int32_t* occupancy) {
  orc_unit_fill_tau(W, D, bits, dtype, budget, Kin, Vin, n, 0.0f, NULL, K, V, codes, occupancy);
}

/*
 * Runs `nsteps` tokens through the step.  Inputs per token t: q[t][G][D],
 * k[t][D], v[t][D].  Per token it records evicted[t] (slot overwritten, or -1
 * when the token was appended to a cache not yet full), written[t] (the slot
 * the token now occupies) and, when want_out is NULL or want_out[t] != 0,
 * one [G][D] block of fp64 attention output, packed in token order into out.  dist_log, when not NULL, receives the distances of
 * the scored slots, dist_log[t][budget] (0 for appended tokens).
 */
/*
 * The same stream with a binarisation threshold tau and, when `score` is not
 * NULL, score memory gamma = `decay`: score[budget] holds A(s) (zero after a
 * fill) and is updated in place.  With score == NULL the eviction uses the
 * step's distances directly.
 */
void orc_unit_stream_ext(const void* W, int32_t D, int32_t G, int32_t bits, int32_t dtype,
                         int32_t budget, void* K, void* V, uint64_t* codes, float* score,
                         int32_t* occupancy, int32_t nsteps, const void* q, const void* k,
                         const void* v, float tau, const float* tauv, float decay,
                         int32_t* evicted, int32_t* written, const uint8_t* want_out,
                         double* out, int32_t* dist_log) {
  size_t row = (size_t)D * elem_bytes(dtype);
  int32_t* dist = (int32_t*)malloc(sizeof(int32_t) * (size_t)budget);
  uint64_t* code_q = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)G);
  size_t n_out = 0;
  for (int32_t t = 0; t < nsteps; ++t) {
    const char* qt = (const char*)q + (size_t)t * (size_t)G * row;
    const char* kt = (const char*)k + (size_t)t * row;
    const char* vt = (const char*)v + (size_t)t * row;
    int32_t slot;
    if (*occupancy == budget) {
      /* steps 1-3: code the query heads of the group and score every slot */
      for (int32_t g = 0; g < G; ++g)
        code_q[g] = orc_code_thr(qt + (size_t)g * row, dtype, D, W, bits, tau, tauv);
      for (int32_t s = 0; s < budget; ++s) dist[s] = orc_group_distance(code_q, G, codes[s]);
      /* step 4 */
      if (score) {
        for (int32_t s = 0; s < budget; ++s) {
#if ORACLE_MUTANT == 9 /* planted: the memory weighs the new distance, not the old score */
          score[s] = fmaf(decay, (float)dist[s], score[s]);
#else
          score[s] = fmaf(decay, score[s], (float)dist[s]);
#endif
        }
        slot = orc_most_dissimilar_score(score, budget);
      } else {
        slot = orc_most_dissimilar(dist, budget);
      }
      evicted[t] = slot;
      if (dist_log) memcpy(dist_log + (size_t)t * budget, dist, sizeof(int32_t) * (size_t)budget);
    } else {
      slot = *occupancy;
      *occupancy += 1;
      evicted[t] = -1;
      if (dist_log) memset(dist_log + (size_t)t * budget, 0, sizeof(int32_t) * (size_t)budget);
    }
    written[t] = slot;
    /* step 5: the current token replaces the evicted one */
    memcpy((char*)K + (size_t)slot * row, kt, row);
    memcpy((char*)V + (size_t)slot * row, vt, row);
    codes[slot] = orc_code_thr(kt, dtype, D, W, bits, tau, tauv);
#if ORACLE_MUTANT != 10 /* (planted when 10: the new token inherits the evicted score) */
    if (score) score[slot] = 0.0f; /* the new token has not been scored yet */
#endif
#if ORACLE_MUTANT == 8 /* planted: the new token's value is not written */
    memset((char*)V + (size_t)slot * row, 0, row);
#endif
    /* attention over the retained cache */
    if (!want_out || want_out[t])
      orc_attend(qt, K, V, *occupancy, D, G, dtype, out + (n_out++) * (size_t)G * (size_t)D);
  }
  free(dist);
  free(code_q);
}

/* ------------------------------------------------------------------------- */
/* Quantised value cache: one byte per value element with one fp32 scale per  */
/* row.  Reading (DASH-KV page: values tolerate coarser compression than      */
/* keys; TTKV page: keys get more bits than values): the row is stored in one */
/* of two byte formats, fmt:                                                 */
/*   1 (int8): s = max_d |v_d| / 127 in fp32, q_d = v_d / s (fp32 division)   */
/*     rounded half to even, clamped to [-127, 127]; stored value q_d * s;    */
/*   2 (fp8, the E4M3 format of the OCP 8-bit floating point specification): */
/*     s = max_d |v_d| / 448 in fp32 (448 is the format's largest finite      */
/*     magnitude), c_d = E4M3 nearest to v_d / s (fp32 division), ties to the */
/*     even mantissa, magnitudes beyond 448 saturating to 448; stored value   */
/*     e4m3(c_d) * s.                                                         */
/* A zero row has s = 0 and every code 0.  Keys stay in the element type:    */
/* codes and logits are those of the method.                                 */
/* ------------------------------------------------------------------------- */

/* E4M3: sign bit, 4 exponent bits (bias 7), 3 mantissa bits.  Exponent field 0
 * holds the subnormals m/8 * 2^-6; field 1..15 the normals (1 + m/8) * 2^(e-7);
 * S.1111.111 is NaN (the format has no infinities), so the largest finite
 * magnitude is 1.75 * 2^8 = 448. */
double orc_e4m3_decode(uint8_t c) {
  const int sgn = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  double a;
#if ORACLE_MUTANT == 20 /* planted: subnormals decoded with the implicit leading bit */
  a = ldexp((double)(8 + m), (e == 0 ? 1 : e) - 10);
  if (e == 0 && m == 0) a = 0.0;
#else
  if (e == 0)
    a = ldexp((double)m, -9);
  else
    a = ldexp((double)(8 + m), e - 10);
#endif
  return sgn ? -a : a;
}

/* The E4M3 code nearest to x: ties to the even mantissa (the even multiple of
 * the binade's step), magnitudes beyond 448 saturate to 448, the sign is kept
 * (a negative x that rounds to zero gives -0, code 0x80), NaN gives 0x7F. */
uint8_t orc_e4m3_encode(float x) {
  if (isnan(x)) return 0x7F;
  const uint8_t sgn = signbit(x) ? 0x80 : 0x00;
  const double a = fabs((double)x);
  if (a >= 448.0) return sgn | 0x7E;
  /* the binade [2^e, 2^(e+1)) holds 8 values 2^(e-3) apart; below 2^-6 the
   * subnormals are 2^-9 apart */
  int e;
  (void)frexp(a, &e); /* a = f 2^e with f in [0.5, 1) */
  e -= 1;
  if (e < -6) e = -6;
  const double step = ldexp(1.0, e - 3);
#if ORACLE_MUTANT == 18 /* planted: ties rounded away from zero */
  const double n = round(a / step);
#else
  const double n = nearbyint(a / step); /* a / step is exact; half to even */
#endif
  const double r = n * step; /* (n = 16 carries into the next binade) */
  if (r == 0.0) return sgn;
  int er;
  (void)frexp(r, &er);
  er -= 1;
  if (er < -6) return sgn | (uint8_t)(r / ldexp(1.0, -9)); /* subnormal: m = r / 2^-9 */
  const int m = (int)(r / ldexp(1.0, er - 3)) - 8;
  return sgn | (uint8_t)(((er + 7) << 3) | m);
}

/* The value a stored byte stands for before its row's scale. */
double orc_value_decode(int32_t fmt, uint8_t c) {
  return fmt == 2 ? orc_e4m3_decode(c) : (double)(int8_t)c;
}

void orc_quantize_row(const void* v, int32_t dtype, int32_t D, int32_t fmt, uint8_t* q,
                      float* scale) {
  float m = 0.0f;
  for (int32_t d = 0; d < D; ++d) {
    float a = fabsf(elem(v, dtype, (size_t)d));
    if (a > m) m = a;
  }
  float s;
  if (fmt == 2) {
#if ORACLE_MUTANT == 19 /* planted: fp8 rows scaled by max / 256 */
    s = m / 256.0f;
#else
    s = m / 448.0f;
#endif
  } else {
#if ORACLE_MUTANT == 13 /* planted: scale by 128 */
    s = m / 128.0f;
#else
    s = m / 127.0f;
#endif
  }
  *scale = s;
  for (int32_t d = 0; d < D; ++d) {
    if (!(s > 0.0f)) {
      q[d] = 0;
      continue;
    }
    float x = elem(v, dtype, (size_t)d) / s;
    if (fmt == 2) {
      q[d] = orc_e4m3_encode(x);
      continue;
    }
    float r;
#if ORACLE_MUTANT == 14 /* planted: rounds half away from zero */
    r = roundf(x);
#else
    r = nearbyintf(x); /* round half to even (default rounding mode) */
#endif
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    q[d] = (uint8_t)(int8_t)r;
  }
}

/* Attention of G query heads over n rows with keys K (element type) and
 * values decode(q[s][d]) * scale[s] (format fmt), in fp64. */
void orc_attend_vq(const void* qv, const void* K, const uint8_t* Vq, const float* Vs, int32_t n,
                   int32_t D, int32_t G, int32_t dtype, int32_t fmt, double* out) {
  double* logit = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  const double scale = 1.0 / sqrt((double)D);
  for (int32_t g = 0; g < G; ++g) {
    double m = -INFINITY;
    for (int32_t s = 0; s < n; ++s) {
      double dot = 0.0;
      for (int32_t d = 0; d < D; ++d)
        dot += (double)elem(qv, dtype, (size_t)g * D + d) *
               (double)elem(K, dtype, (size_t)s * D + d);
      logit[s] = dot * scale;
      if (logit[s] > m) m = logit[s];
    }
    double den = 0.0;
    for (int32_t s = 0; s < n; ++s) den += exp(logit[s] - m);
    for (int32_t d = 0; d < D; ++d) {
      double num = 0.0;
      for (int32_t s = 0; s < n; ++s)
        num += exp(logit[s] - m) * orc_value_decode(fmt, Vq[(size_t)s * D + d]) * (double)Vs[s];
      out[(size_t)g * D + d] = n > 0 ? num / den : 0.0;
    }
  }
  free(logit);
}

/* Fill of a unit with a quantised value cache (format fmt): K copied, V
 * quantised row by row. */
void orc_unit_fill_vq(const void* W, int32_t D, int32_t bits, int32_t dtype, int32_t budget,
                      const void* Kin, const void* Vin, int32_t n, float tau,
                      const float* tauv, int32_t fmt, void* K, uint8_t* Vq, float* Vs,
                      uint64_t* codes, int32_t* occupancy) {
  size_t row = (size_t)D * elem_bytes(dtype);
  (void)budget;
  memcpy(K, Kin, row * (size_t)n);
  for (int32_t s = 0; s < n; ++s) {
    orc_quantize_row((const char*)Vin + (size_t)s * row, dtype, D, fmt, Vq + (size_t)s * D,
                     Vs + s);
    codes[s] = orc_code_thr((const char*)Kin + (size_t)s * row, dtype, D, W, bits, tau, tauv);
  }
  *occupancy = n;
}

/* The step with a quantised value cache (format fmt): as orc_unit_stream_ext,
 * but the new token's value is quantised when written and attention reads the
 * stored values decode(q) * scale. */
void orc_unit_stream_vq(const void* W, int32_t D, int32_t G, int32_t bits, int32_t dtype,
                        int32_t budget, int32_t fmt, void* K, uint8_t* Vq, float* Vs,
                        uint64_t* codes, float* score, int32_t* occupancy, int32_t nsteps,
                        const void* q, const void* k, const void* v, float tau,
                        const float* tauv, float decay, int32_t* evicted, int32_t* written,
                        const uint8_t* want_out, double* out) {
  size_t row = (size_t)D * elem_bytes(dtype);
  int32_t* dist = (int32_t*)malloc(sizeof(int32_t) * (size_t)budget);
  uint64_t* code_q = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)G);
  size_t n_out = 0;
  for (int32_t t = 0; t < nsteps; ++t) {
    const char* qt = (const char*)q + (size_t)t * (size_t)G * row;
    const char* kt = (const char*)k + (size_t)t * row;
    const char* vt = (const char*)v + (size_t)t * row;
    int32_t slot;
    if (*occupancy == budget) {
      for (int32_t g = 0; g < G; ++g)
        code_q[g] = orc_code_thr(qt + (size_t)g * row, dtype, D, W, bits, tau, tauv);
      for (int32_t s = 0; s < budget; ++s) dist[s] = orc_group_distance(code_q, G, codes[s]);
      if (score) {
        for (int32_t s = 0; s < budget; ++s) score[s] = fmaf(decay, score[s], (float)dist[s]);
        slot = orc_most_dissimilar_score(score, budget);
      } else {
        slot = orc_most_dissimilar(dist, budget);
      }
      evicted[t] = slot;
    } else {
      slot = *occupancy;
      *occupancy += 1;
      evicted[t] = -1;
    }
    written[t] = slot;
    memcpy((char*)K + (size_t)slot * row, kt, row);
    orc_quantize_row(vt, dtype, D, fmt, Vq + (size_t)slot * D, Vs + slot);
    codes[slot] = orc_code_thr(kt, dtype, D, W, bits, tau, tauv);
    if (score) score[slot] = 0.0f;
    if (!want_out || want_out[t])
      orc_attend_vq(qt, K, Vq, Vs, *occupancy, D, G, dtype, fmt,
                    out + (n_out++) * (size_t)G * (size_t)D);
  }
  free(dist);
  free(code_q);
}

/* ------------------------------------------------------------------------- */
/* Chunk eviction (ChunkKV page: chunks of about 10 contiguous tokens, here  */
/* scored by the method's distances).  Reading: the budget B is cut into     */
/* B / c aligned chunks of c slots; while the cache is full, new tokens are  */
/* staged in the c - 1 slots after the budget (and attended); the token that */
/* would fill the stage evicts the chunk with the largest sum of its slots'  */
/* group-summed distances (ties: lowest chunk), and the c - 1 staged tokens, */
/* in order, then the token itself take the chunk's slots.  c = 1 is the     */
/* method.                                                                   */
/* State: K, V [B + c - 1][D], codes [B + c - 1]; occupancy counts staged.    */
/* ------------------------------------------------------------------------- */

void orc_unit_stream_chunk(const void* W, int32_t D, int32_t G, int32_t bits, int32_t dtype,
                           int32_t budget, int32_t chunk, void* K, void* V, uint64_t* codes,
                           int32_t* occupancy, int32_t nsteps, const void* q, const void* k,
                           const void* v, float tau, const float* tauv, int32_t* evicted,
                           int32_t* written, const uint8_t* want_out, double* out) {
  size_t row = (size_t)D * elem_bytes(dtype);
  const int32_t nch = budget / chunk;
  int32_t* dsum = (int32_t*)malloc(sizeof(int32_t) * (size_t)(nch > 0 ? nch : 1));
  uint64_t* code_q = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)G);
  size_t n_out = 0;
  for (int32_t t = 0; t < nsteps; ++t) {
    const char* qt = (const char*)q + (size_t)t * (size_t)G * row;
    const char* kt = (const char*)k + (size_t)t * row;
    const char* vt = (const char*)v + (size_t)t * row;
    int32_t slot;
    if (*occupancy < budget + chunk - 1) {
      /* a free slot of the budget, or a staging slot */
      slot = *occupancy;
      *occupancy += 1;
      evicted[t] = -1;
    } else {
      for (int32_t g = 0; g < G; ++g)
        code_q[g] = orc_code_thr(qt + (size_t)g * row, dtype, D, W, bits, tau, tauv);
      for (int32_t i = 0; i < nch; ++i) {
        dsum[i] = 0;
        for (int32_t j = 0; j < chunk; ++j) {
#if ORACLE_MUTANT == 15 /* planted: a chunk scores by its first slot only */
          if (j > 0) break;
#endif
#if ORACLE_MUTANT == 17 /* planted: a chunk scores its slots shifted by one */
          dsum[i] += orc_group_distance(code_q, G, codes[(i * chunk + j + 1) % budget]);
#else
          dsum[i] += orc_group_distance(code_q, G, codes[i * chunk + j]);
#endif
        }
      }
      const int32_t e = orc_most_dissimilar(dsum, nch);
      /* the staged tokens, in order, then this token take the chunk's slots */
      for (int32_t j = 0; j < chunk - 1; ++j) {
#if ORACLE_MUTANT == 16 /* planted: the staged tokens land in reverse order */
        const int32_t from = budget + chunk - 2 - j;
#else
        const int32_t from = budget + j;
#endif
        memcpy((char*)K + (size_t)(e * chunk + j) * row, (char*)K + (size_t)from * row, row);
        memcpy((char*)V + (size_t)(e * chunk + j) * row, (char*)V + (size_t)from * row, row);
        codes[e * chunk + j] = codes[from];
      }
      slot = e * chunk + chunk - 1;
      *occupancy = budget;
      evicted[t] = e * chunk;
    }
    written[t] = slot;
    memcpy((char*)K + (size_t)slot * row, kt, row);
    memcpy((char*)V + (size_t)slot * row, vt, row);
    codes[slot] = orc_code_thr(kt, dtype, D, W, bits, tau, tauv);
    if (!want_out || want_out[t])
      orc_attend(qt, K, V, *occupancy, D, G, dtype, out + (n_out++) * (size_t)G * (size_t)D);
  }
  free(dsum);
  free(code_q);
}

/* The method as described: threshold 0, the step's own distances. */
void orc_unit_stream(const void* W, int32_t D, int32_t G, int32_t bits, int32_t dtype,
                     int32_t budget, void* K, void* V, uint64_t* codes, int32_t* occupancy,
                     int32_t nsteps, const void* q, const void* k, const void* v,
                     int32_t* evicted, int32_t* written, const uint8_t* want_out, double* out,
                     int32_t* dist_log) {
  orc_unit_stream_ext(W, D, G, bits, dtype, budget, K, V, codes, NULL, occupancy, nsteps, q, k,
                      v, 0.0f, NULL, 0.0f, evicted, written, want_out, out, dist_log);
}
