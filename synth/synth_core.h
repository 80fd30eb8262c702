/*
 * synth_core.h — seeded synthetic workload generator (inputs only).
 *
 * This module produces the token stream that the HashEvict step is fed with:
 * cached keys and values, per-step queries, keys and values.  It holds none of
 * the method's arithmetic (no projection, no code, no distance, no attention);
 * it is shared, as plain source, by a host build (synth_host.c) and a device
 * build (synth_gpu.cu) so that a tensor generated on either side is bit-identical.
 *
 * Workload shape (HashEvict page, abstract and "technical framework"; the
 * LLM-shaped heads follow the ChunkKV and TTKV pages' Llama-3.1-8B setting):
 *   mode 0 ("llama", bf16):
 *     key[d]   = bf16( z * (d is one of 4 outlier channels ? 8 : 1) )
 *     value[d] = bf16( z )
 *     query[d] = bf16( 0.5 * key_past[d] + z )   key_past: a uniformly drawn
 *                earlier token (0..t-1) of the query's KV head; query = bf16(z) at t = 0
 *   mode 1 ("iid", fp32):  key, value, query = z, no outliers, no past-key mix.
 *   z ~ approximately N(0,1): Irwin-Hall sum of 12 uniform 16-bit integers,
 *       z = (sum - 393210) / 65536, exact in fp32 (support +-6, variance ~1).
 *
 * Counter hash: SplitMix64 finaliser (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014), chained over the tensor tag
 * and the indices (seed, tag, layer, batch, head, token) and then over the
 * element index.  bf16 conversion is round-to-nearest-even on the fp32 bits.
 */
#ifndef SYNTH_CORE_H
#define SYNTH_CORE_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYNTH_HD __host__ __device__ __forceinline__
#else
#define SYNTH_HD static inline
#endif

#define SYNTH_TAG_KEY 1u
#define SYNTH_TAG_VALUE 2u
#define SYNTH_TAG_QNOISE 3u
#define SYNTH_TAG_QPAST 4u
#define SYNTH_TAG_OUTLIER 5u

#define SYNTH_MODE_LLAMA_BF16 0
#define SYNTH_MODE_IID_F32 1

#define SYNTH_N_OUTLIERS 4
#define SYNTH_OUTLIER_SCALE 8.0f

typedef struct {
  uint64_t seed;
  int32_t layer;
  int32_t batch;
  int32_t heads;
  int32_t kv_heads;
  int32_t head_dim;
  int32_t mode; /* SYNTH_MODE_* */
  int32_t outliers[SYNTH_N_OUTLIERS]; /* filled by synth_pick_outliers (mode 0) */
} synth_cfg;

SYNTH_HD uint64_t synth_mix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* Stream key for one (tag, layer, batch, head, token) vector. */
SYNTH_HD uint64_t synth_stream(uint64_t seed, uint32_t tag, int32_t layer, int32_t b,
                               int32_t head, int32_t t) {
  uint64_t h = synth_mix64(seed ^ ((uint64_t)tag * 0xD1B54A32D192ED03ull));
  h = synth_mix64(h ^ (uint64_t)(uint32_t)layer);
  h = synth_mix64(h ^ (uint64_t)(uint32_t)b);
  h = synth_mix64(h ^ (uint64_t)(uint32_t)head);
  h = synth_mix64(h ^ (uint64_t)(uint32_t)t);
  return h;
}

/* Irwin-Hall(12) normal for element d of a stream. Exact in fp32. */
SYNTH_HD float synth_normal(uint64_t stream, int32_t d) {
  int32_t s = 0;
  for (int r = 0; r < 3; ++r) {
    uint64_t u = synth_mix64(stream + 3ull * (uint64_t)(uint32_t)d + (uint64_t)r);
    s += (int32_t)(u & 0xFFFFu) + (int32_t)((u >> 16) & 0xFFFFu) +
         (int32_t)((u >> 32) & 0xFFFFu) + (int32_t)((u >> 48) & 0xFFFFu);
  }
  return (float)(s - 393210) * (1.0f / 65536.0f);
}

SYNTH_HD uint32_t synth_f32_bits(float f) {
  union { float f; uint32_t u; } c;
  c.f = f;
  return c.u;
}

SYNTH_HD float synth_bits_f32(uint32_t u) {
  union { float f; uint32_t u; } c;
  c.u = u;
  return c.f;
}

/* fp32 -> bf16 bit pattern, round to nearest, ties to even (finite inputs). */
SYNTH_HD uint16_t synth_bf16_rne(float f) {
  uint32_t u = synth_f32_bits(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

SYNTH_HD float synth_bf16_to_f32(uint16_t h) { return synth_bits_f32((uint32_t)h << 16); }

/* Lemire's multiply-shift: uniform integer in [0, n) from 32 random bits. */
SYNTH_HD uint32_t synth_below(uint64_t r, uint32_t n) {
  return (uint32_t)(((uint64_t)(uint32_t)r * (uint64_t)n) >> 32);
}

/* Four distinct outlier channels in [0, head_dim), one set per run (seed). */
SYNTH_HD void synth_pick_outliers(synth_cfg* c) {
  uint64_t st = synth_stream(c->seed, SYNTH_TAG_OUTLIER, 0, 0, 0, 0);
  int n = 0;
  for (uint64_t i = 0; n < SYNTH_N_OUTLIERS; ++i) {
    int32_t ch = (int32_t)synth_below(synth_mix64(st + i), (uint32_t)c->head_dim);
    int dup = 0;
    for (int k = 0; k < n; ++k) dup |= (c->outliers[k] == ch);
    if (!dup) c->outliers[n++] = ch;
  }
}

SYNTH_HD int synth_is_outlier(const synth_cfg* c, int32_t d) {
  int o = 0;
  for (int k = 0; k < SYNTH_N_OUTLIERS; ++k) o |= (c->outliers[k] == d);
  return o;
}

/* Key element d of the vector whose stream is `st`, as the exact fp32 value
 * of the stored element. */
SYNTH_HD float synth_key_elem(const synth_cfg* c, uint64_t st, int32_t d) {
  float z = synth_normal(st, d);
  if (c->mode == SYNTH_MODE_IID_F32) return z;
  if (synth_is_outlier(c, d)) z = z * SYNTH_OUTLIER_SCALE;
  return synth_bf16_to_f32(synth_bf16_rne(z));
}

SYNTH_HD float synth_value_elem(const synth_cfg* c, uint64_t st, int32_t d) {
  float z = synth_normal(st, d);
  if (c->mode == SYNTH_MODE_IID_F32) return z;
  return synth_bf16_to_f32(synth_bf16_rne(z));
}

SYNTH_HD uint64_t synth_key_stream(const synth_cfg* c, int32_t b, int32_t j, int32_t t) {
  return synth_stream(c->seed, SYNTH_TAG_KEY, c->layer, b, j, t);
}

SYNTH_HD uint64_t synth_value_stream(const synth_cfg* c, int32_t b, int32_t j, int32_t t) {
  return synth_stream(c->seed, SYNTH_TAG_VALUE, c->layer, b, j, t);
}

/* Index of the past token whose key a query mixes in (mode 0, t > 0). */
SYNTH_HD int32_t synth_query_past(const synth_cfg* c, int32_t b, int32_t h, int32_t t) {
  return (int32_t)synth_below(synth_stream(c->seed, SYNTH_TAG_QPAST, c->layer, b, h, t),
                              (uint32_t)t);
}

/* Query element d of head h at token t.  `kst` is the key stream of the past
 * token (synth_query_past) of the head's KV group; unused in mode 1 or at t = 0.
 * 0.5 * key is exact (power-of-two scaling), so a fused multiply-add and a
 * separate multiply and add give the same fp32 sum. */
SYNTH_HD float synth_query_elem(const synth_cfg* c, uint64_t qst, uint64_t kst, int32_t t,
                                int32_t d) {
  float z = synth_normal(qst, d);
  if (c->mode == SYNTH_MODE_IID_F32) return z;
  if (t > 0) z = 0.5f * synth_key_elem(c, kst, d) + z;
  return synth_bf16_to_f32(synth_bf16_rne(z));
}

SYNTH_HD uint64_t synth_qnoise_stream(const synth_cfg* c, int32_t b, int32_t h, int32_t t) {
  return synth_stream(c->seed, SYNTH_TAG_QNOISE, c->layer, b, h, t);
}

/* Key stream of the past token a query (b, h, t) mixes in. */
SYNTH_HD uint64_t synth_query_key_stream(const synth_cfg* c, int32_t b, int32_t h, int32_t t) {
  if (c->mode == SYNTH_MODE_IID_F32 || t == 0) return 0;
  int32_t group = c->heads / c->kv_heads;
  return synth_key_stream(c, b, h / group, synth_query_past(c, b, h, t));
}

#endif /* SYNTH_CORE_H */
