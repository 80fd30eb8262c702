/*
 * synth_host.c — host build of the synthetic workload generator (synth_core.h).
 *
 * Element type: mode 0 writes bf16 bit patterns (uint16), mode 1 writes fp32.
 * Layouts:
 *   cache layout  [batch][kv_heads][nt][head_dim]   (token_major = 0)
 *   step layout   [nt][batch][kv_heads][head_dim]   (token_major = 1)
 *   queries       [nt][batch][heads][head_dim]
 *   unit vectors  [nt][head_dim] (keys/values of one (batch, kv head)),
 *                 [nt][group][head_dim] (queries of one KV group)
 */
#include <string.h>
#include "synth_core.h"

static void put(const synth_cfg* c, void* out, size_t idx, float v) {
  if (c->mode == SYNTH_MODE_IID_F32)
    ((float*)out)[idx] = v;
  else
    ((uint16_t*)out)[idx] = synth_bf16_rne(v); /* v is already a bf16 value */
}

void synth_host_init(synth_cfg* c) {
  for (int k = 0; k < SYNTH_N_OUTLIERS; ++k) c->outliers[k] = -1;
  if (c->mode == SYNTH_MODE_LLAMA_BF16) synth_pick_outliers(c);
}

static void kv_vec(const synth_cfg* c, int which, int32_t b, int32_t j, int32_t t, void* out,
                   size_t base) {
  uint64_t st = which == 0 ? synth_key_stream(c, b, j, t) : synth_value_stream(c, b, j, t);
  for (int32_t d = 0; d < c->head_dim; ++d)
    put(c, out, base + (size_t)d,
        which == 0 ? synth_key_elem(c, st, d) : synth_value_elem(c, st, d));
}

static void q_vec(const synth_cfg* c, int32_t b, int32_t h, int32_t t, void* out, size_t base) {
  uint64_t qst = synth_qnoise_stream(c, b, h, t);
  uint64_t kst = synth_query_key_stream(c, b, h, t);
  for (int32_t d = 0; d < c->head_dim; ++d)
    put(c, out, base + (size_t)d, synth_query_elem(c, qst, kst, t, d));
}

void synth_host_kv(const synth_cfg* c, int which, int32_t t0, int32_t nt, int token_major,
                   void* out) {
  const size_t D = (size_t)c->head_dim;
  for (int32_t b = 0; b < c->batch; ++b)
    for (int32_t j = 0; j < c->kv_heads; ++j)
      for (int32_t i = 0; i < nt; ++i) {
        size_t row = token_major
                         ? (((size_t)i * c->batch + b) * c->kv_heads + j)
                         : (((size_t)b * c->kv_heads + j) * (size_t)nt + i);
        kv_vec(c, which, b, j, t0 + i, out, row * D);
      }
}

void synth_host_queries(const synth_cfg* c, int32_t t0, int32_t nt, void* out) {
  const size_t D = (size_t)c->head_dim;
  for (int32_t i = 0; i < nt; ++i)
    for (int32_t b = 0; b < c->batch; ++b)
      for (int32_t h = 0; h < c->heads; ++h) {
        size_t row = ((size_t)i * c->batch + b) * c->heads + h;
        q_vec(c, b, h, t0 + i, out, row * D);
      }
}

void synth_host_unit_kv(const synth_cfg* c, int which, int32_t b, int32_t j, int32_t t0,
                        int32_t nt, void* out) {
  for (int32_t i = 0; i < nt; ++i) kv_vec(c, which, b, j, t0 + i, out, (size_t)i * c->head_dim);
}

void synth_host_unit_queries(const synth_cfg* c, int32_t b, int32_t j, int32_t t0, int32_t nt,
                             void* out) {
  const int32_t G = c->heads / c->kv_heads;
  for (int32_t i = 0; i < nt; ++i)
    for (int32_t g = 0; g < G; ++g)
      q_vec(c, b, j * G + g, t0 + i, out, ((size_t)i * G + g) * c->head_dim);
}

/* Raw generator access for the generator's own tests. */
uint64_t synth_host_mix64(uint64_t x) { return synth_mix64(x); }
float synth_host_normal(uint64_t stream, int32_t d) { return synth_normal(stream, d); }
uint16_t synth_host_bf16(float f) { return synth_bf16_rne(f); }
int32_t synth_host_query_past(const synth_cfg* c, int32_t b, int32_t h, int32_t t) {
  return synth_query_past(c, b, h, t);
}
