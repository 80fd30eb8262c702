/*
 * synth_gpu.cu — device build of the synthetic workload generator (synth_core.h).
 * Same layouts and element types as synth_host.c; one thread per element.
 * Used to stage large workloads directly in HBM; bit-identical to the host build.
 */
#include <cuda_runtime.h>
#include "synth_core.h"

template <typename T>
__device__ __forceinline__ void put_elem(T* out, size_t i, float v);
template <>
__device__ __forceinline__ void put_elem<float>(float* out, size_t i, float v) { out[i] = v; }
template <>
__device__ __forceinline__ void put_elem<uint16_t>(uint16_t* out, size_t i, float v) {
  out[i] = synth_bf16_rne(v);
}

template <typename T>
__global__ void kv_kernel(synth_cfg c, int which, int32_t t0, int32_t nt, int token_major,
                          T* out) {
  const size_t D = (size_t)c.head_dim;
  const size_t total = (size_t)c.batch * c.kv_heads * (size_t)nt * D;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total;
       e += (size_t)gridDim.x * blockDim.x) {
    int32_t d = (int32_t)(e % D);
    size_t row = e / D;
    int32_t b, j, i;
    if (token_major) {
      j = (int32_t)(row % c.kv_heads);
      b = (int32_t)((row / c.kv_heads) % c.batch);
      i = (int32_t)(row / ((size_t)c.kv_heads * c.batch));
    } else {
      i = (int32_t)(row % nt);
      j = (int32_t)((row / nt) % c.kv_heads);
      b = (int32_t)(row / ((size_t)nt * c.kv_heads));
    }
    int32_t t = t0 + i;
    float v = which == 0 ? synth_key_elem(&c, synth_key_stream(&c, b, j, t), d)
                         : synth_value_elem(&c, synth_value_stream(&c, b, j, t), d);
    put_elem(out, e, v);
  }
}

template <typename T>
__global__ void q_kernel(synth_cfg c, int32_t t0, int32_t nt, T* out) {
  const size_t D = (size_t)c.head_dim;
  const size_t total = (size_t)nt * c.batch * c.heads * D;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total;
       e += (size_t)gridDim.x * blockDim.x) {
    int32_t d = (int32_t)(e % D);
    size_t row = e / D;
    int32_t h = (int32_t)(row % c.heads);
    int32_t b = (int32_t)((row / c.heads) % c.batch);
    int32_t i = (int32_t)(row / ((size_t)c.heads * c.batch));
    int32_t t = t0 + i;
    float v = synth_query_elem(&c, synth_qnoise_stream(&c, b, h, t),
                               synth_query_key_stream(&c, b, h, t), t, d);
    put_elem(out, e, v);
  }
}

static unsigned grid_for(size_t total) {
  size_t g = (total + 255) / 256;
  return (unsigned)(g > 148u * 64u ? 148u * 64u : (g == 0 ? 1 : g));
}

extern "C" int synth_gpu_kv(const synth_cfg* c, int which, int32_t t0, int32_t nt,
                            int token_major, void* out, void* stream) {
  size_t total = (size_t)c->batch * c->kv_heads * (size_t)nt * c->head_dim;
  if (total == 0) return 0;
  cudaStream_t s = (cudaStream_t)stream;
  if (c->mode == SYNTH_MODE_IID_F32)
    kv_kernel<float><<<grid_for(total), 256, 0, s>>>(*c, which, t0, nt, token_major, (float*)out);
  else
    kv_kernel<uint16_t><<<grid_for(total), 256, 0, s>>>(*c, which, t0, nt, token_major,
                                                         (uint16_t*)out);
  return (int)cudaGetLastError();
}

extern "C" int synth_gpu_queries(const synth_cfg* c, int32_t t0, int32_t nt, void* out,
                                 void* stream) {
  size_t total = (size_t)nt * c->batch * c->heads * c->head_dim;
  if (total == 0) return 0;
  cudaStream_t s = (cudaStream_t)stream;
  if (c->mode == SYNTH_MODE_IID_F32)
    q_kernel<float><<<grid_for(total), 256, 0, s>>>(*c, t0, nt, (float*)out);
  else
    q_kernel<uint16_t><<<grid_for(total), 256, 0, s>>>(*c, t0, nt, (uint16_t*)out);
  return (int)cudaGetLastError();
}
