// he_noalloc.cu — he_attend_noalloc: decode attention over a caller-owned bf16
// cache that allocates no device memory.
//
// Some callers cannot let a library call cudaMalloc: runtimes whose device
// memory is entirely owned by their own pool or arena (a second allocator
// would fragment it or break its accounting), and deployments that must fix
// every byte of device memory up front.  For them this entry point runs the
// same split-K attention kernel as he_step (tensor-core stream over 64-slot
// tiles, then a log-sum-exp merge) with its partial results in a file-scope
// static device array instead of in handle-owned memory.  The caller passes
// the cache, the queries and the output.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "hashevict.h"
#include "he_pipeline.cuh"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kFlagFloats = 64;  // the first 256 bytes hold the kernels' error flag

// Scratch of every call: [error flag area][partial records].  Every GPU that
// loads the library holds it until the process exits.
static __device__ __align__(256) float g_noalloc_scratch[HE_NOALLOC_SCRATCH_BYTES / 4];

struct DeviceSetup {
  float* scratch = nullptr;  // device address of g_noalloc_scratch
  int num_sms = 0;
  int ctas_per_sm[4][2] = {};  // [G = 1, 2, 4, 8][D = 64, 128]
  bool ready = false;
};
DeviceSetup g_setup[kMaxDevices];

constexpr int kStages = 2;
constexpr bool kPSplit = true;

int g_index(int G) { return G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3; }

template <int D, int G>
const void* stream_fn() {
  return reinterpret_cast<const void*>(&he::stream_kernel<D, G, kStages, kPSplit>);
}

constexpr int kAttendMergeThreads = 512;
constexpr int kStreamThreads = he::StreamShape<128, 4, kStages>::NT;  // the same for every shape

// Log-sum-exp merge of a unit's partials (no eviction, no new token).  If a
// stream CTA of this call gave up a bounded wait (the flag word of the array
// is set), its partials are missing: the unit's output is written as NaN.
template <int D, int G>
__global__ void __launch_bounds__(kAttendMergeThreads) attend_merge_kernel(const he::StepParams p,
                                                                       int stream_ctas) {
  using R = he::PRec<G, D>;
  constexpr int GD4 = G * D / 4;
  constexpr int NQ = kAttendMergeThreads / GD4;
  __shared__ float4 sacc[kAttendMergeThreads];
  __shared__ float smax[kAttendMergeThreads];
  __shared__ float ssum[kAttendMergeThreads];
  const int tid = threadIdx.x;
  const int u = blockIdx.x;
  const int64_t TT = p.total_tiles, NCT = stream_ctas;
  const int first = (int)((((int64_t)u * p.tpu + 1) * NCT - 1) / TT);
  const int last = (int)((((int64_t)u * p.tpu + p.tpu) * NCT - 1) / TT);
  const int n = last - first + 1;
  const float* recs = p.partials + (size_t)(first + u) * R::FLOATS;
  const int q = tid / GD4, o = tid - q * GD4;
  const int g = (4 * o) / D;
  float mx = -1e30f, sum = 0.0f;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c = q; c < n; c += NQ) {
    const float* r = recs + (size_t)c * R::FLOATS;
    const float mc = __ldcg(r + g), lc = __ldcg(r + G + g);
    const float4 x = __ldcg(reinterpret_cast<const float4*>(r + R::HDR) + o);
    const float mn = fmaxf(mx, mc);
    const float so = exp2f(mx - mn), sn = exp2f(mc - mn);
    sum = sum * so + lc * sn;
    a.x = a.x * so + x.x * sn;
    a.y = a.y * so + x.y * sn;
    a.z = a.z * so + x.z * sn;
    a.w = a.w * so + x.w * sn;
    mx = mn;
  }
  sacc[tid] = a;
  smax[tid] = mx;
  ssum[tid] = sum;
  __syncthreads();
  if (tid < GD4) {
    float m2 = -1e30f;
    for (int q2 = 0; q2 < NQ; ++q2) m2 = fmaxf(m2, smax[q2 * GD4 + tid]);
    float l2 = 0.0f;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q2 = 0; q2 < NQ; ++q2) {
      const float w = exp2f(smax[q2 * GD4 + tid] - m2);
      const float4 y = sacc[q2 * GD4 + tid];
      l2 += ssum[q2 * GD4 + tid] * w;
      s.x += y.x * w;
      s.y += y.y * w;
      s.z += y.z * w;
      s.w += y.w * w;
    }
    const float inv = __ldcg(p.err) != 0 ? __int_as_float(0x7fc00000) : 1.0f / l2;
    const int b = u / p.kv_heads, j = u - b * p.kv_heads;
    reinterpret_cast<float4*>(p.out + ((size_t)b * p.kv_heads * G + (size_t)j * G) * D)[tid] =
        make_float4(s.x * inv, s.y * inv, s.z * inv, s.w * inv);
  }
}

template <int D, int G>
const void* merge_fn() {
  return reinterpret_cast<const void*>(&attend_merge_kernel<D, G>);
}

const void* pick_stream(int D, int G) {
  if (D == 64) {
    switch (G) {
      case 1: return stream_fn<64, 1>();
      case 2: return stream_fn<64, 2>();
      case 4: return stream_fn<64, 4>();
      case 8: return stream_fn<64, 8>();
    }
  } else if (D == 128) {
    switch (G) {
      case 1: return stream_fn<128, 1>();
      case 2: return stream_fn<128, 2>();
      case 4: return stream_fn<128, 4>();
      case 8: return stream_fn<128, 8>();
    }
  }
  return nullptr;
}

const void* pick_merge(int D, int G) {
  if (D == 64) {
    switch (G) {
      case 1: return merge_fn<64, 1>();
      case 2: return merge_fn<64, 2>();
      case 4: return merge_fn<64, 4>();
      case 8: return merge_fn<64, 8>();
    }
  } else if (D == 128) {
    switch (G) {
      case 1: return merge_fn<128, 1>();
      case 2: return merge_fn<128, 2>();
      case 4: return merge_fn<128, 4>();
      case 8: return merge_fn<128, 8>();
    }
  }
  return nullptr;
}

int stream_smem(int D, int G) {
  if (D == 64) {
    switch (G) {
      case 1: return he::StreamShape<64, 1, kStages>::SMEM_ALLOC;
      case 2: return he::StreamShape<64, 2, kStages>::SMEM_ALLOC;
      case 4: return he::StreamShape<64, 4, kStages>::SMEM_ALLOC;
      default: return he::StreamShape<64, 8, kStages>::SMEM_ALLOC;
    }
  }
  switch (G) {
    case 1: return he::StreamShape<128, 1, kStages>::SMEM_ALLOC;
    case 2: return he::StreamShape<128, 2, kStages>::SMEM_ALLOC;
    case 4: return he::StreamShape<128, 4, kStages>::SMEM_ALLOC;
    default: return he::StreamShape<128, 8, kStages>::SMEM_ALLOC;
  }
}

// Once per device, with that device current: the scratch array's device
// address (host code cannot use the array's name as a device pointer) and the
// stream kernels' launch shapes.
int setup_device(int dev) {
  DeviceSetup& s = g_setup[dev];
  if (s.ready) return HE_OK;
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
    (void)cudaGetLastError();
    return HE_ECUDA;
  }
  if (cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return HE_ECUDA;
  }
  const int Gs[4] = {1, 2, 4, 8}, Ds[2] = {64, 128};
  for (int gi = 0; gi < 4; ++gi)
    for (int di = 0; di < 2; ++di) {
      const void* fn = pick_stream(Ds[di], Gs[gi]);
      const int smem = stream_smem(Ds[di], Gs[gi]);
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
              cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s.ctas_per_sm[gi][di], fn, kStreamThreads, smem) !=
              cudaSuccess ||
          s.ctas_per_sm[gi][di] < 1) {
        (void)cudaGetLastError();
        return HE_ECUDA;
      }
    }
  s.scratch = static_cast<float*>(ptr);
  s.ready = true;
  return HE_OK;
}

// The driver's tensor-map encoder, resolved once per process (thread-safe).
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool encode_map(CUtensorMap* map, const void* base, uint64_t rows, int D) {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess && fn)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    else
      (void)cudaGetLastError();
  });
  const PFN_cuTensorMapEncodeTiled_v12000 encode = g_encode;
  if (!encode) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int he_attend_noalloc(int32_t batch, int32_t heads, int32_t kv_heads, int32_t head_dim,
                                 int32_t budget, int32_t n, const void* K, const void* V,
                                 const void* q, float* out, void* stream) {
  if (batch < 1 || heads < 1 || kv_heads < 1 || heads % kv_heads != 0) return HE_EINVAL;
  const int G = heads / kv_heads;
  if ((G != 1 && G != 2 && G != 4 && G != 8) || (head_dim != 64 && head_dim != 128))
    return HE_EINVAL;
  if (budget < 1 || n < 1 || n > budget || (int64_t)batch * kv_heads > 65536) return HE_EINVAL;
  if (!K || !V || !q || !out || !aligned16(K) || !aligned16(V) || !aligned16(q) ||
      !aligned16(out))
    return HE_EINVAL;
  const int64_t U = (int64_t)batch * kv_heads;
  if (U * budget >= ((int64_t)1 << 31)) return HE_EINVAL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return HE_ECUDA;
  }
  int rc = setup_device(dev);
  if (rc != HE_OK) return rc;
  const DeviceSetup& s = g_setup[dev];

  const int tile = 64;
  const int tpu = (n + tile - 1) / tile;
  const int64_t total = U * tpu;
  const int max_ctas = s.num_sms * s.ctas_per_sm[g_index(G)][head_dim == 64 ? 0 : 1];
  const int ctas = total < max_ctas ? (int)total : max_ctas;
  const int rec_floats = (2 * G + 3) / 4 * 4 + G * head_dim;
  const size_t need = ((size_t)ctas + (size_t)U) * rec_floats * 4 + kFlagFloats * 4;
  if (need > (size_t)HE_NOALLOC_SCRATCH_BYTES || total > INT32_MAX) return HE_EINVAL;

  CUtensorMap tmK, tmV;
  if (!encode_map(&tmK, K, (uint64_t)U * budget, head_dim) ||
      !encode_map(&tmV, V, (uint64_t)U * budget, head_dim))
    return HE_EINVAL;

  he::StepParams p{};
  p.K = const_cast<void*>(K);
  p.V = const_cast<void*>(V);
  p.q = q;
  p.out = out;
  p.partials = s.scratch + kFlagFloats;
  p.err = reinterpret_cast<int32_t*>(s.scratch);
  p.U = (int32_t)U;
  p.kv_heads = kv_heads;
  p.budget = budget;
  p.occ = n;
  p.tile = tile;
  p.tpu = tpu;
  p.total_tiles = (int32_t)total;
  p.append_slot = 0;
  p.qscale = (float)(1.4426950408889634 / std::sqrt((double)head_dim));

  cudaStream_t st = (cudaStream_t)stream;
  // the flag word starts each call at zero (a kernel that gives up a wait sets it)
  if (cudaMemsetAsync(s.scratch, 0, sizeof(int32_t), st) != cudaSuccess) {
    (void)cudaGetLastError();
    return HE_ECUDA;
  }
  void* sa[] = {(void*)&p, (void*)&tmK, (void*)&tmV};
  if (cudaLaunchKernel(pick_stream(head_dim, G), dim3(ctas), dim3(kStreamThreads), sa,
                       (size_t)stream_smem(head_dim, G), st) != cudaSuccess) {
    (void)cudaGetLastError();
    return HE_ECUDA;
  }
  int sc = ctas;
  void* ma[] = {(void*)&p, (void*)&sc};
  if (cudaLaunchKernel(pick_merge(head_dim, G), dim3((unsigned)U), dim3(kAttendMergeThreads), ma, 0,
                       st) != cudaSuccess) {
    (void)cudaGetLastError();
    return HE_ECUDA;
  }
  return HE_OK;
}
