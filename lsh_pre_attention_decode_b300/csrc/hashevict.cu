// hashevict.cu — the C ABI of libhashevict.so (declared in include/hashevict.h):
// handle life cycle, argument checks, launch shapes and the kernel dispatch.
// Every step of the decode path runs in the kernels of he_step.cuh.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>
#include <type_traits>

#include <cudaTypedefs.h>

#include "hashevict.h"
#include "he_pipeline.cuh"
#include "he_step_simt.cuh"

namespace {

using he::bf16_t;
using he::StepParams;

// Launch configuration of the two step engines.
constexpr int kSimtStages = 4;    // CUDA-core engine (fp32 caches): 32-slot tiles
constexpr int kTcStages = 2;      // tensor-core pipeline (bf16 caches): 64-slot tiles
constexpr int kTcStagesVq = 3;    // the same with a quantised value cache (smaller stages),
                                  // where two such CTAs and a prep CTA fit an SM
constexpr bool kPSplit = true;    // attention weights as bf16 hi + lo parts
// Stream CTAs that start behind the previous step's merge CTAs (a 512-thread
// merge CTA leaves no room for a stream CTA on its SM) take this many tiles
// fewer than the others.
constexpr double kLateTiles = 2.0;
// The same for the fused step: the CTAs that start behind the previous step's
// merging CTAs (its last contributors, one per unit at most).
constexpr double kLateTilesFused = 0.0;

struct Kernels {
  const void* step;    // fp32: the fused step; bf16: the stream kernel
  const void* prep;    // bf16 pipeline
  const void* prep_mem;  // bf16 pipeline with score memory
  const void* merge;   // bf16 pipeline
  const void* merge_mu;  // bf16 pipeline, several units per merge CTA
  const void* merge_chunk_mu;
  const void* score;
  const void* code;
  int step_smem;
  int step_threads;
  int prep_smem;
  int merge_smem;                  // dynamic shared memory of the largest merge CTA
  // merge launch shape for U units of at most n partials: threads per CTA
  // (and nq, units per CTA, smem)
  int (*merge_cfg)(int n, int U, bool multi, int* nq, int* upc, int* smem);
  int tile;
  int rec_floats;
  bool tc;  // tensor-core pipeline (tensor maps, programmatic dependent launch)
  const void* vq_fill;  // quantised value cache: quantisation of filled value rows
  const void* prep_chunk;   // bf16 pipeline with chunk eviction
  const void* merge_chunk;
  int chunk_floats;         // floats of the per-unit chunk record
  const void* fused;        // bf16, the method: the whole step in one kernel
  int fused_smem;
  int fused_threads;
  int fused_rec_floats;
  int fused_stages;
  int stages;  // ring stages of the step kernel
};

// Ring stages of the fused step: two (with the hash warp's copy of W, a third
// stage would leave one CTA per SM).
template <int D, int G>
constexpr int fused_stages() {
  return 2 * (he::StreamShape<D, G, 3, false, true>::SMEM_ALLOC + 1024) <= 233472 ? 3 : 2;
}

// Ring stages of the stream kernel: kTcStagesVq for a quantised value cache
// when two stream CTAs and one prep CTA still fit an SM's shared memory (each
// CTA also reserves 1 KiB), else kTcStages.
template <int D, int G, int VQ>
constexpr int stream_stages() {
  constexpr int kSmemPerSm = 233472;
  return VQ && 2 * (he::StreamShape<D, G, kTcStagesVq, VQ>::SMEM_ALLOC + 1024) +
                       he::PrepShape<D, G>::SMEM + 1024 <= kSmemPerSm
             ? kTcStagesVq
             : kTcStages;
}

template <int D, int G>
int merge_cfg(int n, int U, bool multi, int* nq, int* upc, int* smem) {
  he::MergeShape<D, G>::config(n, U, multi, nq, upc);
  const int t = *nq * *upc * he::MergeShape<D, G>::GD4;
  *smem = he::merge_smem_bytes<D, G>(t);
  return t;
}

template <typename T, int D, int G, int VQ = 0>
Kernels kernels_for() {
  Kernels k{};
  k.score = reinterpret_cast<const void*>(&he::score_kernel<T, D, G>);
  k.code = reinterpret_cast<const void*>(&he::code_kernel<T, D>);
  if constexpr (std::is_same<T, bf16_t>::value) {
    constexpr int NS = stream_stages<D, G, VQ>();
    using S = he::StreamShape<D, G, NS, VQ>;
    k.step = reinterpret_cast<const void*>(&he::stream_kernel<D, G, NS, kPSplit, VQ>);
    k.stages = NS;
    k.prep = reinterpret_cast<const void*>(&he::prep_kernel<D, G, false, VQ>);
    k.prep_mem = reinterpret_cast<const void*>(&he::prep_kernel<D, G, true, VQ>);
    k.merge = reinterpret_cast<const void*>(&he::merge_kernel<D, G, VQ>);
    k.merge_mu = reinterpret_cast<const void*>(&he::merge_kernel<D, G, VQ, false, true>);
    k.vq_fill = VQ ? reinterpret_cast<const void*>(&he::vq_fill_kernel<D, VQ ? VQ : he::kVqInt8>)
                   : nullptr;
    if constexpr (!VQ) {
      constexpr int NSF = fused_stages<D, G>();
      using SF = he::StreamShape<D, G, NSF, false, true>;
      k.fused = reinterpret_cast<const void*>(&he::stream_kernel<D, G, NSF, kPSplit, false, true>);
      k.fused_smem = SF::SMEM_ALLOC;
      k.fused_threads = SF::NT;
      k.fused_rec_floats = he::FRec<G, D>::FLOATS;
      k.fused_stages = NSF;
      k.prep_chunk = reinterpret_cast<const void*>(&he::prep_kernel<D, G, false, false, true>);
      k.merge_chunk = reinterpret_cast<const void*>(&he::merge_kernel<D, G, false, true>);
      k.merge_chunk_mu = reinterpret_cast<const void*>(&he::merge_kernel<D, G, false, true, true>);
      k.chunk_floats = he::ChunkRec<G, D>::FLOATS;
    }
    k.step_smem = S::SMEM_ALLOC;
    k.step_threads = S::NT;
    k.prep_smem = he::PrepShape<D, G>::SMEM;
    k.merge_smem = he::merge_smem_bytes<D, G>(he::kMergeMaxThreads);
    k.merge_cfg = &merge_cfg<D, G>;
    k.tile = S::TS;
    k.rec_floats = he::PRec<G, D>::FLOATS;
    k.tc = true;
  } else {
    using S = he::SimtShape<T, D, G, kSimtStages>;
    k.step = reinterpret_cast<const void*>(&he::step_kernel_simt<T, D, G, kSimtStages>);
    k.step_smem = S::SMEM;
    k.step_threads = he::kThreads;
    k.stages = kSimtStages;
    k.tile = he::kTile;
    k.rec_floats = he::Record<G, D>::FLOATS;
    k.tc = false;
  }
  return k;
}

// Launch with programmatic stream serialisation: the kernel may start before
// the previous kernel in the stream finishes; it orders itself with
// griddepcontrol.wait.
cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

template <typename T, int D, int VQ = 0>
bool pick_g(int G, Kernels* k) {
  switch (G) {
    case 1: *k = kernels_for<T, D, 1, VQ>(); return true;
    case 2: *k = kernels_for<T, D, 2, VQ>(); return true;
    case 4: *k = kernels_for<T, D, 4, VQ>(); return true;
    case 8: *k = kernels_for<T, D, 8, VQ>(); return true;
    default: return false;
  }
}

// vq: 0, he::kVqInt8 or he::kVqFp8 (the value cache's byte format)
bool pick_kernels(int dtype, int D, int G, int vq, Kernels* k) {
  if (dtype == HE_DTYPE_BF16 && vq == he::kVqInt8) {
    if (D == 64) return pick_g<bf16_t, 64, he::kVqInt8>(G, k);
    if (D == 128) return pick_g<bf16_t, 128, he::kVqInt8>(G, k);
  } else if (dtype == HE_DTYPE_BF16 && vq == he::kVqFp8) {
    if (D == 64) return pick_g<bf16_t, 64, he::kVqFp8>(G, k);
    if (D == 128) return pick_g<bf16_t, 128, he::kVqFp8>(G, k);
  } else if (dtype == HE_DTYPE_BF16 && vq == 0) {
    if (D == 64) return pick_g<bf16_t, 64>(G, k);
    if (D == 128) return pick_g<bf16_t, 128>(G, k);
  } else if (dtype == HE_DTYPE_FP32 && vq == 0) {
    if (D == 64) return pick_g<float, 64>(G, k);
    if (D == 128) return pick_g<float, 128>(G, k);
  }
  return false;
}

// 2-D tensor map over a cache viewed as [rows][D] bf16 rows; boxes of
// 64 elements (128 bytes) x `box_rows` rows, 128B swizzle.
bool encode_cache_map(CUtensorMap* map, void* base, uint64_t rows, int D, int box_rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D tensor map over a quantised value cache viewed as [rows][D] bytes; boxes of
// one whole row (D bytes) x `box_rows` rows, 16-byte chunks swizzled within the
// row (128B swizzle for D = 128, 64B for D = 64; the stream kernel's
// vq_tile_off reads that layout).
bool encode_vq_map(CUtensorMap* map, void* base, uint64_t rows, int D, int box_rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)D};
  const cuuint32_t box[2] = {(cuuint32_t)D, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE,
                D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device memory cap of one he_create (0: none), see he_set_alloc_limit.
uint64_t g_alloc_limit = 0;

// One thread waits on a barrier that nothing completes, through the library's
// bounded wait; when the wait gives up it records the error flag, as the step
// kernels do.
__global__ void wait_probe_kernel(int32_t* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    he::mbar_init(&bar, 1);
    he::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !he::mbar_wait_bounded(&bar, 0u, limit_ns)) atomicExch(err, 1);
}

// Keeps the caller's current device and switches to the handle's for the call.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) {
      ok = false;
      return;
    }
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

}  // namespace

#ifdef HE_TIMELINE
extern "C" int he_debug_set_timeline(int64_t* dev) {
  return cudaMemcpyToSymbol(he::g_he_timeline, &dev, sizeof dev) == cudaSuccess ? HE_OK : HE_ECUDA;
}
#endif

struct he_ctx {
  he_cfg cfg;
  int device = 0;
  int G = 0;
  int U = 0;
  int eb = 0;           // element bytes
  int code_bytes = 0;   // bits / 8
  int code_stride = 0;  // bytes per unit row of codes, multiple of 16
  Kernels kern{};
  CUtensorMap tmK{};  // tensor-core engine: 2-D maps over K and V
  CUtensorMap tmV{};
  void* K = nullptr;
  void* V = nullptr;
  void* W = nullptr;
  unsigned char* codes = nullptr;
  int32_t* evicted = nullptr;
  float* score = nullptr;  // per-slot scores with score memory (decay > 0), else null
  float* tauv = nullptr;   // per-bit thresholds [U][bits] (tau_mode HE_TAU_MEDIAN), else null
  bool vq = false;         // quantised value cache: V holds byte rows (int8 or E4M3 codes),
                           // vs their scales
  float* vs = nullptr;     // [U][vs_stride]
  int vs_stride = 0;       // budget rounded up to whole 64-slot tiles
  int32_t* counters = nullptr;
  int32_t* err = nullptr;
  float* partials = nullptr;
  he::UnitOut* uo = nullptr;  // bf16 pipeline: per-unit results of prep
  int kpar = 0;               // parity of the next step's eviction key
  int prev_w1 = 0;            // the previous step's written slot (StepParams::prev_w1)
  int chunk = 1;              // slots per evicted chunk (1: the method)
  int rows = 0;               // rows per unit: budget + chunk - 1 (the stride of K, V, codes)
  float* cstar = nullptr;     // chunk eviction: the evicted chunk's softmax parts, per unit
  int nopre = 0;              // the previous step moved rows (StepParams::nopre)
  int merge_ctas = 0;         // merge CTAs of the previous step (each holds an SM)
  bool fused = false;         // the method on bf16: one kernel per step
  int prev_tpu = 0;           // fused: the split of the previous step (StepParams::prev_*)
  int prev_nc = 0;
  int prev_e = 0;
  int prev_t1 = 0;
  int32_t* evlog = nullptr;   // test exports (caller-owned device buffers, or null)
  int32_t* evcnt = nullptr;
  int32_t evcap = 0;
  int32_t* dist = nullptr;
  void* sq = nullptr;  // he_step_host staging
  void* sk = nullptr;
  void* sv = nullptr;
  float* sout = nullptr;
  int occupancy = 0;
  bool filled = false;
  int sticky = HE_OK;
  int num_sms = 0;
  int ctas_per_sm = 0;
  int max_ctas = 0;
  // kernel timing mode: four events per profiled step (before the cache
  // stream, after it, after codes/eviction, after merge)
  std::vector<cudaEvent_t> prof_ev;
  int prof_cap = 0;
  int prof_n = 0;
};

namespace {

int fail_cuda(he_ctx* h, cudaError_t e) {
  (void)cudaGetLastError();
  if (h) h->sticky = HE_ECUDA;
  (void)e;
  return HE_ECUDA;
}

#define HE_TRY(h, call)                         \
  do {                                          \
    cudaError_t e_ = (call);                    \
    if (e_ != cudaSuccess) return fail_cuda((h), e_); \
  } while (0)

size_t vec_bytes(const he_ctx* h, int heads) {
  return (size_t)h->cfg.batch * heads * h->cfg.head_dim * h->eb;
}

void free_profile(he_ctx* h) {
  for (cudaEvent_t e : h->prof_ev)
    if (e) cudaEventDestroy(e);
  h->prof_ev.clear();
  h->prof_cap = 0;
  h->prof_n = 0;
}

void free_all(he_ctx* h) {
  free_profile(h);
  void* ptrs[] = {h->K, h->V, h->W, h->codes, h->evicted, h->counters, h->err, h->partials,
                  h->score, h->vs, h->cstar, h->tauv,
                  h->uo, h->sq, h->sk, h->sv, h->sout};
  for (void* p : ptrs)
    if (p) cudaFree(p);
}

StepParams base_params(const he_ctx* h) {
  StepParams p{};
  p.K = h->K;
  p.V = h->V;
  p.codes = h->codes;
  p.W = h->W;
  p.evicted = h->evicted;
  p.partials = h->partials;
  p.counters = h->counters;
  p.err = h->err;
  p.U = h->U;
  p.kv_heads = h->cfg.kv_heads;
  p.budget = h->rows;
  p.lbudget = h->cfg.budget;
  p.chunk = h->chunk;
  p.cstar = h->cstar;
  p.occ = h->occupancy;
  p.tile = h->kern.tile;
  p.tpu = (h->occupancy + p.tile - 1) / p.tile;
  p.total_tiles = h->U * p.tpu;
  p.bits = h->cfg.bits;
  p.code_stride = h->code_stride;
  p.append_slot = h->occupancy < h->rows ? h->occupancy : -1;  // (or staged)
  p.qscale = (float)(1.4426950408889634 / std::sqrt((double)h->cfg.head_dim));
  p.vs = h->vs;
  p.vs_stride = h->vs_stride;
  p.tau = h->cfg.threshold;
  p.tauv = h->tauv;
  p.decay = h->cfg.decay;
  p.score = h->score;
  p.evlog = h->evlog;
  p.evcnt = h->evcnt;
  p.evcap = h->evcap;
  p.dist = h->dist;
  return p;
}

// Codes (or, with proj, the projections) of rows of x; unit_tau: the rows are
// the units' cache rows (per_unit each), coded with the handle's per-bit
// thresholds when it has them.
int launch_codes(he_ctx* h, const void* x, int64_t rows, int64_t per_unit, int64_t x_unit_rows,
                 unsigned char* out, int64_t out_unit_bytes, cudaStream_t s,
                 bool unit_tau = true, float* proj = nullptr) {
  if (rows == 0) return HE_OK;
  const int vb = he::kAuxThreads / h->cfg.bits;
  int64_t blocks = (rows + vb - 1) / vb;
  const int64_t cap = (int64_t)h->num_sms * 16;
  if (blocks > cap) blocks = cap;
  const void* W = h->W;
  int bits = h->cfg.bits;
  float tau = h->cfg.threshold;
  const float* tauv = unit_tau ? h->tauv : nullptr;
  void* args[] = {(void*)&x,    (void*)&rows, (void*)&per_unit, (void*)&x_unit_rows,
                  (void*)&W,    (void*)&bits, (void*)&tau,      (void*)&tauv,
                  (void*)&out,  (void*)&out_unit_bytes, (void*)&proj};
  HE_TRY(h, cudaLaunchKernel(h->kern.code, dim3((unsigned)blocks), dim3(he::kAuxThreads), args, 0,
                             s));
  return HE_OK;
}

// Scratch of the fill's key projections: at most this many bytes at a time
// (or one unit's, if that is more).
constexpr int64_t kMedianScratchBytes = (int64_t)1 << 30;

// Per-bit lower-median thresholds of the n filled keys of every unit (n >= 1)
// into h->tauv: the keys' projections (the code's arithmetic) into a scratch
// buffer, a group of units at a time, then one radix select per (unit, bit).
int fill_median_thresholds(he_ctx* h, int64_t n, cudaStream_t s) {
  const int bits = h->cfg.bits;
  const int64_t per_unit = (int64_t)bits * n * (int64_t)sizeof(float);
  int64_t group = kMedianScratchBytes / per_unit;
  if (group < 1) group = 1;
  if (group > h->U) group = h->U;
  float* proj = nullptr;
  if (g_alloc_limit != 0 && (uint64_t)(group * per_unit) > g_alloc_limit) return HE_ENOMEM;
  if (cudaMallocAsync((void**)&proj, (size_t)(group * per_unit), s) != cudaSuccess) {
    (void)cudaGetLastError();
    return HE_ENOMEM;
  }
  int rc = HE_OK;
  const size_t unit_bytes = (size_t)h->rows * h->cfg.head_dim * h->eb;
  for (int64_t u0 = 0; u0 < h->U && rc == HE_OK; u0 += group) {
    const int64_t g = group < h->U - u0 ? group : h->U - u0;
    const void* x = reinterpret_cast<const unsigned char*>(h->K) + (size_t)u0 * unit_bytes;
    rc = launch_codes(h, x, g * n, n, h->rows, nullptr, 0, s, false, proj);
    if (rc != HE_OK) break;
    float* tau = h->tauv + u0 * bits;
    void* args[] = {(void*)&proj, (void*)&n, (void*)&tau};
    if (cudaLaunchKernel((const void*)&he::median_select_kernel, dim3((unsigned)(g * bits)),
                         dim3(he::kAuxThreads), args, 0, s) != cudaSuccess)
      rc = fail_cuda(h, cudaGetLastError());
  }
  if (cudaFreeAsync(proj, s) != cudaSuccess && rc == HE_OK) rc = fail_cuda(h, cudaGetLastError());
  return rc;
}

}  // namespace

extern "C" {

const char* he_strerror(int code) {
  switch (code) {
    case HE_OK: return "ok";
    case HE_EINVAL: return "invalid argument (configuration, size, pointer or alignment)";
    case HE_ENOTFILLED: return "the cache has not been filled (call he_fill first)";
    case HE_ECUDA: return "a CUDA call failed; the handle refuses further work";
    case HE_ENOMEM: return "device memory allocation failed";
    case HE_EDEVICE: return "a kernel reported an internal error (a wait gave up)";
    default: return "unknown error code";
  }
}

int he_create(const he_cfg* cfg, he_handle* out) {
  if (!cfg || !out) return HE_EINVAL;
  *out = nullptr;
  const he_cfg c = *cfg;
  if (c.batch < 1 || c.heads < 1 || c.kv_heads < 1 || c.heads % c.kv_heads != 0) return HE_EINVAL;
  if (c.bits != 8 && c.bits != 16 && c.bits != 32 && c.bits != 64) return HE_EINVAL;
  if (c.budget < 1 || c.budget > (1 << 24)) return HE_EINVAL;
  if (c.v_format != HE_VFMT_ELEM &&
      !((c.v_format == HE_VFMT_INT8 || c.v_format == HE_VFMT_FP8) && c.dtype == HE_DTYPE_BF16))
    return HE_EINVAL;
  if (!std::isfinite(c.threshold) || !(c.decay >= 0.0f && c.decay <= 1.0f)) return HE_EINVAL;
  if (c.chunk < 0 || c.chunk > he::kMaxChunk) return HE_EINVAL;
  if (c.tau_mode != HE_TAU_FIXED && c.tau_mode != HE_TAU_MEDIAN) return HE_EINVAL;
  if (c.engine != HE_ENGINE_PIPELINE &&
      !(c.engine == HE_ENGINE_FUSED && c.dtype == HE_DTYPE_BF16 && c.decay == 0.0f &&
        c.v_format == HE_VFMT_ELEM && c.chunk <= 1))
    return HE_EINVAL;
  const int chunk = c.chunk > 1 ? c.chunk : 1;
  if (chunk > 1 && (c.dtype != HE_DTYPE_BF16 || c.v_format != HE_VFMT_ELEM || c.decay != 0.0f ||
                    c.budget % chunk != 0))
    return HE_EINVAL;
  const int rows = c.budget + chunk - 1;
  if ((int64_t)c.batch * c.kv_heads > 65536) return HE_EINVAL;
  const int G = c.heads / c.kv_heads;
  Kernels kern;
  const int vfmt = c.v_format == HE_VFMT_INT8 ? he::kVqInt8
                   : c.v_format == HE_VFMT_FP8 ? he::kVqFp8
                                               : 0;
  const bool vq = vfmt != 0;
  if (!pick_kernels(c.dtype, c.head_dim, G, vfmt, &kern)) return HE_EINVAL;
  const int64_t U = (int64_t)c.batch * c.kv_heads;
  if (U * ((rows + kern.tile - 1) / kern.tile) > INT32_MAX) return HE_EINVAL;
  if (U * rows + kern.tile >= ((int64_t)1 << 31)) return HE_EINVAL;  // TMA row coordinate

  he_ctx* h = new (std::nothrow) he_ctx();
  if (!h) return HE_ENOMEM;
  h->cfg = c;
  h->G = G;
  h->U = (int)U;
  h->eb = c.dtype == HE_DTYPE_FP32 ? 4 : 2;
  h->code_bytes = c.bits / 8;
  h->code_stride = (int)(((int64_t)rows * h->code_bytes + 15) / 16 * 16);
  h->kern = kern;
  h->vq = vq;
  h->chunk = chunk;
  h->rows = rows;
  h->vs_stride = (rows + 63) / 64 * 64;
  if (cudaGetDevice(&h->device) != cudaSuccess) {
    (void)cudaGetLastError();
    delete h;
    return HE_ECUDA;
  }
  int rc = HE_OK;
  do {
    if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) !=
        cudaSuccess) { rc = HE_ECUDA; break; }
    if (cudaFuncSetAttribute(kern.step, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kern.step_smem) != cudaSuccess) { rc = HE_ECUDA; break; }
    if (chunk > 1 &&
        (cudaFuncSetAttribute(kern.prep_chunk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kern.prep_smem) != cudaSuccess ||
         cudaFuncSetAttribute(kern.prep_chunk, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
         cudaFuncSetAttribute(kern.merge_chunk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kern.merge_smem) != cudaSuccess ||
         cudaFuncSetAttribute(kern.merge_chunk, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
         cudaFuncSetAttribute(kern.merge_chunk_mu, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kern.merge_smem) != cudaSuccess ||
         cudaFuncSetAttribute(kern.merge_chunk_mu, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)) {
      rc = HE_ECUDA;
      break;
    }
    // the three kernels of the bf16 pipeline run side by side on an SM: give
    // them one L1/shared split so that none waits for the SM to reconfigure
    if (kern.tc &&
        (cudaFuncSetAttribute(kern.prep, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kern.prep_smem) != cudaSuccess ||
         cudaFuncSetAttribute(kern.merge, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kern.merge_smem) != cudaSuccess ||
         cudaFuncSetAttribute(kern.step, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
         cudaFuncSetAttribute(kern.prep, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
         cudaFuncSetAttribute(kern.prep_mem, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kern.prep_smem) != cudaSuccess ||
         cudaFuncSetAttribute(kern.prep_mem, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
         cudaFuncSetAttribute(kern.merge, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
         (kern.merge_mu != nullptr &&
          (cudaFuncSetAttribute(kern.merge_mu, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kern.merge_smem) != cudaSuccess ||
           cudaFuncSetAttribute(kern.merge_mu, cudaFuncAttributePreferredSharedMemoryCarveout,
                                (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)))) {
      rc = HE_ECUDA;
      break;
    }

    h->fused = c.engine == HE_ENGINE_FUSED && kern.fused != nullptr;
    if (h->fused &&
        (cudaFuncSetAttribute(kern.fused, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kern.fused_smem) != cudaSuccess ||
         cudaFuncSetAttribute(kern.fused, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)) {
      rc = HE_ECUDA;
      break;
    }
    if ((h->fused ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                        &h->ctas_per_sm, kern.fused, kern.fused_threads, kern.fused_smem)
                  : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                        &h->ctas_per_sm, kern.step, kern.step_threads, kern.step_smem)) !=
            cudaSuccess ||
        h->ctas_per_sm < 1) { rc = HE_ECUDA; break; }
    h->max_ctas = h->num_sms * h->ctas_per_sm;
    // one spare tile of rows after the last unit keeps every tile load in bounds;
    // the cache starts zeroed so rows no token has written are finite
    const size_t cache = ((size_t)U * rows + kern.tile) * c.head_dim * h->eb;
    const size_t vcache = vq ? ((size_t)U * rows + kern.tile) * c.head_dim : cache;
    const size_t nrec = (size_t)h->max_ctas + (size_t)U;
    struct { void** p; size_t bytes; } allocs[] = {
        {&h->K, cache},
        {&h->V, vcache},
        {(void**)&h->vs, vq ? (size_t)U * h->vs_stride * sizeof(float) : 0},
        {&h->W, (size_t)c.head_dim * c.bits * h->eb},
        {(void**)&h->codes, (size_t)U * h->code_stride},
        {(void**)&h->evicted, (size_t)U * sizeof(int32_t)},
        {(void**)&h->counters, (size_t)U * sizeof(int32_t)},
        {(void**)&h->err, sizeof(int32_t)},
        {(void**)&h->partials,
         nrec * (h->fused ? kern.fused_rec_floats : kern.rec_floats) * sizeof(float)},
        {(void**)&h->uo, (size_t)U * sizeof(he::UnitOut)},
        {(void**)&h->score, c.decay > 0.0f ? (size_t)U * rows * sizeof(float) : 0},
        {(void**)&h->cstar, chunk > 1 ? (size_t)U * kern.chunk_floats * sizeof(float) : 0},
        {(void**)&h->tauv,
         c.tau_mode == HE_TAU_MEDIAN ? (size_t)U * c.bits * sizeof(float) : 0},
    };
    uint64_t total = 0;
    for (auto& a : allocs) total += a.bytes;
    if (g_alloc_limit != 0 && total > g_alloc_limit) {
      rc = HE_ENOMEM;
      break;
    }
    for (auto& a : allocs) {
      if (a.bytes == 0) continue;
      if (cudaMalloc(a.p, a.bytes) != cudaSuccess) {
        (void)cudaGetLastError();
        rc = HE_ENOMEM;
        break;
      }
    }
    if (rc != HE_OK) break;
    if (cudaMemset(h->K, 0, cache) != cudaSuccess || cudaMemset(h->V, 0, vcache) != cudaSuccess ||
        (vq && cudaMemset(h->vs, 0, (size_t)U * h->vs_stride * sizeof(float)) != cudaSuccess) ||
        cudaMemset(h->codes, 0, (size_t)U * h->code_stride) != cudaSuccess ||
        cudaMemset(h->counters, 0, (size_t)U * sizeof(int32_t)) != cudaSuccess ||
        cudaMemset(h->uo, 0, (size_t)U * sizeof(he::UnitOut)) != cudaSuccess ||
        cudaMemset(h->err, 0, sizeof(int32_t)) != cudaSuccess ||
        cudaMemset(h->evicted, 0xFF, (size_t)U * sizeof(int32_t)) != cudaSuccess ||
        (h->tauv && cudaMemset(h->tauv, 0, (size_t)U * c.bits * sizeof(float)) != cudaSuccess)) {
      rc = HE_ECUDA;
      break;
    }
    const uint64_t mrows = (uint64_t)U * rows + kern.tile;
    if (kern.tc && (!encode_cache_map(&h->tmK, h->K, mrows, c.head_dim, kern.tile) ||
                     !(vq ? encode_vq_map(&h->tmV, h->V, mrows, c.head_dim, kern.tile)
                          : encode_cache_map(&h->tmV, h->V, mrows, c.head_dim, kern.tile)))) {
      rc = HE_ECUDA;
      break;
    }
    const int n = c.head_dim * c.bits;
    he::projection_kernel<<<(n + 255) / 256, 256>>>(c.seed, c.head_dim, c.bits,
                                                   c.dtype == HE_DTYPE_FP32 ? 1 : 0, h->W);
    if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
      rc = HE_ECUDA;
      break;
    }
  } while (0);
  if (rc != HE_OK) {
    (void)cudaGetLastError();
    free_all(h);
    delete h;
    return rc;
  }
  *out = h;
  return HE_OK;
}

int he_destroy(he_handle h) {
  if (!h) return HE_OK;
  DeviceGuard g(h->device);
  cudaDeviceSynchronize();
  (void)cudaGetLastError();
  free_all(h);
  delete h;
  return HE_OK;
}

int he_fill(he_handle h, const void* K, const void* V, int32_t n, void* stream) {
  if (!h || n < 0 || n > h->cfg.budget) return HE_EINVAL;
  if (n > 0 && (!K || !V || !aligned16(K) || !aligned16(V))) return HE_EINVAL;
  if (h->sticky) return h->sticky;
  DeviceGuard g(h->device);
  if (!g.ok) return fail_cuda(h, cudaErrorInvalidDevice);
  cudaStream_t s = (cudaStream_t)stream;
  const size_t row = (size_t)h->cfg.head_dim * h->eb;
  // a fill that fails part-way (the threshold scratch) leaves the handle
  // unfilled rather than mixing the new rows with the old codes
  h->filled = false;
  if (n > 0) {
    HE_TRY(h, cudaMemcpy2DAsync(h->K, (size_t)h->rows * row, K, (size_t)n * row,
                                (size_t)n * row, (size_t)h->U, cudaMemcpyDeviceToDevice, s));
    if (h->vq) {  // value rows quantised into the byte cache
      const int64_t rows = (int64_t)h->U * n;
      int64_t blocks = (rows + 7) / 8;
      if (blocks > (int64_t)h->num_sms * 16) blocks = (int64_t)h->num_sms * 16;
      int nn = n, budget = h->rows, vstride = h->vs_stride;
      uint8_t* Vq = reinterpret_cast<uint8_t*>(h->V);
      float* vs = h->vs;
      void* args[] = {(void*)&V, (void*)&rows, (void*)&nn, (void*)&budget, (void*)&Vq,
                      (void*)&vs, (void*)&vstride};
      HE_TRY(h, cudaLaunchKernel(h->kern.vq_fill, dim3((unsigned)blocks), dim3(256), args, 0, s));
    } else {
      HE_TRY(h, cudaMemcpy2DAsync(h->V, (size_t)h->rows * row, V, (size_t)n * row,
                                  (size_t)n * row, (size_t)h->U, cudaMemcpyDeviceToDevice, s));
    }
    if (h->tauv) {
      const int rc = fill_median_thresholds(h, n, s);
      if (rc != HE_OK) return rc;
    }
    const int rc = launch_codes(h, h->K, (int64_t)h->U * n, n, h->rows, h->codes,
                                h->code_stride, s);
    if (rc != HE_OK) return rc;
  } else if (h->tauv) {  // no keys: the sign test
    HE_TRY(h, cudaMemsetAsync(h->tauv, 0, (size_t)h->U * h->cfg.bits * sizeof(float), s));
  }
  HE_TRY(h, cudaMemsetAsync(h->counters, 0, (size_t)h->U * sizeof(int32_t), s));
  if (h->uo) HE_TRY(h, cudaMemsetAsync(h->uo, 0, (size_t)h->U * sizeof(he::UnitOut), s));
  if (h->score)  // filled slots start with no accumulated score
    HE_TRY(h, cudaMemsetAsync(h->score, 0, (size_t)h->U * h->rows * sizeof(float), s));
  // The first step after a fill reads the (zeroed) eviction key for the slot
  // the step before it wrote, and with chunk eviction fetches no tile before it
  // waits: the same parameters a step gets after an evicting step, so that a
  // step sequence captured from here (whole eviction cycles, an even number
  // of steps) replays on the cache state it leaves.
  h->prev_w1 = -1;
  h->nopre = h->chunk > 1 ? 1 : 0;
  h->prev_tpu = h->prev_nc = h->prev_e = h->prev_t1 = 0;  // no hash warp folds a key
  h->occupancy = n;
  h->filled = true;
  return HE_OK;
}

int he_step(he_handle h, const void* q, const void* k, const void* v, float* out, void* stream) {
  if (!h || !q || !k || !v || !out) return HE_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return HE_EINVAL;
  if (h->sticky) return h->sticky;
  if (!h->filled) return HE_ENOTFILLED;
  DeviceGuard g(h->device);
  if (!g.ok) return fail_cuda(h, cudaErrorInvalidDevice);
  StepParams p = base_params(h);
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
#ifdef HE_TIMELINE
  static int tl_counter = 0;
  p.tl_step = (tl_counter++) & 7;
#endif
  cudaStream_t s = (cudaStream_t)stream;
  // kernel timing mode: events between the launches serialise the kernels
  cudaEvent_t* ev = h->prof_n < h->prof_cap ? &h->prof_ev[4 * (size_t)h->prof_n] : nullptr;
  if (ev) HE_TRY(h, cudaEventRecord(ev[0], s));
  const int stream_ctas = p.total_tiles == 0
                              ? 0
                              : (p.total_tiles < h->max_ctas ? p.total_tiles : h->max_ctas);
  if (h->fused) {
    // the whole step in one kernel (he_fused.cuh); an empty cache runs one CTA per unit
    p.uo = h->uo;
    p.kpar = h->kpar;
    p.prev_w1 = h->prev_w1;
    p.nopre = 0;
    p.prev_tpu = h->prev_tpu;
    p.prev_nc = h->prev_nc;
    p.prev_e = h->prev_e;
    p.prev_t1 = h->prev_t1;
    // every CTA of the step passes its dependency wait at about the same time
    // (the previous step's CTAs all finish before it returns): an even split
    const int64_t TT = p.total_tiles;
    if (kLateTilesFused > 0.0 && stream_ctas == h->max_ctas && TT > stream_ctas) {
      const int64_t late = h->U < h->max_ctas ? h->U : h->max_ctas;
      const int64_t E = (int64_t)h->max_ctas - late;
      if (E > 0 && E < stream_ctas) {
        const double per = ((double)TT + (double)(stream_ctas - E) * kLateTilesFused) / stream_ctas;
        int64_t T1 = (int64_t)std::llround(per * (double)E);
        if (T1 > TT - (stream_ctas - E)) T1 = TT - (stream_ctas - E);  // a tile per late CTA
        if (T1 < E) T1 = E;
        p.split_e = (int32_t)E;
        p.split_t1 = (int32_t)T1;
      }
    }
    const int grid = stream_ctas == 0 ? h->U : stream_ctas;
    void* sa[] = {(void*)&p, (void*)&h->tmK, (void*)&h->tmV};
    HE_TRY(h, launch_pdl(h->kern.fused, dim3(grid), dim3(h->kern.fused_threads),
                         (size_t)h->kern.fused_smem, s, sa));
    if (ev) {
      HE_TRY(h, cudaEventRecord(ev[1], s));
      HE_TRY(h, cudaEventRecord(ev[2], s));
    }
    h->prev_tpu = p.tpu;
    h->prev_nc = stream_ctas;
    h->prev_e = p.split_e;
    h->prev_t1 = p.split_t1;
  } else if (!h->kern.tc) {
    const int grid = stream_ctas == 0 ? h->U : stream_ctas;
    void* args[] = {(void*)&p};
    HE_TRY(h, cudaLaunchKernel(h->kern.step, dim3(grid), dim3(h->kern.step_threads), args,
                               (size_t)h->kern.step_smem, s));
    if (ev) {
      HE_TRY(h, cudaEventRecord(ev[1], s));
      HE_TRY(h, cudaEventRecord(ev[2], s));
    }
  } else {
    const bool full = p.append_slot < 0;
    const bool ch = h->chunk > 1;
    // prep items: code slots of the budget per CTA (the chunk path: whole chunks)
    const int item = ch ? he::chunk_item_slots(h->chunk, h->cfg.bits)
                        : he::prep_item_slots(h->cfg.bits);
    int splits = full ? (h->cfg.budget + item - 1) / item : 1;
    if (splits < 1) splits = 1;
    he::UnitOut* uo = h->uo;
    p.uo = uo;
    p.kpar = h->kpar;
    p.prev_w1 = h->prev_w1;
    p.nopre = h->nopre;
    // two-group stream-K split (he::TileSplit): when every CTA slot is used,
    // the CTAs placed on SMs free of the previous step's merge CTAs (one per
    // unit, at most one per SM) start first and take more tiles
    const int64_t TT = p.total_tiles;
    if (stream_ctas == h->max_ctas && TT > stream_ctas) {
      const int mc = h->merge_ctas > 0 ? h->merge_ctas : h->U;
      const int merge_sms = mc < h->num_sms ? mc : h->num_sms;
      const int64_t E = (int64_t)h->ctas_per_sm * (h->num_sms - merge_sms);
      if (E > 0 && E < stream_ctas) {
        const double per = ((double)TT + (double)(stream_ctas - E) * kLateTiles) / stream_ctas;
        int64_t T1 = (int64_t)std::llround(per * (double)E);
        if (T1 > TT - (stream_ctas - E)) T1 = TT - (stream_ctas - E);  // a tile per late CTA
        if (T1 < E) T1 = E;
        p.split_e = (int32_t)E;
        p.split_t1 = (int32_t)T1;
      }
    }
    // partials per unit: at most ceil(tiles per unit / fewest tiles of a CTA) + 1
    int nmax = 0;
    if (TT > 0 && stream_ctas > 0) {
      const he::TileSplit sp{TT, stream_ctas, p.split_e, p.split_t1};
      int64_t fewest = TT;
      for (int64_t c : {(int64_t)0, (int64_t)stream_ctas - 1})
        fewest = std::min(fewest, sp.begin(c + 1) - sp.begin(c));
      if (p.split_e > 0) fewest = std::min(fewest, sp.begin(p.split_e) - sp.begin(p.split_e - 1));
      nmax = (int)((p.tpu + fewest - 1) / fewest) + 1;
    }
    // more partials than merge holds in registers: its loads take longest, so
    // it releases the next step only once they are issued
    p.late_release = nmax > he::kMergeRegs ? 1 : 0;
    if (stream_ctas > 0) {
      void* sa[] = {(void*)&p, (void*)&h->tmK, (void*)&h->tmV};
      HE_TRY(h, launch_pdl(h->kern.step, dim3(stream_ctas), dim3(h->kern.step_threads),
                           (size_t)h->kern.step_smem, s, sa));
    }
    if (ev) HE_TRY(h, cudaEventRecord(ev[1], s));
    int first_of_step = stream_ctas > 0 ? 0 : 1;
    void* pa[] = {(void*)&p, (void*)&uo, (void*)&splits, (void*)&first_of_step};
    const int prep_ctas = h->U * splits < h->num_sms ? h->U * splits : h->num_sms;
    HE_TRY(h, launch_pdl(ch ? h->kern.prep_chunk : (h->score ? h->kern.prep_mem : h->kern.prep),
                         dim3(prep_ctas),
                         dim3(he::kPrepThreads),
                         (size_t)h->kern.prep_smem, s, pa));
    if (ev) HE_TRY(h, cudaEventRecord(ev[2], s));
    int sc = stream_ctas;
    // several units per merge CTA only when the units outnumber the SMs (one
    // wave of merge CTAs instead of several); else one unit per CTA
    int msmem = 0, nq = 1, upc = 1;
    const bool multi = h->U > h->num_sms;
    const int mthreads = h->kern.merge_cfg(nmax, h->U, multi, &nq, &upc, &msmem);
    void* ma[] = {(void*)&p, (void*)&uo, (void*)&sc, (void*)&nq};
    const void* mfn = ch ? (upc > 1 ? h->kern.merge_chunk_mu : h->kern.merge_chunk)
                         : (upc > 1 ? h->kern.merge_mu : h->kern.merge);
    HE_TRY(h, launch_pdl(mfn, dim3(h->U / upc), dim3(mthreads), (size_t)msmem, s, ma));
    h->merge_ctas = h->U / upc;
  }
  if (ev) {
    HE_TRY(h, cudaEventRecord(ev[3], s));
    h->prof_n += 1;
  }
  if (h->kern.tc) {
    h->prev_w1 = p.append_slot >= 0 ? p.append_slot + 1 : -1;
    h->nopre = h->chunk > 1 && p.append_slot < 0;  // a chunk eviction moved c rows
    h->kpar ^= 1;
  }
  // append (or stage); a chunk eviction returns the cache to its budget
  if (h->occupancy < h->rows)
    h->occupancy += 1;
  else
    h->occupancy = h->cfg.budget;
  return HE_OK;
}

int he_step_host(he_handle h, const void* q, const void* k, const void* v, float* out,
                 void* stream) {
  if (!h || !q || !k || !v || !out) return HE_EINVAL;
  if (h->sticky) return h->sticky;
  if (!h->filled) return HE_ENOTFILLED;
  DeviceGuard g(h->device);
  if (!g.ok) return fail_cuda(h, cudaErrorInvalidDevice);
  const size_t qb = vec_bytes(h, h->cfg.heads), kb = vec_bytes(h, h->cfg.kv_heads);
  const size_t ob = (size_t)h->cfg.batch * h->cfg.heads * h->cfg.head_dim * sizeof(float);
  if (!h->sq) {
    if (cudaMalloc(&h->sq, qb) != cudaSuccess || cudaMalloc(&h->sk, kb) != cudaSuccess ||
        cudaMalloc(&h->sv, kb) != cudaSuccess || cudaMalloc((void**)&h->sout, ob) != cudaSuccess) {
      (void)cudaGetLastError();
      return HE_ENOMEM;
    }
  }
  cudaStream_t s = (cudaStream_t)stream;
  HE_TRY(h, cudaMemcpyAsync(h->sq, q, qb, cudaMemcpyHostToDevice, s));
  HE_TRY(h, cudaMemcpyAsync(h->sk, k, kb, cudaMemcpyHostToDevice, s));
  HE_TRY(h, cudaMemcpyAsync(h->sv, v, kb, cudaMemcpyHostToDevice, s));
  const int rc = he_step(h, h->sq, h->sk, h->sv, h->sout, stream);
  if (rc != HE_OK) return rc;
  HE_TRY(h, cudaMemcpyAsync(out, h->sout, ob, cudaMemcpyDeviceToHost, s));
  HE_TRY(h, cudaStreamSynchronize(s));
  return HE_OK;
}

static int check_device_error(he_ctx* h) {
  int32_t e = 0;
  HE_TRY(h, cudaDeviceSynchronize());
  HE_TRY(h, cudaMemcpy(&e, h->err, sizeof e, cudaMemcpyDeviceToHost));
  if (e != 0) {
    h->sticky = HE_EDEVICE;
    return HE_EDEVICE;
  }
  return HE_OK;
}

int he_last_evicted(he_handle h, int32_t* host_slots) {
  if (!h || !host_slots) return HE_EINVAL;
  DeviceGuard g(h->device);
  const int rc = check_device_error(h);
  if (rc != HE_OK) return rc;
  HE_TRY(h, cudaMemcpy(host_slots, h->evicted, (size_t)h->U * sizeof(int32_t),
                       cudaMemcpyDeviceToHost));
  return h->sticky;
}

int he_read_state(he_handle h, void* K, void* V, void* codes, int32_t* occupancy) {
  if (!h) return HE_EINVAL;
  DeviceGuard g(h->device);
  const int rc = check_device_error(h);
  if (rc != HE_OK) return rc;
  const size_t cache = (size_t)h->U * h->rows * h->cfg.head_dim * h->eb;
  if (K) HE_TRY(h, cudaMemcpy(K, h->K, cache, cudaMemcpyDeviceToHost));
  if (V) HE_TRY(h, cudaMemcpy(V, h->V, h->vq ? cache / h->eb : cache, cudaMemcpyDeviceToHost));
  if (codes) {
    const size_t w = (size_t)h->rows * h->code_bytes;
    HE_TRY(h, cudaMemcpy2D(codes, w, h->codes, (size_t)h->code_stride, w, (size_t)h->U,
                           cudaMemcpyDeviceToHost));
  }
  if (occupancy) *occupancy = h->occupancy;
  return h->sticky;
}

int he_get_projection(he_handle h, void* host_W) {
  if (!h || !host_W) return HE_EINVAL;
  DeviceGuard g(h->device);
  HE_TRY(h, cudaDeviceSynchronize());
  HE_TRY(h, cudaMemcpy(host_W, h->W, (size_t)h->cfg.head_dim * h->cfg.bits * h->eb,
                       cudaMemcpyDeviceToHost));
  return HE_OK;
}

int he_codes(he_handle h, const void* x, int32_t n, void* codes, void* stream) {
  if (!h || n < 0 || h->tauv) return HE_EINVAL;
  if (n > 0 && (!x || !codes || !aligned16(x) || !aligned16(codes))) return HE_EINVAL;
  if (h->sticky) return h->sticky;
  DeviceGuard g(h->device);
  return launch_codes(h, x, n, n > 0 ? n : 1, n, (unsigned char*)codes,
                      (int64_t)n * h->code_bytes, (cudaStream_t)stream, false);
}

int he_scores(he_handle h, const void* q, int32_t* dist, void* stream) {
  if (!h || !q || !dist || !aligned16(q) || !aligned16(dist)) return HE_EINVAL;
  if (h->sticky) return h->sticky;
  if (!h->filled) return HE_ENOTFILLED;
  DeviceGuard g(h->device);
  StepParams p = base_params(h);
  p.q = q;
  void* args[] = {(void*)&p, (void*)&dist};
  HE_TRY(h, cudaLaunchKernel(h->kern.score, dim3(h->U), dim3(he::kAuxThreads), args, 0,
                             (cudaStream_t)stream));
  return HE_OK;
}

int he_recompute_count(he_handle h, int64_t* total) {
  if (!h || !total) return HE_EINVAL;
  DeviceGuard g(h->device);
  *total = 0;
  if (!h->kern.tc) return HE_OK;
  HE_TRY(h, cudaDeviceSynchronize());
  int32_t* host = new (std::nothrow) int32_t[h->U];
  if (!host) return HE_ENOMEM;
  const cudaError_t e = cudaMemcpy(host, h->counters, (size_t)h->U * sizeof(int32_t),
                                   cudaMemcpyDeviceToHost);
  if (e == cudaSuccess)
    for (int i = 0; i < h->U; ++i) *total += host[i];
  delete[] host;
  if (e != cudaSuccess) return fail_cuda(h, e);
  return HE_OK;
}

int he_set_alloc_limit(uint64_t bytes) {
  g_alloc_limit = bytes;
  return HE_OK;
}

int he_wait_probe(he_handle h, uint32_t limit_us, void* stream) {
  if (!h || limit_us < 1 || limit_us > 1000000) return HE_EINVAL;
  if (h->sticky) return h->sticky;
  DeviceGuard g(h->device);
  if (!g.ok) return fail_cuda(h, cudaErrorInvalidDevice);
  wait_probe_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(h->err, (uint64_t)limit_us * 1000u);
  HE_TRY(h, cudaGetLastError());
  return HE_OK;
}

int he_read_scores(he_handle h, float* host_scores) {
  if (!h || !host_scores || !h->score) return HE_EINVAL;
  if (h->sticky) return h->sticky;
  DeviceGuard g(h->device);
  if (!g.ok) return fail_cuda(h, cudaErrorInvalidDevice);
  const int rc = check_device_error(h);
  if (rc != HE_OK) return rc;
  HE_TRY(h, cudaMemcpy(host_scores, h->score, (size_t)h->U * h->rows * sizeof(float),
                       cudaMemcpyDeviceToHost));
  return HE_OK;
}

int he_read_vscales(he_handle h, float* host_scales) {
  if (!h || !host_scales || !h->vq) return HE_EINVAL;
  if (h->sticky) return h->sticky;
  DeviceGuard g(h->device);
  if (!g.ok) return fail_cuda(h, cudaErrorInvalidDevice);
  const int rc = check_device_error(h);
  if (rc != HE_OK) return rc;
  const size_t w = (size_t)h->rows * sizeof(float);
  HE_TRY(h, cudaMemcpy2D(host_scales, w, h->vs, (size_t)h->vs_stride * sizeof(float), w,
                         (size_t)h->U, cudaMemcpyDeviceToHost));
  return HE_OK;
}

int he_read_thresholds(he_handle h, float* host_tau) {
  if (!h || !host_tau) return HE_EINVAL;
  const size_t n = (size_t)h->U * h->cfg.bits;
  if (!h->tauv) {
    for (size_t i = 0; i < n; ++i) host_tau[i] = h->cfg.threshold;
    return HE_OK;
  }
  if (h->sticky) return h->sticky;
  DeviceGuard g(h->device);
  if (!g.ok) return fail_cuda(h, cudaErrorInvalidDevice);
  const int rc = check_device_error(h);
  if (rc != HE_OK) return rc;
  HE_TRY(h, cudaMemcpy(host_tau, h->tauv, n * sizeof(float), cudaMemcpyDeviceToHost));
  return HE_OK;
}

int he_occupancy(he_handle h, int32_t* occupancy) {
  if (!h || !occupancy) return HE_EINVAL;
  *occupancy = h->occupancy;
  return HE_OK;
}

int he_step_bytes(he_handle h, uint64_t* bytes) {
  if (!h || !bytes) return HE_EINVAL;
  const uint64_t U = (uint64_t)h->U, B = (uint64_t)h->cfg.budget, D = (uint64_t)h->cfg.head_dim;
  const uint64_t e = (uint64_t)h->eb, w = (uint64_t)h->code_bytes;
  const uint64_t Bt = (uint64_t)h->cfg.batch, H = (uint64_t)h->cfg.heads;
  const uint64_t kv = h->vq ? D * e + D + 4 : 2 * D * e;  // bytes of one slot's key and value
  // chunk eviction: over a cycle of c steps the resident rows average
  // B + (c - 1) / 2, and the c - 1 staged rows are read and written once more
  const uint64_t c = (uint64_t)h->chunk;
  *bytes = U * (2 * B + c - 1) / 2 * (kv + w)  // retained K, V and codes read
           + U * (kv + w)                 // the overwritten slot
           + U * 2 * (c - 1) * (kv + w) / c  // staged rows moved into the evicted chunk
           + Bt * H * D * e + U * 2 * D * e  // q, k, v in
           + Bt * H * D * 4                // out
           + D * (uint64_t)h->cfg.bits * e;  // W
  if (h->score) *bytes += U * B * 2 * sizeof(float);  // scores read and written
  return HE_OK;
}

int he_profile_start(he_handle h, int32_t max_steps) {
  if (!h || max_steps < 1 || max_steps > (1 << 16)) return HE_EINVAL;
  if (h->sticky) return h->sticky;
  DeviceGuard g(h->device);
  if (!g.ok) return fail_cuda(h, cudaErrorInvalidDevice);
  free_profile(h);
  h->prof_ev.assign(4 * (size_t)max_steps, nullptr);
  for (cudaEvent_t& e : h->prof_ev) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      e = nullptr;
      free_profile(h);
      (void)cudaGetLastError();
      return HE_ENOMEM;
    }
  }
  h->prof_cap = max_steps;
  h->prof_n = 0;
  return HE_OK;
}

int he_profile_stop(he_handle h, float* ms, int32_t* steps) {
  if (!h || !ms || !steps) return HE_EINVAL;
  if (h->sticky) return h->sticky;
  DeviceGuard g(h->device);
  if (!g.ok) return fail_cuda(h, cudaErrorInvalidDevice);
  double sum[4] = {0, 0, 0, 0};
  const int n = h->prof_n;
  for (int i = 0; i < n; ++i) {
    cudaEvent_t* ev = &h->prof_ev[4 * (size_t)i];
    float t = 0.f;
    for (int k = 0; k < 3; ++k) {
      HE_TRY(h, cudaEventSynchronize(ev[k + 1]));
      HE_TRY(h, cudaEventElapsedTime(&t, ev[k], ev[k + 1]));
      sum[k] += t;
    }
    HE_TRY(h, cudaEventElapsedTime(&t, ev[0], ev[3]));
    sum[3] += t;
  }
  for (int k = 0; k < 4; ++k) ms[k] = (float)sum[k];
  *steps = n;
  free_profile(h);
  return HE_OK;
}

int he_set_evict_log(he_handle h, int32_t* log, int32_t* count, int32_t capacity) {
  if (!h) return HE_EINVAL;
  if (log != nullptr && (count == nullptr || capacity < 1)) return HE_EINVAL;
  h->evlog = log;
  h->evcnt = log ? count : nullptr;
  h->evcap = log ? capacity : 0;
  return HE_OK;
}

int he_set_dist_log(he_handle h, int32_t* dist) {
  if (!h) return HE_EINVAL;
  h->dist = dist;
  return HE_OK;
}

int he_launch_info(he_handle h, int32_t* ctas, int32_t* ctas_per_sm, int32_t* tiles,
                   int32_t* stages) {
  if (!h) return HE_EINVAL;
  const int tpu = (h->occupancy + h->kern.tile - 1) / h->kern.tile;
  const int T = h->U * tpu;
  if (ctas) *ctas = T == 0 ? h->U : (T < h->max_ctas ? T : h->max_ctas);
  if (ctas_per_sm) *ctas_per_sm = h->ctas_per_sm;
  if (tiles) *tiles = T;
  if (stages) *stages = h->fused ? h->kern.fused_stages : h->kern.stages;
  return HE_OK;
}

}  // extern "C"
