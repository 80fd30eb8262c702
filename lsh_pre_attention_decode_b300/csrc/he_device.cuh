// he_device.cuh — device-side building blocks of the HashEvict step kernels:
// element conversion, TMA bulk copies with mbarrier completion (bounded waits),
// the fixed-order projection that yields the code bits, warp reductions.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace he {

constexpr uint32_t kFull = 0xFFFFFFFFu;

// Element types: bf16 is carried as its raw 16-bit pattern; fp32 as float.
struct bf16_t {
  uint16_t bits;
};

template <typename T>
struct ElemTraits;
template <>
struct ElemTraits<bf16_t> {
  static constexpr int kBytes = 2;
};
template <>
struct ElemTraits<float> {
  static constexpr int kBytes = 4;
};

__device__ __forceinline__ float to_f32(bf16_t x) { return __uint_as_float((uint32_t)x.bits << 16); }
__device__ __forceinline__ float to_f32(float x) { return x; }
// Read-only cached load of one element, converted exactly to fp32.
__device__ __forceinline__ float ldg_f32(const bf16_t* p) {
  return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p)) << 16);
}
__device__ __forceinline__ float ldg_f32(const float* p) { return __ldg(p); }
// The two bf16 values packed in a 32-bit word (low half first), exactly.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---------------------------------------------------------------------------
// mbarrier + TMA bulk copy (global -> shared), PTX ISA "cp.async.bulk" and
// "mbarrier" sections.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase with the given parity to complete; gives up after about
// `limit_ns` nanoseconds and returns false (the caller records an error and
// unwinds instead of hanging).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// 1-D bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned)
// from global to this CTA's shared memory; completion is signalled on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------------------
// Method steps 1-2 for one bit: the projection of x onto column j of W, summed
// in fp32 with fused multiply-adds in the fixed order d = 0..D-1 from +0, and
// test against the threshold tau (with tau = 0, the sign test: an exact zero
// gives 0).  x is staged in shared memory as fp32
// (exact copies of the stored elements).
// ---------------------------------------------------------------------------
template <typename T, int D>
__device__ __forceinline__ float projection_value(const float* __restrict__ x,
                                                  const T* __restrict__ W, int bits, int j) {
  float acc = 0.0f;
#pragma unroll 16
  for (int d = 0; d < D; ++d) acc = __fmaf_rn(x[d], ldg_f32(W + (size_t)d * bits + j), acc);
  return acc;
}

template <typename T, int D>
__device__ __forceinline__ uint32_t projection_bit(const float* __restrict__ x,
                                                   const T* __restrict__ W, int bits, int j,
                                                   float tau) {
  return projection_value<T, D>(x, W, bits, j) > tau ? 1u : 0u;
}

// Extract the `bits`-bit code number `idx` from a packed bit string (32-bit words).
__device__ __forceinline__ uint64_t code_from_bits(const uint32_t* s_bits, int bits, int idx) {
  const int off = idx * bits;
  if (bits == 64) return (uint64_t)s_bits[off >> 5] | ((uint64_t)s_bits[(off >> 5) + 1] << 32);
  const uint32_t wrd = s_bits[off >> 5];
  if (bits == 32) return wrd;
  return (wrd >> (off & 31)) & ((1u << bits) - 1u);
}

__device__ __forceinline__ int popc64(uint64_t x) { return __popcll(x); }

// Bounds checks of the debug build (-DHE_DEBUG; compute-sanitizer is not
// available): a failed check records error 3 in the handle's flag, which the
// host reports as HE_EDEVICE, and the caller skips the access.  Without
// HE_DEBUG every check is the constant true and costs nothing.
#ifdef HE_DEBUG
__device__ __forceinline__ bool debug_check(bool ok, int32_t* err) {
  if (!ok) atomicExch(err, 3);
  return ok;
}
#define HE_CHECK(cond, err) (he::debug_check((cond), (err)))
#else
#define HE_CHECK(cond, err) true
#endif

// Packed eviction key: larger distance wins, then the lower slot.
__device__ __forceinline__ uint64_t evict_key(uint32_t dist, uint32_t slot) {
  return ((uint64_t)dist << 32) | (uint64_t)(0xFFFFFFFFu - slot);
}
__device__ __forceinline__ uint32_t evict_key_slot(uint64_t key) {
  return 0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFu);
}
__device__ __forceinline__ uint32_t evict_key_dist(uint64_t key) { return (uint32_t)(key >> 32); }

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    uint64_t w = __shfl_xor_sync(kFull, v, o);
    v = w > v ? w : v;
  }
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// Phase timer (diagnostic builds with -DHE_TIMELINE only; compiled out
// otherwise): thread 0 of a step CTA accumulates nanoseconds per phase in the
// CTA's shared block and, at exit, writes [start, end, phase 0..21] to
// g_he_timeline[cta * 24 ..].
// ---------------------------------------------------------------------------
#ifdef HE_TIMELINE
static __device__ int64_t* g_he_timeline = nullptr;
struct PhaseTimer {
  int64_t acc[22];
  int64_t last;
  int64_t start;
};
#define HE_TL_FIELDS he::PhaseTimer tl;
#define HE_TL_INIT(m)                                 \
  if (tid == 0) {                                     \
    for (int k_ = 0; k_ < 22; ++k_) (m).tl.acc[k_] = 0; \
    (m).tl.start = (m).tl.last = (int64_t)he::global_ns(); \
  }
#define HE_TL_MARK(m, k)                              \
  if (tid == 0) {                                     \
    const int64_t n_ = (int64_t)he::global_ns();      \
    (m).tl.acc[k] += n_ - (m).tl.last;                \
    (m).tl.last = n_;                                 \
  }
#define HE_TL_COUNT(m, k, inc) \
  if (tid == 0) (m).tl.acc[k] += (inc);
#define HE_TL_DONE(m)                                                  \
  if (tid == 0 && he::g_he_timeline) {                                 \
    int64_t* o_ = he::g_he_timeline + (size_t)blockIdx.x * 24;         \
    o_[0] = (m).tl.start;                                              \
    o_[1] = (int64_t)he::global_ns();                                  \
    for (int k_ = 0; k_ < 22; ++k_) o_[2 + k_] = (m).tl.acc[k_];       \
  }
// Stamps: thread 0 of a CTA writes the time at a numbered point of a kernel
// (region r: prep 0, stream 1, merge 2; step slot s = p.tl_step, 0..7) to
// g_he_timeline[((s*3 + r)*4096 + cta)*8 + k].
#define HE_STAMP(r, k)                                                              \
  if (threadIdx.x == 0 && he::g_he_timeline && blockIdx.x < 4096)                  \
    he::g_he_timeline[(((size_t)p.tl_step * 3 + (r)) * 4096 + blockIdx.x) * 8 + (k)] = \
        (int64_t)he::global_ns();
// The same for any thread that passes `c`, and a stored value instead of the time.
#define HE_STAMP_IF(c, r, k)                                                         \
  if ((c) && he::g_he_timeline && blockIdx.x < 4096)                                 \
    he::g_he_timeline[(((size_t)p.tl_step * 3 + (r)) * 4096 + blockIdx.x) * 8 + (k)] = \
        (int64_t)he::global_ns();
#define HE_STAMP_VAL(c, r, k, v)                                                     \
  if ((c) && he::g_he_timeline && blockIdx.x < 4096)                                 \
    he::g_he_timeline[(((size_t)p.tl_step * 3 + (r)) * 4096 + blockIdx.x) * 8 + (k)] = (v);
#else
#define HE_STAMP_IF(c, r, k)
#define HE_STAMP_VAL(c, r, k, v)
#define HE_TL_FIELDS
#define HE_TL_INIT(m)
#define HE_TL_MARK(m, k)
#define HE_TL_COUNT(m, k, inc)
#define HE_TL_DONE(m)
#define HE_STAMP(r, k)
#endif

}  // namespace he
