// he_pipeline.cuh — the bf16 HashEvict decode step as three kernels chained by
// programmatic dependent launch (PDL), so that no latency-bound work runs
// inside the kernel that streams the cache at HBM bandwidth.
//
//   prep   (one CTA per unit and code chunk)  method steps 1-4: project the G
//          query heads and the new key onto W and binarise (the fixed-order
//          fp32 chains of the specification), form the new token's attention
//          logits, scan a chunk of the unit's packed codes (XOR + popcount,
//          group-summed) and fold the chunk's best (distance, slot) into the
//          unit's eviction key with an order-independent atomicMax.
//   stream (stream-K over 64-slot tiles, one producer + four consumer warps)
//          the decode attention over the resident slots except the evicted
//          one: 2-D tensor TMA into a 3-stage ring, logits and value
//          accumulation on the tensor cores (mma.sync m16n8k16 bf16), online
//          softmax in fp32; one partial (max, sum, accumulator) per CTA and unit.
//   merge  (one CTA per unit) log-sum-exp merge of the unit's partials plus the
//          new token, the output, and method step 5: the new token's key,
//          value and code overwrite the evicted slot.
//
// The arithmetic is the specification's "score, evict, overwrite, attend":
// the evicted slot never enters the softmax and the new token always does.
// PDL ordering: prep waits for the previous step to finish, then lets stream
// launch; stream may prefetch K/V and read q before its own wait (everything
// it reads was final before prep's wait returned) and reads the eviction keys
// only after it; merge waits for stream (hence for prep) before reading.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "he_common.cuh"

namespace he {

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" :::);
}

// 2-D tensor TMA load (global -> shared), completion on an mbarrier.  x is the
// innermost (element) coordinate: a multiple of 64 here, so 16-byte aligned.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D = A . B + D, A 16x16 bf16 (row), B 16x8 bf16 (col), D 16x8 fp32.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Per-unit results of prep, read by stream and merge.
struct UnitOut {
  unsigned long long key;  // eviction key (distance << 32 | ~slot); 0 between steps
  unsigned long long codek;
  float lnew[8];           // the new token's base-2 logits, per query head
};

// Partial record of one (stream CTA, unit): [m G][l G] padded to 4, acc [G][D].
template <int G, int D>
struct PRec {
  static constexpr int HDR = (2 * G + 3) / 4 * 4;
  static constexpr int FLOATS = HDR + G * D;
};

// ---------------------------------------------------------------------------
// prep
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 256;
constexpr int kPrepChunk = 4096;  // code slots scanned per CTA

template <int D, int G>
struct PrepShape {
  static constexpr int OFF_W = 0;                         // [D][bits] bf16, <= 16 KiB
  static constexpr int OFF_X = OFF_W + D * 64 * 2;        // (G+1) vectors [D] bf16
  static constexpr int OFF_C = OFF_X + ((G + 1) * D * 2 + 15) / 16 * 16;  // code chunk
  static constexpr int OFF_BITS = OFF_C + kPrepChunk * 8;
  static constexpr int OFF_RED = OFF_BITS + ((G + 1) * 64 / 32) * 4;
  static constexpr int OFF_BAR = (OFF_RED + 8 * 8 + 15) / 16 * 16;
  static constexpr int SMEM = OFF_BAR + 16;
};

template <int D, int G>
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const StepParams p, UnitOut* uo,
                                                            int splits) {
  using S = PrepShape<D, G>;
  extern __shared__ __align__(16) unsigned char smem_prep[];
  unsigned char* smem = smem_prep;
  const uint16_t* Ws = reinterpret_cast<const uint16_t*>(smem + S::OFF_W);
  const uint16_t* xs = reinterpret_cast<const uint16_t*>(smem + S::OFF_X);
  const unsigned char* cs = smem + S::OFF_C;
  uint32_t* sbits = reinterpret_cast<uint32_t*>(smem + S::OFF_BITS);
  uint64_t* red = reinterpret_cast<uint64_t*>(smem + S::OFF_RED);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + S::OFF_BAR);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int u = blockIdx.x / splits, split = blockIdx.x - u * splits;
  const int bits = p.bits, wb = bits >> 3;
  const bool full = p.append_slot < 0;
  const int s0 = split * kPrepChunk;
  const int s1 = full ? min(s0 + kPrepChunk, p.occ) : s0;

  pdl_wait();     // the previous step is complete: codes, cache and W are final
  pdl_trigger();  // stream may launch and prefetch the cache

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    const int b = u / p.kv_heads, j = u - b * p.kv_heads;
    const uint32_t wbytes = (uint32_t)(D * bits * 2), qbytes = (uint32_t)(G * D * 2),
                   kbytes = (uint32_t)(D * 2);
    const uint32_t cbytes = s1 > s0 ? (uint32_t)(((s1 - s0) * wb + 15) & ~15) : 0u;
    mbar_arrive_expect_tx(bar, wbytes + qbytes + kbytes + cbytes);
    bulk_g2s(smem + S::OFF_W, p.W, wbytes, bar);
    bulk_g2s(smem + S::OFF_X,
             reinterpret_cast<const uint16_t*>(p.q) + (size_t)(b * p.kv_heads + j) * G * D, qbytes,
             bar);
    bulk_g2s(smem + S::OFF_X + qbytes, reinterpret_cast<const uint16_t*>(p.k) + (size_t)u * D,
             kbytes, bar);
    if (cbytes)
      bulk_g2s(smem + S::OFF_C, p.codes + (size_t)u * p.code_stride + (size_t)s0 * wb, cbytes,
               bar);
  }
  __syncthreads();
  if (!__syncthreads_and(mbar_wait_bounded(bar, 0u))) {
    // gave up: record it and leave once the copies have landed
    if (tid == 0) {
      atomicExch(p.err, 1);
      (void)mbar_wait_bounded(bar, 0u, 500000000ull);
    }
    return;
  }

  // method steps 1-2: bit j of vector v (v < G: query head, v == G: the key) is
  // the sign of the fp32 fused multiply-add chain over d = 0..D-1 from +0
  const int ntask = (G + 1) * bits;
  for (int t0 = warp * 32; t0 < ntask; t0 += kPrepThreads) {
    const int t = t0 + lane;
    const int v = t < ntask ? t / bits : G, jj = t - (t / bits) * bits;
    uint32_t bit = 0;
    if (t < ntask && (full || v == G)) {
      const uint16_t* x = xs + v * D;
      float acc = 0.0f;
#pragma unroll 16
      for (int d = 0; d < D; ++d)
        acc = __fmaf_rn(__uint_as_float((uint32_t)x[d] << 16),
                        __uint_as_float((uint32_t)Ws[d * bits + jj] << 16), acc);
      bit = acc > 0.0f ? 1u : 0u;
    }
    const uint32_t word = __ballot_sync(kFull, bit);
    if (lane == 0) sbits[t0 >> 5] = word;
  }
  // the new token's logits (only the first chunk's CTA publishes them)
  if (split == 0) {
    for (int g = warp; g < G; g += kPrepThreads / 32) {
      float a = 0.0f;
      for (int d = lane; d < D; d += 32)
        a = fmaf(__uint_as_float((uint32_t)xs[g * D + d] << 16),
                 __uint_as_float((uint32_t)xs[G * D + d] << 16), a);
      a = warp_sum(a);
      if (lane == 0) uo[u].lnew[g] = a * p.qscale;
    }
  }
  __syncthreads();
  if (split == 0 && tid == 0) uo[u].codek = code_from_bits(sbits, bits, G);
  if (!full) return;

  // method steps 3-4 on this chunk: the largest group-summed distance, lowest slot
  uint64_t cq[G];
#pragma unroll
  for (int g = 0; g < G; ++g) cq[g] = code_from_bits(sbits, bits, g);
  uint64_t best = 0;
  for (int s = s0 + tid; s < s1; s += kPrepThreads) {
    const unsigned char* c = cs + (size_t)(s - s0) * wb;
    uint64_t code;
    switch (wb) {
      case 1: code = *c; break;
      case 2: code = *reinterpret_cast<const uint16_t*>(c); break;
      case 4: code = *reinterpret_cast<const uint32_t*>(c); break;
      default: code = *reinterpret_cast<const uint64_t*>(c); break;
    }
    const uint64_t key = evict_key(group_distance<G>(cq, code), (uint32_t)s);
    best = key > best ? key : best;
  }
  best = warp_max_u64(best);
  if (lane == 0) red[warp] = best;
  __syncthreads();
  if (tid == 0) {
    uint64_t b2 = 0;
    for (int w2 = 0; w2 < kPrepThreads / 32; ++w2) b2 = red[w2] > b2 ? red[w2] : b2;
    if (b2) atomicMax(&uo[u].key, (unsigned long long)b2);
  }
}

// ---------------------------------------------------------------------------
// stream
// ---------------------------------------------------------------------------
template <int D, int G, int NS>
struct StreamShape {
  static constexpr int NCW = 4;              // consumer warps
  static constexpr int NC = NCW * 32;        // consumer threads
  static constexpr int NT = NC + 32;         // + the producer warp
  static constexpr int TS = 16 * NCW;        // slots per tile
  static constexpr int NHALF = D / 64;       // 128-byte column boxes per row
  static constexpr int BOXB = TS * 128;      // bytes per TMA box
  static constexpr int TILEB = NHALF * BOXB; // bytes per K (or V) tile
  static constexpr int STAGEB = 2 * TILEB;   // K + V
  static constexpr int KS = D / 16;          // k-steps of the logit MMA
  static constexpr int MT = D / 16;          // d blocks of the value MMA
  static constexpr int PB = 8 * 16 * 2;      // bytes of one P^T block [8 heads][16 slots] bf16
  static constexpr int WACC = NCW * G * D;   // floats of the warp-merge area
  static constexpr int OFF_STAGE = 0;        // 1024-byte aligned (128B swizzle)
  static constexpr int OFF_WACC = NS * STAGEB;
  static constexpr int OFF_P = OFF_WACC + WACC * 4;
  static constexpr int OFF_WM = OFF_P + NCW * 2 * PB;
  static constexpr int OFF_FLAG = OFF_WM + 2 * NCW * G * 4;
  static constexpr int OFF_BAR = OFF_FLAG + 16;
  static constexpr int SMEM = OFF_BAR + 2 * NS * 8;
  static constexpr int SMEM_ALLOC = SMEM + 1024;  // slack to align the base to 1024
  static_assert(D % 64 == 0 && G >= 1 && G <= 8 && (G & (G - 1)) == 0, "shape");
  static_assert(STAGEB % 1024 == 0 && BOXB % 1024 == 0, "swizzle atoms");
};

template <int D, int G, int NS, bool PSPLIT>
__global__ void __launch_bounds__(StreamShape<D, G, NS>::NT, 2)
    stream_kernel(const StepParams p, const UnitOut* uo, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV) {
  using S = StreamShape<D, G, NS>;
  using R = PRec<G, D>;
  constexpr int NC = S::NC;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* stage = smem + S::OFF_STAGE;
  float* wacc = reinterpret_cast<float*>(smem + S::OFF_WACC);
  float* wm = reinterpret_cast<float*>(smem + S::OFF_WM);
  float* wl = wm + S::NCW * G;
  volatile int32_t* v_abort = reinterpret_cast<int32_t*>(smem + S::OFF_FLAG);
  volatile int32_t* v_issued = v_abort + 1;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + S::OFF_BAR);
  uint64_t* empty_bar = full_bar + NS;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool full = p.append_slot < 0;
  const int64_t TT = p.total_tiles, NCTA = gridDim.x;
  const int tb = (int)((int64_t)blockIdx.x * TT / NCTA);
  const int te = (int)(((int64_t)blockIdx.x + 1) * TT / NCTA);
  const int ntiles = te - tb;

  pdl_trigger();  // merge may launch; it waits for this grid before reading
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], S::NCW);
    }
    v_abort[0] = 0;
    v_issued[0] = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // ---------------- producer warp ----------------
  if (warp == S::NCW) {
    if (lane == 0) {
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % NS;
        if (i >= NS && !mbar_wait_bounded(&empty_bar[st], (uint32_t)(((i / NS) - 1) & 1))) {
          atomicExch(p.err, 1);
          break;
        }
        const int t = tb + i;
        const int u = t / p.tpu;
        const int y = u * p.budget + (t - u * p.tpu) * S::TS;
        unsigned char* dst = stage + st * S::STAGEB;
        mbar_arrive_expect_tx(&full_bar[st], (uint32_t)S::STAGEB);
#pragma unroll
        for (int h = 0; h < S::NHALF; ++h)
          tma_load_2d(dst + h * S::BOXB, &tmK, 64 * h, y, &full_bar[st]);
#pragma unroll
        for (int h = 0; h < S::NHALF; ++h)
          tma_load_2d(dst + S::TILEB + h * S::BOXB, &tmV, 64 * h, y, &full_bar[st]);
        *v_issued = i + 1;
      }
    }
    return;
  }

  // ---------------- consumer warps ----------------
  const int cw = warp;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int h0 = 2 * t4, h1 = 2 * t4 + 1;
  const bool real0 = h0 < G, real1 = h1 < G;
  __nv_bfloat16* Phi = reinterpret_cast<__nv_bfloat16*>(smem + S::OFF_P + cw * 2 * S::PB);
  __nv_bfloat16* Plo = Phi + 8 * 16;
  const float qscale = p.qscale;
  const int u_first = tb / p.tpu, u_last = (te - 1) / p.tpu;

  int i = 0;            // CTA-local tile counter
  int drain_from = -1;  // first tile this warp did not wait for (after a give-up)
  bool waited = false;  // prep's results are visible once the grid dependency resolved
  for (int u = u_first; u <= u_last; ++u) {
    const int seg_t0 = max(tb, u * p.tpu), seg_t1 = min(te, (u + 1) * p.tpu);
    const int hi = min((seg_t1 - u * p.tpu) * S::TS, p.occ);

    // query fragments (B operand of the logit MMA): head g8, d = 16ks + 8r + 2t4 (+1)
    uint32_t qb[S::KS][2];
    {
      const int b = u / p.kv_heads, jj = u - b * p.kv_heads;
      const uint32_t* qw = reinterpret_cast<const uint32_t*>(
          reinterpret_cast<const uint16_t*>(p.q) + ((size_t)(b * p.kv_heads + jj) * G) * D);
#pragma unroll
      for (int ks = 0; ks < S::KS; ++ks)
#pragma unroll
        for (int r = 0; r < 2; ++r)
          qb[ks][r] = g8 < G ? __ldg(qw + (g8 * D + 16 * ks + 8 * r + 2 * t4) / 2) : 0u;
    }
    if (!waited) {
      pdl_wait();
      waited = true;
    }
    // the slot this step evicts is left out of the softmax (method step 4)
    const int evict = full ? (int)evict_key_slot(__ldcg(&uo[u].key)) : -1;

    float mrun0 = -1e30f, mrun1 = -1e30f, lrun0 = 0.0f, lrun1 = 0.0f;
    float acc[S::MT][4];
#pragma unroll
    for (int mt = 0; mt < S::MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.0f;

    for (int lt = seg_t0 - u * p.tpu; lt < seg_t1 - u * p.tpu; ++lt, ++i) {
      const int st = i % NS;
      if (drain_from < 0) {
        if (*v_abort) {
          drain_from = i;
        } else if (!mbar_wait_bounded(&full_bar[st], (uint32_t)((i / NS) & 1))) {
          atomicExch(p.err, 1);
          *v_abort = 1;
          drain_from = i;
        }
      }
      const unsigned char* Ks = stage + st * S::STAGEB;
      const unsigned char* Vs = Ks + S::TILEB;
      const int row0 = 16 * cw;
      const int slot_base = lt * S::TS + row0;

      // logits for this warp's 16 slots x 8 (padded) heads
      float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int ks = 0; ks < S::KS; ++ks) {
        const int row = row0 + (lane & 15);
        const int chunk = ((ks & 3) << 1) + (lane >> 4);
        uint32_t a[4];
        ldsm_x4(a, smem_u32(Ks + (ks >> 2) * S::BOXB + row * 128 + ((chunk ^ (row & 7)) << 4)));
        mma_bf16_16816(c, a, qb[ks][0], qb[ks][1]);
      }
      // c[0]: slot g8, head h0; c[1]: slot g8, h1; c[2]: slot g8+8, h0; c[3]: slot g8+8, h1
      float x00 = c[0] * qscale, x01 = c[1] * qscale, x10 = c[2] * qscale, x11 = c[3] * qscale;
      const int sA = slot_base + g8, sB = sA + 8;
      if (sA >= hi || sA == evict) x00 = x01 = -INFINITY;
      if (sB >= hi || sB == evict) x10 = x11 = -INFINITY;
      if (!real0) x00 = x10 = -INFINITY;
      if (!real1) x01 = x11 = -INFINITY;

      // online softmax per head over the warp's slots (lanes sharing t4)
      float t0m = fmaxf(x00, x10), t1m = fmaxf(x01, x11);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        t0m = fmaxf(t0m, __shfl_xor_sync(kFull, t0m, o));
        t1m = fmaxf(t1m, __shfl_xor_sync(kFull, t1m, o));
      }
      const float mn0 = fmaxf(mrun0, t0m), mn1 = fmaxf(mrun1, t1m);
      const float sc0 = exp2f(mrun0 - mn0), sc1 = exp2f(mrun1 - mn1);
      mrun0 = mn0;
      mrun1 = mn1;
      const float p00 = exp2f(x00 - mn0), p10 = exp2f(x10 - mn0);
      const float p01 = exp2f(x01 - mn1), p11 = exp2f(x11 - mn1);
      lrun0 = lrun0 * sc0 + (p00 + p10);
      lrun1 = lrun1 * sc1 + (p01 + p11);
#pragma unroll
      for (int mt = 0; mt < S::MT; ++mt) {
        acc[mt][0] *= sc0;
        acc[mt][2] *= sc0;
        acc[mt][1] *= sc1;
        acc[mt][3] *= sc1;
      }

      // P^T [8 heads][16 slots] in bf16 (hi, and the rounding remainder lo)
      {
        const __nv_bfloat16 a00 = __float2bfloat16_rn(p00), a01 = __float2bfloat16_rn(p01);
        const __nv_bfloat16 a10 = __float2bfloat16_rn(p10), a11 = __float2bfloat16_rn(p11);
        Phi[h0 * 16 + g8] = a00;
        Phi[h1 * 16 + g8] = a01;
        Phi[h0 * 16 + g8 + 8] = a10;
        Phi[h1 * 16 + g8 + 8] = a11;
        if (PSPLIT) {
          Plo[h0 * 16 + g8] = __float2bfloat16_rn(p00 - __bfloat162float(a00));
          Plo[h1 * 16 + g8] = __float2bfloat16_rn(p01 - __bfloat162float(a01));
          Plo[h0 * 16 + g8 + 8] = __float2bfloat16_rn(p10 - __bfloat162float(a10));
          Plo[h1 * 16 + g8 + 8] = __float2bfloat16_rn(p11 - __bfloat162float(a11));
        }
      }
      __syncwarp();
      const uint32_t* Phw = reinterpret_cast<const uint32_t*>(Phi);
      const uint32_t* Plw = reinterpret_cast<const uint32_t*>(Plo);
      const uint32_t bh0 = Phw[g8 * 8 + t4], bh1 = Phw[g8 * 8 + 4 + t4];
      const uint32_t bl0 = PSPLIT ? Plw[g8 * 8 + t4] : 0u;
      const uint32_t bl1 = PSPLIT ? Plw[g8 * 8 + 4 + t4] : 0u;

      // values: O^T[d][head] += V^T[d][slots] P^T[slots][head]
#pragma unroll
      for (int mt = 0; mt < S::MT; ++mt) {
        const int row = row0 + (lane & 7) + ((lane >> 4) << 3);
        const int chunk = ((mt & 3) << 1) + ((lane >> 3) & 1);
        uint32_t a[4];
        ldsm_x4_trans(a, smem_u32(Vs + (mt >> 2) * S::BOXB + row * 128 +
                                  ((chunk ^ (row & 7)) << 4)));
        mma_bf16_16816(acc[mt], a, bh0, bh1);
        if (PSPLIT) mma_bf16_16816(acc[mt], a, bl0, bl1);
      }
      __syncwarp();
      if (lane == 0 && drain_from < 0) mbar_arrive(&empty_bar[st]);  // stage free for refill
    }

    // warp states -> shared memory -> this CTA's partial for unit u
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      lrun0 += __shfl_xor_sync(kFull, lrun0, o);
      lrun1 += __shfl_xor_sync(kFull, lrun1, o);
    }
    if (g8 == 0) {
      if (real0) {
        wm[cw * G + h0] = mrun0;
        wl[cw * G + h0] = lrun0;
      }
      if (real1) {
        wm[cw * G + h1] = mrun1;
        wl[cw * G + h1] = lrun1;
      }
    }
#pragma unroll
    for (int mt = 0; mt < S::MT; ++mt) {
      const int d = 16 * mt + g8;
      if (real0) {
        wacc[(cw * G + h0) * D + d] = acc[mt][0];
        wacc[(cw * G + h0) * D + d + 8] = acc[mt][2];
      }
      if (real1) {
        wacc[(cw * G + h1) * D + d] = acc[mt][1];
        wacc[(cw * G + h1) * D + d + 8] = acc[mt][3];
      }
    }
    group_sync<NC, 1>();
    if (*v_abort) {
      // a wait gave up: let the copies already issued land, then leave
      if (tid == 0) {
        const int issued = *v_issued;
        for (int r = drain_from < 0 ? i : drain_from; r < issued; ++r)
          (void)mbar_wait_bounded(&full_bar[r % NS], (uint32_t)((r / NS) & 1), 500000000ull);
      }
      return;
    }
    float* rec = p.partials + (size_t)(blockIdx.x + u) * R::FLOATS;
    for (int idx = tid; idx < G * D; idx += NC) {
      const int g = idx / D, d = idx - g * D;
      float mx = -1e30f;
#pragma unroll
      for (int w2 = 0; w2 < S::NCW; ++w2) mx = fmaxf(mx, wm[w2 * G + g]);
      float a = 0.0f;
#pragma unroll
      for (int w2 = 0; w2 < S::NCW; ++w2)
        a += wacc[(w2 * G + g) * D + d] * exp2f(wm[w2 * G + g] - mx);
      rec[R::HDR + idx] = a;
    }
    if (tid < G) {
      const int g = tid;
      float mx = -1e30f, sum = 0.0f;
#pragma unroll
      for (int w2 = 0; w2 < S::NCW; ++w2) mx = fmaxf(mx, wm[w2 * G + g]);
#pragma unroll
      for (int w2 = 0; w2 < S::NCW; ++w2) sum += wl[w2 * G + g] * exp2f(wm[w2 * G + g] - mx);
      rec[g] = mx;
      rec[G + g] = sum;
    }
    group_sync<NC, 1>();  // the merge area is reused by the next segment
  }
}

// ---------------------------------------------------------------------------
// merge
// ---------------------------------------------------------------------------
constexpr int kMergeThreads = 512;

// Dynamic shared memory of merge: headers/weights of up to `max_contrib`
// partials ([c][2G] floats) + the per-group sums [NQ][G*D/4] float4.
template <int D, int G>
__host__ __device__ constexpr int merge_smem(int max_contrib) {
  return (max_contrib * 2 * G * 4 + 15) / 16 * 16 + kMergeThreads * 16 + 80;
}

template <int D, int G>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const StepParams p, UnitOut* uo,
                                                              int stream_ctas) {
  using R = PRec<G, D>;
  constexpr int GD4 = G * D / 4;              // float4 outputs per unit
  constexpr int NQ = kMergeThreads / GD4;     // contributor groups
  static_assert(GD4 <= kMergeThreads && kMergeThreads % GD4 == 0, "merge shape");
  extern __shared__ __align__(16) unsigned char smem_merge[];
  unsigned char* smem = smem_merge;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int u = blockIdx.x;
  const bool full = p.append_slot < 0;

  pdl_wait();     // stream (and so prep) is complete and visible
  pdl_trigger();  // the next step's prep may launch; it waits for this grid

  int first = 0, n = 0;
  if (p.total_tiles > 0) {
    const int64_t TT = p.total_tiles, NC = stream_ctas;
    first = (int)((((int64_t)u * p.tpu + 1) * NC - 1) / TT);
    const int last = (int)((((int64_t)u * p.tpu + p.tpu) * NC - 1) / TT);
    n = last - first + 1;
  }
  float* wts = reinterpret_cast<float*>(smem);                  // [n][G]: m, then weight
  float* lsum = wts + (size_t)n * G;                            // [n][G]: l
  float4* part = reinterpret_cast<float4*>(smem + (((size_t)n * 2 * G * 4 + 15) & ~(size_t)15));
  float* hm = reinterpret_cast<float*>(part + kMergeThreads);   // [G]
  float* hl = hm + 8;                                           // [G]
  int* win = reinterpret_cast<int*>(hl + 8);
  const float* recs = p.partials + (size_t)(first + u) * R::FLOATS;

  for (int c = tid; c < n; c += kMergeThreads) {
    const float* r = recs + (size_t)c * R::FLOATS;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      wts[c * G + g] = __ldcg(r + g);
      lsum[c * G + g] = __ldcg(r + G + g);
    }
  }
  __syncthreads();
  // per-head stabiliser and denominator (fixed order: lanes then the warp tree)
  for (int g = warp; g < G; g += kMergeThreads / 32) {
    const float ln = __ldcg(&uo[u].lnew[g]);
    float mx = ln;
    for (int c = lane; c < n; c += 32) mx = fmaxf(mx, wts[c * G + g]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    float sum = 0.0f;
    for (int c = lane; c < n; c += 32) sum += lsum[c * G + g] * exp2f(wts[c * G + g] - mx);
    sum = warp_sum(sum);
    if (lane == 0) {
      hm[g] = mx;
      hl[g] = sum + exp2f(ln - mx);
    }
  }
  if (tid == 0) {
    const unsigned long long key = __ldcg(&uo[u].key);
    *win = full ? (key ? (int)evict_key_slot(key) : -1) : p.append_slot;
  }
  __syncthreads();
  for (int i2 = tid; i2 < n * G; i2 += kMergeThreads) {
    const int g = i2 - (i2 / G) * G;
    wts[i2] = exp2f(wts[i2] - hm[g]);
  }
  __syncthreads();

  // accumulators: group q sums the contributors c = q, q + NQ, ... (fixed order)
  const int q = tid / GD4, o = tid - q * GD4;
  const int g_o = (4 * o) / D;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int c = q; c < n; c += NQ) {
    const float4 x = __ldcg(reinterpret_cast<const float4*>(recs + (size_t)c * R::FLOATS + R::HDR) + o);
    const float w = wts[c * G + g_o];
    a.x += x.x * w;
    a.y += x.y * w;
    a.z += x.z * w;
    a.w += x.w * w;
  }
  part[q * GD4 + o] = a;
  __syncthreads();

  const int winner = *win;
  if (winner < 0 || winner >= p.budget) {  // cannot happen: never write outside the cache
    if (tid == 0) atomicExch(p.err, 2);
    return;
  }
  const int b = u / p.kv_heads, j = u - b * p.kv_heads;
  const uint16_t* vt = reinterpret_cast<const uint16_t*>(p.v) + (size_t)u * D;
  if (tid < GD4) {
    float4 s = part[tid];
    for (int q2 = 1; q2 < NQ; ++q2) {
      const float4 y = part[q2 * GD4 + tid];
      s.x += y.x;
      s.y += y.y;
      s.z += y.z;
      s.w += y.w;
    }
    const int g = (4 * tid) / D, d = 4 * tid - g * D;
    const float wn = exp2f(__ldcg(&uo[u].lnew[g]) - hm[g]);
    const float inv = 1.0f / hl[g];
    float4 r;
    r.x = (s.x + wn * __uint_as_float((uint32_t)vt[d] << 16)) * inv;
    r.y = (s.y + wn * __uint_as_float((uint32_t)vt[d + 1] << 16)) * inv;
    r.z = (s.z + wn * __uint_as_float((uint32_t)vt[d + 2] << 16)) * inv;
    r.w = (s.w + wn * __uint_as_float((uint32_t)vt[d + 3] << 16)) * inv;
    reinterpret_cast<float4*>(p.out + ((size_t)b * p.kv_heads * G + (size_t)j * G) * D)[tid] = r;
  }

  // method step 5: the current token's key, value and code replace the slot
  uint16_t* Kw = reinterpret_cast<uint16_t*>(p.K) + ((size_t)u * p.budget + winner) * D;
  uint16_t* Vw = reinterpret_cast<uint16_t*>(p.V) + ((size_t)u * p.budget + winner) * D;
  const uint16_t* kt = reinterpret_cast<const uint16_t*>(p.k) + (size_t)u * D;
  for (int d = tid; d < D; d += kMergeThreads) {
    Kw[d] = kt[d];
    Vw[d] = vt[d];
  }
  if (tid == 0) {
    store_code(p.codes + (size_t)u * p.code_stride + (size_t)winner * (p.bits >> 3), p.bits,
               __ldcg(&uo[u].codek));
    p.evicted[u] = full ? winner : -1;
    uo[u].key = 0;  // ready for the next step's atomicMax
  }
}

}  // namespace he
