// he_pipeline.cuh — the bf16 HashEvict decode step as three kernels chained by
// programmatic dependent launch (PDL).  The eviction decision is off the
// critical path: it is computed concurrently with the attention, and the
// evicted slot is taken out of the attention afterwards.
//
//   prep   (one CTA per unit and code item)  method steps 1-4: project the G
//          query heads and the new key onto W and binarise (the fixed-order
//          fp32 chains of the specification), form the new token's attention
//          logits, scan a chunk of the unit's packed codes (XOR + popcount,
//          group-summed) and fold the chunk's best (distance, slot) into the
//          unit's eviction key with an order-independent atomicMax.
//   stream (stream-K over 64-slot tiles, one producer + four consumer warps;
//          runs while prep runs) the decode attention over every resident
//          slot: 2-D tensor TMA into an NS-stage ring, logits and value
//          accumulation on the tensor cores (mma.sync m16n8k16 bf16), online
//          softmax in fp32; one partial (max, sum, accumulator) per CTA and unit.
//   merge  (one CTA per unit) removes the evicted slot from the one partial that
//          contains it, log-sum-exp merges the partials, adds the new token,
//          writes the output, and does method step 5: the new token's key,
//          value and code overwrite the evicted slot.
//
// Removal: with p the evicted slot's weight in its partial (same max), the
// partial becomes (l - p, A - p V).  When p <= l / 2 the subtraction loses at
// most one bit of the partial's sum; otherwise merge recomputes that partial
// from the cache without the slot (CUDA cores) — so the result is the
// specification's "score, evict, overwrite, attend" to fp32 accuracy either way.
//
// Launch order and PDL: stream, prep, merge.  stream waits for the previous
// step, then lets prep launch (prep's CTAs take the room stream's CTAs leave on
// each SM, so they never delay the stream); prep reads a final cache without
// waiting and waits for stream at its very end (it cannot complete before
// stream has); merge waits for prep, hence for both.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "he_common.cuh"
#include "he_fused.cuh"
#include "he_layout.cuh"
#include "he_tc.cuh"

namespace he {

// ---------------------------------------------------------------------------
// Quantised value cache (template argument VQ of the bf16 kernels): 0 = value
// rows in bf16; else one byte per value and one fp32 scale s per slot, the row
// stored as codes of v / s with s = max |v| / range:
//   kVqInt8: int8, v / s rounded half to even (range 127);
//   kVqFp8:  E4M3 (OCP 8-bit floating point), v / s rounded to the nearest
//            value, ties to the even mantissa, saturating at 448 (range 448).
// ---------------------------------------------------------------------------
constexpr int kVqInt8 = 1;
constexpr int kVqFp8 = 2;

template <int VQ>
__device__ __forceinline__ float vq_range() {
  return VQ == kVqFp8 ? 448.0f : 127.0f;
}

// The stored byte of x = v / s (s > 0).
template <int VQ>
__device__ __forceinline__ uint8_t vq_encode(float x) {
  if constexpr (VQ == kVqFp8) {
    uint16_t r;  // (the second operand lands in the low byte)
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
    return (uint8_t)(r & 0xFF);
  } else {
    return (uint8_t)(int8_t)(int)fminf(fmaxf(rintf(x), -127.0f), 127.0f);
  }
}

// The value a stored byte stands for before its slot's scale (exact in fp32).
template <int VQ>
__device__ __forceinline__ float vq_decode(uint8_t c) {
  if constexpr (VQ == kVqFp8) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)c));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
  } else {
    return (float)(int8_t)c;
  }
}

// Byte words of two slots s (even) and s + 1 of one value-tile row position:
// byte i of each word is the same column.  -> four f16 pairs (slot s in the
// lower half), pair i from bytes i, exact (|int8| < 2^11; every E4M3 value is an
// f16 normal).
template <int VQ>
__device__ __forceinline__ void vq_pairs_f16(uint32_t we, uint32_t wo, uint32_t (&pr)[4]) {
  if constexpr (VQ == kVqFp8) {
    const uint32_t x01 = __byte_perm(we, wo, 0x5140), x23 = __byte_perm(we, wo, 0x7362);
    asm("{\n\t.reg .b16 a, b, c, d;\n\tmov.b32 {a, b}, %4;\n\tmov.b32 {c, d}, %5;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t"
        "cvt.rn.f16x2.e4m3x2 %2, c;\n\tcvt.rn.f16x2.e4m3x2 %3, d;\n\t}"
        : "=r"(pr[0]), "=r"(pr[1]), "=r"(pr[2]), "=r"(pr[3])
        : "r"(x01), "r"(x23));
  } else {
    // byte b ^ 0x80 as the low mantissa bits of f16 1024: 1024 + b + 128;
    // minus 1152 gives b (both steps exact)
    const uint32_t ue = we ^ 0x80808080u, uo = wo ^ 0x80808080u;
    const __half2 off = __float2half2_rn(1152.0f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t t =
          (__byte_perm(ue, uo, (uint32_t)(i | ((4 + i) << 8))) & 0x00FF00FFu) | 0x64006400u;
      const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&t), off);
      pr[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
  }
}

// Byte offset of (slot row s, byte b) in a value tile of D-byte rows as the
// tensor copy lays it out: 16-byte chunks swizzled within 128-byte (D = 128)
// or 64-byte (D = 64) rows, so that the four slot rows a thread reads per
// column fall in different banks.
template <int D>
__device__ __forceinline__ int vq_tile_off(int s, int b) {
  static_assert(D == 64 || D == 128, "value tile rows of 64 or 128 bytes");
  const int x = D == 128 ? (s & 7) : ((s >> 1) & 3);
  return s * D + ((((b >> 4) ^ x)) << 4) + (b & 15);
}

// Power-of-two exponent bound of the f16 value-MMA weights (see stream_kernel).
constexpr int kVqExpMax = 100;

// ---------------------------------------------------------------------------
// prep
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 128;  // one warp per SM sub-partition: fits beside two stream CTAs
constexpr int kPrepItem = 4096;  // code slots scanned per CTA item, at most (prep_item_slots)
constexpr int kPrepCodeBytes = 16384;  // the item's codes in shared memory, at most

template <int D, int G>
struct PrepShape {
  static constexpr int OFF_W = 0;                         // [D][bits] bf16, <= 16 KiB
  static constexpr int OFF_X = OFF_W + D * 64 * 2;        // (G+1) vectors [D] bf16
  static constexpr int OFF_C = OFF_X + ((G + 1) * D * 2 + 15) / 16 * 16;  // the item's codes
  static constexpr int OFF_BITS = OFF_C + kPrepCodeBytes;
  static constexpr int OFF_RED = OFF_BITS + ((G + 1) * 64 / 32) * 4;
  static constexpr int OFF_BAR = (OFF_RED + 8 * 8 + 16 + 15) / 16 * 16;
  static constexpr int SMEM = OFF_BAR + 16;
};

// MEM: score memory (p.score, p.decay), a separate instantiation because its
// register use is higher.  CH: chunk eviction (p.chunk slots per chunk; the
// chunks of the first p.lbudget slots score the sum of their slots' distances).
// One CTA per SM at most: a CTA takes the (unit, code item) items
// blockIdx.x, blockIdx.x + gridDim.x, ... in turn, so that prep never crowds
// the stream kernel's CTAs off an SM.
template <int D, int G, bool MEM, int VQ = 0, bool CH = false>
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const StepParams p, UnitOut* uo,
                                                            int splits, int first_of_step) {
  static_assert(!(CH && (MEM || VQ)), "chunk eviction takes neither option");
  using S = PrepShape<D, G>;
  extern __shared__ __align__(16) unsigned char smem_prep[];
  unsigned char* smem = smem_prep;
  const uint16_t* Ws = reinterpret_cast<const uint16_t*>(smem + S::OFF_W);
  const uint16_t* xs = reinterpret_cast<const uint16_t*>(smem + S::OFF_X);
  const unsigned char* cs = smem + S::OFF_C;
  uint32_t* sbits = reinterpret_cast<uint32_t*>(smem + S::OFF_BITS);
  uint64_t* red = reinterpret_cast<uint64_t*>(smem + S::OFF_RED);
  int* last = reinterpret_cast<int*>(red + kPrepThreads / 32);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + S::OFF_BAR);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bits = p.bits, wb = bits >> 3;
  const bool full = p.append_slot < 0;
  const int nitems = p.U * splits;

  HE_STAMP(0, 0);
  // launched behind stream, which waited for the previous step before letting
  // prep launch: codes, cache and W are final.  With an empty cache there is no
  // stream kernel and prep waits for the previous step itself.
  if (first_of_step) pdl_wait();
  pdl_trigger();  // merge may launch; it waits for this grid before reading
  HE_STAMP(0, 1);

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();

  uint32_t phase = 0;
  for (int it = blockIdx.x; it < nitems; it += gridDim.x, phase ^= 1u) {
    const int u = it / splits, split = it - u * splits;
    const int item = CH ? chunk_item_slots(p.chunk, bits) : prep_item_slots(bits);
    const int s0 = split * item;
    const int s1 = full ? min(s0 + item, CH ? p.lbudget : p.occ) : s0;
    if (tid == 0) {
      const int b = u / p.kv_heads, j = u - b * p.kv_heads;
      const uint32_t wbytes = it == (int)blockIdx.x ? (uint32_t)(D * bits * 2) : 0u;
      const uint32_t qbytes = (uint32_t)(G * D * 2), kbytes = (uint32_t)(D * 2);
      uint32_t cbytes = s1 > s0 ? (uint32_t)(((s1 - s0) * wb + 15) & ~15) : 0u;
      if (!HE_CHECK((int64_t)s0 * wb + cbytes <= p.code_stride, p.err)) cbytes = 0;
      mbar_arrive_expect_tx(bar, wbytes + qbytes + kbytes + cbytes);
      if (wbytes) bulk_g2s(smem + S::OFF_W, p.W, wbytes, bar);
      bulk_g2s(smem + S::OFF_X,
               reinterpret_cast<const uint16_t*>(p.q) + (size_t)(b * p.kv_heads + j) * G * D,
               qbytes, bar);
      bulk_g2s(smem + S::OFF_X + qbytes, reinterpret_cast<const uint16_t*>(p.k) + (size_t)u * D,
               kbytes, bar);
      if (cbytes)
        bulk_g2s(smem + S::OFF_C, p.codes + (size_t)u * p.code_stride + (size_t)s0 * wb, cbytes,
                 bar);
    }
    // (quantised value cache: the new token's value row, for the first item,
    // loaded while the copies are in flight)
    float vnew = 0.0f;
    if constexpr (VQ) {
      static_assert(D <= kPrepThreads, "one value element per thread");
      if (split == 0 && tid < D)
        vnew = __uint_as_float((uint32_t)__ldcg(reinterpret_cast<const uint16_t*>(p.v) +
                                                (size_t)u * D + tid)
                               << 16);
    }
    if (!__syncthreads_and(mbar_wait_bounded(bar, phase))) {
      // gave up: record it and leave once the copies have landed
      if (tid == 0) {
        atomicExch(p.err, 1);
        (void)mbar_wait_bounded(bar, phase, 500000000ull);
      }
      return;
    }
    HE_STAMP(0, 2);

    // method steps 1-2: bit j of vector v (v < G: query head, v == G: the key)
    // is the sign of the fp32 fused multiply-add chain over d = 0..D-1 from +0
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
        bit = acc > (p.tauv ? __ldg(p.tauv + (size_t)u * bits + jj) : p.tau) ? 1u : 0u;
      }
      const uint32_t word = __ballot_sync(kFull, bit);
      if (lane == 0) sbits[t0 >> 5] = word;
    }
    // the new token's logits (only the unit's first item publishes them);
    // with a quantised value cache also its value row, quantised as merge
    // will store it (s = max |v| / range, codes of v / s, both fp32 divisions)
    if (split == 0) {
      for (int g = warp; g < G; g += kPrepThreads / 32) {
        float a = 0.0f;
        for (int d = lane; d < D; d += 32)
          a = fmaf(__uint_as_float((uint32_t)xs[g * D + d] << 16),
                   __uint_as_float((uint32_t)xs[G * D + d] << 16), a);
        a = warp_sum(a);
        if (lane == 0) uo[u].lnew[g] = a * p.qscale;
      }
      if constexpr (VQ) {
        float m = fabsf(vnew);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
        float* wmax = reinterpret_cast<float*>(red + kPrepThreads / 32 + 2);  // [4]
        if (lane == 0) wmax[warp] = m;
        __syncthreads();
        m = 0.0f;
        for (int w2 = 0; w2 < D / 32; ++w2) m = fmaxf(m, wmax[w2]);
        const float sc = __fdiv_rn(m, vq_range<VQ>());
        if (tid < D) uo[u].vqnew[tid] = sc > 0.0f ? vq_encode<VQ>(__fdiv_rn(vnew, sc)) : 0;
        if (tid == 0) uo[u].vsnew = sc;
      }
    }
    __syncthreads();
    HE_STAMP(0, 6);
    if (split == 0 && tid == 0) uo[u].codek = code_from_bits(sbits, bits, G);

    if (full) {
      // method steps 3-4 on this item: the largest group-summed distance, lowest slot
      uint64_t cq[G];
#pragma unroll
      for (int g = 0; g < G; ++g) cq[g] = code_from_bits(sbits, bits, g);
      uint64_t best = 0;
      auto code_at = [&](int s) -> uint64_t {
        const unsigned char* c = cs + (size_t)(s - s0) * wb;
        switch (wb) {
          case 1: return *c;
          case 2: return *reinterpret_cast<const uint16_t*>(c);
          case 4: return *reinterpret_cast<const uint32_t*>(c);
          default: return *reinterpret_cast<const uint64_t*>(c);
        }
      };
      if constexpr (CH) {
        // a chunk [s, s + c) scores the sum of its slots' distances; the key
        // carries its first slot, so ties go to the lowest chunk
        const int c = p.chunk;
        for (int s = s0 + tid * c; s < s1; s += kPrepThreads * c) {
          uint32_t sum = 0;
          for (int i = 0; i < c; ++i) {
            const uint32_t d = group_distance<G>(cq, code_at(s + i));
            if (p.dist != nullptr) p.dist[(size_t)u * p.budget + s + i] = (int32_t)d;
            sum += d;
          }
          const uint64_t key = evict_key(sum, (uint32_t)s);
          best = key > best ? key : best;
        }
      } else if constexpr (!MEM) {  // (the method: 32 registers, so prep fits beside two stream CTAs)
        for (int s = s0 + tid; s < s1; s += kPrepThreads) {
          const uint32_t d = group_distance<G>(cq, code_at(s));
          if (p.dist != nullptr) p.dist[(size_t)u * p.budget + s] = (int32_t)d;
          const uint64_t key = evict_key(d, (uint32_t)s);
          best = key > best ? key : best;
        }
      } else {
        // score memory: A = gamma A + d (a non-negative fp32 orders as its bits).
        // The scores of a batch of this thread's slots are all loaded before any
        // is used (one memory round trip per batch).
        constexpr int NB = 16;
        constexpr int IT = kPrepItem / kPrepThreads;
        static_assert(IT % NB == 0, "score batches");
        float* sc = p.score + (size_t)u * p.budget;
        for (int i0 = 0; i0 < IT; i0 += NB) {
          float a[NB];
#pragma unroll
          for (int i = 0; i < NB; ++i) {
            const int s = s0 + tid + (i0 + i) * kPrepThreads;
            a[i] = s < s1 ? __ldcg(sc + s) : 0.0f;
          }
#pragma unroll
          for (int i = 0; i < NB; ++i) {
            const int s = s0 + tid + (i0 + i) * kPrepThreads;
            if (s < s1) {
              const uint32_t d = group_distance<G>(cq, code_at(s));
              if (p.dist != nullptr) p.dist[(size_t)u * p.budget + s] = (int32_t)d;
              const float v = __fmaf_rn(p.decay, a[i], (float)d);
              sc[s] = v;
              const uint64_t key = evict_key(__float_as_uint(v), (uint32_t)s);
              best = key > best ? key : best;
            }
          }
        }
      }
      HE_STAMP(0, 7);
      best = warp_max_u64(best);
      if (lane == 0) red[warp] = best;
      __syncthreads();
      HE_STAMP(0, 4);
      // a unit of one item decides here: its key is this CTA's best (a plain
      // store; the key was zeroed by the previous step's merge); else the
      // items fold their bests with atomicMax and the last one decides
      uint64_t* s_key = red + kPrepThreads / 32 + 1;  // (after the flag `last`)
      if (tid == 0) {
        uint64_t b2 = 0;
        for (int w2 = 0; w2 < kPrepThreads / 32; ++w2) b2 = red[w2] > b2 ? red[w2] : b2;
        if (splits == 1) {
          uo[u].key[p.kpar] = b2;
          *s_key = b2;
          *last = 1;
        } else {
          if (b2) atomicMax(&uo[u].key[p.kpar], (unsigned long long)b2);
          __threadfence();
          *last = atomicAdd(&uo[u].arrived, 1) == splits - 1;
          __threadfence();
          if (*last) *s_key = __ldcg(&uo[u].key[p.kpar]);
        }
      }
      __syncthreads();
      HE_STAMP(0, 5);
      if (*last) {
        // the unit's eviction is decided: hand merge the evicted slot's logits
        // and value row, so that merge needs no dependent load
        const int winner = (int)evict_key_slot(*s_key);
        if constexpr (CH) {
          // the chunk's softmax parts (see ChunkRec): every key and value row
          // of the chunk loaded at once (rows i = warp, warp + 4, ...), the
          // logits, then per part and head the max, the sum and the accumulator
          using CR = ChunkRec<G, D>;
          constexpr int E = D / 32;  // elements of a row per lane
          float* co = reinterpret_cast<float*>(p.cstar) + (size_t)u * CR::FLOATS;
          // (a chunk outside the budget cannot be chosen; merge reports it)
          const int c = (winner >= 0 && winner + p.chunk <= p.lbudget) ? p.chunk : 0;
          // the item's code buffer is free now: logits [16][8], maxima [2][8],
          // weights [16][8] (fp32), value rows [16][D] (bf16)
          float* sl = reinterpret_cast<float*>(smem + S::OFF_C);
          float* sm = sl + kMaxChunk * 8;
          float* sw = sm + 16;
          uint16_t* sv = reinterpret_cast<uint16_t*>(sw + kMaxChunk * 8);
          const size_t rb = ((size_t)u * p.budget + winner) * D + (size_t)lane * E;
          uint32_t kr[kMaxChunk / 4][E / 2], vr[kMaxChunk / 4][E / 2];
#pragma unroll
          for (int r = 0; r < kMaxChunk / 4; ++r) {
            const int i = warp + 4 * r;
            if (i < c) {
              const uint32_t* kp = reinterpret_cast<const uint32_t*>(
                  reinterpret_cast<const uint16_t*>(p.K) + rb + (size_t)i * D);
              const uint32_t* vp = reinterpret_cast<const uint32_t*>(
                  reinterpret_cast<const uint16_t*>(p.V) + rb + (size_t)i * D);
#pragma unroll
              for (int e = 0; e < E / 2; ++e) {
                kr[r][e] = __ldcg(kp + e);
                vr[r][e] = __ldcg(vp + e);
              }
            }
          }
#pragma unroll
          for (int r = 0; r < kMaxChunk / 4; ++r) {
            const int i = warp + 4 * r;
            if (i < c) {
#pragma unroll
              for (int g = 0; g < G; ++g) {
                float a = 0.0f;
#pragma unroll
                for (int e = 0; e < E / 2; ++e) {
                  a = fmaf(__uint_as_float((uint32_t)xs[g * D + lane * E + 2 * e] << 16),
                           bf16_lo(kr[r][e]), a);
                  a = fmaf(__uint_as_float((uint32_t)xs[g * D + lane * E + 2 * e + 1] << 16),
                           bf16_hi(kr[r][e]), a);
                }
                a = warp_sum(a);
                if (lane == 0) sl[i * 8 + g] = a * p.qscale;
              }
#pragma unroll
              for (int e = 0; e < E / 2; ++e)
                reinterpret_cast<uint32_t*>(sv + i * D + lane * E)[e] = vr[r][e];
            }
          }
          __syncthreads();
          const int t0 = winner / p.tile;
          auto part_of = [&](int i) { return (winner + i) / p.tile != t0 ? 1 : 0; };
          if (tid < 2 * G) {
            const int part = tid / G, g = tid - part * G;
            float m = -1e30f;
            for (int i = 0; i < c; ++i)
              if (part_of(i) == part) m = fmaxf(m, sl[i * 8 + g]);
            float l = 0.0f;
            for (int i = 0; i < c; ++i)
              if (part_of(i) == part) l += exp2f(sl[i * 8 + g] - m);
            sm[part * 8 + g] = m;
            co[CR::M + part * 8 + g] = m;
            co[CR::L + part * 8 + g] = l;
          }
          __syncthreads();
          if (tid < c * G) {
            const int i = tid / G, g = tid - i * G;
            sw[i * 8 + g] = exp2f(sl[i * 8 + g] - sm[part_of(i) * 8 + g]);
          }
          __syncthreads();
          for (int idx = tid; idx < 2 * G * D; idx += kPrepThreads) {
            const int part = idx / (G * D), rem = idx - part * (G * D);
            const int g = rem / D, d = rem - g * D;
            float a = 0.0f;
            for (int i = 0; i < c; ++i)
              if (part_of(i) == part)
                a = fmaf(sw[i * 8 + g], __uint_as_float((uint32_t)sv[i * D + d] << 16), a);
            co[CR::A + idx] = a;
          }
          if (tid == 0) uo[u].arrived = 0;
        } else {
          const uint16_t* Krow =
              reinterpret_cast<const uint16_t*>(p.K) + ((size_t)u * p.budget + winner) * D;
          const uint16_t* Vrow =
              reinterpret_cast<const uint16_t*>(p.V) + ((size_t)u * p.budget + winner) * D;
          // the value row (and scale) and the key row are loaded together: one
          // memory round trip (D <= kPrepThreads: one value element per thread)
          static_assert(D <= kPrepThreads, "one value element per thread");
          uint16_t vh = 0;
          uint8_t vb = 0;
          float vsc = 0.0f;
          if constexpr (VQ) {
            if (tid < D) vb = __ldcg(reinterpret_cast<const uint8_t*>(p.V) +
                                     ((size_t)u * p.budget + winner) * D + tid);
            if (tid == 0) vsc = __ldcg(p.vs + (size_t)u * p.vs_stride + winner);
          } else {
            if (tid < D) vh = __ldcg(Vrow + tid);
          }
          constexpr int KE = D / 32;  // key elements per lane
          uint16_t kv[KE];
#pragma unroll
          for (int e = 0; e < KE; ++e) kv[e] = __ldcg(Krow + lane + 32 * e);
          for (int g = warp; g < G; g += kPrepThreads / 32) {
            float a = 0.0f;
#pragma unroll
            for (int e = 0; e < KE; ++e)
              a = fmaf(__uint_as_float((uint32_t)xs[g * D + lane + 32 * e] << 16),
                       __uint_as_float((uint32_t)kv[e] << 16), a);
            a = warp_sum(a);
            if (lane == 0) uo[u].lstar[g] = a * p.qscale;
          }
          if constexpr (VQ) {
            if (tid < D) uo[u].vqstar[tid] = vb;
            if (tid == 0) uo[u].vsstar = vsc;
          } else {
            if (tid < D) uo[u].vstar[tid] = vh;
          }
          if (tid == 0 && splits > 1) uo[u].arrived = 0;
        }
      }
    }
    __syncthreads();  // the staging buffers are reused by the next item
  }
  HE_STAMP(0, 3);
  // this grid completes only after stream has, so that merge's wait on this
  // grid covers stream's partials too
  if (tid == 0) pdl_wait();
}

// Quantisation of value rows into a quantised value cache (one warp per row):
// row r of V_in [rows][D] (bf16) is slot r % n of unit r / n; s = max |v| /
// range (fp32 division), byte d = the code of v_d / s (fp32 division); a zero
// row gives s = 0 and codes 0.
template <int D, int VQ>
__global__ void __launch_bounds__(256) vq_fill_kernel(const uint16_t* __restrict__ V_in,
                                                      int64_t rows, int n, int budget,
                                                      uint8_t* Vq, float* vs, int vs_stride) {
  static_assert(VQ == kVqInt8 || VQ == kVqFp8, "a byte format");
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows;
       r += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int64_t u = r / n, sl = r - u * n;
    float v[E], m = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      v[e] = __uint_as_float((uint32_t)V_in[r * D + lane * E + e] << 16);
      m = fmaxf(m, fabsf(v[e]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    const float sc = __fdiv_rn(m, vq_range<VQ>());
    uint8_t* dst = Vq + ((size_t)u * budget + sl) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) dst[e] = sc > 0.0f ? vq_encode<VQ>(__fdiv_rn(v[e], sc)) : 0;
    if (lane == 0) vs[(size_t)u * vs_stride + sl] = sc;
  }
}

// ---------------------------------------------------------------------------
// stream
// ---------------------------------------------------------------------------
// Work of one step: the U units' tiles of 64 slots, split statically
// (stream-K): CTA c takes a contiguous range of the U * tpu tiles and keeps one
// partial per unit it touches (record c + u).
//
// A producer warp issues the loads; for every ring stage it writes a
// descriptor (unit, tile, flags, record) that the four consumer warps read
// after the stage's full barrier, and the unit's G query rows come into the
// stage with the first tile of each segment (TMA, so no consumer thread waits
// on a global load).  A sentinel descriptor ends the stream.  Consumer-wide
// synchronisation uses mbarriers with bounded waits, so a wait that gives up
// unwinds every warp without a hang.
constexpr int kL2PrefetchTiles = 1;  // tiles of the range prefetched into L2 before the wait
constexpr int kDescFirst = 1;  // first tile of a segment: load q, reset the state
constexpr int kDescLast = 2;   // last tile of a segment: write the partial
constexpr int kDescEnd = 4;    // no more tiles

// VQ: the value cache holds byte rows with one fp32 scale per slot (a stage is
// the bf16 K tile, the swizzled byte V tile and the tile's scales).  The value
// MMA runs in f16: each consumer warp converts its A fragments from the byte
// tile in registers (an exact conversion), and the weights carry the slots'
// scales times a power of two of the warp's.
// FUSED: the whole step in this kernel (he_fused.cuh): a hash warp after the
// producer warp, and the last CTA of each unit merges it.
template <int D, int G, int NS, int VQ = 0, bool FUSED = false>
struct StreamShape {
  static constexpr int NCW = 4;              // consumer warps
  static constexpr int NC = NCW * 32;        // consumer threads
  static constexpr int NT = NC + 32 + (FUSED ? 32 : 0);  // + the producer (and hash) warp
  static constexpr int TS = 16 * NCW;        // slots per tile
  static constexpr int NHALF = D / 64;       // 128-byte column boxes per row
  static constexpr int BOXB = TS * 128;      // bytes per TMA box
  static constexpr int TILEB = NHALF * BOXB; // bytes per K (or V) tile
  static constexpr int VQT = TS * D;         // VQ: bytes of the V tile
  static constexpr int SCB = TS * 4;         // VQ: bytes of the tile's scales
  static constexpr int STAGEB = VQ ? (TILEB + VQT + SCB + 1023) / 1024 * 1024 : 2 * TILEB;
  static constexpr int QB = G * D * 2;       // the unit's query rows (bf16)
  static constexpr int KS = D / 16;          // k-steps of the logit MMA
  static constexpr int MT = D / 16;          // d blocks of the value MMA
  static constexpr int PB = 8 * 16 * 2;      // bytes of one P^T block [8 heads][16 slots] bf16 (VQ: f16)
  // floats of the warp-merge area (FUSED: also the merge's recompute scratch)
  static constexpr int WACC = NCW * G * (D + (FUSED ? 2 : 0));
  static constexpr int OFF_STAGE = 0;        // 1024-byte aligned (128B swizzle)
  static constexpr int OFF_Q = NS * STAGEB;  // [NS][QB]
  static constexpr int OFF_WACC = (OFF_Q + NS * QB + 15) / 16 * 16;
  static constexpr int OFF_P = OFF_WACC + WACC * 4;
  static constexpr int OFF_WM = OFF_P + NCW * 2 * PB;
  static constexpr int OFF_DESC = OFF_WM + 2 * NCW * G * 4;  // int4 [NS]
  // abort, issued, producer done, hash done, merge flag, last contributor, pad[2]
  static constexpr int OFF_FLAG = OFF_DESC + 16 * NS;
  static constexpr int OFF_BAR = OFF_FLAG + 32;             // full[NS], empty[NS], sync[3]
  static constexpr int OFF_PREW = OFF_BAR + (2 * NS + 3) * 8;  // int [NS]
  // FUSED: the hash warp's copy of W (up to 64 bits; a bulk-copy destination,
  // so 16-byte aligned) and its barrier
  static constexpr int OFF_W = (OFF_PREW + 16 + 127) / 128 * 128;
  static constexpr int WB = FUSED ? D * 64 * 2 : 0;
  static constexpr int OFF_WBAR = OFF_W + WB;
  static constexpr int OFF_XS = OFF_WBAR + 16;  // FUSED: the hash warp's rows, fp32 [G + 1][D]
  static constexpr int SMEM = FUSED ? OFF_XS + (G + 1) * D * 4 : OFF_WBAR;
  static_assert(OFF_Q % 16 == 0 && OFF_DESC % 16 == 0 && OFF_BAR % 8 == 0 && OFF_W % 16 == 0 &&
                    OFF_WBAR % 8 == 0 && OFF_P % 16 == 0 && OFF_WACC % 16 == 0 &&
                    OFF_XS % 16 == 0,
                "shared-memory alignment (bulk copies 16 bytes, mbarriers 8)");
  static_assert(NS <= 4, "written-slot table");
  static constexpr int SMEM_ALLOC = SMEM + 1024;  // slack to align the base to 1024
  static_assert(D % 64 == 0 && G >= 1 && G <= 8 && (G & (G - 1)) == 0, "shape");
  static_assert(STAGEB % 1024 == 0 && BOXB % 1024 == 0 && QB % 16 == 0, "alignment");
};

template <int D, int G, int NS, bool PSPLIT, int VQ = 0, bool FUSED = false>
__global__ void __launch_bounds__(StreamShape<D, G, NS, VQ, FUSED>::NT, 2)
    stream_kernel(const StepParams p, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV) {
  static_assert(!(FUSED && VQ), "the fused step keeps bf16 values");
  using S = StreamShape<D, G, NS, VQ, FUSED>;
  using R = std::conditional_t<FUSED, FRec<G, D>, PRec<G, D>>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* stage = smem + S::OFF_STAGE;
  const unsigned char* qstage = smem + S::OFF_Q;
  float* wacc = reinterpret_cast<float*>(smem + S::OFF_WACC);
  float* wm = reinterpret_cast<float*>(smem + S::OFF_WM);
  float* wl = wm + S::NCW * G;
  int4* desc = reinterpret_cast<int4*>(smem + S::OFF_DESC);
  volatile int32_t* v_abort = reinterpret_cast<int32_t*>(smem + S::OFF_FLAG);
  volatile int32_t* v_issued = v_abort + 1;   // stages issued (descriptors written)
  volatile int32_t* v_prod_done = v_abort + 2;
  volatile int32_t* v_hash_done = v_abort + 3;  // FUSED: segments the hash warp finished
  int* s_flag = const_cast<int*>(reinterpret_cast<volatile int*>(v_abort + 4));
  volatile int32_t* v_last = v_abort + 5;  // FUSED: this CTA is the unit's last contributor
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + S::OFF_BAR);
  uint64_t* empty_bar = full_bar + NS;
  uint64_t* sync_bar = empty_bar + NS;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tps = p.tpu;
  const TileSplit split{(int64_t)p.U * tps, (int64_t)gridDim.x, p.split_e, p.split_t1};
  const int sb = (int)split.begin(blockIdx.x);
  const int se = (int)split.begin((int64_t)blockIdx.x + 1);
  // tiles fetched before the wait (none after a step that moved whole rows)
  const int npre = p.nopre ? 0 : (se - sb < NS ? se - sb : NS);

  // one stage: its descriptor, then (unless it is the sentinel) K, V and, at a
  // segment's first tile, the unit's query rows, all on the stage's barrier
  // the K/V tiles are read once per step: evict them from L2 first, so that
  // the small data re-read within the step (partial records, prep's results,
  // codes) stays resident for merge and prep
  const uint64_t l2pol = l2_evict_first_policy();
  auto put = [&](int k, int u, int lt, int flags, int rec) {
    const int st = k % NS;
    desc[st] = make_int4(u, lt, flags, rec);
    const int y = u * p.budget + lt * S::TS;
    if ((flags & kDescEnd) ||
        !HE_CHECK(u >= 0 && u < p.U && lt >= 0 &&
                      (int64_t)y + S::TS <= (int64_t)p.U * p.budget + S::TS &&
                      (!VQ || (lt + 1) * S::TS <= p.vs_stride),
                  p.err)) {
      mbar_arrive(&full_bar[st]);  // (a failed check: the stage is left as it was)
    } else {
      unsigned char* dst = stage + st * S::STAGEB;
      constexpr uint32_t tile_bytes = VQ ? S::TILEB + S::VQT + S::SCB : 2 * S::TILEB;
      mbar_arrive_expect_tx(&full_bar[st],
                            tile_bytes + ((flags & kDescFirst) ? (uint32_t)S::QB : 0u));
      if (flags & kDescFirst)
        bulk_g2s(const_cast<unsigned char*>(qstage) + st * S::QB,
                 reinterpret_cast<const uint16_t*>(p.q) + (size_t)u * G * D, (uint32_t)S::QB,
                 &full_bar[st]);
#pragma unroll
      for (int h = 0; h < S::NHALF; ++h)
        tma_load_2d_hint(dst + h * S::BOXB, &tmK, 64 * h, y, &full_bar[st], l2pol);
      if constexpr (VQ) {
        tma_load_2d_hint(dst + S::TILEB, &tmV, 0, y, &full_bar[st], l2pol);
        bulk_g2s(dst + S::TILEB + S::VQT, p.vs + (size_t)u * p.vs_stride + (size_t)lt * S::TS,
                 (uint32_t)S::SCB, &full_bar[st]);
      } else {
#pragma unroll
        for (int h = 0; h < S::NHALF; ++h)
          tma_load_2d_hint(dst + S::TILEB + h * S::BOXB, &tmV, 64 * h, y, &full_bar[st], l2pol);
      }
    }
    *v_issued = k + 1;
  };
  auto put_static = [&](int k) {
    const int t = sb + k;
    const int u = t / tps, lt = t - u * tps;
    const int flags = ((k == 0 || lt == 0) ? kDescFirst : 0) |
                      ((t == se - 1 || lt == tps - 1) ? kDescLast : 0);
    put(k, u, lt, flags, (int)blockIdx.x + u);
  };

  HE_STAMP(1, 0);
  // The first tiles are fetched while the previous step's merge may still be
  // writing: every cache row but the one slot per unit that it overwrites is
  // final already, and the consumers re-read that row after the wait.  (The
  // query rows are this step's input, final before the launch.)  Which slot
  // that is, is final too (the previous step's eviction key, or the host's
  // append slot), so it is read here, while the first tiles are in flight.
  int32_t* prew = reinterpret_cast<int32_t*>(smem + S::OFF_PREW);
  if (warp == S::NCW && lane == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], S::NCW);
    }
    mbar_init(&sync_bar[0], S::NCW);
    mbar_init(&sync_bar[1], S::NCW);
    mbar_init(&sync_bar[2], S::NCW);
    v_abort[0] = 0;
    v_issued[0] = 0;
    v_prod_done[0] = 0;
    v_hash_done[0] = 0;
    v_abort[4] = 0;
    v_abort[5] = 0;
    if constexpr (FUSED) mbar_init(reinterpret_cast<uint64_t*>(smem + S::OFF_WBAR), 1);
    fence_mbar_init();
  }
  if constexpr (FUSED) {
    // the barriers and flags are set up; the hash warp goes its own way (it
    // does its own dependency wait once its work before the wait is done)
    __syncthreads();
    if (warp == S::NCW + 1) {
      hash_warp<D, G>(p, sb, se, v_hash_done, lane, reinterpret_cast<uint16_t*>(smem + S::OFF_W),
                      reinterpret_cast<uint64_t*>(smem + S::OFF_WBAR),
                      reinterpret_cast<float*>(smem + S::OFF_XS));
      return;
    }
  }
  if (warp == S::NCW && lane == 0) {
    for (int k = 0; k < npre; ++k) put_static(k);
    // the next tile of the range into L2 as well, while the previous step's
    // merge (latency bound, little DRAM traffic) finishes: a stale copy of the
    // one row that merge overwrites is harmless, L2 sees merge's write
    const int pfe =
        p.nopre ? 0 : (se - sb < npre + kL2PrefetchTiles ? se - sb : npre + kL2PrefetchTiles);
    for (int k = npre; k < pfe; ++k) {
      const int t = sb + k;
      const int u = t / tps, lt = t - u * tps;
      const int y = u * p.budget + lt * S::TS;
#pragma unroll
      for (int h = 0; h < S::NHALF; ++h) {
        tma_prefetch_2d(&tmK, 64 * h, y);
        if constexpr (!VQ) tma_prefetch_2d(&tmV, 64 * h, y);
      }
      if constexpr (VQ) tma_prefetch_2d(&tmV, 0, y);
    }
  }
  if (tid < npre) {
    const int u = (sb + tid) / tps;  // the unit of tile tid
    int w = -1;
    if (p.prev_w1 > 0) {
      w = p.prev_w1 - 1;  // the previous step appended here
    } else if (p.prev_w1 < 0 && p.uo != nullptr) {
      if constexpr (FUSED) {
        // the previous step's key is final once all its hash warps counted in
        // (they do so early in that step); if not yet, read the slot after the wait
        if (ld_acquire_gpu(&p.uo[u].hcnt[p.kpar ^ 1]) == prev_hash_count(p, u)) {
          const unsigned long long key = __ldcg(&p.uo[u].key[p.kpar ^ 1]);
          w = key ? (int)evict_key_slot(key) : -1;
        } else {
          w = -2;
        }
      } else {
        const unsigned long long key = __ldcg(&p.uo[u].key[p.kpar ^ 1]);
        w = key ? (int)evict_key_slot(key) : -1;
      }
    }
    prew[tid] = w;
  }
  group_sync<S::NC + 32, FUSED ? 1 : 0>();  // (FUSED: the hash warp has gone its own way)
  pdl_wait();     // the previous step is complete: the cache is final
  HE_STAMP_IF(FUSED && tid == 0, 1, 2);
  pdl_trigger();  // prep may launch now: its CTAs take the room stream leaves

  // ---------------- producer warp ----------------
  if (warp == S::NCW) {
    if (lane == 0) {
      int k = npre;
      bool ok = true;
      auto acquire = [&](int kk) {  // the stage of kk is free again
        if (kk >= NS && !mbar_wait_bounded(&empty_bar[kk % NS], (uint32_t)(((kk / NS) - 1) & 1))) {
          atomicExch(p.err, 1);
          *v_abort = 1;
          return false;
        }
        return *v_abort == 0;
      };
      for (; k < se - sb && ok; ++k) {
        ok = acquire(k);
        if (ok) put_static(k);
      }
      if (ok && acquire(k)) put(k, -1, 0, kDescEnd, 0);
      __threadfence_block();
      *v_prod_done = 1;
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
  const int row0 = 16 * cw;

  uint32_t qb[S::KS][2];
  float mrun0 = -1e30f, mrun1 = -1e30f, lrun0 = 0.0f, lrun1 = 0.0f;
  float acc[S::MT][4];
  int wslot = -1;
  int ew = kVqExpMax;  // VQ: the warp's weight exponent in this segment
  uint32_t sync_phase[3] = {0u, 0u, 0u};
  int seg = 0;     // FUSED: segments finished by this CTA
  int merges = 0;  // FUSED: units this CTA merged
  int k = 0;
  bool aborted = false;
  for (;; ++k) {
    const int st = k % NS;
    if (!mbar_wait_bounded(&full_bar[st], (uint32_t)((k / NS) & 1))) {
      atomicExch(p.err, 1);
      *v_abort = 1;
      aborted = true;
      break;
    }
    const int4 dsc = desc[st];
    if (dsc.z & kDescEnd) break;
    const int u = dsc.x, lt = dsc.y;
    const unsigned char* Ks = stage + st * S::STAGEB;
    const unsigned char* Vs = Ks + S::TILEB;
    const int slot_base = lt * S::TS + row0;
    const int hi = p.occ;

    if (dsc.z & kDescFirst) {
      // query fragments (B operand of the logit MMA): head g8, d = 16ks + 8r + 2t4 (+1)
      const uint32_t* qw = reinterpret_cast<const uint32_t*>(qstage + st * S::QB);
#pragma unroll
      for (int ks = 0; ks < S::KS; ++ks)
#pragma unroll
        for (int r = 0; r < 2; ++r)
          qb[ks][r] = g8 < G ? qw[(g8 * D + 16 * ks + 8 * r + 2 * t4) / 2] : 0u;
      mrun0 = mrun1 = -1e30f;
      lrun0 = lrun1 = 0.0f;
#pragma unroll
      for (int mt = 0; mt < S::MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.0f;
      ew = kVqExpMax;
      // the slot the previous step of this cache wrote in unit u (the evicted
      // slot, or the last appended one): stale in a tile fetched before the wait
      wslot = k < npre ? prew[k] : -1;
      if (FUSED && wslot == -2) wslot = __ldcg(&p.evicted[u]);  // (final after the wait)
    }
    if (VQ && k < npre && (unsigned)(wslot - slot_base) < 16u &&
        HE_CHECK(wslot < p.budget, p.err)) {
      // re-read the row written by the previous step (now visible) into the
      // tile: its bf16 key (swizzled), byte value row and scale
      const int row = wslot - lt * S::TS;
      constexpr int CK = D / 8, CV = D / 16;  // 16-byte chunks of the key and value rows
      const size_t r = (size_t)u * p.budget + wslot;
      unsigned char* Kd = const_cast<unsigned char*>(Ks);
      if (lane < CK) {
        const uint4 x = __ldcg(reinterpret_cast<const uint4*>(
            reinterpret_cast<const uint16_t*>(p.K) + r * D + 8 * lane));
        *reinterpret_cast<uint4*>(Kd + (lane >> 3) * S::BOXB + row * 128 +
                                  (((lane & 7) ^ (row & 7)) << 4)) = x;
      } else if (lane < CK + CV) {
        const int c = lane - CK;
        const uint4 x = __ldcg(reinterpret_cast<const uint4*>(
            reinterpret_cast<const uint8_t*>(p.V) + r * D + 16 * c));
        *reinterpret_cast<uint4*>(Kd + S::TILEB + vq_tile_off<D>(row, 16 * c)) = x;
      } else if (lane == CK + CV) {
        *reinterpret_cast<float*>(Kd + S::TILEB + S::VQT + 4 * row) =
            __ldcg(p.vs + (size_t)u * p.vs_stride + wslot);
      }
      fence_proxy_async_smem();  // the stage is refilled by TMA later
      __syncwarp();
    }
    if (!VQ && k < npre && (unsigned)(wslot - slot_base) < 16u &&
        HE_CHECK(wslot < p.budget, p.err)) {
      // re-read the row written by the previous step (now visible) into the tile
      const int row = wslot - lt * S::TS;
      constexpr int CH = D / 8;  // 16-byte chunks per row
      if (lane < 2 * CH) {
        const int c = lane < CH ? lane : lane - CH;
        const uint16_t* src = reinterpret_cast<const uint16_t*>(lane < CH ? p.K : p.V) +
                              ((size_t)u * p.budget + wslot) * D + 8 * c;
        const uint4 x = __ldcg(reinterpret_cast<const uint4*>(src));
        unsigned char* dst = const_cast<unsigned char*>(lane < CH ? Ks : Vs) +
                             (c >> 3) * S::BOXB + row * 128 + (((c & 7) ^ (row & 7)) << 4);
        *reinterpret_cast<uint4*>(dst) = x;
        fence_proxy_async_smem();  // the stage is refilled by TMA later
      }
      __syncwarp();
    }

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
    if (sA >= hi) x00 = x01 = -INFINITY;
    if (sB >= hi) x10 = x11 = -INFINITY;
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
    // VQ: the value MMA's weights are p * s * 2^ew in f16, ew the largest
    // exponent (at most kVqExpMax) that keeps the warp's largest scale times
    // 2^ew below 2^15 in every tile so far (weights p <= 1: no f16 overflow);
    // the accumulator holds 2^ew times the values' sum, and shrinking ew
    // rescales it (exact powers of two)
    float sa = 0.0f, sb = 0.0f, fvq = 1.0f;
    if constexpr (VQ) {
      const float* scl = reinterpret_cast<const float*>(Ks + S::TILEB + S::VQT);
      sa = sA < hi ? scl[row0 + g8] : 0.0f;
      sb = sB < hi ? scl[row0 + g8 + 8] : 0.0f;
      float smx = fmaxf(sa, sb);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) smx = fmaxf(smx, __shfl_xor_sync(kFull, smx, o));
      // smx in [2^(E-127), 2^(E-126)) for its biased exponent E >= 1
      const int en = smx > 0.0f ? min(141 - ((__float_as_int(smx) >> 23) & 0xFF), kVqExpMax)
                                : kVqExpMax;
      if (en < ew) {
        fvq = en - ew >= -126 ? __int_as_float((127 + en - ew) << 23) : 0.0f;
        ew = en;
      }
    }
    const float ac0 = sc0 * fvq, ac1 = sc1 * fvq;
#pragma unroll
    for (int mt = 0; mt < S::MT; ++mt) {
      acc[mt][0] *= ac0;
      acc[mt][2] *= ac0;
      acc[mt][1] *= ac1;
      acc[mt][3] *= ac1;
    }

    // P^T [8 heads][16 slots] in bf16 (hi, and the rounding remainder lo); with
    // a quantised value cache in f16, each slot's weight times its scale and 2^ew
    if constexpr (VQ) {
      const float pw = __int_as_float((127 + ew) << 23);
      const float ea = sa * pw, eb = sb * pw;  // (exact)
      const float w00 = p00 * ea, w01 = p01 * ea, w10 = p10 * eb, w11 = p11 * eb;
      __half* Ph = reinterpret_cast<__half*>(Phi);
      __half* Pl = reinterpret_cast<__half*>(Plo);
      const __half a00 = __float2half_rn(w00), a01 = __float2half_rn(w01);
      const __half a10 = __float2half_rn(w10), a11 = __float2half_rn(w11);
      Ph[h0 * 16 + g8] = a00;
      Ph[h1 * 16 + g8] = a01;
      Ph[h0 * 16 + g8 + 8] = a10;
      Ph[h1 * 16 + g8 + 8] = a11;
      if (PSPLIT) {
        Pl[h0 * 16 + g8] = __float2half_rn(w00 - __half2float(a00));
        Pl[h1 * 16 + g8] = __float2half_rn(w01 - __half2float(a01));
        Pl[h0 * 16 + g8 + 8] = __float2half_rn(w10 - __half2float(a10));
        Pl[h1 * 16 + g8 + 8] = __float2half_rn(w11 - __half2float(a11));
      }
    } else {
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
    // VQ: this thread's value words, the value MMA's A fragments before
    // conversion.  Block mt = 4 q + i of the MMA takes row g8 + 8 h as
    // d = 64 q + 32 h + 4 g8 + i, so one 32-bit word of a slot row holds a
    // thread's four blocks; its slots are the fragment's columns 2 t4, 2 t4 + 1,
    // 2 t4 + 8, 2 t4 + 9.  Then the stage is free.
    uint32_t wv[VQ ? D / 64 : 1][2][4];
    if constexpr (VQ) {
      const unsigned char* vt = Ks + S::TILEB;
#pragma unroll
      for (int q = 0; q < D / 64; ++q)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int s = row0 + 2 * t4 + (j & 1) + 8 * (j >> 1);
            wv[q][h][j] = *reinterpret_cast<const uint32_t*>(
                vt + vq_tile_off<D>(s, 64 * q + 32 * h + 4 * g8));
          }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[st]);  // stage free for refill
    }
    __syncwarp();
    const uint32_t* Phw = reinterpret_cast<const uint32_t*>(Phi);
    const uint32_t* Plw = reinterpret_cast<const uint32_t*>(Plo);
    const uint32_t bh0 = Phw[g8 * 8 + t4], bh1 = Phw[g8 * 8 + 4 + t4];
    const uint32_t bl0 = PSPLIT ? Plw[g8 * 8 + t4] : 0u;
    const uint32_t bl1 = PSPLIT ? Plw[g8 * 8 + 4 + t4] : 0u;

    // values: O^T[d][head] += V^T[d][slots] P^T[slots][head]
    if constexpr (VQ) {
#pragma unroll
      for (int q = 0; q < D / 64; ++q) {
        uint32_t r0[4], r1[4], r2[4], r3[4];
        vq_pairs_f16<VQ>(wv[q][0][0], wv[q][0][1], r0);  // row g8, columns 2 t4, 2 t4 + 1
        vq_pairs_f16<VQ>(wv[q][1][0], wv[q][1][1], r1);  // row g8 + 8
        vq_pairs_f16<VQ>(wv[q][0][2], wv[q][0][3], r2);  // row g8, columns 2 t4 + 8, + 9
        vq_pairs_f16<VQ>(wv[q][1][2], wv[q][1][3], r3);  // row g8 + 8
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t a[4] = {r0[i], r1[i], r2[i], r3[i]};
          mma_f16_16816(acc[4 * q + i], a, bh0, bh1);
          if (PSPLIT) mma_f16_16816(acc[4 * q + i], a, bl0, bl1);
        }
      }
    } else {
#pragma unroll
      for (int mt = 0; mt < S::MT; ++mt) {
        const int row = row0 + (lane & 7) + ((lane >> 4) << 3);
        const int chunk = ((mt & 3) << 1) + ((lane >> 3) & 1);
        uint32_t a[4];
        ldsm_x4_trans(a, smem_u32(Vs + (mt >> 2) * S::BOXB + row * 128 + ((chunk ^ (row & 7)) << 4)));
        mma_bf16_16816(acc[mt], a, bh0, bh1);
        if (PSPLIT) mma_bf16_16816(acc[mt], a, bl0, bl1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[st]);  // stage free for refill
    }

    if (dsc.z & kDescLast) {
      // warp states -> shared memory -> the partial record of this segment
      float l0 = lrun0, l1 = lrun1;
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        l0 += __shfl_xor_sync(kFull, l0, o);
        l1 += __shfl_xor_sync(kFull, l1, o);
      }
      if (g8 == 0) {
        if (real0) {
          wm[cw * G + h0] = mrun0;
          wl[cw * G + h0] = l0;
        }
        if (real1) {
          wm[cw * G + h1] = mrun1;
          wl[cw * G + h1] = l1;
        }
      }
      // (VQ: the accumulator holds 2^ew times the sums, its rows in the value
      // MMA's column order)
      const float uvq = VQ ? __int_as_float((127 - ew) << 23) : 1.0f;
#pragma unroll
      for (int mt = 0; mt < S::MT; ++mt) {
        const int d = VQ ? 64 * (mt >> 2) + 4 * g8 + (mt & 3) : 16 * mt + g8;
        const int d8 = VQ ? d + 32 : d + 8;
        if (real0) {
          wacc[(cw * G + h0) * D + d] = acc[mt][0] * uvq;
          wacc[(cw * G + h0) * D + d8] = acc[mt][2] * uvq;
        }
        if (real1) {
          wacc[(cw * G + h1) * D + d] = acc[mt][1] * uvq;
          wacc[(cw * G + h1) * D + d8] = acc[mt][3] * uvq;
        }
      }
      if (!consumer_sync<S::NCW>(&sync_bar[0], sync_phase[0], lane)) {
        atomicExch(p.err, 1);
        *v_abort = 1;
        aborted = true;
        break;
      }
      float* rec = p.partials +
                   (size_t)(HE_CHECK(dsc.w >= 0 && dsc.w < (int)gridDim.x + p.U, p.err) ? dsc.w : 0) *
                       R::FLOATS;
      for (int idx = tid; idx < G * D; idx += S::NC) {
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
      // the merge area is reused by the next segment
      if (!consumer_sync<S::NCW>(&sync_bar[1], sync_phase[1], lane)) {
        atomicExch(p.err, 1);
        *v_abort = 1;
        aborted = true;
        break;
      }
      if constexpr (FUSED) {
        // the segment's state is written: the next tile starts a segment, so
        // these hold nothing while this CTA counts in and perhaps merges
        mrun0 = mrun1 = -1e30f;
        lrun0 = lrun1 = 0.0f;
#pragma unroll
        for (int mt = 0; mt < S::MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.0f;
#pragma unroll
        for (int ks = 0; ks < S::KS; ++ks) qb[ks][0] = qb[ks][1] = 0u;
        // count in once the hash warp has stored this segment's candidate; the
        // unit's last contributor merges it
        int first, n;
        unit_contributors(split, u, tps, first, n);
        if (tid == 0) {
          *v_last = 0;
          const uint64_t t0 = global_ns();
          HE_STAMP_IF(true, 1, 3);
          while (*v_hash_done <= seg && global_ns() - t0 < 2000000000ull) {
          }
          HE_STAMP_IF(true, 1, 4);
          if (*v_hash_done <= seg) {
            atomicExch(p.err, 1);
            *v_abort = 1;
          } else {
            const int prev = atom_add_acq_rel_gpu(&p.uo[u].arrived, 1);
            *v_last = prev == n - 1 ? 1 : 0;
          }
          HE_STAMP_IF(true, 1, 5);
        }
        if (!consumer_sync<S::NCW>(&sync_bar[2], sync_phase[2], lane) || *v_abort) {
          atomicExch(p.err, 1);
          *v_abort = 1;
          aborted = true;
          break;
        }
        if (*v_last &&
            !fused_merge<D, G, S::NCW>(p, split, u, first, n, wacc, s_flag, ++merges, tid,
                                       &sync_bar[2], sync_phase[2])) {
          atomicExch(p.err, 1);
          *v_abort = 1;
          aborted = true;
          break;
        }
        HE_STAMP_IF(tid == 0 && *v_last, 1, 6);
        ++seg;
      }
    }
  }
  if constexpr (FUSED) {
    // an empty cache (no tiles; CTA u per unit): the new token alone
    if (!aborted && p.tpu == 0) {
      if (tid == 0) {
        const uint64_t t0 = global_ns();
        while (*v_hash_done < 1 && global_ns() - t0 < 2000000000ull) {
        }
        if (*v_hash_done < 1) {
          atomicExch(p.err, 1);
          *v_abort = 1;
        }
      }
      if (!consumer_sync<S::NCW>(&sync_bar[2], sync_phase[2], lane) || *v_abort ||
          !fused_merge<D, G, S::NCW>(p, split, (int)blockIdx.x, 0, 0, wacc, s_flag, ++merges,
                                     tid, &sync_bar[2], sync_phase[2])) {
        atomicExch(p.err, 1);
        *v_abort = 1;
        aborted = true;
      }
    }
  }
  if (aborted && tid == 0) {
    // a wait gave up: once the producer has stopped, let every copy it issued
    // land before the CTA's shared memory is released
    const uint64_t t0 = global_ns();
    while (*v_prod_done == 0 && global_ns() - t0 < 500000000ull) {
    }
    const int issued = *v_issued;
    for (int r = issued - NS > 0 ? issued - NS : 0; r < issued; ++r)
      (void)mbar_wait_bounded(&full_bar[r % NS], (uint32_t)((r / NS) & 1), 500000000ull);
  }
  HE_STAMP(1, 1);
}

// ---------------------------------------------------------------------------
// merge
// ---------------------------------------------------------------------------
// A merge CTA has GD4 * NQ threads: NQ contributor groups of GD4 = G * D / 4
// threads (one float4 of the unit's output each).  Every shape runs 512
// threads.  A merge CTA fits beside two stream CTAs only with at most four
// warps of at most 64 registers (an SM's registers are four sub-partitions of
// 16384, and two stream CTAs put three warps of 136 registers on two of them);
// such CTAs, with the partial records staged in shared memory, let all the next
// step's stream CTAs start together but did not shorten the step.
constexpr int kMergeMaxThreads = 512;
constexpr int kMergeMinThreads = 512;
constexpr int kMergeRegs = 12;  // partials held in registers per thread (more are looped)
// Chunk eviction: the chunk is subtracted from its partials unless its weight
// exceeds this many times the weight that remains (every partial and the new
// token, per head); the subtraction's rounding error is then at most about
// (1 + this) times the partials' own relative error, else merge recomputes.
constexpr float kChunkRemoveMax = 16.0f;

template <int D, int G>
struct MergeShape {
  static constexpr int GD4 = G * D / 4;  // float4 outputs per unit
  static constexpr int NQ_MIN = GD4 >= kMergeMinThreads ? 1 : kMergeMinThreads / GD4;
  static constexpr int NQ_MAX = GD4 >= kMergeMaxThreads ? 1 : kMergeMaxThreads / GD4;
  static_assert(GD4 <= kMergeMaxThreads && D <= kMergeMinThreads, "merge shape");
  // threads for units with at most n partials each
  static int threads(int n) {
    int nq = (n + kMergeRegs - 1) / kMergeRegs;
    nq = nq < NQ_MIN ? NQ_MIN : (nq > NQ_MAX ? NQ_MAX : nq);
    return GD4 * nq;
  }
  // Launch shape for U units with at most n partials each: nq groups of GD4
  // threads per unit and upc units per CTA.  With `multi` a CTA takes up to
  // four units of ceil(n / kMergeRegs) groups each (and at least D threads)
  // when U is a multiple of that count; else one unit of threads(n) threads.
  static void config(int n, int U, bool multi, int* nq, int* upc) {
    // (at least D threads per unit: they write the new token's key and value rows)
    constexpr int QMIN = (D + GD4 - 1) / GD4;
    int q = (n + kMergeRegs - 1) / kMergeRegs;
    q = q < QMIN ? QMIN : (q > NQ_MAX ? NQ_MAX : q);
    if (multi) {
      int up = kMergeMaxThreads / (q * GD4);
      up = up >= 4 ? 4 : up;
      while (up > 1 && U % up != 0) --up;
      if (up > 1) {
        *nq = q;
        *upc = up;
        return;
      }
    }
    *nq = threads(n) / GD4;
    *upc = 1;
  }
};

// Exact partial over slots [lo, hi) of unit u without the slots [skip,
// skip + nskip) (CUDA cores, fp32): per head the base-2 max, sum and
// accumulator -> xm, xl, xa [G][D].
// Every warp of the CTA runs an online softmax over a strided share of the
// slots (lane owns D/32 elements), then the warp states merge in a fixed order.
template <int D, int G, int VQ>
__device__ void recompute_partial(const StepParams& p, int u, int lo, int hi, int skip,
                                  int nskip, const float* qf, float* wstate, float* xm, float* xl,
                                  float* xa, int tid) {
  constexpr int E = D / 32;
  const int RW = (int)(blockDim.x >> 5);
  const int lane = tid & 31, warp = tid >> 5;
  {
    const uint16_t* Kc = reinterpret_cast<const uint16_t*>(p.K) + (size_t)u * p.budget * D;
    // (a quantised value cache: bytes instead of bf16, one scale per slot)
    const uint16_t* Vc = VQ ? reinterpret_cast<const uint16_t*>(reinterpret_cast<const int8_t*>(p.V) +
                                                                (size_t)u * p.budget * D)
                            : reinterpret_cast<const uint16_t*>(p.V) + (size_t)u * p.budget * D;
    float mr[G], lr[G], ar[G][E];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      mr[g] = -1e30f;
      lr[g] = 0.0f;
#pragma unroll
      for (int e = 0; e < E; ++e) ar[g][e] = 0.0f;
    }
    // a warp takes RU consecutive slots at a time, every row of the group
    // loaded before any is used (one memory round trip per group); lane l
    // holds elements [l E, l E + E) of each row
    constexpr int RU = 4;
    for (int s0 = lo + warp * RU; s0 < hi; s0 += RW * RU) {
      float kx[RU][E], vx[RU][E];
#pragma unroll
      for (int r = 0; r < RU; ++r) {
        const int s = s0 + r < hi ? s0 + r : hi - 1;  // (a slot past the range is not folded)
        const size_t at = (size_t)s * D + lane * E;
        if constexpr (E == 4) {
          const uint2 kw = __ldcg(reinterpret_cast<const uint2*>(Kc + at));
          kx[r][0] = bf16_lo(kw.x);
          kx[r][1] = bf16_hi(kw.x);
          kx[r][2] = bf16_lo(kw.y);
          kx[r][3] = bf16_hi(kw.y);
        } else {
          const uint32_t kw = __ldcg(reinterpret_cast<const uint32_t*>(Kc + at));
          kx[r][0] = bf16_lo(kw);
          kx[r][1] = bf16_hi(kw);
        }
        if constexpr (VQ) {
          const int8_t* vb = reinterpret_cast<const int8_t*>(Vc) + at;
          const float sc = __ldcg(p.vs + (size_t)u * p.vs_stride + s);
#pragma unroll
          for (int e = 0; e < E; ++e) vx[r][e] = vq_decode<VQ>((uint8_t)__ldcg(vb + e)) * sc;
        } else if constexpr (E == 4) {
          const uint2 vw = __ldcg(reinterpret_cast<const uint2*>(Vc + at));
          vx[r][0] = bf16_lo(vw.x);
          vx[r][1] = bf16_hi(vw.x);
          vx[r][2] = bf16_lo(vw.y);
          vx[r][3] = bf16_hi(vw.y);
        } else {
          const uint32_t vw = __ldcg(reinterpret_cast<const uint32_t*>(Vc + at));
          vx[r][0] = bf16_lo(vw);
          vx[r][1] = bf16_hi(vw);
        }
      }
#pragma unroll
      for (int r = 0; r < RU; ++r) {
        const int s = s0 + r;
        if (s >= hi || (unsigned)(s - skip) < (unsigned)nskip) continue;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float dot = 0.0f;
#pragma unroll
          for (int e = 0; e < E; ++e) dot = fmaf(qf[g * D + lane * E + e], kx[r][e], dot);
          const float x = warp_sum(dot) * p.qscale;
          const float mn = fmaxf(mr[g], x);
          const float so = exp2f(mr[g] - mn), sn = exp2f(x - mn);
          lr[g] = lr[g] * so + sn;
#pragma unroll
          for (int e = 0; e < E; ++e) ar[g][e] = ar[g][e] * so + sn * vx[r][e];
          mr[g] = mn;
        }
      }
    }
    // warp state -> wstate [warp][G][2 + D]
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float* ws = wstate + ((size_t)warp * G + g) * (2 + D);
      if (lane == 0) {
        ws[0] = mr[g];
        ws[1] = lr[g];
      }
#pragma unroll
      for (int e = 0; e < E; ++e) ws[2 + lane * E + e] = ar[g][e];
    }
  }
  __syncthreads();
  for (int idx = tid; idx < G * D; idx += (int)blockDim.x) {
    const int g = idx / D, d = idx - g * D;
    float mx = -1e30f;
    for (int w = 0; w < RW; ++w) mx = fmaxf(mx, wstate[((size_t)w * G + g) * (2 + D)]);
    float a = 0.0f, l = 0.0f;
    for (int w = 0; w < RW; ++w) {
      const float* ws = wstate + ((size_t)w * G + g) * (2 + D);
      const float sc = exp2f(ws[0] - mx);
      a += ws[2 + d] * sc;
      l += ws[1] * sc;
    }
    xa[idx] = a;
    if (d == 0) {
      xm[g] = mx;
      xl[g] = l;
    }
  }
  __syncthreads();
}

// One CTA per unit.  Every load is issued up front (one memory round trip):
// thread (q, o) holds the partials of contributors c = q, q + NQ, ... (four
// outputs o each), folds them into a running (max, sum, accumulator), taking
// the evicted slot out of its partial; the NQ group states are merged in a
// fixed order, the new token is added, the output written and the slot
// overwritten.  If the evicted slot carries more than half of its partial's
// mass, that partial is recomputed exactly and the fold redone.

template <int D, int G>
__device__ __forceinline__ void fold_one(float mc, float lc, float4 x, bool is_crel,
                                         float lst, const float4& vs, float& mx, float& sum,
                                         float4& a) {
  if (is_crel) {  // take the evicted slot out (its weight is at most half)
    const float pw = exp2f(lst - mc);
    lc -= pw;
    x.x -= pw * vs.x;
    x.y -= pw * vs.y;
    x.z -= pw * vs.z;
    x.w -= pw * vs.w;
  }
  const float mn = fmaxf(mx, mc);
  const float so = exp2f(mx - mn), sn = exp2f(mc - mn);
  sum = sum * so + lc * sn;
  a.x = a.x * so + x.x * sn;
  a.y = a.y * so + x.y * sn;
  a.z = a.z * so + x.z * sn;
  a.w = a.w * so + x.w * sn;
  mx = mn;
}

// Chunk eviction: take part(s) of the evicted chunk (ChunkRec) out of a
// partial (mc, lc, x); returns the weight taken out, which the caller compares
// with half the partial's sum.
__device__ __forceinline__ float take_part(float cm, float cl, const float4& ca, float mc,
                                          float& lc, float4& x) {
  const float sc = exp2f(cm - mc);
  const float w = cl * sc;
  lc -= w;
  x.x -= ca.x * sc;
  x.y -= ca.y * sc;
  x.z -= ca.z * sc;
  x.w -= ca.w * sc;
  return w;
}

// CH: chunk eviction.  At a full step the key names the evicted chunk's first
// slot; its c slots leave the (at most two) partials that hold them, the
// staged rows [lbudget, lbudget + c - 1) move to the chunk's first c - 1
// slots and the new token takes its last.  Other steps append (stage) the
// token at p.append_slot, as the method does.
// MU: a CTA merges MT / (nq * GD4) units, one group of nq * GD4 threads each
// (for steps with more units than SMs: the merge CTAs then run in one wave
// instead of several); else one unit per CTA.
template <int D, int G, int VQ = 0, bool CH = false, bool MU = false>
__global__ void __launch_bounds__(kMergeMaxThreads)
    merge_kernel(const StepParams p, UnitOut* uo, int stream_ctas, int nq) {
  static_assert(!(CH && VQ), "chunk eviction keeps bf16 values");
  using R = PRec<G, D>;
  constexpr int GD4 = MergeShape<D, G>::GD4;
  const int MT = (int)blockDim.x, NQ = MU ? nq : MT / GD4, GT = NQ * GD4, UPC = MU ? MT / GT : 1;
  extern __shared__ __align__(16) unsigned char smem_merge[];
  float4* sacc = reinterpret_cast<float4*>(smem_merge);  // [MT]
  float* smax = reinterpret_cast<float*>(sacc + MT);      // [MT]
  float* ssum = smax + MT;                                // [MT]
  float* qf = ssum + MT;                                  // [G][D] query heads (fp32)
  float* xa = qf + G * D;                                           // [G][D] recomputed partial
  float* xm = xa + G * D;                                           // [8]
  float* xl = xm + 8;                                               // [8]
  int* sflag = reinterpret_cast<int*>(xl + 8);                      // [4] per group
  int* rparam = sflag + 4;                                          // [4][4] per group
  float* wstate = reinterpret_cast<float*>(rparam + 16);            // recompute scratch
  const int ctid = threadIdx.x;              // thread of the CTA
  const int grp = MU ? ctid / GT : 0;        // the unit group
  const int tid = ctid - grp * GT;           // thread of the group
  // VQ, per group: [D] the new row, [32] maxima
  float* vqrow = wstate + (MT / 32) * G * (2 + D) + grp * (D + 32);
  const int u = blockIdx.x * UPC + grp;
  const bool full = p.append_slot < 0;

  HE_STAMP(2, 0);
  pdl_wait();  // stream (and so prep) is complete and visible
  // the next step's stream kernel may launch (it waits for this grid): at once,
  // so that its first tiles load while this grid works, unless the units have
  // many partials each: then after this CTA's loads are issued, which go ahead
  // of that flood of tile loads (the loads of such units take longest)
  if (!p.late_release) pdl_trigger();
  HE_STAMP(2, 1);

  // contributors: the CTAs whose ranges cover the unit's tiles (records first+u ..)
  const int tps = p.tpu;
  const int64_t TSS = (int64_t)p.U * tps, NCT = stream_ctas;
  const TileSplit split{TSS, NCT, p.split_e, p.split_t1};
  int first = 0, n = 0;
  if (TSS > 0 && NCT > 0) {
    first = (int)split.owner((int64_t)u * tps);
    const int last = (int)split.owner((int64_t)u * tps + tps - 1);
    n = last - first + 1;
  }
  if (!HE_CHECK(first + u + n <= stream_ctas + p.U, p.err)) n = 0;
  const float* recs = p.partials + (size_t)(first + u) * R::FLOATS;
  auto rec_of = [&](int c) { return recs + (size_t)c * R::FLOATS; };
  const int b = u / p.kv_heads, j = u - b * p.kv_heads;
  const int q = tid / GD4, o = tid - q * GD4;
  const int g = (4 * o) / D;
  const int d0 = 4 * o - g * D;

  // ---- loads, all independent ----
  const unsigned long long key = full ? __ldcg(&uo[u].key[p.kpar]) : 0ull;
  const float lst = (full && !CH) ? __ldcg(&uo[u].lstar[g]) : 0.0f;
  const uint2 vs2 = (full && !CH) ? __ldcg(reinterpret_cast<const uint2*>(uo[u].vstar + d0))
                                  : make_uint2(0u, 0u);
  const float ln = __ldcg(&uo[u].lnew[g]);
  const float lng = (CH && tid < G) ? __ldcg(&uo[u].lnew[tid]) : 0.0f;  // head tid's
  const unsigned long long codek = __ldcg(&uo[u].codek);
  const uint16_t* kt = reinterpret_cast<const uint16_t*>(p.k) + (size_t)u * D;
  const uint16_t* vtp = reinterpret_cast<const uint16_t*>(p.v) + (size_t)u * D;
  // (quantised value cache: the evicted slot's codes and scale, and the new
  // token's codes and scale, as prep staged them)
  const uint32_t w4 = (VQ && full) ? __ldcg(reinterpret_cast<const uint32_t*>(uo[u].vqstar + d0))
                                   : 0u;
  const float ss = (VQ && full) ? __ldcg(&uo[u].vsstar) : 0.0f;
  const uint8_t vqn = (VQ && tid < D) ? __ldcg(&uo[u].vqnew[tid]) : (uint8_t)0;
  const float vsn = VQ ? __ldcg(&uo[u].vsnew) : 0.0f;
  const uint16_t kt1 = tid < D ? __ldcg(kt + tid) : (uint16_t)0;
  const uint16_t vt1 = tid < D ? __ldcg(vtp + tid) : (uint16_t)0;
  const uint2 vt2 = __ldcg(reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(p.v) +
                                                          (size_t)u * D + d0));
  // chunk eviction: the chunk's two softmax parts and the staged rows (one
  // 16-byte piece per thread; their addresses do not depend on the decision)
  float cm0 = -1e30f, cl0 = 0.0f, cm1 = -1e30f, cl1 = 0.0f;
  float4 ca0 = make_float4(0.f, 0.f, 0.f, 0.f), ca1 = ca0;
  uint4 srow = make_uint4(0u, 0u, 0u, 0u);
  uint64_t scode = 0;
  if constexpr (CH) {
    if (full) {
      using CR = ChunkRec<G, D>;
      const float* cr = reinterpret_cast<const float*>(p.cstar) + (size_t)u * CR::FLOATS;
      cm0 = __ldcg(cr + CR::M + g);
      cl0 = __ldcg(cr + CR::L + g);
      ca0 = __ldcg(reinterpret_cast<const float4*>(cr + CR::A) + o);
      cm1 = __ldcg(cr + CR::M + 8 + g);
      cl1 = __ldcg(cr + CR::L + 8 + g);
      ca1 = __ldcg(reinterpret_cast<const float4*>(cr + CR::A + G * D) + o);
      const int CH8 = D / 8, npc = (p.chunk - 1) * CH8;
      if (tid < 2 * npc) {
        const int arr = tid / npc, r = tid - arr * npc;
        const uint16_t* base = reinterpret_cast<const uint16_t*>(arr ? p.V : p.K);
        srow = __ldcg(reinterpret_cast<const uint4*>(
                          base + ((size_t)u * p.budget + p.lbudget + r / CH8) * D) + r % CH8);
      }
      if (tid < p.chunk - 1) {
        const int wb = p.bits >> 3;
        const unsigned char* src =
            p.codes + (size_t)u * p.code_stride + (size_t)(p.lbudget + tid) * wb;
        for (int bb = 0; bb < wb; ++bb) scode |= (uint64_t)__ldcg(src + bb) << (8 * bb);
      }
    }
  }
  float rm[kMergeRegs], rl[kMergeRegs];
  float4 rx[kMergeRegs];
#pragma unroll
  for (int i = 0; i < kMergeRegs; ++i) {
    const int c = q + i * NQ;
    if (c < n) {
      const float* r = rec_of(c);
      rm[i] = __ldcg(r + g);
      rl[i] = __ldcg(r + G + g);
      rx[i] = __ldcg(reinterpret_cast<const float4*>(r + R::HDR) + o);
    }
  }

  HE_STAMP(2, 3);  // (the loads are issued; the key is the first to be used)
  if (p.late_release) pdl_trigger();
  int winner = full ? (key ? (int)evict_key_slot(key) : -1) : p.append_slot;
  // slots evicted, and the end of the slots eviction may choose from
  const int nev = (CH && full) ? p.chunk : 1;
  const int wend = (CH && full) ? p.lbudget : p.budget;
  // (cannot happen: never write outside the cache; the group writes nothing
  // but still takes part in the CTA's barriers)
  const bool bad = winner < 0 || winner + nev > wend;
  if (bad) {
    if (tid == 0) atomicExch(p.err, 2);
    if (!MU) return;
    winner = 0;
  }
  // the evicted slot's contributor: the owner of tile winner / tile (with a
  // chunk, crel .. crel_hi own its first and last slot)
  const int crel = (full && n > 0)
                       ? (int)split.owner((int64_t)u * tps + winner / p.tile) - first
                       : -1;
  const int crel_hi =
      (CH && full && n > 0)
          ? (int)split.owner((int64_t)u * tps + (winner + nev - 1) / p.tile) - first
          : crel;

  float4 vs = make_float4(__uint_as_float(vs2.x << 16), __uint_as_float(vs2.x & 0xFFFF0000u),
                          __uint_as_float(vs2.y << 16), __uint_as_float(vs2.y & 0xFFFF0000u));
  // quantised value cache: the evicted row as stored (decode(q) * s), and the
  // new row's codes and scale from prep
  if constexpr (VQ) {
    if (full) {
      vs = make_float4(vq_decode<VQ>((uint8_t)(w4 & 0xFF)) * ss,
                       vq_decode<VQ>((uint8_t)((w4 >> 8) & 0xFF)) * ss,
                       vq_decode<VQ>((uint8_t)((w4 >> 16) & 0xFF)) * ss,
                       vq_decode<VQ>((uint8_t)(w4 >> 24)) * ss);
    }
    // the new token's row as stored (prep quantised it): its codes' values
    if (tid < D) vqrow[tid] = vq_decode<VQ>(vqn);
  }
  if (tid == 0) sflag[grp] = 0;
  __syncthreads();
  const float vscale = VQ ? vsn : 0.0f;

  float mx = -1e30f, sum = 0.0f;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  float rw = 0.0f;  // chunk eviction: the weight taken out, in the running max's frame
#pragma unroll
  for (int i = 0; i < kMergeRegs; ++i) {
    const int c = q + i * NQ;
    if (c < n) {
      if constexpr (CH) {
        if (full && (c == crel || c == crel_hi)) {
          float w = 0.0f;
          if (c == crel) w += take_part(cm0, cl0, ca0, rm[i], rl[i], rx[i]);
          if (c == crel_hi) w += take_part(cm1, cl1, ca1, rm[i], rl[i], rx[i]);
          const float mn = fmaxf(mx, rm[i]);
          rw = rw * exp2f(mx - mn) + w * exp2f(rm[i] - mn);
        }
        fold_one<D, G>(rm[i], rl[i], rx[i], false, lst, vs, mx, sum, a);
      } else {
        if (c == crel && d0 == 0 && !(exp2f(lst - rm[i]) <= 0.5f * rl[i])) atomicExch(&sflag[grp], 1);
        fold_one<D, G>(rm[i], rl[i], rx[i], c == crel, lst, vs, mx, sum, a);
      }
    }
  }
  for (int c = q + kMergeRegs * NQ; c < n; c += NQ) {
    const float* r = rec_of(c);
    const float mc = __ldcg(r + g);
    float lc = __ldcg(r + G + g);
    float4 x = __ldcg(reinterpret_cast<const float4*>(r + R::HDR) + o);
    if constexpr (CH) {
      if (full && (c == crel || c == crel_hi)) {
        float w = 0.0f;
        if (c == crel) w += take_part(cm0, cl0, ca0, mc, lc, x);
        if (c == crel_hi) w += take_part(cm1, cl1, ca1, mc, lc, x);
        const float mn = fmaxf(mx, mc);
        rw = rw * exp2f(mx - mn) + w * exp2f(mc - mn);
      }
      fold_one<D, G>(mc, lc, x, false, lst, vs, mx, sum, a);
    } else {
      if (c == crel && d0 == 0 && !(exp2f(lst - mc) <= 0.5f * lc)) atomicExch(&sflag[grp], 1);
      fold_one<D, G>(mc, lc, x, c == crel, lst, vs, mx, sum, a);
    }
  }
  if constexpr (CH) {
    if (full) {
      // the weight taken out against the weight that remains, per head
      // (one unit per CTA with chunks: ctid == tid)
      smax[ctid] = mx;
      ssum[ctid] = sum;
      wstate[ctid] = rw;
      __syncthreads();
      if (tid < G) {
        const int og = tid * (D / 4);  // head tid's first output group
        float M = lng;
        for (int q2 = 0; q2 < NQ; ++q2) M = fmaxf(M, smax[grp * GT + q2 * GD4 + og]);
        float rem = exp2f(lng - M), out_w = 0.0f;
        for (int q2 = 0; q2 < NQ; ++q2) {
          const float f = exp2f(smax[grp * GT + q2 * GD4 + og] - M);
          rem += ssum[grp * GT + q2 * GD4 + og] * f;
          out_w += wstate[grp * GT + q2 * GD4 + og] * f;
        }
        if (!(out_w <= kChunkRemoveMax * rem)) atomicExch(&sflag[grp], 1);
      }
    }
  }
  HE_STAMP(2, 4);
  bool recomputed;
  if constexpr (!MU) {
    __syncthreads();
    recomputed = sflag[0] != 0;
    if (recomputed) {
      // the evicted slot dominates its partial: recompute that partial without it
      const uint16_t* qg =
          reinterpret_cast<const uint16_t*>(p.q) + (size_t)(b * p.kv_heads + j) * G * D;
      for (int i2 = tid; i2 < G * D; i2 += MT) qf[i2] = __uint_as_float((uint32_t)qg[i2] << 16);
      __syncthreads();
      // the slots of that contributor (with a chunk: of contributors crel .. crel_hi)
      const int c = first + crel, ch = first + crel_hi;
      const int tb = (int)split.begin(c), te = (int)split.begin((int64_t)ch + 1);
      const int lo = (max(tb, u * tps) - u * tps) * p.tile;
      const int hi = min((min(te, (u + 1) * tps) - u * tps) * p.tile, p.occ);
      recompute_partial<D, G, VQ>(p, u, lo,
                                  HE_CHECK(0 <= lo && lo <= hi && hi <= p.budget, p.err) ? hi : lo,
                                  winner, nev, qf, wstate, xm, xl, xa, tid);
      mx = -1e30f;
      sum = 0.0f;
      a = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int c2 = q; c2 < n; c2 += NQ) {
        if (c2 > crel && c2 <= crel_hi) continue;  // (a chunk's second contributor: in the first)
        if (c2 == crel) {
          fold_one<D, G>(xm[g], xl[g], reinterpret_cast<const float4*>(xa)[o], false, lst, vs, mx,
                         sum, a);
        } else {
          const float* r = rec_of(c2);
          fold_one<D, G>(__ldcg(r + g), __ldcg(r + G + g),
                         __ldcg(reinterpret_cast<const float4*>(r + R::HDR) + o), false, lst, vs,
                         mx, sum, a);
        }
      }
    }
  } else {
    // the slots an exact recompute would cover (contributor crel .. crel_hi's
    // part of the unit), for whichever thread of the CTA runs it
    if (tid == 0) {
      const int c = first + crel, ch = first + crel_hi;
      int lo = 0, hi = 0;
      if (full && n > 0) {
        const int tb = (int)split.begin(c), te = (int)split.begin((int64_t)ch + 1);
        lo = (max(tb, u * tps) - u * tps) * p.tile;
        hi = min((min(te, (u + 1) * tps) - u * tps) * p.tile, p.occ);
      }
      rparam[grp * 4 + 0] = lo;
      rparam[grp * 4 + 1] = hi;
      rparam[grp * 4 + 2] = winner;
      rparam[grp * 4 + 3] = nev;
    }
    __syncthreads();
    const bool recomputed_mu = sflag[grp] != 0;
    // a unit whose evicted slot dominates its partial: the whole CTA recomputes
    // that partial without it, then the unit's group folds again (one unit at a
    // time; the loop is the same for every thread)
    for (int gi = 0; gi < UPC; ++gi) {
      if (sflag[gi] == 0) continue;
      const int ug = blockIdx.x * UPC + gi;
      const uint16_t* qg = reinterpret_cast<const uint16_t*>(p.q) + (size_t)ug * G * D;
      for (int i2 = ctid; i2 < G * D; i2 += MT) qf[i2] = __uint_as_float((uint32_t)qg[i2] << 16);
      __syncthreads();
      const int lo = rparam[gi * 4 + 0], hi = rparam[gi * 4 + 1];
      recompute_partial<D, G, VQ>(p, ug, lo,
                                  HE_CHECK(0 <= lo && lo <= hi && hi <= p.budget, p.err) ? hi : lo,
                                  rparam[gi * 4 + 2], rparam[gi * 4 + 3], qf, wstate, xm, xl, xa,
                                  ctid);
      if (grp == gi) {
        mx = -1e30f;
        sum = 0.0f;
        a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c2 = q; c2 < n; c2 += NQ) {
          if (c2 > crel && c2 <= crel_hi) continue;  // (a chunk's second contributor: in the first)
          if (c2 == crel) {
            fold_one<D, G>(xm[g], xl[g], reinterpret_cast<const float4*>(xa)[o], false, lst, vs, mx,
                           sum, a);
          } else {
            const float* r = rec_of(c2);
            fold_one<D, G>(__ldcg(r + g), __ldcg(r + G + g),
                           __ldcg(reinterpret_cast<const float4*>(r + R::HDR) + o), false, lst, vs,
                           mx, sum, a);
          }
        }
      }
      __syncthreads();  // (qf, xa and the scratch serve the next unit)
    }
    recomputed = recomputed_mu;
  }
  sacc[ctid] = a;
  smax[ctid] = mx;
  ssum[ctid] = sum;
  __syncthreads();

  const int gb = grp * GT;  // the group's first thread
  if (tid < GD4 && !bad) {
    // fold the groups in order, then the new token
    float m2 = ln;
    for (int q2 = 0; q2 < NQ; ++q2) m2 = fmaxf(m2, smax[gb + q2 * GD4 + tid]);
    float l2 = 0.0f;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q2 = 0; q2 < NQ; ++q2) {
      const float w = exp2f(smax[gb + q2 * GD4 + tid] - m2);
      const float4 y = sacc[gb + q2 * GD4 + tid];
      l2 += ssum[gb + q2 * GD4 + tid] * w;
      s.x += y.x * w;
      s.y += y.y * w;
      s.z += y.z * w;
      s.w += y.w * w;
    }
    const float wn = exp2f(ln - m2);
    const float inv = 1.0f / (l2 + wn);
    float4 vt = make_float4(__uint_as_float(vt2.x << 16), __uint_as_float(vt2.x & 0xFFFF0000u),
                            __uint_as_float(vt2.y << 16), __uint_as_float(vt2.y & 0xFFFF0000u));
    if constexpr (VQ)  // the new token's value as stored
      vt = make_float4(vqrow[d0] * vscale, vqrow[d0 + 1] * vscale, vqrow[d0 + 2] * vscale,
                       vqrow[d0 + 3] * vscale);
    float4 r;
    r.x = (s.x + wn * vt.x) * inv;
    r.y = (s.y + wn * vt.y) * inv;
    r.z = (s.z + wn * vt.z) * inv;
    r.w = (s.w + wn * vt.w) * inv;
    reinterpret_cast<float4*>(p.out + ((size_t)b * p.kv_heads * G + (size_t)j * G) * D)[tid] = r;
  }

  // chunk eviction: the staged rows, keys, values and codes, in arrival order
  // take the chunk's first c - 1 slots (rows of the stage are only read here)
  int wslot = winner;
  if constexpr (CH) {
    if (full && !bad) {
      const int c = nev, CH8 = D / 8, npc = (c - 1) * CH8;  // 16-byte pieces per array
      const size_t ub = (size_t)u * p.budget;
      for (int t = tid; t < 2 * npc; t += GT) {
        const int arr = t / npc, r = t - arr * npc;
        const int i = r / CH8, w = r - i * CH8;
        uint16_t* base = reinterpret_cast<uint16_t*>(arr ? p.V : p.K);
        // (the piece of this thread was loaded up front; more threads than pieces)
        const uint4 x = t == tid ? srow
                                 : __ldcg(reinterpret_cast<const uint4*>(
                                              base + (ub + p.lbudget + i) * D) + w);
        reinterpret_cast<uint4*>(base + (ub + winner + i) * D)[w] = x;
      }
      if (tid < c - 1)
        store_code(p.codes + (size_t)u * p.code_stride + (size_t)(winner + tid) * (p.bits >> 3),
                   p.bits, scode);
      wslot = winner + c - 1;
    }
  }
  HE_STAMP(2, 5);
  // method step 5: the current token's key, value and code replace the slot
  if (bad) return;
  if (!HE_CHECK(wslot >= 0 && wslot < p.budget &&
                    (!(CH && full) || p.lbudget + nev - 1 <= p.budget),
                p.err))
    return;
  uint16_t* Kw = reinterpret_cast<uint16_t*>(p.K) + ((size_t)u * p.budget + wslot) * D;
  if (tid < D) {
    Kw[tid] = kt1;
    if constexpr (VQ)
      reinterpret_cast<uint8_t*>(p.V)[((size_t)u * p.budget + winner) * D + tid] = vqn;
    else
      reinterpret_cast<uint16_t*>(p.V)[((size_t)u * p.budget + wslot) * D + tid] = vt1;
  }
  if (VQ && tid == 0) p.vs[(size_t)u * p.vs_stride + winner] = vscale;
  if (tid == 0) {
    store_code(p.codes + (size_t)u * p.code_stride + (size_t)wslot * (p.bits >> 3), p.bits,
               codek);
    p.evicted[u] = full ? winner : -1;
    log_eviction(p, u, full ? winner : -1);
    if (p.score != nullptr) p.score[(size_t)u * p.budget + winner] = 0.0f;  // not scored yet
    uo[u].key[p.kpar ^ 1] = 0;  // ready for the next step's atomicMax
    if (recomputed) atomicAdd(p.counters + u, 1);  // how often the exact path ran
  }
  HE_STAMP(2, 2);
}

// Dynamic shared memory of merge.
template <int D, int G>
constexpr int merge_smem_bytes(int threads) {
  return threads * (16 + 4 + 4) + (G * D + G * D + 8 + 8) * 4 + 16 + 64 +
         (threads / 32) * G * (2 + D) * 4 + 4 * (D + 32) * 4;
}

}  // namespace he
