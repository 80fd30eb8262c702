// he_fused.cuh — the bf16 HashEvict decode step in one launch (tensor cores).
//
// Stream-K over 64-slot cache tiles (he_common.cuh explains the split, the
// local eviction candidates and the last-CTA combine).  Per CTA: one producer
// warp and four consumer warps, two CTAs per SM.
//   producer  first a prologue item by TMA (the projection W and the query
//             heads and keys of the CTA's first units), then the K/V tiles by
//             2-D tensor TMA (128-byte boxes, 128B swizzle, L2 evict-first) into a
//             2-stage ring with full/empty mbarriers (bounded waits);
//   consumers method steps 1-2 from shared memory (the fixed-order fp32 chains
//             of the specification, ballot bit-packing), steps 3-4 on the CTA's
//             own slots (codes prefetched into registers at kernel start) giving
//             the local candidate; then, per tile and per warp of 16 slots,
//             logits S = K . Q^T and values O^T += V^T . P^T on the tensor cores
//             (mma.sync m16n8k16 bf16, the G query heads of a KV group on N,
//             padded to 8), online softmax in fp32 with the local candidate held
//             out (its logits kept for the combine), P as bf16 hi + lo parts;
//             per unit a partial record; the unit's last CTA combines (global
//             candidate, LSE merge, non-winning candidates and the new token
//             added back) and overwrites the evicted slot (step 5).
// Programmatic dependent launch: the kernel waits for the previous step's
// kernel before touching memory, and lets the next step's kernel launch early.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "he_common.cuh"
#include "he_tc.cuh"

namespace he {

template <int D, int G, int NS>
struct FusedShape {
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
  static constexpr int MAXU = 3;             // units per prologue batch
  static constexpr int XV = G + 1;           // staged vectors per unit (queries, key)
  static constexpr int WACC = NCW * G * D;   // floats of the warp-merge / combine area
  static constexpr int CPR = 4;              // code words (16 B) prefetched per thread
  static constexpr int BITW = (MAXU * XV * 64 + 31) / 32;
  static constexpr int OFF_STAGE = 0;        // 1024-byte aligned (128B swizzle)
  static constexpr int OFF_W = NS * STAGEB;  // W [D][bits] bf16 (bits <= 64)
  static constexpr int OFF_X = OFF_W + D * 64 * 2;
  static constexpr int OFF_WACC = OFF_X + (MAXU * XV * D * 2 + 15) / 16 * 16;
  static constexpr int OFF_P = OFF_WACC + WACC * 4;
  static constexpr int OFF_WM = OFF_P + NCW * 2 * PB;
  static constexpr int OFF_UB = OFF_WM + 2 * NCW * G * 4;
  static constexpr int UB = 1024;
  static constexpr int OFF_MISC = OFF_UB + UB;
  static constexpr int OFF_BAR = OFF_MISC + kMiscBytes;
  static constexpr int SMEM = OFF_BAR + (2 * NS + 1) * 8;
  static constexpr int SMEM_ALLOC = SMEM + 1024;  // slack to align the base to 1024
  static_assert(D % 64 == 0 && G >= 1 && G <= 8 && (G & (G - 1)) == 0, "shape");
  static_assert(STAGEB % 1024 == 0 && BOXB % 1024 == 0, "swizzle atoms");
  static_assert(WACC >= G * D + D, "empty-cache staging fits the merge area");
};

// Per-batch unit information: code bits, the new key's code, the new token's
// logits, the local candidate key of the CTA's segment of each unit.
template <int G, int MAXU, int BITW>
struct FusedUnits {
  uint32_t bits[BITW];
  unsigned long long best[MAXU];
  uint64_t codek[MAXU];
  float lnew[MAXU][G];
};

// Method steps 1-2 for the batch's staged vectors x [nb][G+1][D] (bf16) with W
// [D][bits] (bf16), both in shared memory.  Task t codes bit t % bits of vector
// t / bits; thread tid owns tasks tid + c * NC (one W column), four chains at a
// time, each the sequential fp32 fused multiply-add over d = 0..D-1 from +0.
template <int D, int G, int NC, int MAXU, int BITW>
__device__ __forceinline__ void fused_codes(const uint16_t* Ws, const uint16_t* xs, int nb,
                                            int bits, bool queries,
                                            FusedUnits<G, MAXU, BITW>& fu, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  const int nvec = nb * (G + 1);
  const int j = tid % bits;
  const int ntask = nvec * bits;
  const int nchain = (ntask + NC - 1) / NC;
  for (int c0 = 0; c0 < nchain; c0 += 4) {
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const uint16_t* xv[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int v = (tid + (c0 + c) * NC) / bits;
      xv[c] = xs + (v < nvec ? v : nvec - 1) * D;
    }
#pragma unroll 8
    for (int d = 0; d < D; ++d) {
      const float w = __uint_as_float((uint32_t)Ws[d * bits + j] << 16);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        acc[c] = __fmaf_rn(__uint_as_float((uint32_t)xv[c][d] << 16), w, acc[c]);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (c0 + c < nchain) {
        const int task0 = (c0 + c) * NC + warp * 32;
        const int tk = task0 + lane;
        const bool is_key = ((tk / bits) % (G + 1)) == G;
        const uint32_t bit = (tk < ntask && (queries || is_key) && acc[c] > 0.0f) ? 1u : 0u;
        const uint32_t word = __ballot_sync(kFull, bit);
        if (lane == 0 && task0 < ntask) fu.bits[task0 >> 5] = word;
      }
    }
  }
}

// Best eviction key among the codes held in one 16-byte word (word index c of
// the unit's code row) restricted to slots [lo, hi).
template <int G, int WB>
__device__ __forceinline__ uint64_t best_in_word_w(const uint4& w4, int c, int lo, int hi,
                                                   const uint64_t (&cq)[G]) {
  constexpr int PER = 16 / WB;
  const uint32_t wd[4] = {w4.x, w4.y, w4.z, w4.w};
  uint64_t best = 0;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    uint64_t code;
    if (WB == 8) code = (uint64_t)wd[2 * e] | ((uint64_t)wd[2 * e + 1] << 32);
    else if (WB == 4) code = wd[e];
    else if (WB == 2) code = (wd[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
    else code = (wd[e >> 2] >> (8 * (e & 3))) & 0xFFu;
    const int s = c * PER + e;
    if (s >= lo && s < hi) {
      const uint64_t key = evict_key(group_distance<G>(cq, code), (uint32_t)s);
      best = key > best ? key : best;
    }
  }
  return best;
}

template <int G>
__device__ __forceinline__ uint64_t best_in_word(const uint4& w4, int wb, int c, int lo, int hi,
                                                 const uint64_t (&cq)[G]) {
  switch (wb) {
    case 1: return best_in_word_w<G, 1>(w4, c, lo, hi, cq);
    case 2: return best_in_word_w<G, 2>(w4, c, lo, hi, cq);
    case 4: return best_in_word_w<G, 4>(w4, c, lo, hi, cq);
    default: return best_in_word_w<G, 8>(w4, c, lo, hi, cq);
  }
}

template <int D, int G, int NS, bool PSPLIT>
__global__ void __launch_bounds__(FusedShape<D, G, NS>::NT, 2)
    step_kernel_tc(const StepParams p, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV) {
  using S = FusedShape<D, G, NS>;
  using R = Record<G, D>;
  using T = bf16_t;
  using FU = FusedUnits<G, S::MAXU, S::BITW>;
  static_assert(sizeof(FU) <= S::UB, "unit batch");
  constexpr int NC = S::NC;
  constexpr int CAP = S::WACC / (3 * G + 1);  // combine: contributors per scratch chunk
  extern __shared__ __align__(16) unsigned char smem_tc[];
  unsigned char* smem = smem_tc + ((1024u - (smem_u32(smem_tc) & 1023u)) & 1023u);
  unsigned char* stage = smem + S::OFF_STAGE;
  uint16_t* Ws = reinterpret_cast<uint16_t*>(smem + S::OFF_W);
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + S::OFF_X);
  float* wacc = reinterpret_cast<float*>(smem + S::OFF_WACC);
  float* wm = reinterpret_cast<float*>(smem + S::OFF_WM);
  float* wl = wm + S::NCW * G;
  FU& fu = *reinterpret_cast<FU*>(smem + S::OFF_UB);
  Misc& m = *reinterpret_cast<Misc*>(smem + S::OFF_MISC);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + S::OFF_BAR);
  uint64_t* empty_bar = full_bar + NS;
  uint64_t* pro_bar = empty_bar + NS;
  volatile int32_t* v_abort = &m.abort;
  volatile int32_t* v_issued = &m.issued;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool full = p.append_slot < 0;

  HE_STAMP(1, 0);
  pdl_wait();     // the previous step is complete: the cache, codes and records are final
  pdl_trigger();  // the next step may launch; it waits for this grid the same way
  HE_STAMP(1, 1);

  if (p.total_tiles == 0) {  // empty cache: the new token alone
    if ((int)blockIdx.x < p.U && warp < S::NCW) {
      unit_prologue<T, D, G, NC, 1>(p, blockIdx.x, wacc, wacc + G * D, m, tid);
      combine_unit<T, D, G, NC, 1>(p, blockIdx.x, 0, 0, m, tid, wacc, CAP);
    }
    return;
  }

  const int64_t TT = p.total_tiles, NCTA = gridDim.x;
  const int tb = (int)((int64_t)blockIdx.x * TT / NCTA);
  const int te = (int)(((int64_t)blockIdx.x + 1) * TT / NCTA);
  const int ntiles = te - tb;
  const int u_first = tb / p.tpu, u_last = (te - 1) / p.tpu;
  const int nb0 = min(S::MAXU, u_last - u_first + 1);

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], S::NCW);
    }
    mbar_init(pro_bar, 1);
    m.abort = 0;
    m.issued = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // ---------------- producer warp ----------------
  if (warp == S::NCW) {
    if (lane == 0) {
      // prologue item first, ahead of the cache stream: W and the batch's vectors
      const uint32_t wbytes = (uint32_t)(D * p.bits * 2);
      mbar_arrive_expect_tx(pro_bar, wbytes + (uint32_t)(nb0 * (G + 1) * D * 2));
      bulk_g2s(Ws, p.W, wbytes, pro_bar);
      for (int k = 0; k < nb0; ++k) {
        const int u = u_first + k;
        const int b = u / p.kv_heads, jh = u - b * p.kv_heads;
        bulk_g2s(xs + k * (G + 1) * D,
                 reinterpret_cast<const uint16_t*>(p.q) + (size_t)(b * p.kv_heads + jh) * G * D,
                 (uint32_t)(G * D * 2), pro_bar);
        bulk_g2s(xs + (k * (G + 1) + G) * D,
                 reinterpret_cast<const uint16_t*>(p.k) + (size_t)u * D, (uint32_t)(D * 2),
                 pro_bar);
      }
      const uint64_t pol = l2_evict_first_policy();
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
          tma_load_2d_hint(dst + h * S::BOXB, &tmK, 64 * h, y, &full_bar[st], pol);
#pragma unroll
        for (int h = 0; h < S::NHALF; ++h)
          tma_load_2d_hint(dst + S::TILEB + h * S::BOXB, &tmV, 64 * h, y, &full_bar[st], pol);
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
  const int wb = p.bits >> 3;

  // prefetch the first segment's codes (16-byte words) into registers
  const int lo0 = (max(tb, u_first * p.tpu) - u_first * p.tpu) * S::TS;
  const int hi0 = min((min(te, (u_first + 1) * p.tpu) - u_first * p.tpu) * S::TS, p.occ);
  const uint4* crow0 = reinterpret_cast<const uint4*>(p.codes + (size_t)u_first * p.code_stride);
  const int cw0 = (lo0 * wb) >> 4, cw1 = (hi0 * wb + 15) >> 4;
  uint4 creg[S::CPR];
#pragma unroll
  for (int r = 0; r < S::CPR; ++r) {
    const int c = cw0 + tid + r * NC;
    creg[r] = (full && c < cw1) ? __ldcg(crow0 + c) : make_uint4(0u, 0u, 0u, 0u);
  }

  int i = 0;            // CTA-local tile counter
  int drain_from = -1;  // first tile this warp did not wait for (after a give-up)
  int batch_u0 = u_first, batch_n = 0;
  for (int u = u_first; u <= u_last; ++u) {
    const int seg_t0 = max(tb, u * p.tpu), seg_t1 = min(te, (u + 1) * p.tpu);
    const int lo = (seg_t0 - u * p.tpu) * S::TS;
    const int hi = min((seg_t1 - u * p.tpu) * S::TS, p.occ);

    if (u >= batch_u0 + batch_n) {
      // prologue batch: units u .. u + nb - 1
      const int nb = min(S::MAXU, u_last - u + 1);
      if (u == u_first) {
        if (!mbar_wait_bounded(pro_bar, 0u)) {
          atomicExch(p.err, 1);
          *v_abort = 1;
        }
        HE_STAMP(1, 6);
      } else {  // later batches: stage the vectors with plain loads (W stays in place)
        for (int e = tid; e < nb * (G + 1) * D / 8; e += NC) {
          const int v = e / (D / 8), w8 = e - v * (D / 8);
          const int k = v / (G + 1), h = v - k * (G + 1);
          const int uu = u + k;
          const int b = uu / p.kv_heads, jh = uu - b * p.kv_heads;
          const uint4* src = h < G ? reinterpret_cast<const uint4*>(
                                         reinterpret_cast<const uint16_t*>(p.q) +
                                         ((size_t)(b * p.kv_heads + jh) * G + h) * D)
                                   : reinterpret_cast<const uint4*>(
                                         reinterpret_cast<const uint16_t*>(p.k) + (size_t)uu * D);
          reinterpret_cast<uint4*>(xs)[e] = __ldcg(src + w8);
        }
        group_sync<NC, 1>();
      }
      batch_u0 = u;
      batch_n = nb;
      fused_codes<D, G, NC, S::MAXU, S::BITW>(Ws, xs, nb, p.bits, full, fu, tid);
      // the new token's logits
      for (int w2 = warp; w2 < nb * G; w2 += S::NCW) {
        const int k = w2 / G, g = w2 - k * G;
        float a = 0.0f;
        for (int d = lane; d < D; d += 32)
          a = fmaf(__uint_as_float((uint32_t)xs[(k * (G + 1) + g) * D + d] << 16),
                   __uint_as_float((uint32_t)xs[(k * (G + 1) + G) * D + d] << 16), a);
        a = warp_sum(a);
        if (lane == 0) fu.lnew[k][g] = a * p.qscale;
      }
      if (tid < S::MAXU) fu.best[tid] = 0ull;
      group_sync<NC, 1>();
      if (u == u_first) HE_STAMP(1, 7);
      if (tid < nb) fu.codek[tid] = code_from_bits(fu.bits, p.bits, tid * (G + 1) + G);
      if (full) {
        // method steps 3-4 on this CTA's slots of each unit of the batch
        for (int k = 0; k < nb; ++k) {
          const int uu = u + k;
          const int klo = (max(tb, uu * p.tpu) - uu * p.tpu) * S::TS;
          const int khi = min((min(te, (uu + 1) * p.tpu) - uu * p.tpu) * S::TS, p.occ);
          uint64_t cq[G];
#pragma unroll
          for (int g = 0; g < G; ++g) cq[g] = code_from_bits(fu.bits, p.bits, k * (G + 1) + g);
          const uint4* crow =
              reinterpret_cast<const uint4*>(p.codes + (size_t)uu * p.code_stride);
          const int c0 = (klo * wb) >> 4, c1 = (khi * wb + 15) >> 4;
          uint64_t best = 0;
          for (int c = c0 + tid, r = 0; c < c1; c += NC, ++r) {
            uint4 w4;
            if (uu == u_first && r < S::CPR) {
              w4 = creg[0];
#pragma unroll
              for (int rr = 1; rr < S::CPR; ++rr)
                if (rr == r) w4 = creg[rr];
            } else {
              w4 = __ldcg(crow + c);
            }
            const uint64_t kb2 = best_in_word<G>(w4, wb, c, klo, khi, cq);
            best = kb2 > best ? kb2 : best;
          }
          best = warp_max_u64(best);
          if (lane == 0 && best) atomicMax(&fu.best[k], (unsigned long long)best);
        }
      }
      group_sync<NC, 1>();
    }
    HE_STAMP(1, 2);
    const int kb = u - batch_u0;
    if (tid < G) {
      m.lnew[tid] = fu.lnew[kb][tid];
      m.candlog[tid] = -INFINITY;
    }
    if (tid == 0) {
      m.codek = fu.codek[kb];
      m.cand_slot = full ? (int)evict_key_slot(fu.best[kb]) : -1;
      m.cand_dist = full ? (int)evict_key_dist(fu.best[kb]) : 0;
    }
    group_sync<NC, 1>();
    const int cand = m.cand_slot;

    // query fragments (B operand of the logit MMA) from the staged vectors
    uint32_t qb[S::KS][2];
    {
      const uint32_t* xw = reinterpret_cast<const uint32_t*>(xs + kb * (G + 1) * D);
#pragma unroll
      for (int ks = 0; ks < S::KS; ++ks)
#pragma unroll
        for (int r = 0; r < 2; ++r)
          qb[ks][r] = g8 < G ? xw[(g8 * D + 16 * ks + 8 * r + 2 * t4) >> 1] : 0u;
    }

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
      if (sA >= hi) {
        x00 = x01 = -INFINITY;
      } else if (sA == cand) {
        if (real0) m.candlog[h0] = x00;
        if (real1) m.candlog[h1] = x01;
        x00 = x01 = -INFINITY;
      }
      if (sB >= hi) {
        x10 = x11 = -INFINITY;
      } else if (sB == cand) {
        if (real0) m.candlog[h0] = x10;
        if (real1) m.candlog[h1] = x11;
        x10 = x11 = -INFINITY;
      }
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

    // warp states -> shared memory; merge into this CTA's record for unit u
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
        (void)mbar_wait_bounded(pro_bar, 0u, 500000000ull);
      }
      return;
    }
    HE_STAMP(1, 3);
    write_partial<G, D, NC>(p.partials + (size_t)(blockIdx.x + u) * R::FLOATS, wm, wl, wacc,
                            S::NCW, m, cand, full, tid);
    finish_segment<T, D, G, NC, 1>(p, u, m, tid, wacc, CAP);
    HE_STAMP(1, 4);
  }
  HE_STAMP(1, 5);
}

}  // namespace he
