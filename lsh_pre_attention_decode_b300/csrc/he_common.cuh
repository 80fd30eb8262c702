// he_common.cuh — pieces shared by the two step-kernel engines (CUDA-core and
// tensor-core): per-step parameters, the per-unit prologue (method steps 1-2 for
// the query heads and the new key), the packed-code scan (steps 3-4), the
// partial-result record, the last-CTA combine (step 5 and the merge of the
// attention partials), and the stand-alone code / score / projection kernels.
//
// Method: "HashEvict: A Pre-Attention KV Cache Eviction Strategy using
// Locality-Sensitive Hashing" (arXiv 2412.16187), abstract and technical
// framework steps 1-5; attention over the retained cache as in the TTKV page's
// introduction (each decode step attends the whole cache).
//
// Work decomposition shared by both engines (stream-K over cache tiles):
//   the resident slots of every (batch, KV head) unit are cut into tiles; the
//   U * tiles_per_unit tiles form one list split into equal contiguous ranges,
//   one per CTA.  A range may cover the end of one unit and the start of the
//   next; the CTA emits one partial per unit it touches, into record cta + u.
//   Per unit segment a CTA codes the queries and the key, finds its local
//   eviction candidate (largest group-summed Hamming distance, lowest slot),
//   runs an online softmax over its slots with the candidate held out (its
//   logits kept aside), writes its partial and counts itself in; the last CTA
//   of the unit (atomic counter, no waiting) picks the global candidate,
//   merges the partials, adds back every non-winning candidate and the new
//   token, writes the output and overwrites the evicted slot.  The evicted
//   slot therefore never enters the softmax and the new token always does —
//   the same arithmetic as "evict, overwrite, then attend".
#pragma once

#include "he_device.cuh"

namespace he {

struct UnitOut;  // bf16 pipeline: per-unit results of the codes/eviction kernel

struct StepParams {
  void* K;               // cache keys   [U][budget][D] (budget: rows per unit, the stride)
  void* V;               // cache values [U][budget][D]
  unsigned char* codes;  // [U][code_stride] words of bits/8 bytes
  const void* W;         // projection [D][bits]
  const void* q;         // [batch][heads][D]
  const void* k;         // [batch][kv_heads][D]
  const void* v;         // [batch][kv_heads][D]
  float* out;            // [batch][heads][D]
  int32_t* evicted;      // [U]
  float* partials;       // [ctas + U][record]
  int32_t* counters;     // [U], zero between steps
  int32_t* err;          // set nonzero when a kernel gives up (bounded waits)
  int32_t U;
  int32_t kv_heads;
  int32_t budget;
  int32_t occ;           // resident slots before the step
  int32_t tile;          // slots per tile (engine-specific)
  int32_t tpu;           // tiles per unit = ceil(occ / tile)
  int32_t total_tiles;   // U * tpu
  int32_t bits;
  int32_t code_stride;   // bytes per unit row of codes (multiple of 16)
  int32_t append_slot;   // -1: cache full, evict; else the slot the token is appended to
  float qscale;          // log2(e) / sqrt(D): logits kept in base 2
  float tau;             // binarisation threshold: bit = (projection > tau)
  const float* tauv;     // or one threshold per bit and unit [U][bits] (null: tau)
  float decay;           // score memory gamma (with score != nullptr)
  float* score;          // per-slot scores [U][budget] (null: evict by the step's distances)
  float* vs;             // quantised value cache: per-slot scales [U][vs_stride] (V holds byte rows)
  int32_t vs_stride;
  // bf16 pipeline: per-unit results, the parity of this step's eviction key,
  // and the slot the previous step of this cache wrote: 0 none (or not
  // tracked), s + 1 appended at slot s, -1 evicted (slot in the other key)
  UnitOut* uo;
  int32_t kpar;
  int32_t prev_w1;
  // chunk eviction (bf16 pipeline): chunk c > 1 evicts aligned chunks of c
  // slots of the first lbudget (a multiple of c); the rows [lbudget, budget)
  // stage the newest tokens; cstar holds the evicted chunk's logits and value
  // rows (per unit); nopre: the previous step moved rows, so the stream kernel
  // fetches no tile before it waits for that step
  int32_t lbudget;
  int32_t chunk;
  int32_t nopre;
  void* cstar;
  // bf16 pipeline: stream-K split of the tiles in two groups (TileSplit);
  // split_e = split_t1 = 0 is the even split
  int32_t split_e;
  int32_t split_t1;
  // bf16 pipeline: merge lets the next step launch only once its loads are
  // issued (1; units of many partials), else as soon as its wait returns (0)
  int32_t late_release;
  // fused step: the split of this cache's previous step (prev_tpu tiles per
  // unit over prev_nc CTAs, prev_e / prev_t1 as split_e / split_t1; prev_nc = 0:
  // no CTA), which fixes how many hash warps fold that step's eviction key
  int32_t prev_tpu;
  int32_t prev_nc;
  int32_t prev_e;
  int32_t prev_t1;
  // test exports (null: off): a per-step eviction log written on the device
  // (evlog [evcap][U], evcnt [U] entries written per unit) and the group-summed
  // distance of every slot scored by a full-cache step (dist [U][budget])
  int32_t* evlog;
  int32_t* evcnt;
  int32_t evcap;
  int32_t* dist;
#ifdef HE_TIMELINE
  int32_t tl_step;       // diagnostic builds: step slot of the stamps
#endif
};

// Misc shared-memory block of a step CTA.
struct Misc {
  uint32_t bits[32];  // packed code bits of the G queries and the key
  uint64_t cq[8];     // query codes
  uint64_t codek;     // the new key's code
  uint64_t pad0;
  float lnew[8];      // new token's base-2 logits
  float candlog[8];   // local candidate's base-2 logits
  float hm[8];        // combine: per-head max
  float hl[8];        // combine: per-head sum
  float redf[8][8];   // combine: per-warp per-head maxima
  uint64_t red64[8];
  int32_t cand_slot;
  int32_t cand_dist;
  int32_t is_last;
  int32_t winner;
  int32_t abort;
  int32_t issued;
  int32_t pad1[2];
  HE_TL_FIELDS
};
static_assert(sizeof(Misc) <= 1024, "misc");
constexpr int kMiscBytes = 1024;

// Partial record of one (CTA, unit): header [m G][l G][cand logit G][slot][dist]
// padded to 4 floats, then the accumulator [G][D].
template <int G, int D>
struct Record {
  static constexpr int HDR = ((3 * G + 2) + 3) / 4 * 4;
  static constexpr int FLOATS = HDR + G * D;
};

// Barrier over the first NT threads of the CTA (ID 0 = the whole CTA).
template <int NT, int ID>
__device__ __forceinline__ void group_sync() {
  if constexpr (ID == 0) {
    __syncthreads();
  } else {
    asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(NT) : "memory");
  }
}

__device__ __forceinline__ void store_code(unsigned char* dst, int bits, uint64_t code) {
  switch (bits) {
    case 8: *dst = (unsigned char)code; break;
    case 16: *reinterpret_cast<uint16_t*>(dst) = (uint16_t)code; break;
    case 32: *reinterpret_cast<uint32_t*>(dst) = (uint32_t)code; break;
    default: *reinterpret_cast<uint64_t*>(dst) = code; break;
  }
}

// Test export: appends the slot a step wrote in unit u to the device eviction
// log.  Steps of one cache are ordered on the device (each waits for the
// previous one), so the per-unit count needs no atomic.
__device__ __forceinline__ void log_eviction(const StepParams& p, int u, int32_t slot) {
  if (p.evlog == nullptr) return;
  const int32_t i = p.evcnt[u];
  if (i < p.evcap) p.evlog[(size_t)i * p.U + u] = slot;
  p.evcnt[u] = i + 1;
}

// Method step 3: group-summed Hamming distance of one cached code.
template <int G>
__device__ __forceinline__ uint32_t group_distance(const uint64_t (&cq)[G], uint64_t code) {
  uint32_t d = 0;
#pragma unroll
  for (int g = 0; g < G; ++g) d += (uint32_t)popc64(cq[g] ^ code);
  return d;
}

// Best eviction key over the codes of slots [lo, hi) of one unit row, read as
// 16-byte chunks of 16/WB codes (WB = bits/8 bytes per code); per-thread result.
// When dist_out is set, the distances are stored too.
template <int G, int WB>
__device__ __forceinline__ uint64_t scan_codes_w(const unsigned char* row, int lo, int hi,
                                                 const uint64_t (&cq)[G], int tid, int nthreads,
                                                 int32_t* dist_out, float* score, float decay) {
  constexpr int PER = 16 / WB;
  const int c0 = (lo * WB) >> 4;
  const int c1 = (hi * WB + 15) >> 4;
  uint64_t best = 0;
  for (int c = c0 + tid; c < c1; c += nthreads) {
    const uint4 ch = __ldg(reinterpret_cast<const uint4*>(row) + c);
    const uint32_t wd[4] = {ch.x, ch.y, ch.z, ch.w};
    const int s0 = c * PER;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      uint64_t code;
      if (WB == 8) code = (uint64_t)wd[2 * e] | ((uint64_t)wd[2 * e + 1] << 32);
      else if (WB == 4) code = wd[e];
      else if (WB == 2) code = (wd[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
      else code = (wd[e >> 2] >> (8 * (e & 3))) & 0xFFu;
      const int s = s0 + e;
      if (s >= lo && s < hi) {
        const uint32_t dist = group_distance<G>(cq, code);
        if (dist_out) dist_out[s] = (int32_t)dist;
        uint32_t rank = dist;
        if (score) {  // score memory: A = gamma A + d; a non-negative fp32 orders as its bits
          const float a = __fmaf_rn(decay, score[s], (float)dist);
          score[s] = a;
          rank = __float_as_uint(a);
        }
        const uint64_t key = evict_key(rank, (uint32_t)s);
        best = key > best ? key : best;
      }
    }
  }
  return best;
}

template <int G>
__device__ __forceinline__ uint64_t scan_codes(const unsigned char* row, int bits, int lo, int hi,
                                               const uint64_t (&cq)[G], int tid, int nthreads,
                                               int32_t* dist_out, float* score = nullptr,
                                               float decay = 0.0f) {
  switch (bits) {
    case 8: return scan_codes_w<G, 1>(row, lo, hi, cq, tid, nthreads, dist_out, score, decay);
    case 16: return scan_codes_w<G, 2>(row, lo, hi, cq, tid, nthreads, dist_out, score, decay);
    case 32: return scan_codes_w<G, 4>(row, lo, hi, cq, tid, nthreads, dist_out, score, decay);
    default: return scan_codes_w<G, 8>(row, lo, hi, cq, tid, nthreads, dist_out, score, decay);
  }
}

// Method steps 1-2 for the G query heads (when `with_queries`) and the key
// staged in shared memory (s_q [G][D], s_k [D]) -> m.cq[], m.codek.  Bit tasks
// are head-major (task = head * bits + j; head G is the key), packed by warp
// ballots.  Run by the first NT threads; ends with a group barrier.
// tauv: the unit's per-bit thresholds [bits], or null for tau on every bit.
template <typename T, int D, int G, int NT, int BAR>
__device__ __forceinline__ void code_queries_and_key(const float* s_q, const float* s_k,
                                                     const T* W, int bits, float tau,
                                                     const float* tauv, bool with_queries,
                                                     Misc& m, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  const int ntask = (G + 1) * bits;
  for (int t0 = warp * 32; t0 < ntask; t0 += NT) {
    const int t = t0 + lane;
    uint32_t bit = 0;
    if (t < ntask) {
      const int h = t / bits, j = t - h * bits;
      const float tj = tauv ? tauv[j] : tau;
      if (h == G)
        bit = projection_bit<T, D>(s_k, W, bits, j, tj);
      else if (with_queries)
        bit = projection_bit<T, D>(s_q + h * D, W, bits, j, tj);
    }
    const uint32_t word = __ballot_sync(kFull, bit);
    if (lane == 0) m.bits[t0 >> 5] = word;
  }
  group_sync<NT, BAR>();
  if (tid <= G) {
    const uint64_t c = code_from_bits(m.bits, bits, tid);
    if (tid < G) m.cq[tid] = c;
    else m.codek = c;
  }
  group_sync<NT, BAR>();
}

// Stages unit u's query heads and new key (fp32, exact) and computes the codes
// and the new token's base-2 logits.
template <typename T, int D, int G, int NT, int BAR>
__device__ __forceinline__ void unit_prologue(const StepParams& p, int u, float* s_q, float* s_k,
                                              Misc& m, int tid) {
  constexpr int NW = NT / 32;
  const int lane = tid & 31, warp = tid >> 5;
  const int b = u / p.kv_heads, j = u - b * p.kv_heads;
  const T* qg = reinterpret_cast<const T*>(p.q) + ((size_t)b * p.kv_heads * G + (size_t)j * G) * D;
  const T* kg = reinterpret_cast<const T*>(p.k) + (size_t)u * D;
  for (int i = tid; i < G * D; i += NT) s_q[i] = to_f32(qg[i]);
  for (int i = tid; i < D; i += NT) s_k[i] = to_f32(kg[i]);
  group_sync<NT, BAR>();
  for (int g = warp; g < G; g += NW) {
    float a = 0.0f;
    for (int d = lane; d < D; d += 32) a = fmaf(s_q[g * D + d], s_k[d], a);
    a = warp_sum(a);
    if (lane == 0) m.lnew[g] = a * p.qscale;
  }
  code_queries_and_key<T, D, G, NT, BAR>(s_q, s_k, reinterpret_cast<const T*>(p.W), p.bits,
                                         p.tau, p.tauv ? p.tauv + (size_t)u * p.bits : nullptr,
                                         p.append_slot < 0, m, tid);
}

// Local eviction candidate over slots [lo, hi) of unit u -> m.cand_slot/dist;
// resets m.candlog.  Group barriers inside.
template <int G, int NT, int BAR>
__device__ __forceinline__ void local_candidate(const StepParams& p, int u, int lo, int hi, Misc& m,
                                                int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  uint64_t cq[G];
#pragma unroll
  for (int g = 0; g < G; ++g) cq[g] = m.cq[g];
  uint64_t best = scan_codes<G>(p.codes + (size_t)u * p.code_stride, p.bits, lo, hi, cq, tid, NT,
                                p.dist ? p.dist + (size_t)u * p.budget : nullptr,
                                p.score ? p.score + (size_t)u * p.budget : nullptr, p.decay);
  best = warp_max_u64(best);
  if (lane == 0) m.red64[warp] = best;
  group_sync<NT, BAR>();
  if (tid == 0) {
    uint64_t b2 = 0;
    for (int w2 = 0; w2 < NT / 32; ++w2) b2 = m.red64[w2] > b2 ? m.red64[w2] : b2;
    m.cand_slot = (int)evict_key_slot(b2);
    m.cand_dist = (int)evict_key_dist(b2);
#pragma unroll
    for (int g = 0; g < G; ++g) m.candlog[g] = -INFINITY;
  }
  group_sync<NT, BAR>();
}

// Merges NW warp states (wm/wl [NW][G], wacc [NW][G][D]) into this CTA's record
// for unit u.  Caller has synchronised after writing the warp states.
template <int G, int D, int NT>
__device__ __forceinline__ void write_partial(float* rec, const float* wm, const float* wl,
                                              const float* wacc, int nw, const Misc& m, int cand,
                                              bool full, int tid) {
  using R = Record<G, D>;
  for (int idx = tid; idx < G * D; idx += NT) {
    const int g = idx / D, d = idx - g * D;
    float mx = -1e30f;
    for (int w2 = 0; w2 < nw; ++w2) mx = fmaxf(mx, wm[w2 * G + g]);
    float a = 0.0f;
    for (int w2 = 0; w2 < nw; ++w2) a += wacc[(w2 * G + g) * D + d] * exp2f(wm[w2 * G + g] - mx);
    __stcg(rec + R::HDR + idx, a);
  }
  if (tid < G) {
    const int g = tid;
    float mx = -1e30f, sum = 0.0f;
    for (int w2 = 0; w2 < nw; ++w2) mx = fmaxf(mx, wm[w2 * G + g]);
    for (int w2 = 0; w2 < nw; ++w2) sum += wl[w2 * G + g] * exp2f(wm[w2 * G + g] - mx);
    __stcg(rec + g, mx);
    __stcg(rec + G + g, sum);
    __stcg(rec + 2 * G + g, full ? m.candlog[g] : -INFINITY);
  }
  if (tid == 0) {
    __stcg(rec + 3 * G, __int_as_float(cand));
    __stcg(rec + 3 * G + 1, __int_as_float(full ? m.cand_dist : 0));
  }
}

// The last CTA of unit u merges the unit's partials (records of CTAs
// first .. first+n-1, stored at index cta + u), adds back the non-winning
// candidates and the new token, writes the output and overwrites the slot.
// `scratch` (cap * (3G + 1) floats of shared memory) holds per-contributor
// weights; contributors are taken in chunks of `cap`.  Every sum runs in a
// fixed order, so the result does not depend on which CTA combines.
template <typename T, int D, int G, int NT, int BAR>
__device__ void combine_unit(const StepParams& p, int u, int first, int n, Misc& m, int tid,
                             float* scratch, int cap) {
  using R = Record<G, D>;
  constexpr int NW = NT / 32;
  constexpr int SW = 3 * G + 1;                  // scratch floats per contributor
  constexpr int OPT = (G * D + NT - 1) / NT;     // outputs per thread
  const int lane = tid & 31, warp = tid >> 5;
  const bool full = p.append_slot < 0;
  const float* recs = p.partials + (size_t)(first + u) * R::FLOATS;

  // pass A: eviction choice (largest local key) and per-head stabiliser (the max
  // over every partial max and every candidate logit; any upper bound works)
  uint64_t best = 0;
  float mx[G];
#pragma unroll
  for (int g = 0; g < G; ++g) mx[g] = -1e30f;
  for (int c = tid; c < n; c += NT) {
    const float* r = recs + (size_t)c * R::FLOATS;
    const int slot = __float_as_int(__ldcg(r + 3 * G));
    const int dist = __float_as_int(__ldcg(r + 3 * G + 1));
    if (full && slot >= 0) {
      const uint64_t key = evict_key((uint32_t)dist, (uint32_t)slot);
      best = key > best ? key : best;
    }
#pragma unroll
    for (int g = 0; g < G; ++g) mx[g] = fmaxf(mx[g], fmaxf(__ldcg(r + g), __ldcg(r + 2 * G + g)));
  }
  best = warp_max_u64(best);
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx[g] = fmaxf(mx[g], __shfl_xor_sync(kFull, mx[g], o));
  if (lane == 0) {
    m.red64[warp] = best;
#pragma unroll
    for (int g = 0; g < G; ++g) m.redf[warp][g] = mx[g];
  }
  group_sync<NT, BAR>();
  if (tid == 0) {
    uint64_t b2 = 0;
    for (int w2 = 0; w2 < NW; ++w2) b2 = m.red64[w2] > b2 ? m.red64[w2] : b2;
    m.winner = full ? (int)evict_key_slot(b2) : p.append_slot;
    for (int g = 0; g < G; ++g) {
      float x = m.lnew[g];
      for (int w2 = 0; w2 < NW; ++w2) x = fmaxf(x, m.redf[w2][g]);
      m.hm[g] = x;
      m.hl[g] = exp2f(m.lnew[g] - x);
    }
  }
  group_sync<NT, BAR>();
  HE_TL_MARK(m, 12);
  const int winner = m.winner;
  if (winner < 0 || winner >= p.budget) {  // cannot happen for a non-empty unit; never write
    if (tid == 0) {
      atomicExch(p.err, 2);
      p.counters[u] = 0;
    }
    return;
  }

  const T* Vc = reinterpret_cast<const T*>(p.V) + (size_t)u * p.budget * D;
  float a[OPT];
#pragma unroll
  for (int k = 0; k < OPT; ++k) a[k] = 0.0f;
  for (int c0 = 0; c0 < n; c0 += cap) {
    const int cn = min(cap, n - c0);
    // pass B: weights of this chunk of contributors
    for (int c = tid; c < cn; c += NT) {
      const float* r = recs + (size_t)(c0 + c) * R::FLOATS;
      const int slot = __float_as_int(__ldcg(r + 3 * G));
      const bool keep = full && slot >= 0 && slot != winner;
      float* sc = scratch + c * SW;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float w = exp2f(__ldcg(r + g) - m.hm[g]);
        sc[g] = w;
        sc[G + g] = keep ? exp2f(__ldcg(r + 2 * G + g) - m.hm[g]) : 0.0f;
        sc[2 * G + g] = __ldcg(r + G + g) * w;
      }
      sc[3 * G] = __int_as_float(keep ? slot : -1);
    }
    group_sync<NT, BAR>();
    for (int g = warp; g < G; g += NW) {
      float sum = 0.0f;
      for (int c = lane; c < cn; c += 32) sum += scratch[c * SW + 2 * G + g] + scratch[c * SW + G + g];
      sum = warp_sum(sum);
      if (lane == 0) m.hl[g] += sum;
    }
    // pass C: accumulators of this chunk (independent loads, fixed order)
#pragma unroll
    for (int k = 0; k < OPT; ++k) {
      const int idx = tid + k * NT;
      if (idx < G * D) {
        const int g = idx / D, d = idx - g * D;
        float acc = a[k];
#pragma unroll 4
        for (int c = 0; c < cn; ++c) {
          acc += __ldcg(recs + (size_t)(c0 + c) * R::FLOATS + R::HDR + idx) * scratch[c * SW + g];
          const int slot = __float_as_int(scratch[c * SW + 3 * G]);
          if (slot >= 0) acc += scratch[c * SW + G + g] * to_f32(Vc[(size_t)slot * D + d]);
        }
        a[k] = acc;
      }
    }
    group_sync<NT, BAR>();
  }
  HE_TL_MARK(m, 13);

  const int b = u / p.kv_heads, j = u - b * p.kv_heads;
  const T* vt = reinterpret_cast<const T*>(p.v) + (size_t)u * D;
#pragma unroll
  for (int k = 0; k < OPT; ++k) {
    const int idx = tid + k * NT;
    if (idx < G * D) {
      const int g = idx / D, d = idx - g * D;
      const float acc = a[k] + exp2f(m.lnew[g] - m.hm[g]) * to_f32(vt[d]);
      p.out[((size_t)b * p.kv_heads * G + (size_t)j * G + g) * D + d] = acc / m.hl[g];
    }
  }

  // method step 5: the current token's key, value and code replace the slot
  T* Kw = reinterpret_cast<T*>(p.K) + ((size_t)u * p.budget + winner) * D;
  T* Vw = reinterpret_cast<T*>(p.V) + ((size_t)u * p.budget + winner) * D;
  const T* kt = reinterpret_cast<const T*>(p.k) + (size_t)u * D;
  for (int d = tid; d < D; d += NT) {
    Kw[d] = kt[d];
    Vw[d] = vt[d];
  }
  if (tid == 0) {
    store_code(p.codes + (size_t)u * p.code_stride + (size_t)winner * (p.bits >> 3), p.bits,
               m.codek);
    if (p.score) p.score[(size_t)u * p.budget + winner] = 0.0f;  // not scored yet
    p.evicted[u] = full ? winner : -1;
    p.counters[u] = 0;
    log_eviction(p, u, full ? winner : -1);
  }
}

// After this CTA's record for unit u is written: fence, count in, and combine
// if this CTA is the unit's last contributor.  CTA c owns tiles
// [floor(c*TT/NC), floor((c+1)*TT/NC)); the owner of tile t is ((t+1)*NC-1)/TT.
template <typename T, int D, int G, int NT, int BAR>
__device__ __forceinline__ void finish_segment(const StepParams& p, int u, Misc& m, int tid,
                                               float* scratch, int cap) {
  // every thread's record stores are ordered before thread 0's release fence by
  // the barrier; the last contributor's acquire fence orders its reads after
  group_sync<NT, BAR>();
  HE_TL_MARK(m, 8);
  const int64_t TT = p.total_tiles, NC = gridDim.x;
  const int first = (int)((((int64_t)u * p.tpu + 1) * NC - 1) / TT);
  const int last = (int)((((int64_t)u * p.tpu + p.tpu) * NC - 1) / TT);
  if (tid == 0) {
    __threadfence();
    const int prev = atomicAdd(&p.counters[u], 1);
    __threadfence();
    m.is_last = (prev == last - first);
  }
  group_sync<NT, BAR>();
  HE_TL_MARK(m, 9);
  if (m.is_last) {
    combine_unit<T, D, G, NT, BAR>(p, u, first, last - first + 1, m, tid, scratch, cap);
    HE_TL_MARK(m, 10);
  }
  group_sync<NT, BAR>();
}

// ---------------------------------------------------------------------------
// Stand-alone kernels
// ---------------------------------------------------------------------------

constexpr int kAuxThreads = 256;

// Codes of rows of x (method steps 1-2).  Row r (r < rows) is vector
// (r / per_unit, r % per_unit) at x + ((r / per_unit) * x_unit_rows + r % per_unit) * D;
// its code goes to out + (r / per_unit) * out_unit_bytes + (r % per_unit) * bits/8.
// Bit j's threshold: tauv[(r / per_unit) * bits + j], or tau with tauv null.
// With proj non-null the kernel writes the projections instead of the codes:
// proj[((r / per_unit) * bits + j) * per_unit + r % per_unit] (fp32).
template <typename T, int D>
__global__ void __launch_bounds__(kAuxThreads) code_kernel(const T* __restrict__ x, int64_t rows,
                                                           int64_t per_unit, int64_t x_unit_rows,
                                                           const T* __restrict__ W, int bits,
                                                           float tau, const float* tauv,
                                                           unsigned char* out,
                                                           int64_t out_unit_bytes, float* proj) {
  __shared__ float xs[kAuxThreads / 8][D];  // up to 32 vectors (bits = 8)
  __shared__ uint32_t sbits[kAuxThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int vb = kAuxThreads / bits;  // vectors per block pass
  for (int64_t r0 = (int64_t)blockIdx.x * vb; r0 < rows; r0 += (int64_t)gridDim.x * vb) {
    for (int i = tid; i < vb * D; i += kAuxThreads) {
      const int vi = i / D, d = i - vi * D;
      const int64_t r = r0 + vi;
      float val = 0.0f;
      if (r < rows) {
        const int64_t unit = r / per_unit, s = r - unit * per_unit;
        val = to_f32(x[(unit * x_unit_rows + s) * D + d]);
      }
      xs[vi][d] = val;
    }
    __syncthreads();
    const int vi = tid / bits, j = tid - vi * bits;
    const int64_t r = r0 + vi;
    if (proj != nullptr) {
      if (r < rows) {
        const int64_t unit = r / per_unit, s = r - unit * per_unit;
        proj[(unit * bits + j) * per_unit + s] = projection_value<T, D>(xs[vi], W, bits, j);
      }
    } else {
      float tj = tau;
      if (tauv != nullptr && r < rows) tj = tauv[(r / per_unit) * bits + j];
      const uint32_t bit = r < rows ? projection_bit<T, D>(xs[vi], W, bits, j, tj) : 0u;
      const uint32_t word = __ballot_sync(kFull, bit);
      if (lane == 0) sbits[warp] = word;
      __syncthreads();
      if (tid < vb && r0 + tid < rows) {
        const int64_t r2 = r0 + tid;
        const int64_t unit = r2 / per_unit, s = r2 - unit * per_unit;
        store_code(out + unit * out_unit_bytes + s * (bits >> 3), bits,
                   code_from_bits(sbits, bits, tid));
      }
    }
    __syncthreads();
  }
}

// Order-preserving map of fp32 bit patterns to unsigned integers (a negative
// value's bits are complemented, a non-negative one gets its sign bit set).
__device__ __forceinline__ uint32_t float_order_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float float_from_order_key(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Per-bit lower-median thresholds: CTA c takes row c of proj ([rows][n] fp32,
// the n keys' projections onto one column of W) and writes element (n - 1) / 2
// of its ascending order to tau[c], by a radix select on the order-preserving
// keys (four passes of 8 bits, a shared-memory histogram each).  n >= 1.
static __global__ void __launch_bounds__(kAuxThreads)
    median_select_kernel(const float* __restrict__ proj, int64_t n, float* tau) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_prefix, s_rank;
  const int tid = threadIdx.x;
  const float* row = proj + (size_t)blockIdx.x * n;
  uint32_t prefix = 0, rank = (uint32_t)((n - 1) / 2);
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += kAuxThreads) hist[i] = 0;
    __syncthreads();
    for (int64_t i = tid; i < n; i += kAuxThreads) {
      const uint32_t k = float_order_key(__ldcg(row + i));
      // (keys that agree with the digits chosen so far)
      if (pass == 0 || (k >> (shift + 8)) == (prefix >> (shift + 8)))
        atomicAdd(&hist[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t c = 0;
      int b = 0;
      for (; b < 255; ++b) {
        if (c + hist[b] > rank) break;
        c += hist[b];
      }
      s_rank = rank - c;
      s_prefix = prefix | ((uint32_t)b << shift);
    }
    __syncthreads();
    prefix = s_prefix;
    rank = s_rank;
    __syncthreads();
  }
  if (tid == 0) tau[blockIdx.x] = float_from_order_key(prefix);
}

// Group-summed distances of every resident slot to the step's query codes
// (method step 3), one CTA per unit; slots occ..budget-1 get 0.
template <typename T, int D, int G>
__global__ void __launch_bounds__(kAuxThreads) score_kernel(const StepParams p, int32_t* dist) {
  __shared__ float s_q[G * D];
  __shared__ float s_k[D];
  __shared__ Misc m;
  const int tid = threadIdx.x;
  const int u = blockIdx.x;
  const int b = u / p.kv_heads, j = u - b * p.kv_heads;
  const T* qg = reinterpret_cast<const T*>(p.q) + ((size_t)b * p.kv_heads * G + (size_t)j * G) * D;
  for (int i = tid; i < G * D; i += kAuxThreads) s_q[i] = to_f32(qg[i]);
  for (int i = tid; i < D; i += kAuxThreads) s_k[i] = 0.0f;
  __syncthreads();
  code_queries_and_key<T, D, G, kAuxThreads, 0>(s_q, s_k, reinterpret_cast<const T*>(p.W),
                                                p.bits, p.tau,
                                                p.tauv ? p.tauv + (size_t)u * p.bits : nullptr,
                                                true, m, tid);
  uint64_t cq[G];
#pragma unroll
  for (int g = 0; g < G; ++g) cq[g] = m.cq[g];
  int32_t* drow = dist + (size_t)u * p.budget;
  for (int s = p.occ + tid; s < p.budget; s += kAuxThreads) drow[s] = 0;
  if (p.occ > 0)
    (void)scan_codes<G>(p.codes + (size_t)u * p.code_stride, p.bits, 0, p.occ, cq, tid,
                        kAuxThreads, drow);
}

// The projection matrix W[d][j] drawn from the seed: SplitMix64 finaliser over a
// counter (Steele, Lea, Flood 2014), Irwin-Hall sum of twelve 16-bit uniforms.
__device__ __forceinline__ uint64_t splitmix_finalise(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static __global__ void projection_kernel(uint64_t seed, int D, int bits, int is_fp32, void* W) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= D * bits) return;
  const uint64_t st = splitmix_finalise(seed ^ 0x48455F50524F4A57ull);
  int32_t sum = 0;
  for (int r = 0; r < 3; ++r) {
    const uint64_t w = splitmix_finalise(st + 3ull * (uint64_t)e + (uint64_t)r);
    sum += (int32_t)(w & 0xFFFF) + (int32_t)((w >> 16) & 0xFFFF) + (int32_t)((w >> 32) & 0xFFFF) +
           (int32_t)(w >> 48);
  }
  const float z = (float)(sum - 393210) * (1.0f / 65536.0f);
  if (is_fp32) {
    reinterpret_cast<float*>(W)[e] = z;
  } else {
    uint32_t u = __float_as_uint(z);
    u += 0x7FFFu + ((u >> 16) & 1u);  // round to nearest even
    reinterpret_cast<uint16_t*>(W)[e] = (uint16_t)(u >> 16);
  }
}

}  // namespace he
