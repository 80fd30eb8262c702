// he_fused.cuh — pieces of the fused bf16 step (one kernel per decode step for
// the method): the hash warp (method steps 1-4 for the CTA's own slots) and the
// merge that the last CTA to finish a unit's tiles runs (removal of the evicted
// slot, the new token, the output, and method step 5).
//
// A stream CTA owns a contiguous range of the step's 64-slot tiles; its range
// cuts the units it touches into segments (one per unit).  For each segment:
//   * the hash warp codes the unit's G query heads (and, in the CTA holding
//     the unit's first tile, the new key, with the new token's logits), scans
//     the codes of the segment's slots, folds the segment's best (distance,
//     slot) into the unit's eviction key with an order-independent atomicMax,
//     and stores that candidate's logits and value row in the CTA's record;
//   * the consumer warps stream the segment's tiles (attention over every
//     resident slot, the candidate included), write the partial (max, sum,
//     accumulator) into the same record and count the CTA in; the last CTA of
//     the unit merges.
// The unit's eviction key is the maximum over its segments' candidates, so the
// evicted slot is the candidate of exactly one record, whose logits and value
// row the merge takes out of that record's partial.  If the slot carries more
// than half of that partial's weight, the partial is recomputed exactly
// without it instead (CUDA cores), as the three-kernel pipeline does.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <type_traits>

#include "he_common.cuh"
#include "he_layout.cuh"
#include "he_tc.cuh"

namespace he {

constexpr int kFusedTile = 64;  // slots per tile of the fused step

// Atomic add with release and acquire semantics at GPU scope: this thread's
// (and, through barriers, its CTA's) writes before it are visible to whoever
// sees the count, and what the previous adders wrote is visible after it.
__device__ __forceinline__ int32_t atom_add_acq_rel_gpu(int32_t* p, int32_t v) {
  int32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ int32_t ld_acquire_gpu(const int32_t* p) {
  int32_t v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Contributors (stream CTAs) of unit u's tiles in a split of U * tps tiles.
__device__ __forceinline__ void unit_contributors(const TileSplit& sp, int u, int tps, int& first,
                                                  int& n) {
  first = (int)sp.owner((int64_t)u * tps);
  n = (int)sp.owner((int64_t)u * tps + tps - 1) - first + 1;
}

// Hash warps that fold the previous step's eviction key of unit u (0 when that
// step had no stream CTA).
__device__ __forceinline__ int prev_hash_count(const StepParams& p, int u) {
  if (p.prev_tpu <= 0 || p.prev_nc <= 0) return 0;
  const TileSplit ps{(int64_t)p.U * p.prev_tpu, (int64_t)p.prev_nc, p.prev_e, p.prev_t1};
  int first, n;
  unit_contributors(ps, u, p.prev_tpu, first, n);
  return n;
}

// Row of D bf16 (D / 2 words) into registers: lane l holds words l, l + 32, ...
template <int D>
__device__ __forceinline__ void load_row_words(const uint16_t* src, uint32_t (&w)[D / 64],
                                               int lane) {
  const uint32_t* s = reinterpret_cast<const uint32_t*>(src);
#pragma unroll
  for (int i = 0; i < D / 64; ++i) w[i] = __ldcg(s + i * 32 + lane);
}

// Dot product of a row held as load_row_words with an fp32 row in shared
// memory (lane-local sums, then the warp sum).
template <int D>
__device__ __forceinline__ float row_dot_s(const float* xs, const uint32_t (&b)[D / 64], int lane) {
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < D / 64; ++i) {
    const float2 x = *reinterpret_cast<const float2*>(xs + 2 * (i * 32 + lane));
    s = fmaf(x.x, bf16_lo(b[i]), s);
    s = fmaf(x.y, bf16_hi(b[i]), s);
  }
  return warp_sum(s);
}

// Method steps 1-2 for NV vectors on one warp: bit j of vector v is
// (sum_d x_v[d] W[d][j] > tau), each sum in fp32 with fused multiply-adds in
// the fixed order d = 0..D-1 from +0 (the specification's chains; bf16 products
// are exact, so only that order matters).  Lane j owns bit j (and j + 32 for
// 64-bit codes).  xs: the vectors as fp32 [NV][D] (exact copies of the bf16
// elements) and Ws: W [D][bits] (bf16), both in shared memory.
// tauv: per-bit thresholds [bits] (null: tau on every bit).
template <int D, int NV>
__device__ __forceinline__ void hash_codes(const float* xs, const uint16_t* Ws, int bits,
                                           float tau, const float* tauv, int lane,
                                           uint64_t (&code)[NV]) {
  const bool two = bits == 64;
  const bool ok0 = lane < bits;
  const int j0 = ok0 ? lane : 0, j1 = two ? lane + 32 : 0;
  const float t0 = tauv ? __ldg(tauv + j0) : tau, t1 = tauv && two ? __ldg(tauv + j1) : tau;
  float a0[NV], a1[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) a0[v] = a1[v] = 0.0f;
#pragma unroll 2
  for (int d = 0; d < D; d += 4) {
    float w0[4], w1[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      w0[e] = __uint_as_float((uint32_t)Ws[(d + e) * bits + j0] << 16);
      w1[e] = __uint_as_float((uint32_t)Ws[(d + e) * bits + j1] << 16);
    }
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const float4 x = *reinterpret_cast<const float4*>(xs + v * D + d);  // (a broadcast)
      a0[v] = __fmaf_rn(x.x, w0[0], a0[v]);
      a0[v] = __fmaf_rn(x.y, w0[1], a0[v]);
      a0[v] = __fmaf_rn(x.z, w0[2], a0[v]);
      a0[v] = __fmaf_rn(x.w, w0[3], a0[v]);
      if (two) {
        a1[v] = __fmaf_rn(x.x, w1[0], a1[v]);
        a1[v] = __fmaf_rn(x.y, w1[1], a1[v]);
        a1[v] = __fmaf_rn(x.z, w1[2], a1[v]);
        a1[v] = __fmaf_rn(x.w, w1[3], a1[v]);
      }
    }
  }
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const uint32_t lo = __ballot_sync(kFull, ok0 && a0[v] > t0);
    const uint32_t hi = __ballot_sync(kFull, two && a1[v] > t1);
    code[v] = (uint64_t)lo | ((uint64_t)hi << 32);
  }
}

// Best eviction key over the codes of slots [lo, hi) of one unit row (method
// steps 3-4), read as 16-byte chunks through L2 (lanes take chunks lane,
// lane + 32, ...; NBATCH chunks per lane are loaded before any is used); the
// warp's maximum.  dist_out (test export, may be null): every slot's distance.
template <int G, int WB>
__device__ __forceinline__ uint64_t hash_scan_w(const unsigned char* row, int lo, int hi,
                                                const uint64_t (&cq)[G], int lane,
                                                int32_t* dist_out) {
  constexpr int PER = 16 / WB;
  constexpr int NBATCH = 8;
  const int c0 = (lo * WB) >> 4;
  const int c1 = (hi * WB + 15) >> 4;
  uint64_t best = 0;
  for (int cb = c0; cb < c1; cb += 32 * NBATCH) {
    uint4 ch[NBATCH];
#pragma unroll
    for (int b = 0; b < NBATCH; ++b) {
      const int c = cb + lane + 32 * b;
      ch[b] = c < c1 ? __ldcg(reinterpret_cast<const uint4*>(row) + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int b = 0; b < NBATCH; ++b) {
      const int c = cb + lane + 32 * b;
      const uint32_t wd[4] = {ch[b].x, ch[b].y, ch[b].z, ch[b].w};
      const int s0 = c * PER;
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        uint64_t code;
        if (WB == 8) code = (uint64_t)wd[2 * e] | ((uint64_t)wd[2 * e + 1] << 32);
        else if (WB == 4) code = wd[e];
        else if (WB == 2) code = (wd[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
        else code = (wd[e >> 2] >> (8 * (e & 3))) & 0xFFu;
        const int s = s0 + e;
        if (c < c1 && s >= lo && s < hi) {
          const uint32_t dist = group_distance<G>(cq, code);
          if (dist_out != nullptr) dist_out[s] = (int32_t)dist;
          const uint64_t key = evict_key(dist, (uint32_t)s);
          best = key > best ? key : best;
        }
      }
    }
  }
  return warp_max_u64(best);
}

template <int G>
__device__ __forceinline__ uint64_t hash_scan(const unsigned char* row, int bits, int lo, int hi,
                                              const uint64_t (&cq)[G], int lane,
                                              int32_t* dist_out) {
  switch (bits) {
    case 8: return hash_scan_w<G, 1>(row, lo, hi, cq, lane, dist_out);
    case 16: return hash_scan_w<G, 2>(row, lo, hi, cq, lane, dist_out);
    case 32: return hash_scan_w<G, 4>(row, lo, hi, cq, lane, dist_out);
    default: return hash_scan_w<G, 8>(row, lo, hi, cq, lane, dist_out);
  }
}

// The hash warp of a fused-step CTA holding tiles [sb, se), with W [D][bits]
// brought into Ws by one bulk copy and xs ((G + 1) x D fp32, shared) holding
// the rows of the unit at hand: for each segment in tile order, the work
// described at the top of this file.  The codes depend on this step's inputs
// only, so the first segment's are computed before the dependency wait;
// everything that reads the cache (codes, candidate rows) comes after it.
// After segment i, i + 1 goes to *hash_done for the consumer warps.  With an
// empty cache (no tiles) CTA u only codes unit u's new key and logits.
template <int D, int G>
__device__ void hash_warp(const StepParams& p, int sb, int se, volatile int32_t* hash_done,
                          int lane, uint16_t* Ws, uint64_t* wbar, float* xs) {
  using FR = FRec<G, D>;
  const int tps = p.tpu;
  const bool full = p.append_slot < 0;
  const bool empty = tps == 0;
  if (lane == 0) {
    const uint32_t wbytes = (uint32_t)(D * p.bits * 2);
    mbar_arrive_expect_tx(wbar, wbytes);
    bulk_g2s(Ws, p.W, wbytes, wbar);
  }
  HE_STAMP_IF(lane == 0, 0, 0);
  // method steps 1-2 for unit u: its rows into xs, the G query codes and the
  // new key's code into code[], the new token's base-2 logits into lnew[]
  uint64_t code[G + 1];
  float lnew[G];
  auto prepare = [&](int u) {
    __syncwarp();
#pragma unroll
    for (int r = 0; r <= G; ++r) {
      const uint16_t* src = r < G ? reinterpret_cast<const uint16_t*>(p.q) + ((size_t)u * G + r) * D
                                  : reinterpret_cast<const uint16_t*>(p.k) + (size_t)u * D;
      uint32_t w[D / 64];
      load_row_words<D>(src, w, lane);
#pragma unroll
      for (int i = 0; i < D / 64; ++i)
        *reinterpret_cast<float2*>(xs + r * D + 2 * (i * 32 + lane)) =
            make_float2(bf16_lo(w[i]), bf16_hi(w[i]));
    }
    __syncwarp();
    hash_codes<D, G + 1>(xs, Ws, p.bits, p.tau,
                         p.tauv ? p.tauv + (size_t)u * p.bits : nullptr, lane, code);
    uint32_t kw[D / 64];
    load_row_words<D>(reinterpret_cast<const uint16_t*>(p.k) + (size_t)u * D, kw, lane);
#pragma unroll
    for (int g = 0; g < G; ++g) lnew[g] = row_dot_s<D>(xs + g * D, kw, lane) * p.qscale;
  };
  bool ok = mbar_wait_bounded(wbar, 0u);
  if (!ok) atomicExch(p.err, 1);  // (the consumers give up waiting for this warp)
  if (ok && (empty || sb < se)) prepare(empty ? (int)blockIdx.x : sb / tps);
  HE_STAMP_IF(lane == 0, 0, 1);
  pdl_wait();  // the previous step is complete: codes and cache are final
  HE_STAMP_IF(lane == 0, 0, 2);
  int seg = 0;
  for (int t = empty ? 0 : sb; ok && (empty ? seg == 0 : t < se); ++seg) {
    const int u = empty ? (int)blockIdx.x : t / tps;
    const int te = empty ? 0 : min(se, (u + 1) * tps);
    if (seg > 0) prepare(u);
    if ((empty || t == u * tps) && lane == 0) {
      // this CTA holds the unit's first tile: the new token's code and logits
      // for the unit's merge
      p.uo[u].codek = code[G];
#pragma unroll
      for (int g = 0; g < G; ++g) p.uo[u].lnew[g] = lnew[g];
    }
    if (full && !empty) {
      uint64_t cq[G];
#pragma unroll
      for (int g = 0; g < G; ++g) cq[g] = code[g];
      const int lo = (t - u * tps) * kFusedTile;
      const int hi = min((te - u * tps) * kFusedTile, p.occ);
      const uint64_t best =
          hash_scan<G>(p.codes + (size_t)u * p.code_stride, p.bits, lo, hi, cq, lane,
                       p.dist != nullptr ? p.dist + (size_t)u * p.budget : nullptr);
      if (lane == 0 && best != 0) atomicMax(&p.uo[u].key[p.kpar], (unsigned long long)best);
      // the candidate's logits and value row into this CTA's record
      const int cand = best != 0 ? (int)evict_key_slot(best) : lo;
      float* rec = p.partials + ((size_t)blockIdx.x + u) * FR::FLOATS;
      if (HE_CHECK(cand >= lo && cand < hi && (int64_t)blockIdx.x + u < (int64_t)gridDim.x + p.U,
                   p.err)) {
        uint32_t kr[D / 64], vr[D / 64];
        const size_t row = ((size_t)u * p.budget + cand) * D;
        load_row_words<D>(reinterpret_cast<const uint16_t*>(p.K) + row, kr, lane);
        load_row_words<D>(reinterpret_cast<const uint16_t*>(p.V) + row, vr, lane);
        uint32_t* vdst = reinterpret_cast<uint32_t*>(rec + FR::VR);
#pragma unroll
        for (int i = 0; i < D / 64; ++i) __stcg(vdst + i * 32 + lane, vr[i]);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float l = row_dot_s<D>(xs + g * D, kr, lane) * p.qscale;
          if (lane == 0) __stcg(rec + FR::LC + g, l);
        }
        if (lane == 0)
          __stcg(reinterpret_cast<unsigned long long*>(rec + FR::KEY), (unsigned long long)best);
      }
    }
    // the key fold (and the record) before the count that says it is final
    __threadfence();
    __syncwarp();
    if (lane == 0) {
      if (!empty) atomicAdd(&p.uo[u].hcnt[p.kpar], 1);
      __threadfence_block();
      *hash_done = seg + 1;
    }
    HE_STAMP_IF(lane == 0 && seg == 0, 0, 3);
    __syncwarp();
    t = te;
  }
  HE_STAMP_IF(lane == 0, 0, 4);
}

// Exact partial of unit u over slots [lo, hi) without slot `skip` (CUDA cores,
// fp32), by the NW consumer warps: each warp runs an online softmax over a
// strided share of the slots (lane l holds elements [l E, l E + E)), the warp
// states meet in wst [NW][G][2 + D] (shared memory), and the result (base-2
// max, sum, accumulator) replaces the partial fields of record `rec`.
// Returns false if a consumer barrier gave up.
template <int D, int G, int NW>
__device__ bool recompute_record(const StepParams& p, int u, int lo, int hi, int skip,
                                 float* wst, float* rec, int tid, uint64_t* bar,
                                 uint32_t& phase) {
  using FR = FRec<G, D>;
  constexpr int E = D / 32;
  constexpr int NT = NW * 32;
  const int lane = tid & 31, warp = tid >> 5;
  {
    float qf[G][E];
    const uint16_t* qg = reinterpret_cast<const uint16_t*>(p.q) + (size_t)u * G * D;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < E; ++e)
        qf[g][e] = __uint_as_float((uint32_t)__ldcg(qg + g * D + lane * E + e) << 16);
    const uint16_t* Kc = reinterpret_cast<const uint16_t*>(p.K) + (size_t)u * p.budget * D;
    const uint16_t* Vc = reinterpret_cast<const uint16_t*>(p.V) + (size_t)u * p.budget * D;
    float mr[G], lr[G], ar[G][E];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      mr[g] = -1e30f;
      lr[g] = 0.0f;
#pragma unroll
      for (int e = 0; e < E; ++e) ar[g][e] = 0.0f;
    }
    constexpr int RU = G >= 8 ? 1 : 2;  // slots loaded per round trip
    for (int s0 = lo + warp * RU; s0 < hi; s0 += NW * RU) {
      float kx[RU][E], vx[RU][E];
#pragma unroll
      for (int r = 0; r < RU; ++r) {
        const int s = s0 + r < hi ? s0 + r : hi - 1;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          kx[r][e] = __uint_as_float((uint32_t)__ldcg(Kc + (size_t)s * D + lane * E + e) << 16);
          vx[r][e] = __uint_as_float((uint32_t)__ldcg(Vc + (size_t)s * D + lane * E + e) << 16);
        }
      }
#pragma unroll
      for (int r = 0; r < RU; ++r) {
        const int s = s0 + r;
        if (s >= hi || s == skip) continue;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float dot = 0.0f;
#pragma unroll
          for (int e = 0; e < E; ++e) dot = fmaf(qf[g][e], kx[r][e], dot);
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
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float* ws = wst + ((size_t)warp * G + g) * (2 + D);
      if (lane == 0) {
        ws[0] = mr[g];
        ws[1] = lr[g];
      }
#pragma unroll
      for (int e = 0; e < E; ++e) ws[2 + lane * E + e] = ar[g][e];
    }
  }
  if (!consumer_sync<NW>(bar, phase, lane)) return false;
  for (int idx = tid; idx < G * D; idx += NT) {
    const int g = idx / D, d = idx - g * D;
    float mx = -1e30f;
    for (int w = 0; w < NW; ++w) mx = fmaxf(mx, wst[((size_t)w * G + g) * (2 + D)]);
    float a = 0.0f, l = 0.0f;
    for (int w = 0; w < NW; ++w) {
      const float* ws = wst + ((size_t)w * G + g) * (2 + D);
      const float sc = exp2f(ws[0] - mx);
      a += ws[2 + d] * sc;
      l += ws[1] * sc;
    }
    __stcg(rec + FR::HDR + idx, a);
    if (d == 0) {
      __stcg(rec + g, mx);
      __stcg(rec + G + g, l);
    }
  }
  __threadfence_block();
  return consumer_sync<NW>(bar, phase, lane);
}

// The merge of unit u by the NW consumer warps of its last contributor
// (contributors first .. first + n - 1, records first + u ..): the evicted slot
// out of the record that holds it (or that record recomputed without it), the
// log-sum-exp merge of every record in a fixed order, the new token, the
// output; then method step 5 (the new token's key, value and code into the
// slot) and the resets the next steps of this cache rely on.  wst: shared
// scratch of NW * G * (2 + D) floats; flag: one shared int, set to mseq (this
// CTA's merge number, from 1) when the exact path is needed.
// Returns false if a consumer barrier gave up.
template <int D, int G, int NW>
__device__ bool fused_merge(const StepParams& p, const TileSplit& split, int u, int first, int n,
                            float* wst, int* flag, int mseq, int tid, uint64_t* bar,
                            uint32_t& phase) {
  using FR = FRec<G, D>;
  constexpr int NT = NW * 32;
  constexpr int GD4 = G * D / 4;
  constexpr int OPT = (GD4 + NT - 1) / NT;  // float4 outputs per thread
  const int lane = tid & 31;
  const bool full = p.append_slot < 0;
  const int tps = p.tpu;
  const float* recs = p.partials + (size_t)(first + u) * FR::FLOATS;
  int og[OPT], od[OPT];
#pragma unroll
  for (int k = 0; k < OPT; ++k) {
    const int o = tid + k * NT < GD4 ? tid + k * NT : 0;
    og[k] = (4 * o) / D;
    od[k] = 4 * o - og[k] * D;
  }
  // everything that does not depend on the decision, with the decision itself
  float lnw[OPT];
  uint2 vtw[OPT];
  const uint16_t* vt = reinterpret_cast<const uint16_t*>(p.v) + (size_t)u * D;
#pragma unroll
  for (int k = 0; k < OPT; ++k) {
    lnw[k] = __ldcg(&p.uo[u].lnew[og[k]]);
    vtw[k] = __ldcg(reinterpret_cast<const uint2*>(vt + od[k]));
  }
  const unsigned long long key = full ? __ldcg(&p.uo[u].key[p.kpar]) : 0ull;
  const int winner = full ? (key ? (int)evict_key_slot(key) : -1) : p.append_slot;
  if (!HE_CHECK(n >= 0 && (int64_t)first + u + n <= (int64_t)gridDim.x + p.U, p.err)) n = 0;

  // The records are loaded a batch at a time with every field the merge may
  // need, so the decision (the unit's key, loaded with the first batch) costs no
  // round trip of its own: the record that holds the evicted slot is the one
  // whose candidate key equals the unit's key.
  float mx[OPT], sum[OPT];
  float4 acc[OPT];
  float lst[OPT], cm[OPT], cl[OPT];
  float4 vst[OPT];
  bool have_c = false;
  auto fold_all = [&](auto find_tag) {
    constexpr bool find = decltype(find_tag)::value;
    // (fewer records per round trip while looking for the evicted slot's record:
    // each carries its candidate fields too)
    constexpr int NB = find ? (OPT == 1 ? 4 : 2) : (OPT == 1 ? 8 : 4);
#pragma unroll
    for (int k = 0; k < OPT; ++k) {
      mx[k] = -1e30f;
      sum[k] = 0.0f;
      acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int c0 = 0; c0 < n; c0 += NB) {
      float rm[NB][OPT], rl[NB][OPT], rc_l[NB][OPT];
      float4 rx[NB][OPT];
      uint2 rv[NB][OPT];
      unsigned long long rk[NB];
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        const int c = c0 + i < n ? c0 + i : n - 1;
        const float* r = recs + (size_t)c * FR::FLOATS;
        rk[i] = find ? __ldcg(reinterpret_cast<const unsigned long long*>(r + FR::KEY)) : 0ull;
#pragma unroll
        for (int k = 0; k < OPT; ++k) {
          const int o = tid + k * NT < GD4 ? tid + k * NT : 0;
          rm[i][k] = __ldcg(r + og[k]);
          rl[i][k] = __ldcg(r + G + og[k]);
          rx[i][k] = __ldcg(reinterpret_cast<const float4*>(r + FR::HDR) + o);
          rc_l[i][k] = find ? __ldcg(r + FR::LC + og[k]) : 0.0f;
          rv[i][k] = find ? __ldcg(reinterpret_cast<const uint2*>(r + FR::VR) + od[k] / 4)
                          : make_uint2(0u, 0u);
        }
      }
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        if (c0 + i >= n) continue;
        if (find && full && !have_c && rk[i] == key) {
          have_c = true;
#pragma unroll
          for (int k = 0; k < OPT; ++k) {
            lst[k] = rc_l[i][k];
            cm[k] = rm[i][k];
            cl[k] = rl[i][k];
            vst[k] = make_float4(bf16_lo(rv[i][k].x), bf16_hi(rv[i][k].x), bf16_lo(rv[i][k].y),
                                 bf16_hi(rv[i][k].y));
          }
        }
#pragma unroll
        for (int k = 0; k < OPT; ++k) {
          const float mc = rm[i][k], lc = rl[i][k];
          const float4 x = rx[i][k];
          const float mn = fmaxf(mx[k], mc);
          const float so = exp2f(mx[k] - mn), sn = exp2f(mc - mn);
          sum[k] = sum[k] * so + lc * sn;
          acc[k].x = acc[k].x * so + x.x * sn;
          acc[k].y = acc[k].y * so + x.y * sn;
          acc[k].z = acc[k].z * so + x.z * sn;
          acc[k].w = acc[k].w * so + x.w * sn;
          mx[k] = mn;
        }
      }
    }
  };
  fold_all(std::true_type{});
  if (winner < 0 || winner >= p.budget) {  // cannot happen: never write outside the cache
    if (tid == 0) atomicExch(p.err, 2);
    return true;
  }
  // (a full step's key is one of the records' candidates; a missing match is
  // reported and the slot is not taken out)
  if (full && n > 0 && !have_c && tid == 0) atomicExch(p.err, 2);
  // the evicted slot leaves the total, unless it carries more than half of its
  // own record's weight: then that record is recomputed without it
  if (have_c) {
#pragma unroll
    for (int k = 0; k < OPT; ++k)
      if (tid + k * NT < GD4 && !(exp2f(lst[k] - cm[k]) <= 0.5f * cl[k])) *flag = mseq;
  }
  if (!consumer_sync<NW>(bar, phase, lane)) return false;
  const bool recomputed = *flag == mseq;
  if (recomputed) {
    const int crel = (int)split.owner((int64_t)u * tps + winner / kFusedTile) - first;
    const int c = first + crel;
    const int tb = (int)split.begin(c), te = (int)split.begin((int64_t)c + 1);
    const int lo = (max(tb, u * tps) - u * tps) * kFusedTile;
    const int hi = min((min(te, (u + 1) * tps) - u * tps) * kFusedTile, p.occ);
    float* rec = const_cast<float*>(recs) + (size_t)crel * FR::FLOATS;
    if (!recompute_record<D, G, NW>(
            p, u, lo,
            HE_CHECK(0 <= lo && lo <= hi && hi <= p.budget && 0 <= crel && crel < n, p.err) ? hi
                                                                                           : lo,
            winner, wst, rec, tid, bar, phase))
      return false;
    fold_all(std::false_type{});
  } else if (have_c) {
#pragma unroll
    for (int k = 0; k < OPT; ++k) {
      const float pw = exp2f(lst[k] - mx[k]);
      sum[k] -= pw;
      acc[k].x -= pw * vst[k].x;
      acc[k].y -= pw * vst[k].y;
      acc[k].z -= pw * vst[k].z;
      acc[k].w -= pw * vst[k].w;
    }
  }

  // the new token, the output
  float* out = p.out + (size_t)u * G * D;
#pragma unroll
  for (int k = 0; k < OPT; ++k) {
    const int o = tid + k * NT;
    if (o < GD4) {
      const uint2 w2 = vtw[k];
      const float m2 = fmaxf(mx[k], lnw[k]);
      const float so = exp2f(mx[k] - m2), wn = exp2f(lnw[k] - m2);
      const float inv = 1.0f / (sum[k] * so + wn);
      float4 r;
      r.x = (acc[k].x * so + wn * bf16_lo(w2.x)) * inv;
      r.y = (acc[k].y * so + wn * bf16_hi(w2.x)) * inv;
      r.z = (acc[k].z * so + wn * bf16_lo(w2.y)) * inv;
      r.w = (acc[k].w * so + wn * bf16_hi(w2.y)) * inv;
      reinterpret_cast<float4*>(out)[o] = r;
    }
  }

  // method step 5: the current token's key, value and code replace the slot
  constexpr int CH = D / 8;  // 16-byte pieces per row
  const size_t row = ((size_t)u * p.budget + winner) * D;
  if (tid < 2 * CH) {
    const int c = tid < CH ? tid : tid - CH;
    const uint16_t* src = reinterpret_cast<const uint16_t*>(tid < CH ? p.k : p.v) + (size_t)u * D;
    uint16_t* dst = reinterpret_cast<uint16_t*>(tid < CH ? p.K : p.V) + row;
    reinterpret_cast<uint4*>(dst)[c] = __ldcg(reinterpret_cast<const uint4*>(src) + c);
  }
  if (tid == 0) {
    store_code(p.codes + (size_t)u * p.code_stride + (size_t)winner * (p.bits >> 3), p.bits,
               __ldcg(&p.uo[u].codek));
    p.evicted[u] = full ? winner : -1;
    log_eviction(p, u, full ? winner : -1);
    // ready for the next steps: the contributor count, and the other parity's
    // key and hash count (the previous step's, read by this step's CTAs before
    // they waited; every contributor of this unit is past that)
    p.uo[u].arrived = 0;
    p.uo[u].key[p.kpar ^ 1] = 0ull;
    p.uo[u].hcnt[p.kpar ^ 1] = 0;
    if (recomputed) atomicAdd(p.counters + u, 1);  // how often the exact path ran
  }
  return true;
}

}  // namespace he
