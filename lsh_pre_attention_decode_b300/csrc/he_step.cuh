// he_step.cuh — the fused HashEvict decode step: one launch per step does
// method steps 1-5 and the decode attention (HashEvict, arXiv 2412.16187,
// technical framework steps 1-5 and abstract; attention over the retained
// cache as in the TTKV page's introduction).
//
// Work decomposition (stream-K over cache tiles):
//   The resident slots of every (batch, KV head) unit are cut into tiles of 32
//   slots; the U * tiles_per_unit tiles form one list that is split into equal
//   contiguous ranges, one per CTA (grid = SMs x resident CTAs per SM).  A range
//   may cover the end of one unit and the start of the next: the CTA emits one
//   partial result per unit it touches.
//   Per unit segment a CTA
//     (a) codes the G query heads and the new key (fixed-order fp32 projection,
//         sign, ballot bit-pack), and the new token's attention logits;
//     (b) scans its slots' packed codes (16-byte loads, XOR + popcount, summed
//         over the G query codes) for its local eviction candidate: the largest
//         distance, lowest slot on ties;
//     (c) streams its K/V tiles through shared memory (TMA bulk copies,
//         NS-stage mbarrier ring) and runs an online softmax that leaves the
//         local candidate out but keeps its logits aside;
//     (d) writes its partial (max, sum, accumulator, candidate) and counts
//         itself in; the last CTA of a unit (atomic counter, no waiting) picks
//         the global candidate (the largest local key), merges the partials,
//         adds back every non-winning candidate and the new token, writes the
//         output, and overwrites the evicted slot's K, V and code.
//   This is the same arithmetic as "evict, overwrite, then attend": the
//   evicted slot never enters the softmax and the new token always does.
#pragma once

#include "he_device.cuh"

namespace he {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = 32;  // cache slots per tile

struct StepParams {
  void* K;              // cache keys   [U][budget][D]
  void* V;              // cache values [U][budget][D]
  unsigned char* codes; // [U][code_stride] words of bits/8 bytes
  const void* W;        // projection [D][bits]
  const void* q;        // [batch][heads][D]
  const void* k;        // [batch][kv_heads][D]
  const void* v;        // [batch][kv_heads][D]
  float* out;           // [batch][heads][D]
  int32_t* evicted;     // [U]
  float* partials;      // [ctas + U][record]
  int32_t* counters;    // [U], zero between steps
  int32_t* err;         // set to nonzero when a wait gives up
  int32_t U;
  int32_t kv_heads;
  int32_t budget;
  int32_t occ;          // resident slots before the step
  int32_t tpu;          // tiles per unit = ceil(occ / kTile)
  int32_t total_tiles;  // U * tpu
  int32_t bits;
  int32_t code_stride;  // bytes per unit row of codes (multiple of 16)
  int32_t append_slot;  // -1: cache full, evict; else the slot the token is appended to
  float qscale;         // log2(e) / sqrt(D): logits kept in base 2
};

template <typename T, int D, int G, int NS>
struct StepShape {
  static constexpr int EB = ElemTraits<T>::kBytes;
  static constexpr int ROWB = D * EB;               // bytes per cached row
  static constexpr int TILEB = kTile * ROWB;        // bytes per K (or V) tile
  static constexpr int LPS = (G * D / 8 > 64) ? 16 : 8;  // lanes per slot, logit phase
  static constexpr int EPL = D / LPS;               // elements per lane, logit phase
  static constexpr int EPC = 16 / EB;               // elements per 16-byte chunk
  static constexpr int CPL = EPL / EPC;             // chunks per lane, logit phase
  static constexpr int NPASS = kTile * LPS / kThreads;
  static constexpr int SPW = kTile / kWarps;        // slots per warp, value phase
  static constexpr int EPW = D / 32;                // elements per lane, value phase
  static constexpr int HDR = ((3 * G + 2) + 3) / 4 * 4;  // record header floats
  static constexpr int REC = HDR + G * D;           // floats per partial record
  // shared memory carve-up (bytes; every offset a multiple of 16)
  static constexpr int OFF_STAGE = 0;
  static constexpr int OFF_WACC = OFF_STAGE + NS * 2 * TILEB;
  static constexpr int OFF_Q = OFF_WACC + kWarps * G * D * 4;
  static constexpr int OFF_K = OFF_Q + G * D * 4;
  static constexpr int OFF_LG = OFF_K + D * 4;
  static constexpr int OFF_PW = OFF_LG + 2 * kTile * G * 4;
  static constexpr int OFF_WM = OFF_PW + kWarps * SPW * G * 4;
  static constexpr int OFF_MISC = OFF_WM + 2 * kWarps * G * 4;
  static constexpr int MISC = 512;
  static constexpr int OFF_BAR = OFF_MISC + MISC;
  static constexpr int SMEM = OFF_BAR + NS * 8;
  static_assert(D % 64 == 0 && (G & (G - 1)) == 0 && G <= 8, "shape");
  static_assert(CPL >= 1 && NPASS >= 1 && G <= LPS, "logit lane mapping");
  static_assert(SPW * G <= 32, "value-phase softmax lanes");
};

// Misc shared block (inside OFF_MISC .. +512).
struct Misc {
  uint32_t bits[32];    // packed code bits of the G queries and the key
  uint64_t cq[8];       // query codes
  uint64_t codek;       // the new key's code
  uint64_t pad0;
  float lnew[8];        // new token's base-2 logits
  float candlog[8];     // local candidate's base-2 logits
  float hm[8];          // combine: per-head max
  float hl[8];          // combine: per-head sum
  uint64_t red64[kWarps];
  int32_t cand_slot;
  int32_t cand_dist;
  int32_t is_last;
  int32_t winner;
};
static_assert(sizeof(Misc) <= 512, "misc");

// Loads EPW consecutive elements of a row, converted exactly to fp32.
template <typename T, int EPW>
__device__ __forceinline__ void load_row_part(const unsigned char* src, float (&x)[EPW]);
template <>
__device__ __forceinline__ void load_row_part<bf16_t, 4>(const unsigned char* src, float (&x)[4]) {
  uint2 w = *reinterpret_cast<const uint2*>(src);
  x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
}
template <>
__device__ __forceinline__ void load_row_part<bf16_t, 2>(const unsigned char* src, float (&x)[2]) {
  uint32_t w = *reinterpret_cast<const uint32_t*>(src);
  x[0] = bf16_lo(w); x[1] = bf16_hi(w);
}
template <>
__device__ __forceinline__ void load_row_part<float, 4>(const unsigned char* src, float (&x)[4]) {
  float4 w = *reinterpret_cast<const float4*>(src);
  x[0] = w.x; x[1] = w.y; x[2] = w.z; x[3] = w.w;
}
template <>
__device__ __forceinline__ void load_row_part<float, 2>(const unsigned char* src, float (&x)[2]) {
  float2 w = *reinterpret_cast<const float2*>(src);
  x[0] = w.x; x[1] = w.y;
}

// 16-byte chunk -> EPC floats (exact).
template <typename T>
__device__ __forceinline__ void chunk_to_f32(const uint4& c, float* x);
template <>
__device__ __forceinline__ void chunk_to_f32<bf16_t>(const uint4& c, float* x) {
  x[0] = bf16_lo(c.x); x[1] = bf16_hi(c.x); x[2] = bf16_lo(c.y); x[3] = bf16_hi(c.y);
  x[4] = bf16_lo(c.z); x[5] = bf16_hi(c.z); x[6] = bf16_lo(c.w); x[7] = bf16_hi(c.w);
}
template <>
__device__ __forceinline__ void chunk_to_f32<float>(const uint4& c, float* x) {
  x[0] = __uint_as_float(c.x); x[1] = __uint_as_float(c.y);
  x[2] = __uint_as_float(c.z); x[3] = __uint_as_float(c.w);
}

// Store / load one packed code word of w = bits/8 bytes.
__device__ __forceinline__ void store_code(unsigned char* dst, int bits, uint64_t code) {
  switch (bits) {
    case 8: *dst = (unsigned char)code; break;
    case 16: *reinterpret_cast<uint16_t*>(dst) = (uint16_t)code; break;
    case 32: *reinterpret_cast<uint32_t*>(dst) = (uint32_t)code; break;
    default: *reinterpret_cast<uint64_t*>(dst) = code; break;
  }
}

// Group-summed Hamming distance of one cached code to the G query codes.
template <int G>
__device__ __forceinline__ uint32_t group_distance(const uint64_t (&cq)[G], uint64_t code) {
  uint32_t d = 0;
#pragma unroll
  for (int g = 0; g < G; ++g) d += (uint32_t)popc64(cq[g] ^ code);
  return d;
}

// Best eviction key over the codes of slots [lo, hi) of one unit row, read as
// 16-byte chunks of 16/WB codes (WB = bits/8 bytes per code); per-thread result
// (reduce afterwards).  When dist_out is set, the distances are stored too.
template <int G, int WB>
__device__ __forceinline__ uint64_t scan_codes_w(const unsigned char* row, int lo, int hi,
                                                 const uint64_t (&cq)[G], int tid, int nthreads,
                                                 int32_t* dist_out) {
  constexpr int PER = 16 / WB;  // codes per chunk
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
        const uint64_t key = evict_key(dist, (uint32_t)s);
        best = key > best ? key : best;
      }
    }
  }
  return best;
}

template <int G>
__device__ __forceinline__ uint64_t scan_codes(const unsigned char* row, int bits, int lo, int hi,
                                               const uint64_t (&cq)[G], int tid, int nthreads,
                                               int32_t* dist_out) {
  switch (bits) {
    case 8: return scan_codes_w<G, 1>(row, lo, hi, cq, tid, nthreads, dist_out);
    case 16: return scan_codes_w<G, 2>(row, lo, hi, cq, tid, nthreads, dist_out);
    case 32: return scan_codes_w<G, 4>(row, lo, hi, cq, tid, nthreads, dist_out);
    default: return scan_codes_w<G, 8>(row, lo, hi, cq, tid, nthreads, dist_out);
  }
}

// Codes the G query heads (when `with_queries`) and the key staged in shared
// memory (s_q [G][D], s_k [D]) into m.cq[] and m.codek.  Bit tasks are laid out
// head-major (task = head * bits + j; head G is the key) and packed with warp
// ballots.  Ends with a __syncthreads.
template <typename T, int D, int G>
__device__ __forceinline__ void code_queries_and_key(const float* s_q, const float* s_k,
                                                     const T* W, int bits, bool with_queries,
                                                     Misc& m, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  const int ntask = (G + 1) * bits;
  for (int t0 = warp * 32; t0 < ntask; t0 += kThreads) {
    const int t = t0 + lane;
    uint32_t bit = 0;
    if (t < ntask) {
      const int h = t / bits, j = t - h * bits;
      if (h == G)
        bit = projection_bit<T, D>(s_k, W, bits, j);
      else if (with_queries)
        bit = projection_bit<T, D>(s_q + h * D, W, bits, j);
    }
    const uint32_t word = __ballot_sync(kFull, bit);
    if (lane == 0) m.bits[t0 >> 5] = word;
  }
  __syncthreads();
  if (tid <= G) {
    const uint64_t c = code_from_bits(m.bits, bits, tid);
    if (tid < G) m.cq[tid] = c;
    else m.codek = c;
  }
  __syncthreads();
}

template <typename T, int D, int G, int NS>
__device__ __forceinline__ void unit_prologue(const StepParams& p, int u, float* s_q, float* s_k,
                                              Misc& m, int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  const int b = u / p.kv_heads, j = u - b * p.kv_heads;
  const T* qg = reinterpret_cast<const T*>(p.q) + ((size_t)b * p.kv_heads * G + (size_t)j * G) * D;
  const T* kg = reinterpret_cast<const T*>(p.k) + (size_t)u * D;
  for (int i = tid; i < G * D; i += kThreads) s_q[i] = to_f32(qg[i]);
  for (int i = tid; i < D; i += kThreads) s_k[i] = to_f32(kg[i]);
  __syncthreads();
  // the new token's logits (base 2): warp g handles query head g
  if (warp < G) {
    float a = 0.0f;
    for (int d = lane; d < D; d += 32) a = fmaf(s_q[warp * D + d], s_k[d], a);
    a = warp_sum(a);
    if (lane == 0) m.lnew[warp] = a * p.qscale;
  }
  code_queries_and_key<T, D, G>(s_q, s_k, reinterpret_cast<const T*>(p.W), p.bits,
                                p.append_slot < 0, m, tid);
}

// The last CTA of unit u merges the unit's partials (records of CTAs
// first .. first+n-1, stored at index cta + u), adds back the non-winning
// candidates and the new token, writes the output and overwrites the slot.
template <typename T, int D, int G, int NS>
__device__ void combine_unit(const StepParams& p, int u, int first, int n, Misc& m, int tid) {
  using S = StepShape<T, D, G, NS>;
  const int lane = tid & 31, warp = tid >> 5;
  const bool full = p.append_slot < 0;
  const float* recs = p.partials + (size_t)(first + u) * S::REC;

  // global eviction choice: the largest local key
  if (full) {
    uint64_t best = 0;
    for (int c = tid; c < n; c += kThreads) {
      const float* r = recs + (size_t)c * S::REC;
      const int slot = __float_as_int(__ldcg(r + 3 * G));
      const int dist = __float_as_int(__ldcg(r + 3 * G + 1));
      if (slot >= 0) {
        const uint64_t key = evict_key((uint32_t)dist, (uint32_t)slot);
        best = key > best ? key : best;
      }
    }
    best = warp_max_u64(best);
    if (lane == 0) m.red64[warp] = best;
    __syncthreads();
    if (tid == 0) {
      uint64_t b2 = 0;
      for (int w2 = 0; w2 < kWarps; ++w2) b2 = m.red64[w2] > b2 ? m.red64[w2] : b2;
      m.winner = (int)evict_key_slot(b2);
    }
  } else if (tid == 0) {
    m.winner = p.append_slot;
  }
  __syncthreads();
  const int winner = m.winner;
  if (winner < 0 || winner >= p.budget) {  // cannot happen for a non-empty unit; never write
    if (tid == 0) {
      atomicExch(p.err, 2);
      p.counters[u] = 0;
    }
    return;
  }

  // per-head max and sum over partials, surviving candidates and the new token
  if (warp < G) {
    const int g = warp;
    float mx = m.lnew[g];
    for (int c = lane; c < n; c += 32) {
      const float* r = recs + (size_t)c * S::REC;
      mx = fmaxf(mx, __ldcg(r + g));
      const int slot = __float_as_int(__ldcg(r + 3 * G));
      if (full && slot >= 0 && slot != winner) mx = fmaxf(mx, __ldcg(r + 2 * G + g));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    float sum = 0.0f;
    for (int c = lane; c < n; c += 32) {
      const float* r = recs + (size_t)c * S::REC;
      sum += __ldcg(r + G + g) * exp2f(__ldcg(r + g) - mx);
      const int slot = __float_as_int(__ldcg(r + 3 * G));
      if (full && slot >= 0 && slot != winner) sum += exp2f(__ldcg(r + 2 * G + g) - mx);
    }
    sum = warp_sum(sum);
    if (lane == 0) {
      m.hm[g] = mx;
      m.hl[g] = sum + exp2f(m.lnew[g] - mx);
    }
  }
  __syncthreads();

  const int b = u / p.kv_heads, j = u - b * p.kv_heads;
  const T* Vc = reinterpret_cast<const T*>(p.V) + (size_t)u * p.budget * D;
  const T* vt = reinterpret_cast<const T*>(p.v) + (size_t)u * D;
  for (int idx = tid; idx < G * D; idx += kThreads) {
    const int g = idx / D, d = idx - g * D;
    const float mx = m.hm[g];
    float a = 0.0f;
    for (int c = 0; c < n; ++c) {
      const float* r = recs + (size_t)c * S::REC;
      a += __ldcg(r + S::HDR + idx) * exp2f(__ldcg(r + g) - mx);
      const int slot = __float_as_int(__ldcg(r + 3 * G));
      if (full && slot >= 0 && slot != winner)
        a += exp2f(__ldcg(r + 2 * G + g) - mx) * to_f32(Vc[(size_t)slot * D + d]);
    }
    a += exp2f(m.lnew[g] - mx) * to_f32(vt[d]);
    p.out[((size_t)b * p.kv_heads * G + (size_t)j * G + g) * D + d] = a / m.hl[g];
  }

  // method step 5: the current token's key, value and code replace the slot
  T* Kw = reinterpret_cast<T*>(p.K) + ((size_t)u * p.budget + winner) * D;
  T* Vw = reinterpret_cast<T*>(p.V) + ((size_t)u * p.budget + winner) * D;
  const T* kt = reinterpret_cast<const T*>(p.k) + (size_t)u * D;
  for (int d = tid; d < D; d += kThreads) {
    Kw[d] = kt[d];
    Vw[d] = vt[d];
  }
  if (tid == 0) {
    store_code(p.codes + (size_t)u * p.code_stride + (size_t)winner * (p.bits >> 3), p.bits,
               m.codek);
    p.evicted[u] = full ? winner : -1;
    p.counters[u] = 0;
  }
}

template <typename T, int D, int G, int NS>
__global__ void __launch_bounds__(kThreads, (G <= 4 ? 2 : 1)) step_kernel(const StepParams p) {
  using S = StepShape<T, D, G, NS>;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* stage = smem + S::OFF_STAGE;
  float* wacc = reinterpret_cast<float*>(smem + S::OFF_WACC);
  float* s_q = reinterpret_cast<float*>(smem + S::OFF_Q);
  float* s_k = reinterpret_cast<float*>(smem + S::OFF_K);
  float* lgbuf = reinterpret_cast<float*>(smem + S::OFF_LG);
  float* pw = reinterpret_cast<float*>(smem + S::OFF_PW);
  float* wm = reinterpret_cast<float*>(smem + S::OFF_WM);
  float* wl = wm + kWarps * G;
  Misc& m = *reinterpret_cast<Misc*>(smem + S::OFF_MISC);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::OFF_BAR);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool full = p.append_slot < 0;

  if (p.total_tiles == 0) {  // empty cache: the new token alone
    if ((int)blockIdx.x < p.U) {
      unit_prologue<T, D, G, NS>(p, blockIdx.x, s_q, s_k, m, tid);
      combine_unit<T, D, G, NS>(p, blockIdx.x, 0, 0, m, tid);
    }
    return;
  }

  const int64_t TT = p.total_tiles, NC = gridDim.x;
  const int tb = (int)((int64_t)blockIdx.x * TT / NC);
  const int te = (int)(((int64_t)blockIdx.x + 1) * TT / NC);
  const int ntiles = te - tb;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncthreads();

  auto issue = [&](int i) {  // producer: CTA-local tile i -> stage i % NS
    const int t = tb + i;
    const int u = t / p.tpu;
    const int slot0 = (t - u * p.tpu) * kTile;
    const int rows = min(kTile, p.occ - slot0);
    const uint32_t bytes = (uint32_t)rows * S::ROWB;
    unsigned char* dst = stage + (i % NS) * 2 * S::TILEB;
    const size_t off = ((size_t)u * p.budget + slot0) * S::ROWB;
    mbar_arrive_expect_tx(&bars[i % NS], 2u * bytes);
    bulk_g2s(dst, reinterpret_cast<const unsigned char*>(p.K) + off, bytes, &bars[i % NS]);
    bulk_g2s(dst + S::TILEB, reinterpret_cast<const unsigned char*>(p.V) + off, bytes,
             &bars[i % NS]);
  };
  if (tid == 0)
    for (int i = 0; i < NS && i < ntiles; ++i) issue(i);

  const int lps_k = tid % S::LPS;  // lane within the slot group (logit phase)
  int i = 0;                       // CTA-local tile counter
  const int u_first = tb / p.tpu, u_last = (te - 1) / p.tpu;
  for (int u = u_first; u <= u_last; ++u) {
    const int seg_t0 = max(tb, u * p.tpu), seg_t1 = min(te, (u + 1) * p.tpu);
    const int lo = (seg_t0 - u * p.tpu) * kTile;
    const int hi = min((seg_t1 - u * p.tpu) * kTile, p.occ);

    // (a) codes, new-token logits
    unit_prologue<T, D, G, NS>(p, u, s_q, s_k, m, tid);

    // (b) local eviction candidate
    int cand = -1;
    if (full) {
      uint64_t cq[G];
#pragma unroll
      for (int g = 0; g < G; ++g) cq[g] = m.cq[g];
      uint64_t best = scan_codes<G>(p.codes + (size_t)u * p.code_stride, p.bits, lo, hi, cq, tid,
                                    kThreads, nullptr);
      best = warp_max_u64(best);
      if (lane == 0) m.red64[warp] = best;
      __syncthreads();
      if (tid == 0) {
        uint64_t b2 = 0;
        for (int w2 = 0; w2 < kWarps; ++w2) b2 = m.red64[w2] > b2 ? m.red64[w2] : b2;
        m.cand_slot = (int)evict_key_slot(b2);
        m.cand_dist = (int)evict_key_dist(b2);
#pragma unroll
        for (int g = 0; g < G; ++g) m.candlog[g] = -INFINITY;
      }
      __syncthreads();
      cand = m.cand_slot;
    }

    // (c) attention over the segment's tiles
    float qr[G][S::EPL];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int c = 0; c < S::CPL; ++c)
#pragma unroll
        for (int e = 0; e < S::EPC; ++e)
          qr[g][c * S::EPC + e] = s_q[g * D + (lps_k + S::LPS * c) * S::EPC + e] * p.qscale;

    float mrun[G], lrun[G], acc[G][S::EPW];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      mrun[g] = -1e30f;
      lrun[g] = 0.0f;
#pragma unroll
      for (int e = 0; e < S::EPW; ++e) acc[g][e] = 0.0f;
    }

    for (int lt = seg_t0 - u * p.tpu; lt < seg_t1 - u * p.tpu; ++lt, ++i) {
      const int st = i % NS;
      const bool ok = mbar_wait_bounded(&bars[st], (uint32_t)((i / NS) & 1));
      const unsigned char* Kt = stage + st * 2 * S::TILEB;
      const unsigned char* Vt = Kt + S::TILEB;
      const int slot_base = lt * kTile;
      float* lg = lgbuf + (i & 1) * kTile * G;

      // logits: LPS lanes per slot, transpose-reduce of the G partial dots
#pragma unroll
      for (int pass = 0; pass < S::NPASS; ++pass) {
        const int sl = pass * (kThreads / S::LPS) + tid / S::LPS;
        float v[G];
#pragma unroll
        for (int g = 0; g < G; ++g) v[g] = 0.0f;
#pragma unroll
        for (int c = 0; c < S::CPL; ++c) {
          const uint4 ch =
              *reinterpret_cast<const uint4*>(Kt + sl * S::ROWB + (lps_k + S::LPS * c) * 16);
          float x[S::EPC];
          chunk_to_f32<T>(ch, x);
#pragma unroll
          for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < S::EPC; ++e) v[g] = fmaf(qr[g][c * S::EPC + e], x[e], v[g]);
        }
        // reduce-scatter over the slot's lanes: lane keeps one head's sum
#pragma unroll
        for (int nn = G, o = 1; nn > 1; nn >>= 1, o <<= 1) {
          const bool upper = (lane & o) != 0;
#pragma unroll
          for (int i2 = 0; i2 < nn / 2; ++i2) {
            const float send = upper ? v[i2] : v[i2 + nn / 2];
            const float keep = upper ? v[i2 + nn / 2] : v[i2];
            v[i2] = keep + __shfl_xor_sync(kFull, send, o);
          }
        }
#pragma unroll
        for (int o = G; o < S::LPS; o <<= 1) v[0] += __shfl_xor_sync(kFull, v[0], o);
        if (lps_k < G) {
          int h = 0;
#pragma unroll
          for (int l2 = 0, w2 = G >> 1; w2 > 0; ++l2, w2 >>= 1) h += ((lps_k >> l2) & 1) * w2;
          const int slot = slot_base + sl;
          float val = v[0];
          if (slot >= hi) {
            val = -INFINITY;
          } else if (slot == cand) {
            m.candlog[h] = val;
            val = -INFINITY;
          }
          lg[sl * G + h] = val;
        }
      }
      if (!__syncthreads_and(ok)) {
        // a TMA wait gave up: record it, let the copies in flight land, leave
        if (tid == 0) {
          atomicExch(p.err, 1);
          const int issued = min(ntiles, NS + max(0, i - 1));
          for (int r = i; r < issued; ++r)
            (void)mbar_wait_bounded(&bars[r % NS], (uint32_t)((r / NS) & 1), 500000000ull);
        }
        return;
      }
      // stage of tile i-1 is free: every warp is past its value phase
      if (tid == 0 && i >= 1 && i - 1 + NS < ntiles) issue(i - 1 + NS);

      // value phase: warp w owns slots w, w + 8, ... of the tile
      float x = -INFINITY;
      if (lane < S::SPW * G) x = lg[(warp + kWarps * (lane / G)) * G + (lane % G)];
      float tmax = x;
#pragma unroll
      for (int o = G; o < S::SPW * G; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, o));
      float mnew[G], sc[G];
      float mymax = 0.0f;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        mnew[g] = fmaxf(mrun[g], __shfl_sync(kFull, tmax, g));
        sc[g] = exp2f(mrun[g] - mnew[g]);
        if ((lane % G) == g) mymax = mnew[g];
      }
      const float pr = (lane < S::SPW * G) ? exp2f(x - mymax) : 0.0f;
      float* pwarp = pw + warp * S::SPW * G;
      if (lane < S::SPW * G) pwarp[lane] = pr;
      float ps = pr;
#pragma unroll
      for (int o = G; o < S::SPW * G; o <<= 1) ps += __shfl_xor_sync(kFull, ps, o);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        lrun[g] = lrun[g] * sc[g] + __shfl_sync(kFull, ps, g);
        mrun[g] = mnew[g];
#pragma unroll
        for (int e = 0; e < S::EPW; ++e) acc[g][e] *= sc[g];
      }
      __syncwarp();
#pragma unroll
      for (int ii = 0; ii < S::SPW; ++ii) {
        const int sl = warp + kWarps * ii;
        if (slot_base + sl < hi) {
          float vx[S::EPW];
          load_row_part<T, S::EPW>(Vt + sl * S::ROWB + lane * S::EPW * S::EB, vx);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float pg = pwarp[ii * G + g];
#pragma unroll
            for (int e = 0; e < S::EPW; ++e) acc[g][e] = fmaf(pg, vx[e], acc[g][e]);
          }
        }
      }
    }

    // (d) merge the warps' states into this CTA's partial for unit u
    if (lane == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        wm[warp * G + g] = mrun[g];
        wl[warp * G + g] = lrun[g];
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < S::EPW; ++e) wacc[(warp * G + g) * D + lane * S::EPW + e] = acc[g][e];
    __syncthreads();
    float* rec = p.partials + (size_t)(blockIdx.x + u) * S::REC;
    for (int idx = tid; idx < G * D; idx += kThreads) {
      const int g = idx / D;
      float mx = -1e30f;
#pragma unroll
      for (int w2 = 0; w2 < kWarps; ++w2) mx = fmaxf(mx, wm[w2 * G + g]);
      float a = 0.0f;
#pragma unroll
      for (int w2 = 0; w2 < kWarps; ++w2) a += wacc[(w2 * G + g) * D + (idx - g * D)] * exp2f(wm[w2 * G + g] - mx);
      __stcg(rec + S::HDR + idx, a);
    }
    if (tid < G) {
      const int g = tid;
      float mx = -1e30f, sum = 0.0f;
      for (int w2 = 0; w2 < kWarps; ++w2) mx = fmaxf(mx, wm[w2 * G + g]);
      for (int w2 = 0; w2 < kWarps; ++w2) sum += wl[w2 * G + g] * exp2f(wm[w2 * G + g] - mx);
      __stcg(rec + g, mx);
      __stcg(rec + G + g, sum);
      __stcg(rec + 2 * G + g, full ? m.candlog[g] : -INFINITY);
    }
    if (tid == 0) {
      __stcg(rec + 3 * G, __int_as_float(cand));
      __stcg(rec + 3 * G + 1, __int_as_float(full ? m.cand_dist : 0));
    }
    __threadfence();
    __syncthreads();
    // owner of tile t: the CTA c with floor(c*TT/NC) <= t < floor((c+1)*TT/NC),
    // i.e. c = ((t + 1) * NC - 1) / TT
    const int first = (int)((((int64_t)u * p.tpu + 1) * NC - 1) / TT);
    const int last = (int)((((int64_t)u * p.tpu + p.tpu) * NC - 1) / TT);
    if (tid == 0) {
      const int prev = atomicAdd(&p.counters[u], 1);
      m.is_last = (prev == last - first);
    }
    __syncthreads();
    if (m.is_last) {
      __threadfence();
      combine_unit<T, D, G, NS>(p, u, first, last - first + 1, m, tid);
    }
    __syncthreads();
  }
}

// Codes of rows of x (method steps 1-2).  Row r (r < rows) is vector
// (r / per_unit, r % per_unit) at x + ((r / per_unit) * x_unit_rows + r % per_unit) * D;
// its code goes to out + (r / per_unit) * out_unit_bytes + (r % per_unit) * bits/8.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) code_kernel(const T* __restrict__ x, int64_t rows,
                                                        int64_t per_unit, int64_t x_unit_rows,
                                                        const T* __restrict__ W, int bits,
                                                        unsigned char* out,
                                                        int64_t out_unit_bytes) {
  __shared__ float xs[kThreads / 8][D];  // up to 32 vectors (bits = 8)
  __shared__ uint32_t sbits[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int vb = kThreads / bits;  // vectors per block pass
  for (int64_t r0 = (int64_t)blockIdx.x * vb; r0 < rows; r0 += (int64_t)gridDim.x * vb) {
    for (int i = tid; i < vb * D; i += kThreads) {
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
    const uint32_t bit = (r0 + vi < rows) ? projection_bit<T, D>(xs[vi], W, bits, j) : 0u;
    const uint32_t word = __ballot_sync(kFull, bit);
    if (lane == 0) sbits[warp] = word;
    __syncthreads();
    if (tid < vb && r0 + tid < rows) {
      const int64_t r = r0 + tid;
      const int64_t unit = r / per_unit, s = r - unit * per_unit;
      store_code(out + unit * out_unit_bytes + s * (bits >> 3), bits,
                 code_from_bits(sbits, bits, tid));
    }
    __syncthreads();
  }
}

// Group-summed distances of every resident slot to the step's query codes
// (method step 3), one CTA per unit; slots occ..budget-1 get 0.
template <typename T, int D, int G>
__global__ void __launch_bounds__(kThreads) score_kernel(const StepParams p, int32_t* dist) {
  __shared__ float s_q[G * D];
  __shared__ float s_k[D];
  __shared__ Misc m;
  const int tid = threadIdx.x;
  const int u = blockIdx.x;
  const int b = u / p.kv_heads, j = u - b * p.kv_heads;
  const T* qg = reinterpret_cast<const T*>(p.q) + ((size_t)b * p.kv_heads * G + (size_t)j * G) * D;
  for (int i = tid; i < G * D; i += kThreads) s_q[i] = to_f32(qg[i]);
  for (int i = tid; i < D; i += kThreads) s_k[i] = 0.0f;
  __syncthreads();
  code_queries_and_key<T, D, G>(s_q, s_k, reinterpret_cast<const T*>(p.W), p.bits, true, m, tid);
  uint64_t cq[G];
#pragma unroll
  for (int g = 0; g < G; ++g) cq[g] = m.cq[g];
  int32_t* drow = dist + (size_t)u * p.budget;
  for (int s = p.occ + tid; s < p.budget; s += kThreads) drow[s] = 0;
  if (p.occ > 0)
    (void)scan_codes<G>(p.codes + (size_t)u * p.code_stride, p.bits, 0, p.occ, cq, tid, kThreads,
                        drow);
}

// The projection matrix W[d][j] drawn from the seed: SplitMix64 finaliser over a
// counter (Steele, Lea, Flood 2014), Irwin-Hall sum of twelve 16-bit uniforms.
__device__ __forceinline__ uint64_t splitmix_finalise(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void projection_kernel(uint64_t seed, int D, int bits, int is_fp32, void* W) {
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
