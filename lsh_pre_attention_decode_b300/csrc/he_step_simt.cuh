// he_step_simt.cuh — CUDA-core engine of the fused HashEvict step (used for
// fp32 caches): the logits and the value accumulation run as fp32 FMAs on the
// CUDA cores.  Tiles of 32 slots; per tile, 8 lanes per slot form the dot
// products (transpose-reduced over the lanes), then each warp keeps its own
// online-softmax state over 4 slots of the tile.  K/V tiles arrive by 1-D TMA
// bulk copies into an NS-stage mbarrier ring.  Shared pieces: he_common.cuh.
#pragma once

#include "he_common.cuh"

namespace he {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = 32;  // cache slots per tile

template <typename T, int D, int G, int NS>
struct SimtShape {
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
  // shared memory carve-up (bytes; every offset a multiple of 16)
  static constexpr int OFF_STAGE = 0;
  static constexpr int OFF_WACC = OFF_STAGE + NS * 2 * TILEB;
  static constexpr int OFF_Q = OFF_WACC + kWarps * G * D * 4;
  static constexpr int OFF_K = OFF_Q + G * D * 4;
  static constexpr int OFF_LG = OFF_K + D * 4;
  static constexpr int OFF_PW = OFF_LG + 2 * kTile * G * 4;
  static constexpr int OFF_WM = OFF_PW + kWarps * SPW * G * 4;
  static constexpr int OFF_MISC = OFF_WM + 2 * kWarps * G * 4;
  static constexpr int MISC = kMiscBytes;
  static constexpr int OFF_BAR = OFF_MISC + MISC;
  static constexpr int SMEM = OFF_BAR + NS * 8;
  static_assert(D % 64 == 0 && (G & (G - 1)) == 0 && G <= 8, "shape");
  static_assert(CPL >= 1 && NPASS >= 1 && G <= LPS, "logit lane mapping");
  static_assert(SPW * G <= 32, "value-phase softmax lanes");
};

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

template <typename T, int D, int G, int NS>
__global__ void __launch_bounds__(kThreads, (G <= 4 ? 2 : 1)) step_kernel_simt(const StepParams p) {
  using S = SimtShape<T, D, G, NS>;
  using R = Record<G, D>;
  extern __shared__ __align__(128) unsigned char smem_simt[];
  unsigned char* smem = smem_simt;
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
      unit_prologue<T, D, G, kThreads, 0>(p, blockIdx.x, s_q, s_k, m, tid);
      combine_unit<T, D, G, kThreads, 0>(p, blockIdx.x, 0, 0, m, tid, wacc,
                                         kWarps * G * D / (3 * G + 1));
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
    unit_prologue<T, D, G, kThreads, 0>(p, u, s_q, s_k, m, tid);

    // (b) local eviction candidate
    int cand = -1;
    if (full) {
      local_candidate<G, kThreads, 0>(p, u, lo, hi, m, tid);
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
    write_partial<G, D, kThreads>(p.partials + (size_t)(blockIdx.x + u) * R::FLOATS, wm, wl, wacc,
                                  kWarps, m, cand, full, tid);
    finish_segment<T, D, G, kThreads, 0>(p, u, m, tid, wacc, kWarps * G * D / (3 * G + 1));
  }
}

}  // namespace he
