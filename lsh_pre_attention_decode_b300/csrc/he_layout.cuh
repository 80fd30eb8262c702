// he_layout.cuh — data layouts shared by the bf16 step kernels: the per-unit
// results handed between a step's kernels (and to the next step), the stream-K
// split of a step's tiles over the CTAs, and the partial-record layouts.
#pragma once

#include <stdint.h>

namespace he {

// Per-unit results of prep, read by merge.
struct UnitOut {
  // eviction key (distance << 32 | ~slot) of the steps of parity 0 and 1: a
  // step folds into key[kpar] while the next step's stream kernel may still
  // read key[kpar ^ 1] (the previous step's decision); merge zeroes key[kpar ^ 1]
  unsigned long long key[2];
  unsigned long long codek;
  float lnew[8];           // the new token's base-2 logits, per query head
  float lstar[8];          // the evicted slot's base-2 logits, per query head
  int32_t arrived;         // prep CTAs (fused step: stream CTAs) of the unit done,
                           // reset by the last one
  int32_t hcnt[2];         // fused step: hash warps of the unit done, per key parity
  int32_t pad;
  uint16_t vstar[128];     // the evicted slot's value row (bf16)
  uint8_t vqstar[128];     // quantised value cache: the evicted slot's byte row ...
  float vsstar;            // ... and its scale
  uint8_t vqnew[128];      // quantised value cache: the new token's byte row ...
  float vsnew;             // ... and its scale (prep quantises, merge writes them)
  int32_t cready[2];       // fused step: cq[parity] published (1), reset by the unit's merge
  int32_t pad2;
  unsigned long long cq[2][8];  // fused step: the query codes, per key parity
};

// Chunk eviction: what merge needs to take the evicted chunk out of the
// attention, per unit.  The chunk's slots fall in at most two 64-slot tiles
// (part 0: the tile of its first slot, part 1: the next one); per part and
// query head, the base-2 softmax state of the part's slots alone: max m, sum
// l = sum exp2(x - m), accumulator a[D] = sum exp2(x - m) v.  An empty part
// has m = -1e30, l = 0, a = 0.  Layout (floats): m [2][8], l [2][8], a [2][G][D].
constexpr int kMaxChunk = 16;
template <int G, int D>
struct ChunkRec {
  static constexpr int M = 0, L = 16, A = 32;
  static constexpr int FLOATS = A + 2 * G * D;
};

// Code slots a prep CTA scans per item: 16 KiB of codes at most (4096 slots
// of up to 32 bits, 2048 of 64).
__host__ __device__ __forceinline__ int prep_item_slots(int bits) {
  return bits == 64 ? 2048 : 4096;
}

// Slots per prep item with chunks of c slots: a multiple of c and of 16 (so
// that an item's codes start on a 16-byte boundary for the bulk copy).
__host__ __device__ __forceinline__ int chunk_item_slots(int c, int bits) {
  const int l = 16 * c / (c & -c);  // lcm(c, 16) for 1 <= c <= 16
  return prep_item_slots(bits) / l * l;
}

// Stream-K split of a step's TT tiles over NC stream CTAs, in two groups: the
// first E CTAs take tiles [0, T1) and the others [T1, TT), each group split
// evenly (CTA c of a group of n over T tiles: [c T / n, (c + 1) T / n)).  The
// host gives the first group more tiles when the others start later (they wait
// for SMs that the previous step's merge CTAs hold); E = T1 = 0 is the even
// split.  Every CTA holds at least one tile, so the CTAs holding a unit's
// tiles are consecutive and each writes a partial.
struct TileSplit {
  int64_t TT, NC, E, T1;
  __host__ __device__ int64_t begin(int64_t c) const {  // first tile of CTA c (c <= NC)
    if (c <= E) return E > 0 ? c * T1 / E : 0;
    return T1 + (c - E) * (TT - T1) / (NC - E);
  }
  __host__ __device__ int64_t owner(int64_t t) const {  // the CTA whose range holds tile t
    if (t < T1) return ((t + 1) * E - 1) / T1;
    return E + ((t - T1 + 1) * (NC - E) - 1) / (TT - T1);
  }
};

// Partial record of one (stream CTA, unit): [m G][l G] padded to 4, acc [G][D].
template <int G, int D>
struct PRec {
  static constexpr int HDR = (2 * G + 3) / 4 * 4;
  static constexpr int FLOATS = HDR + G * D;
};

// Partial record of the fused step, per (stream CTA, unit): the PRec fields,
// then the segment's eviction candidate (its key (distance << 32 | ~slot), its
// base-2 logits per query head and its value row as bf16 words).
template <int G, int D>
struct FRec {
  static constexpr int HDR = PRec<G, D>::HDR;
  static constexpr int KEY = HDR + G * D;          // u64 (two floats), 8-byte aligned
  static constexpr int LC = KEY + 2;               // [G]
  static constexpr int VR = (LC + G + 3) / 4 * 4;  // D bf16 = D / 2 words, 16-byte aligned
  static constexpr int FLOATS = VR + D / 2;
  static_assert(KEY % 4 == 0 && FLOATS % 4 == 0, "record alignment");
};

}  // namespace he
