// scales.cuh -- stores of one warp's group scales to every destination row
// of a token, in each scale layout (shared by the two dispatch kernels).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace moeperm {

// The warp's 32 lanes hold the 16-element chunks [group_base*GSZ/16, +32) of a
// row; lane l's group exponent is e (active lanes only) or, for the plain fp32
// format, its scale sval. Writes the scales of those groups to the rows
// rows[0..nslots) (negative = dropped), spreading the destinations over lanes.
// Every lane of the warp must call it.
template <int GSZ, int FMT>
__device__ __forceinline__ void store_scales(const ScatterArgs& p, int nslots, const int* rows,
                                             const int* exps, int lane, bool active, int e,
                                             float sval, int group_base, int G, int G4) {
  constexpr int GL = GSZ / 16;  // lanes per group
  constexpr int GPW = 32 / GL;  // groups per warp
  const uint32_t byte = active ? (uint32_t)(e + 127) : 0u;
  if constexpr (FMT == kFmtPacked) {
    static_assert(GSZ == 128, "packed layout is defined for groups of 128");
    const uint32_t word = __shfl_sync(0xffffffffu, byte, 0) |
                          (__shfl_sync(0xffffffffu, byte, 8) << 8) |
                          (__shfl_sync(0xffffffffu, byte, 16) << 16) |
                          (__shfl_sync(0xffffffffu, byte, 24) << 24);
    // the warp's word goes to every destination, one destination per lane
    if (__shfl_sync(0xffffffffu, (int)active, 0)) {
      const int64_t wofs = (int64_t)(group_base / 4) * p.ld_s;
      uint32_t* sc = reinterpret_cast<uint32_t*>(p.scales);
      for (int k = lane; k < nslots; k += 32) {
        const int row = rows[k];
        if (row < 0) continue;
        int64_t pk = row;  // compact / identity: one block
        if (p.mode == kModeMasked) {  // one block per expert (no division: the expert is kept)
          const int ex = exps[k];
          pk = (int64_t)ex * G4 * p.ld_s + (row - ex * p.cap);
        }
        sc[pk + wofs] = word;
      }
    }
  } else if constexpr (FMT == kFmtU8 || FMT == kFmtMX) {
    constexpr int WPW = GPW / 4;  // whole 4-group words per warp
    const int q = lane % WPW;
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) word |= __shfl_sync(0xffffffffu, byte, (4 * q + j) * GL) << (8 * j);
    const bool word_ok = (p.ld_s % 4) == 0;
    uint8_t* sc = reinterpret_cast<uint8_t*>(p.scales);
    // lane = (destination, word): word q of destination k on lane q + WPW * k
    if (word_ok && group_base + 4 * q + 3 < G) {
      for (int k = lane / WPW; k < nslots; k += 32 / WPW)
        if (rows[k] >= 0)
          *reinterpret_cast<uint32_t*>(sc + (int64_t)rows[k] * p.ld_s + group_base + 4 * q) = word;
    }
    // otherwise byte by byte, from the first lane of each group
    const int gidx = group_base + lane / GL;
    const bool by_word = word_ok && ((gidx / 4) * 4 + 3 < G);
    if (active && (lane % GL) == 0 && !by_word) {
      for (int k = 0; k < nslots; ++k)
        if (rows[k] >= 0) sc[(int64_t)rows[k] * p.ld_s + gidx] = (uint8_t)byte;
    }
  } else {  // fp32 scales: 2^e, or the plain amax / 448
    // lane = (destination, group): group q of destination k on lane q + GPW * k,
    // the value taken from the group's first lane
    const float mine = (FMT == kFmtF32) ? sval : __uint_as_float((uint32_t)(e + 127) << 23);
    const int q = lane % GPW;
    const float v = __shfl_sync(0xffffffffu, mine, q * GL);
    const bool q_active = __shfl_sync(0xffffffffu, (int)active, q * GL) != 0;
    if (q_active) {
      float* sc = reinterpret_cast<float*>(p.scales);
      for (int k = lane / GPW; k < nslots; k += 32 / GPW)
        if (rows[k] >= 0) sc[(int64_t)rows[k] * p.ld_s + group_base + q] = v;
    }
  }
}

}  // namespace moeperm
