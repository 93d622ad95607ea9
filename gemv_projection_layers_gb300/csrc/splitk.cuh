// splitk.cuh -- fixed-order split-K combination shared by the tensor-core and
// router kernels.
//
// The CTAs cut the linear order of (tile, k-block) units into G equal
// ranges (part_begin).  A tile whose k-blocks fall into several ranges is
// "split"; its contributors are the CTAs c_first .. c_last in increasing
// order, which is also increasing k.  Two ways to finish a split tile, both
// deterministic (the summation order depends only on the partition):
//
// * owner mode: c_first covers the tile's first k-blocks, and for c_first
//   that range is always its LAST segment, while every other contributor
//   covers its part as its FIRST segment.  The others write fp32 partials
//   early and bump the tile counter; the owner waits (bounded) for S - 1
//   arrivals, sums their partials in CTA order while its own last segment is
//   still streaming, and finishes with own + others.  It then zeroes the
//   counter.  One partial slot per CTA.
// * distributed mode: every contributor writes its partial and bumps the
//   counter; after its main loop each waits for all S, reduces 1/S of the
//   tile's outputs in CTA order, and bumps the counter again; the S-th of
//   those second arrivals zeroes it.  Two partial slots per CTA (first and
//   last segment).
//
// Both wait on other CTAs, so every CTA of the grid must be resident at once:
// the kernels are launched cooperatively with at most one CTA per SM.  Waits
// are bounded and report kStatusTimeoutSplitK in the status word.
#pragma once

#include "kernels.h"
#include "ptx.cuh"

namespace proj {

enum : uint32_t { kStatusTimeoutSplitK = 1u << 7 };

// Spin (bounded) until *p >= target.
__device__ __forceinline__ bool spin_until_ge(const uint32_t* p, uint32_t target,
                                              uint32_t* status) {
  if (ld_acquire_gpu(p) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    __nanosleep(64);
    if (ld_acquire_gpu(p) >= target) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(status, kStatusTimeoutSplitK);
      return false;
    }
  }
}

struct TileSplit {
  int64_t c_first, c_last;
};

__device__ __forceinline__ TileSplit tile_split(int tile, int KB, int64_t U, int64_t G) {
  const int64_t tu0 = static_cast<int64_t>(tile) * KB;
  return {part_owner(tu0, U, G), part_owner(tu0 + KB - 1, U, G)};
}

// Distributed mode: slot of contributor c for `tile` (0 = its first segment).
__device__ __forceinline__ int64_t dist_slot(int64_t c, int tile, int KB, int64_t U, int64_t G) {
  return 2 * c + ((part_begin(c, U, G) / KB) == tile ? 0 : 1);
}

}  // namespace proj
