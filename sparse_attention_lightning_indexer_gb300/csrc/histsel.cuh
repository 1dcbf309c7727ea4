// Histogram-guided exact Top-k pieces for one-query CTAs.
//
// A packed candidate word (topk.cuh) has the score's order-preserving code in its high half. Its
// bin is that code's 12 bits below the sign for non-negative scores (8 exponent bits and the top
// 4 mantissa bits, so a bin spans 1/16 of an octave) and 0 for negative scores. Bins are
// monotone in the word: a larger word never has a smaller bin. Counting words per bin therefore
// answers "how many words are >= the lowest word of bin b" exactly, which is what lets a
// selection cut be raised without ever ordering words.
#pragma once
#include <cstdint>

#include "topk.cuh"

namespace ds4 {

constexpr int kHBins = 4096;

__device__ __forceinline__ uint32_t hbin(uint64_t u) {
  const uint32_t hi = static_cast<uint32_t>(u >> 32);
  return hi >= 0x80000000u ? (hi - 0x80000000u) >> 19 : 0u;
}

// 16-bit counters packed two per 32-bit word (a CTA counts at most a few ten thousand words).
__device__ __forceinline__ void hist16_inc(uint32_t* h, uint32_t bin) {
  atomicAdd(&h[bin >> 1], 1u << ((bin & 1u) << 4));
}
struct Hist16 {
  const uint32_t* h;
  __device__ __forceinline__ uint32_t operator()(uint32_t bin) const {
    return (h[bin >> 1] >> ((bin & 1u) << 4)) & 0xFFFFu;
  }
};
struct Hist32 {
  const uint32_t* h;
  __device__ __forceinline__ uint32_t operator()(uint32_t bin) const { return h[bin]; }
};

// One warp: the highest bin b in [lo, hi] whose count summed over bins >= b reaches K, scanning
// down from hi 32 bins at a time. *count receives that sum. When no bin reaches K, returns lo
// with the total over [lo, hi]. Counters may grow while the scan runs: every value read is then
// a lower bound, so a returned bin still has at least *count words at or above it.
template <int K, class Get>
__device__ __forceinline__ uint32_t warp_find_cut(const Get get, uint32_t lo, uint32_t hi,
                                                  uint32_t* count, int lane) {
  uint32_t acc = 0u;
  for (int top = static_cast<int>(hi); top >= static_cast<int>(lo); top -= 32) {
    const int bin = top - lane;
    uint32_t s = bin >= static_cast<int>(lo) ? get(static_cast<uint32_t>(bin)) : 0u;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {  // inclusive prefix over lanes, highest bin first
      const uint32_t v = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += v;
    }
    const uint32_t hit = __ballot_sync(0xffffffffu, acc + s >= static_cast<uint32_t>(K));
    if (hit) {
      const int l = __ffs(hit) - 1;
      *count = acc + __shfl_sync(0xffffffffu, s, l);
      return static_cast<uint32_t>(top - l);
    }
    acc += __shfl_sync(0xffffffffu, s, 31);
  }
  *count = acc;
  return lo;
}

}  // namespace ds4
