// Histogram-guided exact Top-k pieces for one-query CTAs.
//
// A packed candidate word (topk.cuh) has the score's order-preserving 32-bit code in its high
// half. Its bin is the top 12 bits of that code: the sign, the 8 exponent bits and the top 3
// mantissa bits, so a bin spans 1/8 of an octave on either side of zero. Bins are monotone in
// the word: a larger word never has a smaller bin. Counting words per bin therefore answers
// "how many words are >= the lowest word of bin b" exactly, which is what lets a selection cut
// be raised without ever ordering words.
#pragma once
#include <cstdint>

#include "topk.cuh"

namespace ds4 {

constexpr int kHBins = 4096;

__device__ __forceinline__ uint32_t hbin(uint64_t u) { return static_cast<uint32_t>(u >> 52); }

// The lowest score whose word reaches bin b: the float whose order-preserving code is b << 20.
// Bins below 8 hold no finite score (their codes are NaN patterns and -inf): -inf for them, so
// a threshold test keeps a superset, never fewer keys, than the bin test.
__device__ __forceinline__ float bin_floor_score(uint32_t b) {
  if (b <= 8u) return -__int_as_float(0x7f800000);
  const uint32_t code = b << 20;
  return __uint_as_float((code & 0x80000000u) ? (code & 0x7FFFFFFFu) : ~code);
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

// One warp: the highest bin b in [lo, hi] whose count summed over bins >= b reaches K.
// *count receives that sum. When no bin reaches K, returns lo with the total over [lo, hi].
// Lane l first sums its slice of the range (slices of ceil(range / 32) bins, the highest slice
// on lane 0); a prefix over the lanes locates the slice that holds the cut, which the warp then
// scans 32 bins at a time. Counters may grow while the scan runs: every value read is then a
// lower bound, so a returned bin still has at least *count words at or above it.
template <int K, class Get>
__device__ __forceinline__ uint32_t warp_find_cut(const Get get, uint32_t lo, uint32_t hi,
                                                  uint32_t* count, int lane) {
  const int range = static_cast<int>(hi) - static_cast<int>(lo) + 1;
  const int per = (range + 31) / 32;
  const int ltop = static_cast<int>(hi) - lane * per;
  uint32_t s = 0u;
#pragma unroll 4
  for (int i = 0; i < per; ++i) {
    const int bin = ltop - i;
    if (bin >= static_cast<int>(lo)) s += get(static_cast<uint32_t>(bin));
  }
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {  // inclusive prefix over lanes, highest slice first
    const uint32_t v = __shfl_up_sync(0xffffffffu, s, off);
    if (lane >= off) s += v;
  }
  const uint32_t before = __shfl_up_sync(0xffffffffu, s, 1);
  const uint32_t hit = __ballot_sync(0xffffffffu, s >= static_cast<uint32_t>(K));
  if (!hit) {
    *count = __shfl_sync(0xffffffffu, s, 31);
    return lo;
  }
  const int ls = __ffs(hit) - 1;
  uint32_t acc = __shfl_sync(0xffffffffu, lane == 0 ? 0u : before, ls);
  const int top0 = static_cast<int>(hi) - ls * per;
  const int bottom = top0 - per + 1 > static_cast<int>(lo) ? top0 - per + 1 : static_cast<int>(lo);
  for (int top = top0; top >= bottom; top -= 32) {
    const int bin = top - lane;
    uint32_t c = bin >= bottom ? get(static_cast<uint32_t>(bin)) : 0u;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, c, off);
      if (lane >= off) c += v;
    }
    const uint32_t h = __ballot_sync(0xffffffffu, acc + c >= static_cast<uint32_t>(K));
    if (h) {
      const int l = __ffs(h) - 1;
      *count = acc + __shfl_sync(0xffffffffu, c, l);
      return static_cast<uint32_t>(top - l);
    }
    acc += __shfl_sync(0xffffffffu, c, 31);
  }
  // Not reached: the slice holds the cut. Counters that grew meanwhile can only move it up.
  *count = acc;
  return static_cast<uint32_t>(bottom);
}

// The same search over 16-bit bin counters with 32-bin group counters beside them (grp[g]
// counts the words of bins 32g..32g+31): the groups above lo's group locate the cut's group,
// whose bins are then read one by one, so the cost does not grow with the range. Groups are
// only trusted above lo's group (their bins are all >= lo); lo's own group is read bin by bin.
__device__ __forceinline__ uint32_t warp_find_cut_grouped(uint32_t K, const uint32_t* bins16,
                                                          const uint32_t* grp, uint32_t lo,
                                                          uint32_t hi, uint32_t* count, int lane) {
  const int glo = static_cast<int>(lo >> 5), ghi = static_cast<int>(hi >> 5);
  uint32_t acc = 0u;
  int found = glo;
  for (int top = ghi; top > glo; top -= 32) {
    const int g = top - lane;
    uint32_t s = g > glo ? grp[g] : 0u;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += v;
    }
    const uint32_t before = __shfl_up_sync(0xffffffffu, s, 1);
    const uint32_t hit = __ballot_sync(0xffffffffu, acc + s >= K);
    if (hit) {
      const int l = __ffs(hit) - 1;
      acc += __shfl_sync(0xffffffffu, lane == 0 ? 0u : before, l);
      found = top - l;
      break;
    }
    acc += __shfl_sync(0xffffffffu, s, 31);
  }
  const int btop = found * 32 + 31 < static_cast<int>(hi) ? found * 32 + 31 : static_cast<int>(hi);
  const int bbot = found * 32 > static_cast<int>(lo) ? found * 32 : static_cast<int>(lo);
  const int bin = btop - lane;
  uint32_t s = bin >= bbot ? Hist16{bins16}(static_cast<uint32_t>(bin)) : 0u;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, s, off);
    if (lane >= off) s += v;
  }
  const uint32_t hit = __ballot_sync(0xffffffffu, acc + s >= K);
  if (hit) {
    const int l = __ffs(hit) - 1;
    *count = acc + __shfl_sync(0xffffffffu, s, l);
    return static_cast<uint32_t>(btop - l);
  }
  // No bin reached K (only possible in lo's group): the total at or above bbot.
  *count = acc + __shfl_sync(0xffffffffu, s, 31);
  return static_cast<uint32_t>(bbot);
}

}  // namespace ds4
