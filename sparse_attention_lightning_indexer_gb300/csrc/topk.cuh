// Warp-level streaming Top-k building blocks.
//
// A candidate (score, key index) is packed into one 64-bit word whose unsigned order is the
// selection order: the high half is the score mapped to an order-preserving unsigned code, the
// low half is ~index, so among equal scores the lower index compares larger. Every packed word
// of a real candidate is non-zero, so 0 doubles as the "empty slot" sentinel below all of them.
// Selecting the k largest words is therefore exactly "k best scores, ties to the lower index"
// (the Top-512 rule of "DeepSeek V4 Flash 추론을 1.6초로 줄인 ds4 최적화", 섹션별 상세), with no
// tie left open.
//
// Streaming selection per query (one warp): an unsorted pool holds every candidate that beat
// the running threshold theta (the exact k-th best word seen so far, 0 before k words were
// seen). When the pool nears capacity, an exact radix select finds the k-th largest word,
// compacts the pool to exactly the k largest and raises theta to it. Only the final k words are
// ever sorted, once. The page replaced a bitonic sort plus a merge cascade with a streaming
// Top-512; here no sorting network ever runs on the stream itself. The CTA-wide selects and the
// CTA-wide sort below finish split lists and one-query CTAs.
#pragma once
#include <cstdint>

namespace ds4 {

__device__ __forceinline__ uint64_t pack_key(float score, uint32_t index) {
  uint32_t b = __float_as_uint(score);
  if (b == 0x80000000u) b = 0u;  // -0 and +0 are the same score
  const uint32_t o = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<uint64_t>(o) << 32) | static_cast<uint64_t>(~index);
}
__device__ __forceinline__ float key_score(uint64_t u) {
  const uint32_t o = static_cast<uint32_t>(u >> 32);
  const uint32_t b = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  return __uint_as_float(b);
}
__device__ __forceinline__ int32_t key_index(uint64_t u) {
  return static_cast<int32_t>(~static_cast<uint32_t>(u));
}

__device__ __forceinline__ uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }
__device__ __forceinline__ uint64_t umin64(uint64_t a, uint64_t b) { return a < b ? a : b; }

// Exact radix select over pool[0..n), n > K: afterwards pool[0..K) holds exactly the K largest
// words (unordered) and the K-th largest is returned. One warp; `hist` is 256 words of shared
// scratch owned by this warp. Digits of 8 bits from the top; a digit pass stops as soon as the
// bin holding the K-th word is kept whole, so typical score distributions need 2-4 passes and
// only exact score ties ever reach the index bits.
template <int K>
__device__ __noinline__ uint64_t select_compact(uint64_t* pool, int n, uint32_t* hist, int lane) {
  // Bits above the highest bit in which two pool words differ are common to all of them: the
  // first digit starts right below that, so no pass is spent on a digit every word shares.
  uint64_t diff = 0ull;
  const uint64_t first = pool[0];
  for (int i = lane; i < n; i += 32) diff |= pool[i] ^ first;
  const uint32_t dlo = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(diff));
  const uint32_t dhi = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(diff >> 32));
  const int top = dhi ? 63 - __clz(dhi) : (dlo ? 31 - __clz(dlo) : 0);  // highest differing bit
  int width = top + 1 < 8 ? top + 1 : 8;
  int shift = top + 1 - width;                   // current digit: bits [shift, shift + width)
  uint64_t prefix = shift + width >= 64 ? 0ull : (first & (~0ull << (shift + width)));
  uint32_t need = K;  // rank of the K-th word among words matching `prefix`
  for (;;) {
#pragma unroll
    for (int i = 0; i < 8; ++i) hist[lane * 8 + i] = 0u;
    __syncwarp();
    const uint64_t hi_mask = shift + width >= 64 ? 0ull : (~0ull << (shift + width));
    const uint32_t dmask = (1u << width) - 1u;
    for (int i = lane; i < n; i += 32) {
      const uint64_t u = pool[i];
      if ((u & hi_mask) == prefix) atomicAdd(&hist[static_cast<uint32_t>(u >> shift) & dmask], 1u);
    }
    __syncwarp();
    // Lane l owns bins 8l..8l+7. above = number of matching words in higher bins.
    uint32_t c[8];
    uint32_t s = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      c[j] = hist[lane * 8 + j];
      s += c[j];
    }
    uint32_t incl = s;  // inclusive suffix sum over lanes >= lane
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t v = __shfl_down_sync(0xffffffffu, incl, off);
      if (lane + off < 32) incl += v;
    }
    uint32_t run = incl - s;
    int bin = -1;
    uint32_t bin_above = 0, bin_cnt = 0;
#pragma unroll
    for (int j = 7; j >= 0; --j) {
      if (bin < 0 && run < need && run + c[j] >= need) {
        bin = lane * 8 + j;
        bin_above = run;
        bin_cnt = c[j];
      }
      run += c[j];
    }
    const uint32_t who = __ballot_sync(0xffffffffu, bin >= 0);
    const int src = __ffs(who) - 1;
    bin = __shfl_sync(0xffffffffu, bin, src);
    bin_above = __shfl_sync(0xffffffffu, bin_above, src);
    bin_cnt = __shfl_sync(0xffffffffu, bin_cnt, src);
    prefix |= static_cast<uint64_t>(bin) << shift;
    need -= bin_above;
    if (bin_cnt == need || shift == 0) break;
    width = shift < 8 ? shift : 8;
    shift -= width;
    __syncwarp();
  }
  // Keep exactly the words whose digits down to `shift` are >= the cut.
  const uint64_t cut = prefix >> shift;
  const uint32_t lt_mask = (1u << lane) - 1u;
  int out = 0;
  uint64_t mn = ~0ull;
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    const uint64_t u = i < n ? pool[i] : 0ull;
    const bool keep = i < n && (u >> shift) >= cut;
    const uint32_t m = __ballot_sync(0xffffffffu, keep);
    if (keep) {
      pool[out + __popc(m & lt_mask)] = u;
      mn = umin64(mn, u);
    }
    out += __popc(m);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mn = umin64(mn, __shfl_xor_sync(0xffffffffu, mn, off));
  __syncwarp();
  return mn;
}

// One in-register compare-exchange stage at distance J < R (element e = lane*R + r).
template <int R, int J>
__device__ __forceinline__ void reg_stage(uint64_t (&v)[R], int lane, int k) {
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if ((r & J) == 0) {
      const bool desc = ((lane * R + r) & k) == 0;
      const uint64_t a = v[r], b = v[r | J];
      const bool swap = desc ? (a < b) : (a > b);
      v[r] = swap ? b : a;
      v[r | J] = swap ? a : b;
    }
  }
}

// Bitonic sort, descending, of 32*R words held in registers by one warp, element e = lane*R + r.
// Distances below R are register swaps; larger ones exchange through shuffles. The stage loops
// run at run time and only the per-register work is unrolled: a fully unrolled 512-word network
// is thousands of straight-line instructions that would execute once, from a cold instruction
// cache.
template <int R>
__device__ __forceinline__ void warp_sort_desc(uint64_t (&v)[R], int lane) {
  static_assert(R == 16, "in-register stages are spelled out for 16 words per lane");
  constexpr int N = 32 * R;
#pragma unroll 1
  for (int k = 2; k <= N; k <<= 1) {
#pragma unroll 1
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= R) {
        const int lj = j / R;
        const bool lower = (lane & lj) == 0;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint64_t other = __shfl_xor_sync(0xffffffffu, v[r], lj);
          const bool desc = ((lane * R + r) & k) == 0;
          v[r] = (lower == desc) ? umax64(v[r], other) : umin64(v[r], other);
        }
      } else if (j == 8) {
        reg_stage<R, 8>(v, lane, k);
      } else if (j == 4) {
        reg_stage<R, 4>(v, lane, k);
      } else if (j == 2) {
        reg_stage<R, 2>(v, lane, k);
      } else {
        reg_stage<R, 1>(v, lane, k);
      }
    }
  }
}

// CTA-wide variant of select_compact for the end of a kernel, when every warp is free. All NT
// threads call it. get(i), i in [0, n), yields distinct non-zero words plus any number of zero
// words (empty slots, ignored); `out` receives the min(K, #non-zero) largest words, unordered,
// and that count is returned. hist: 256 shared words; scratch: 8 shared words.
template <int K, int NT, class Get>
__device__ __noinline__ int cta_select_get(const Get get, int n, uint64_t* out, uint32_t* hist,
                                           uint32_t* scratch) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;
  if (tid == 0) {
    scratch[0] = 0u;
    scratch[1] = 0u;
    scratch[5] = 0u;
    scratch[7] = 0u;
  }
  __syncthreads();
  // One pass: non-zero count, and the bits in which non-zero words differ from a reference.
  uint64_t ref = 0ull;
  for (int i = 0; i < n && ref == 0ull; ++i) ref = get(i);  // usually word 0
  uint64_t diff = 0ull;
  uint32_t nnz = 0u;
#pragma unroll 4
  for (int i = tid; i < n; i += NT) {
    const uint64_t u = get(i);
    if (u) {
      diff |= u ^ ref;
      ++nnz;
    }
  }
  const uint32_t wlo = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(diff));
  const uint32_t whi = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(diff >> 32));
  const uint32_t wn = __reduce_add_sync(0xffffffffu, nnz);
  if (lane == 0) {
    atomicOr(&scratch[0], wlo);
    atomicOr(&scratch[1], whi);
    atomicAdd(&scratch[7], wn);
  }
  __syncthreads();
  if (scratch[7] <= static_cast<uint32_t>(K)) {  // everything non-zero is kept
    for (int base = 0; base < n; base += NT) {
      const int i = base + tid;
      const uint64_t u = i < n ? get(i) : 0ull;
      const uint32_t m = __ballot_sync(0xffffffffu, u != 0ull);
      uint32_t slot = 0;
      if (lane == 0 && m) slot = atomicAdd(&scratch[5], __popc(m));
      slot = __shfl_sync(0xffffffffu, slot, 0);
      if (u) out[slot + __popc(m & lt_mask)] = u;
    }
    __syncthreads();
    return static_cast<int>(scratch[7]);
  }
  const uint64_t first = ref;
  const uint32_t dlo = scratch[0], dhi = scratch[1];
  const int top = dhi ? 63 - __clz(dhi) : (dlo ? 31 - __clz(dlo) : 0);
  int width = top + 1 < 8 ? top + 1 : 8;
  int shift = top + 1 - width;
  uint64_t prefix = shift + width >= 64 ? 0ull : (first & (~0ull << (shift + width)));
  uint32_t need = K;
  for (;;) {
    for (int i = tid; i < 256; i += NT) hist[i] = 0u;
    __syncthreads();
    const uint64_t hi_mask = shift + width >= 64 ? 0ull : (~0ull << (shift + width));
    const uint32_t dmask = (1u << width) - 1u;
#pragma unroll 4
    for (int i = tid; i < n; i += NT) {
      const uint64_t u = get(i);
      if ((u & hi_mask) == prefix) atomicAdd(&hist[static_cast<uint32_t>(u >> shift) & dmask], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      uint32_t c[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[lane * 8 + j];
        sum += c[j];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t v = __shfl_down_sync(0xffffffffu, incl, off);
        if (lane + off < 32) incl += v;
      }
      uint32_t run = incl - sum;
#pragma unroll
      for (int j = 7; j >= 0; --j) {
        if (run < need && run + c[j] >= need) {
          scratch[2] = lane * 8 + j;
          scratch[3] = run;
          scratch[4] = c[j];
        }
        run += c[j];
      }
    }
    __syncthreads();
    const uint32_t bin = scratch[2], above = scratch[3], cnt = scratch[4];
    __syncthreads();
    prefix |= static_cast<uint64_t>(bin) << shift;
    need -= above;
    if (cnt == need || shift == 0) break;
    width = shift < 8 ? shift : 8;
    shift -= width;
  }
  // Compaction in two passes (count per warp, then write at the warp's prefix offset), so no
  // pass waits on a returning atomic. Each warp owns a contiguous stripe of the input.
  const uint64_t cut = prefix >> shift;
  constexpr int kWarps = NT / 32;
  const int per_warp = (n + kWarps - 1) / kWarps;
  const int lo = warp * per_warp, hi = lo + per_warp < n ? lo + per_warp : n;
  uint32_t cnt = 0;
  for (int base = lo; base < hi; base += 128) {  // four independent words per lane
    bool keep[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = base + r * 32 + lane;
      keep[r] = i < hi && (get(i) >> shift) >= cut;
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) cnt += __popc(__ballot_sync(0xffffffffu, keep[r]));
  }
  uint32_t* wcount = hist;  // the histogram is no longer needed
  if (lane == 0) wcount[warp] = cnt;
  __syncthreads();
  uint32_t pos = 0;
  for (int w = 0; w < warp; ++w) pos += wcount[w];
  for (int base = lo; base < hi; base += 128) {
    uint64_t u[4];
    bool keep[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = base + r * 32 + lane;
      u[r] = i < hi ? get(i) : 0ull;
      keep[r] = i < hi && (u[r] >> shift) >= cut;
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const uint32_t m = __ballot_sync(0xffffffffu, keep[r]);
      if (keep[r]) out[pos + __popc(m & lt_mask)] = u[r];
      pos += __popc(m);
    }
  }
  __syncthreads();
  return K;
}

struct ArrayWords {
  const uint64_t* p;
  __device__ __forceinline__ uint64_t operator()(int i) const { return p[i]; }
};

// cta_select_get with a sampled pre-filter, for large inputs. 128 evenly spaced words are
// sampled and a high-ranked one (about 3K/n of the way down) becomes a provisional cut; one pass
// keeps every word >= that cut in per-warp segments of `tmp` (capacity `cap` words). When at
// least K words survive and no segment overflows, the K largest of all words are among them
// and the radix select runs on the segments only (about 3K words instead of n); otherwise it
// runs on all n words. Exact either way.
template <int K, int NT, class Get>
__device__ __noinline__ int cta_select_sampled(const Get get, int n, uint64_t* out, uint64_t* tmp,
                                               int cap, uint32_t* hist, uint32_t* scratch) {
  constexpr int kSamples = 128;
  constexpr int kMaxSeg = 256;  // survivor slots per warp (expected ~3K / warps)
  static_assert(NT >= kSamples, "one sample per thread");
  const int tid = threadIdx.x, lane = tid & 31;
  const int rank = static_cast<int>((3ll * K * kSamples) / (n > 1 ? n : 1));  // 0-based
  if (n <= 4 * K || rank >= kSamples - 1 || cap < 4 * K + kSamples)
    return cta_select_get<K, NT>(get, n, out, hist, scratch);
  uint64_t* samples = tmp + cap - kSamples;  // top of tmp; survivors fill it from the bottom
  if (tid == 0) {
    scratch[6] = 0u;  // provisional cut, low and high halves
    scratch[7] = 0u;
    scratch[5] = 0u;  // survivor count
    scratch[4] = 0u;  // segment overflow flag
  }
  if (tid < kSamples) samples[tid] = get(static_cast<int>((static_cast<int64_t>(tid) * n) / kSamples));
  __syncthreads();
  if (tid < kSamples) {
    const uint64_t mine = samples[tid];
    int greater = 0;
#pragma unroll 8
    for (int j = 0; j < kSamples; ++j) greater += samples[j] > mine ? 1 : 0;
    if (greater == rank && mine != 0ull) {  // distinct non-zero words: at most one thread
      scratch[6] = static_cast<uint32_t>(mine);
      scratch[7] = static_cast<uint32_t>(mine >> 32);
    }
  }
  __syncthreads();
  const uint64_t cut = (static_cast<uint64_t>(scratch[7]) << 32) | scratch[6];
  if (cut == 0ull) return cta_select_get<K, NT>(get, n, out, hist, scratch);
  // Survivors go to per-warp segments of kSeg zero-initialised words (a register counter per
  // warp, no atomics); the select then reads every segment and ignores the zero slots.
  constexpr int kWarps = NT / 32;
  const int seg = (cap - kSamples) / kWarps < kMaxSeg ? (cap - kSamples) / kWarps : kMaxSeg;
  const int warp = tid >> 5;
  for (int i = tid; i < kWarps * seg; i += NT) tmp[i] = 0ull;
  __syncthreads();
  uint64_t* mine = tmp + warp * seg;
  const int per_warp = (n + kWarps - 1) / kWarps;
  const int lo = warp * per_warp, hi = lo + per_warp < n ? lo + per_warp : n;
  uint32_t cnt = 0;
  for (int base = lo; base < hi; base += 128) {  // four independent words per lane
    uint64_t u[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = base + r * 32 + lane;
      u[r] = i < hi ? get(i) : 0ull;
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const bool keep = u[r] >= cut && u[r] != 0ull;
      const uint32_t m = __ballot_sync(0xffffffffu, keep);
      const uint32_t at = cnt + __popc(m & ((1u << lane) - 1u));
      if (keep && at < static_cast<uint32_t>(seg)) mine[at] = u[r];
      cnt += __popc(m);
    }
  }
  if (lane == 0) {
    atomicAdd(&scratch[5], cnt);
    if (cnt > static_cast<uint32_t>(seg)) atomicOr(&scratch[4], 1u);  // a segment overflowed
  }
  __syncthreads();
  const int kept = static_cast<int>(scratch[5]);
  const bool overflow = scratch[4] != 0u;
  __syncthreads();
  if (kept < K || overflow) return cta_select_get<K, NT>(get, n, out, hist, scratch);
  return cta_select_get<K, NT>(ArrayWords{tmp}, kWarps * seg, out, hist, scratch);
}

// Bitonic sort, descending, of x[0..N) in shared memory by all NT threads of the CTA (for the
// end of a kernel, when every warp is free): N/2 compare-exchanges per stage, one barrier each.
template <int N, int NT>
__device__ __forceinline__ void cta_sort_desc(uint64_t* x) {
#pragma unroll 1
  for (int k = 2; k <= N; k <<= 1) {
#pragma unroll 1
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int p = threadIdx.x; p < N / 2; p += NT) {
        const int i = ((p & ~(j - 1)) << 1) | (p & (j - 1));
        const int l = i + j;
        const uint64_t a = x[i], b = x[l];
        const bool desc = (i & k) == 0;
        if (desc ? (a < b) : (a > b)) {
          x[i] = b;
          x[l] = a;
        }
      }
      __syncthreads();
    }
  }
}

// cta_select_get over an array of words.
template <int K, int NT>
__device__ __forceinline__ int cta_select(const uint64_t* pool, int n, uint64_t* out,
                                          uint32_t* hist, uint32_t* scratch) {
  return cta_select_get<K, NT>(ArrayWords{pool}, n, out, hist, scratch);
}

}  // namespace ds4
