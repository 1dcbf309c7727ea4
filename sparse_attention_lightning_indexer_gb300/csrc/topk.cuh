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
// The per-query state is a list of k words sorted descending plus an unsorted buffer of
// candidates that beat the list's last word (the running threshold). When the buffer fills,
// one warp sorts it and merges it into the list with bitonic networks in shared memory; the
// threshold can only rise. The page replaced a bitonic sort plus merge cascade over all scores
// with a streaming Top-512; here bitonic networks only ever see the small buffer.
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

__device__ __forceinline__ void cmp_swap_desc(uint64_t* x, int i, int l) {
  const uint64_t a = x[i], b = x[l];
  if (a < b) {
    x[i] = b;
    x[l] = a;
  }
}

// Sorts a bitonic sequence x[0..n) descending (one warp; n a power of two >= 64).
template <int N>
__device__ __forceinline__ void bitonic_merge_desc(uint64_t* x, int lane) {
#pragma unroll 1
  for (int j = N / 2; j > 0; j >>= 1) {
#pragma unroll
    for (int p = lane; p < N / 2; p += 32) {
      const int i = ((p & ~(j - 1)) << 1) | (p & (j - 1));
      cmp_swap_desc(x, i, i + j);
    }
    __syncwarp();
  }
}

// Full bitonic sort of x[0..N) descending (one warp).
template <int N>
__device__ __forceinline__ void bitonic_sort_desc(uint64_t* x, int lane) {
#pragma unroll 1
  for (int k = 2; k <= N; k <<= 1) {
#pragma unroll 1
    for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
      for (int p = lane; p < N / 2; p += 32) {
        const int i = ((p & ~(j - 1)) << 1) | (p & (j - 1));
        const int l = i + j;
        const uint64_t a = x[i], b = x[l];
        const bool desc = (i & k) == 0;
        if (desc ? (a < b) : (a > b)) {
          x[i] = b;
          x[l] = a;
        }
      }
      __syncwarp();
    }
  }
}

// x[0..N/2) and x[N/2..N) are each sorted descending; sorts x[0..N) descending.
template <int N>
__device__ __forceinline__ void merge_sorted_halves_desc(uint64_t* x, int lane) {
#pragma unroll
  for (int i = lane; i < N / 2; i += 32) cmp_swap_desc(x, i, N - 1 - i);
  __syncwarp();
  bitonic_merge_desc<N / 2>(x, lane);
  bitonic_merge_desc<N / 2>(x + N / 2, lane);
}

// list[0..K) sorted descending (0-padded); buf[0..n) unsorted candidates, capacity C <= K.
// Afterwards list holds the K largest of list U buf, sorted descending. One warp.
template <int K, int C>
__device__ __forceinline__ void merge_buffer(uint64_t* list, uint64_t* buf, int n, int lane) {
  static_assert(C <= K, "buffer larger than the list");
  for (int i = n + lane; i < C; i += 32) buf[i] = 0ull;
  __syncwarp();
  bitonic_sort_desc<C>(buf, lane);
  // At most C of the buffer can enter the top K, so list[0..K-C) stays; the top C of
  // list[K-C..K) U buf is the elementwise max against the reversed buffer (a bitonic sequence).
  uint64_t* tail = list + (K - C);
#pragma unroll
  for (int i = lane; i < C; i += 32) {
    const uint64_t a = tail[i], b = buf[C - 1 - i];
    tail[i] = a > b ? a : b;
  }
  __syncwarp();
  bitonic_merge_desc<C>(tail, lane);
  if (K == 2 * C) {
    merge_sorted_halves_desc<K>(list, lane);
  } else {
    static_assert(K == 2 * C || K == C, "unsupported list/buffer ratio");
  }
}

// a[0..K) and b[0..K) sorted descending; a becomes the K largest of a U b, sorted. One warp.
template <int K>
__device__ __forceinline__ void merge_lists(uint64_t* a, const uint64_t* b, int lane) {
#pragma unroll
  for (int i = lane; i < K; i += 32) {
    const uint64_t x = a[i], y = b[K - 1 - i];
    a[i] = x > y ? x : y;
  }
  __syncwarp();
  bitonic_merge_desc<K>(a, lane);
}

}  // namespace ds4
