// Merge of Top-k lists computed over disjoint key ranges of the same queries: the exchange step
// of a key-sharded indexer (each shard scores its keys and keeps its own Top-512; the union of
// the shards' lists holds the global Top-512, because a key in the global Top-512 is also in the
// Top-512 of its own shard). One CTA merges one query row: every list's (score, key) pairs are
// packed into ordered words (topk.cuh: score descending, ties to the lower key), an exact radix
// select keeps the 512 largest and one CTA-wide bitonic sort orders them.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "ds4idx.h"
#include "topk.cuh"

namespace ds4w {
extern std::atomic<uint64_t>* launch_counter();
}

namespace ds4m {

constexpr int kTopK = 512;
constexpr int kMaxLists = 16;
constexpr int kThreads = 256;

struct MergeParams {
  const int32_t* in_idx;    // [n_lists, rows, 512]
  const float* in_score;    // [n_lists, rows, 512]
  int32_t* out_idx;         // [rows, 512]
  float* out_score;         // [rows, 512] or null
  int64_t rows;
  int32_t n_lists;
  int64_t idx_offset[kMaxLists];  // added to list l's key indices
  int64_t row0[kMaxLists];        // list l holds rows row0[l] .. rows-1; earlier rows are empty
};

__global__ void __launch_bounds__(kThreads) merge_topk_kernel(const __grid_constant__ MergeParams p) {
  extern __shared__ uint64_t smem_words[];
  uint64_t* words = smem_words;                    // [n_lists * 512]
  uint64_t* sel = words + p.n_lists * kTopK;       // [512]
  __shared__ uint32_t hist[256];
  __shared__ uint32_t scratch[8];
  const int64_t row = blockIdx.x;
  const int n = p.n_lists * kTopK;
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const int l = i / kTopK, r = i % kTopK;
    uint64_t u = 0ull;
    if (row >= p.row0[l]) {
      const int64_t at = (static_cast<int64_t>(l) * p.rows + row) * kTopK + r;
      const int32_t k = __ldg(p.in_idx + at);
      if (k >= 0) {
        const int64_t key = k + p.idx_offset[l];
        u = ds4::pack_key(__ldg(p.in_score + at), static_cast<uint32_t>(key));
      }
    }
    words[i] = u;
  }
  __syncthreads();
  const int cnt = ds4::cta_select<kTopK, kThreads>(words, n, sel, hist, scratch);
  for (int i = cnt + threadIdx.x; i < kTopK; i += kThreads) sel[i] = 0ull;
  __syncthreads();
  ds4::cta_sort_desc<kTopK, kThreads>(sel);
  for (int i = threadIdx.x; i < kTopK; i += kThreads) {
    const uint64_t u = sel[i];
    p.out_idx[row * kTopK + i] = u ? ds4::key_index(u) : -1;
    if (p.out_score) p.out_score[row * kTopK + i] = u ? ds4::key_score(u) : -__int_as_float(0x7f800000);
  }
}

}  // namespace ds4m

extern "C" int ds4idx_merge_topk(int32_t n_lists, int64_t rows, const int32_t* in_idx,
                                 const float* in_score, const int64_t* idx_offsets,
                                 const int64_t* row0, int32_t topk, int32_t* out_idx,
                                 float* out_score, void* stream) {
  using namespace ds4m;
  if (n_lists < 1 || n_lists > kMaxLists || rows < 0 || rows > 0x7FFFFFFF || topk != kTopK ||
      !idx_offsets)
    return DS4IDX_ERR_INVALID_ARG;
  if (rows == 0) return DS4IDX_OK;
  if (!in_idx || !in_score || !out_idx) return DS4IDX_ERR_INVALID_ARG;
  MergeParams p{};
  p.in_idx = in_idx;
  p.in_score = in_score;
  p.out_idx = out_idx;
  p.out_score = out_score;
  p.rows = rows;
  p.n_lists = n_lists;
  for (int l = 0; l < n_lists; ++l) {
    // merged keys are 32-bit indices (< 2^31)
    if (idx_offsets[l] < 0 || idx_offsets[l] > 0x7FFFFFFF) return DS4IDX_ERR_INVALID_ARG;
    p.idx_offset[l] = idx_offsets[l];
    p.row0[l] = row0 ? row0[l] : 0;
    if (p.row0[l] < 0) return DS4IDX_ERR_INVALID_ARG;
  }
  const size_t smem = static_cast<size_t>(n_lists + 1) * kTopK * sizeof(uint64_t);
  if (cudaFuncSetAttribute(merge_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return DS4IDX_ERR_CUDA;
  merge_topk_kernel<<<static_cast<unsigned>(rows), kThreads, smem,
                      static_cast<cudaStream_t>(stream)>>>(p);
  if (cudaGetLastError() != cudaSuccess) return DS4IDX_ERR_LAUNCH;
  ds4w::launch_counter()->fetch_add(1, std::memory_order_relaxed);
  return DS4IDX_OK;
}
