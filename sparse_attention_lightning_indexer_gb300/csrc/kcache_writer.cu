// FP8 index-cache writer: the step before the indexer. New index keys (and the queries of an FP8
// indexer call) are quantised per token row to OCP E4M3FN codes with one fp32 scale,
//     scale = absmax(row) / 448,   code = E4M3(clamp(x / scale, -448, 448))   (RNE, satfinite),
// a row whose scale is 0 getting codes 0, and the query scale is folded into the head weights,
// w'[t,j] = w[t,j] * qscale[t]. "DeepSeek V4 Flash는 단일 AMD MI300X에서 실행됩니다", section
// 두 가지 핵심 정확성 수정 사항 (FP8 형식 불일치), is about exactly this cache: written as FP8
// E4M3, with the format's largest finite value fixing the scale. Every fp32 operation here is a
// single correctly rounded one (IEEE division and multiplication, the hardware's
// round-to-nearest-even E4M3 conversion), so the codes and scales are bit-exact functions of
// the inputs.
//
// Both kernels are HBM-bound streams: a key row is one warp (128 values, 16-byte loads, one
// 128-byte store of codes); a query token is one CTA (64 x 128 values).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "ds4idx.h"

namespace ds4w {

constexpr int kDim = 128;
constexpr int kHeads = 64;
constexpr float kE4M3Max = 448.f;

extern std::atomic<uint64_t>* launch_counter();

// Two fp32 values to two E4M3FN codes, round to nearest even with saturation to +-448:
// the code of lo in bits 0..7, of hi in bits 8..15.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ float clamp448(float y) { return fminf(kE4M3Max, fmaxf(-kE4M3Max, y)); }

// Four values of a row to four codes packed little-endian into 32 bits.
__device__ __forceinline__ uint32_t encode4(float4 v, float scale) {
  if (scale == 0.f) return 0u;
  const float y0 = clamp448(__fdiv_rn(v.x, scale)), y1 = clamp448(__fdiv_rn(v.y, scale));
  const float y2 = clamp448(__fdiv_rn(v.z, scale)), y3 = clamp448(__fdiv_rn(v.w, scale));
  return e4m3x2(y0, y1) | (e4m3x2(y2, y3) << 16);
}

__device__ __forceinline__ float4 bf16x4_to_float4(uint2 u) {
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
}

template <bool kBf16>
__device__ __forceinline__ float4 load4(const void* base, int64_t elem) {
  if (kBf16) return bf16x4_to_float4(__ldg(reinterpret_cast<const uint2*>(
                                         static_cast<const uint16_t*>(base) + elem)));
  return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem));
}

__device__ __forceinline__ float abs_max4(float4 v) {
  return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
}

// Keys: warp w of the grid-stride loop takes rows w, w + warps, ...; kRows rows per iteration
// with all loads issued before any reduction. Row i goes to cache row dst = slots[i] (slots
// given) or dst_offset + i; destinations outside [0, cache_rows) are skipped.
template <bool kBf16, int kRows>
__global__ void __launch_bounds__(256) quantize_keys_kernel(const void* __restrict__ k, int64_t n,
                                                            const int64_t* __restrict__ slots,
                                                            int64_t dst_offset,
                                                            uint8_t* __restrict__ kcache,
                                                            float* __restrict__ kscale,
                                                            int64_t cache_rows) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r0 = warp0 * kRows; r0 < n; r0 += warps * kRows) {
    float4 v[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
      v[r] = r0 + r < n ? load4<kBf16>(k, (r0 + r) * kDim + lane * 4) : make_float4(0, 0, 0, 0);
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const int64_t row = r0 + r;
      if (row >= n) break;
      // absmax: non-negative floats order like their bit patterns
      const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(abs_max4(v[r]))));
      const float scale = __fdiv_rn(amax, kE4M3Max);
      const int64_t dst = slots ? __ldg(slots + row) : dst_offset + row;
      if (dst < 0 || dst >= cache_rows) continue;
      reinterpret_cast<uint32_t*>(kcache + dst * kDim)[lane] = encode4(v[r], scale);
      if (lane == 0) kscale[dst] = scale;
    }
  }
}

// Queries: CTA t quantises token t (64 heads x 128 = 8192 values, 32 per thread) with one scale
// and folds it into that token's 64 head weights.
template <bool kBf16>
__global__ void __launch_bounds__(256) quantize_queries_kernel(const void* __restrict__ q,
                                                               const float* __restrict__ w,
                                                               int64_t T, uint8_t* __restrict__ qc,
                                                               float* __restrict__ w_out,
                                                               float* __restrict__ qscale) {
  constexpr int kPerThread = kHeads * kDim / 256;  // 32 values = 8 float4
  __shared__ uint32_t s_max[8];
  const int64_t t = blockIdx.x;
  if (t >= T) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t base = t * kHeads * kDim;
  float4 v[kPerThread / 4];
  // element e = (i * 256 + tid) * 4: each float4 load of the CTA is one contiguous 4 KiB span
#pragma unroll
  for (int i = 0; i < kPerThread / 4; ++i) v[i] = load4<kBf16>(q, base + (i * 256 + tid) * 4);
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < kPerThread / 4; ++i) m = fmaxf(m, abs_max4(v[i]));
  const uint32_t wm = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
  if (lane == 0) s_max[warp] = wm;
  __syncthreads();
  uint32_t bm = 0u;
#pragma unroll
  for (int i = 0; i < 8; ++i) bm = max(bm, s_max[i]);
  const float scale = __fdiv_rn(__uint_as_float(bm), kE4M3Max);
  uint32_t* out = reinterpret_cast<uint32_t*>(qc + base);
#pragma unroll
  for (int i = 0; i < kPerThread / 4; ++i) out[i * 256 + tid] = encode4(v[i], scale);
  if (tid < kHeads) w_out[t * kHeads + tid] = __fmul_rn(__ldg(w + t * kHeads + tid), scale);
  if (qscale && tid == 0) qscale[t] = scale;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return sms;
}

}  // namespace ds4w

using namespace ds4w;

extern "C" int ds4idx_quantize_keys(const void* k, int32_t in_dtype, int64_t n,
                                    const int64_t* slots, int64_t dst_offset, uint8_t* kcache,
                                    float* kscale, int64_t cache_rows, void* stream) {
  if (in_dtype != DS4IDX_BF16 && in_dtype != DS4IDX_F32) return DS4IDX_ERR_INVALID_ARG;
  if (n < 0 || cache_rows < 0 || (slots == nullptr && dst_offset < 0)) return DS4IDX_ERR_INVALID_ARG;
  if (n == 0) return DS4IDX_OK;
  if (!k || !kcache || !kscale || !aligned(k, 16) || !aligned(kcache, 16) || !aligned(kscale, 4) ||
      (slots && !aligned(slots, 8)))
    return DS4IDX_ERR_INVALID_ARG;
  if (!slots && dst_offset + n > cache_rows) return DS4IDX_ERR_INVALID_ARG;
  const int sms = sm_count();
  if (sms < 1) return DS4IDX_ERR_CUDA;
  constexpr int kRows = 4;
  const int64_t warps_needed = (n + kRows - 1) / kRows;
  const int64_t ctas = std::min<int64_t>((warps_needed + 7) / 8, static_cast<int64_t>(sms) * 8);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (in_dtype == DS4IDX_BF16)
    quantize_keys_kernel<true, kRows><<<static_cast<unsigned>(ctas), 256, 0, s>>>(
        k, n, slots, dst_offset, kcache, kscale, cache_rows);
  else
    quantize_keys_kernel<false, kRows><<<static_cast<unsigned>(ctas), 256, 0, s>>>(
        k, n, slots, dst_offset, kcache, kscale, cache_rows);
  if (cudaGetLastError() != cudaSuccess) return DS4IDX_ERR_LAUNCH;
  launch_counter()->fetch_add(1, std::memory_order_relaxed);
  return DS4IDX_OK;
}

extern "C" int ds4idx_quantize_queries(const void* q, int32_t in_dtype, int64_t T, const float* w,
                                       uint8_t* q_codes, float* w_out, float* qscale,
                                       void* stream) {
  if (in_dtype != DS4IDX_BF16 && in_dtype != DS4IDX_F32) return DS4IDX_ERR_INVALID_ARG;
  if (T < 0 || T > 0x7FFFFFFF) return DS4IDX_ERR_INVALID_ARG;
  if (T == 0) return DS4IDX_OK;
  if (!q || !w || !q_codes || !w_out || !aligned(q, 16) || !aligned(w, 4) ||
      !aligned(q_codes, 16) || !aligned(w_out, 4) || (qscale && !aligned(qscale, 4)))
    return DS4IDX_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (in_dtype == DS4IDX_BF16)
    quantize_queries_kernel<true><<<static_cast<unsigned>(T), 256, 0, s>>>(q, w, T, q_codes, w_out,
                                                                           qscale);
  else
    quantize_queries_kernel<false><<<static_cast<unsigned>(T), 256, 0, s>>>(q, w, T, q_codes,
                                                                            w_out, qscale);
  if (cudaGetLastError() != cudaSuccess) return DS4IDX_ERR_LAUNCH;
  launch_counter()->fetch_add(1, std::memory_order_relaxed);
  return DS4IDX_OK;
}
