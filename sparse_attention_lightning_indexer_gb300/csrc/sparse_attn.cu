// Sparse attention over the indexer's selected keys, for sm_103a: the step that consumes the
// Top-512 lists ("DeepSeek V4 Flash 추론을 1.6초로 줄인 ds4 최적화", 용어 해설: sparse attention
// computes only some token pairs, and the Lightning Indexer chooses them).
//
// For query token t and head h over its selected positions J(t) (the indexer's out_idx row,
// -1 = empty), with one latent row kv[s] (d_qk = 576) per position shared by all 128 heads:
//     s_j = scale * q[t,h,:] . kv[j,:],   o[t,h,:] = sum_j softmax(s)_j kv[j, 0:512],
//     lse[t,h] = log sum_j exp(s_j).
//
// One CTA per token, all 128 heads (heads = TMEM lanes, so each softmax row lives in the two
// threads of its lane). Warps 0-3 and 8-11 are the softmax / output warps (two per TMEM lane
// quadrant, each owning half of the keys and half of every output block), warps 4-7 gather the
// selected rows with cp.async (eight threads per 128-byte row segment, so every warp instruction
// moves four whole segments) into the 128-byte-swizzled operand layout, warp 12 issues
// tcgen05.mma.
//   A  S[128 heads x 512 keys] = Q K^T accumulates over 9 chunks of 64 dims: per chunk a Q
//      chunk (tiled TMA) and the chunk of all 512 gathered key rows; 4 MMAs of N = 128 keys per
//      16-dim step into TMEM columns 0..511.
//   B  two passes over S in TMEM: the row maximum, then p = exp2(s * scale * log2 e - max),
//      summed in fp32 and stored as bf16 into shared memory in the K-major 128-byte-swizzled
//      layout of an MMA A operand (8 blocks of 64 keys).
//   C  O[128 x 512] = P V in two halves of 256 value dims (TMEM columns 0..255 and 256..511, free
//      once S is read, so the second half's MMAs run while the first half is stored): V chunks of
//      64 keys x 256 dims are gathered again and fed as an MN-major B operand. The output warps
//      scale each half by 1 / sum and store it as bf16.
// Shared memory: phase A's two 80 KB stages and phase C's P (128 KB) + two 32 KB V stages share
// one 192 KB region (the phases of a token never overlap).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "ds4idx.h"
#include "ptx.cuh"

namespace ds4w {
extern std::atomic<uint64_t>* launch_counter();
}

namespace ds4a {

using namespace ds4;

constexpr int kH = 128;          // heads = MMA M = TMEM lanes
constexpr int kDqk = 576;        // key / query width
constexpr int kDv = 512;         // value width (first kDv dims of a row)
constexpr int kK = 512;          // selected keys per token
constexpr int kChunk = 64;       // dims per K chunk (128 bytes of bf16)
constexpr int kNChunks = kDqk / kChunk;  // 9
constexpr int kAStageBytes = kH * 128 + kK * 128;  // Q chunk 16 KB + key chunk 64 KB
constexpr int kVKeys = 64;       // keys per V chunk
constexpr int kVStageBytes = 4 * kVKeys * 128;     // 4 blocks of 64 dims: 32 KB
constexpr int kPBytes = (kK / 64) * kH * 128;      // 8 blocks of 64 keys: 128 KB
constexpr int kOffP = 0;
constexpr int kOffV = kPBytes;
constexpr int kRegion = kPBytes + 2 * kVStageBytes;  // 192 KB
static_assert(2 * kAStageBytes <= kRegion, "phase A stages fit the shared region");
constexpr int kOffRows = kRegion;                   // int32 gather rows [512]
constexpr int kOffMask = kOffRows + kK * 4;         // uint32 validity words [16]
constexpr int kOffRed = kOffMask + 64;              // float [2 halves][2][128]: max, sum
constexpr int kOffBars = kOffRed + 2 * 2 * kH * 4;
constexpr int kNumBars = 2 + 2 + 1 + 1 + 2 + 2 + 1;
constexpr int kOffMisc = kOffBars + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 32 + 1024;
constexpr int kProducer0 = 4, kProducers = 4, kSoftmax1 = 8, kMma = 12;
constexpr int kThreads = (kMma + 1) * 32;
constexpr int kSoftmaxThreads = 8 * 32;
constexpr int kProducerThreads = kProducers * 32;
// B operand of P.V: V chunk rows are keys (the K dimension), 64 value dims per 128-byte row
// (the N dimension): an MN-major operand. Atoms of 8 keys x 64 dims (1 KB) repeat every 1 KB
// along K and every kVKeys * 128 bytes along N.
constexpr uint32_t kVStrideN = kVKeys * 128;
constexpr uint32_t kVStrideK = 1024;

__device__ uint32_t g_err;  // bounded-wait timeouts, read by ds4idx_sparse_attention_status

struct SAParams {
  const int32_t* idx;      // [T, 512]
  const int64_t* row0;     // [T] kv row of key 0 (or null)
  uint16_t* out;           // [T, 128, 512] bf16
  float* lse;              // [T, 128] or null
  int64_t T;
  int64_t kv_rows;
  float scale_log2;        // scale * log2(e)
};

__device__ __forceinline__ void gather4(void* dst, const CUtensorMap* m, uint64_t* bar, int32_t col,
                                        int32_t r0, int32_t r1, int32_t r2, int32_t r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3),
      "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar,
                                            int32_t x, int32_t y, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
// Shared-memory descriptor of an MN-major operand in the 128-byte swizzle layout.
__device__ __forceinline__ uint64_t smem_desc_mn_sw128(uint32_t saddr, uint32_t stride_n,
                                                       uint32_t stride_k) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((stride_n >> 4) & 0x3FFFu) << 16;  // leading byte offset
  d |= static_cast<uint64_t>((stride_k >> 4) & 0x3FFFu) << 32;  // stride byte offset
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}
// L2 policies: the latent rows are gathered many times (keep them), queries and outputs pass once.
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)),
               "l"(src), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void st_global_v4(void* dst, uint4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(dst), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__global__ void __launch_bounds__(kThreads, 1)
    sparse_attn_kernel(const __grid_constant__ CUtensorMap tmap_q, const uint16_t* __restrict__ kv,
                       const __grid_constant__ SAParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  int32_t* s_rows = reinterpret_cast<int32_t*>(smem + kOffRows);
  uint32_t* s_mask = reinterpret_cast<uint32_t*>(smem + kOffMask);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* a_full = bars;        // [2]
  uint64_t* a_empty = bars + 2;   // [2]
  uint64_t* s_ready = bars + 4;
  uint64_t* p_ready = bars + 5;
  uint64_t* v_full = bars + 6;    // [2]
  uint64_t* v_empty = bars + 8;   // [2]
  uint64_t* o_ready = bars + 10;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile uint32_t* s_abort = reinterpret_cast<volatile uint32_t*>(smem + kOffMisc + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&a_full[i], kProducerThreads + 1);  // every gather thread + the Q chunk's TMA
      mbar_init(&a_empty[i], 1);
      mbar_init(&v_full[i], kProducerThreads);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(s_ready, 1);
    mbar_init(p_ready, 8);
    mbar_init(o_ready, 1);
    *s_abort = 0u;
    fence_mbar_init();
  }
  if (warp == kMma) {
    tmem_alloc(s_tmem, 512);
    tmem_relinquish();
  }
  // Gather rows (an empty slot gathers row 0; its score is masked) and validity words.
  const int64_t r0 = p.row0 ? p.row0[t] : 0;
  for (int j = threadIdx.x; j < kK; j += kThreads) {
    const int32_t k = p.idx[t * kK + j];
    const int64_t r = r0 + k;
    const bool ok = k >= 0 && r >= 0 && r < p.kv_rows;
    s_rows[j] = ok ? static_cast<int32_t>(r) : 0;
    const uint32_t m = __ballot_sync(0xffffffffu, ok);
    if (lane == 0) s_mask[j >> 5] = m;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  uint32_t* err = &g_err;

  if (warp >= kProducer0 && warp < kProducer0 + kProducers) {
    // ---------------- gathers: each thread copies its 16-byte pieces, waits for them one stage
    // later (cp.async groups), makes them visible to the tensor core (proxy fence) and arrives.
    const int pt = threadIdx.x - kProducer0 * 32;  // 0..127
    const int pw = pt >> 5;
    const int seg = lane & 7, sub = lane >> 3;      // K rows: 8 threads per 128-byte segment
    const uint64_t keep = policy_evict_last(), pass = policy_evict_first();
    int issued_q = 0;
    bool ok = true;
    for (int c = 0; c < kNChunks; ++c) {
      const int st = c & 1;
      if (!(ok = mbar_wait_warp(&a_empty[st], ((c >> 1) & 1) ^ 1u, s_abort, err))) break;
      uint8_t* base = smem + st * kAStageBytes;
      if (pt == 0) {
        mbar_arrive_expect_tx(&a_full[st], kH * 128);
        tma_load_2d(base, &tmap_q, &a_full[st], c * kChunk, static_cast<int32_t>(t * kH), pass);
        issued_q = c + 1;
      }
      uint8_t* kbase = base + kH * 128;
      for (int i = 0; i < kK / (4 * kProducers); ++i) {
        const int r = (i * kProducers + pw) * 4 + sub;  // key row 0..511
        cp_async16(kbase + r * 128 + ((seg ^ (r & 7)) * 16),
                   kv + static_cast<int64_t>(s_rows[r]) * kDqk + c * kChunk + seg * 8, keep);
      }
      cp_async_commit();
      if (c > 0) {
        cp_async_wait<1>();
        fence_proxy_async_smem();
        mbar_arrive(&a_full[(c - 1) & 1]);
      }
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    if (ok) mbar_arrive(&a_full[(kNChunks - 1) & 1]);
    // phase C reuses the region: wait until every phase-A MMA has completed
    if (ok && mbar_wait_warp(s_ready, 0u, s_abort, err)) {
      for (int i = 0; i < 2 * (kK / kVKeys); ++i) {
        const int half = i / (kK / kVKeys), kc = i % (kK / kVKeys), st = i & 1;
        if (!(ok = mbar_wait_warp(&v_empty[st], ((i >> 1) & 1) ^ 1u, s_abort, err))) break;
        uint8_t* base = smem + kOffV + st * kVStageBytes;
        // V rows: one warp instruction copies one row's 512 bytes (32 x 16)
        for (int j = 0; j < kVKeys / kProducers; ++j) {
          const int r = j * kProducers + pw;  // 0..63 within the chunk
          const int nb = lane >> 3, cc = lane & 7;
          cp_async16(base + nb * kVStrideN + r * 128 + ((cc ^ (r & 7)) * 16),
                     kv + static_cast<int64_t>(s_rows[kc * kVKeys + r]) * kDqk + half * 256 + lane * 8,
                     keep);
        }
        cp_async_commit();
        if (i > 0) {
          cp_async_wait<1>();
          fence_proxy_async_smem();
          mbar_arrive(&v_full[(i - 1) & 1]);
        }
        if (i == 2 * (kK / kVKeys) - 1) {
          cp_async_wait<0>();
          fence_proxy_async_smem();
          mbar_arrive(&v_full[i & 1]);
        }
      }
    }
    cp_async_wait<0>();  // never exit with copies in flight
    if (pt == 0)
      for (int j = issued_q > 2 ? issued_q - 2 : 0; j < issued_q; ++j)
        mbar_drain(&a_full[j & 1], (j >> 1) & 1);
  } else if (warp == kMma) {
    // ---------------- MMA issue (one thread)
    if (lane == 0) {
      constexpr uint32_t kIdescS = instr_desc(1u, 1u, 128, 128);            // K-major A and B
      constexpr uint32_t kIdescO = instr_desc(1u, 1u, 128, 256) | (1u << 16);  // B MN-major
      bool ok = true;
      for (int c = 0; ok && c < kNChunks; ++c) {
        const int st = c & 1;
        if (!(ok = mbar_wait(&a_full[st], (c >> 1) & 1, s_abort, err))) break;
        tc_fence_after();
        const uint32_t qa = smem_u32(smem + st * kAStageBytes);
        const uint32_t kb = qa + kH * 128;
        for (int j = 0; j < 4; ++j)
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem + 128 * j, smem_desc_sw128(qa + ks * 32),
                     smem_desc_sw128(kb + j * 128 * 128 + ks * 32), kIdescS, (c | ks) ? 1u : 0u);
        mma_commit(&a_empty[st]);
      }
      mma_commit(s_ready);
      if (ok) ok = mbar_wait(p_ready, 0u, s_abort, err);
      tc_fence_after();
      const uint32_t pa = smem_u32(smem + kOffP);
      for (int i = 0; ok && i < 2 * (kK / kVKeys); ++i) {
        const int half = i / (kK / kVKeys), kc = i % (kK / kVKeys), st = i & 1;
        if (!(ok = mbar_wait(&v_full[st], (i >> 1) & 1, s_abort, err))) break;
        tc_fence_after();
        const uint32_t vb = smem_u32(smem + kOffV + st * kVStageBytes);
        for (int ks = 0; ks < kVKeys / 16; ++ks)
          mma_bf16(tmem + 256 * half, smem_desc_sw128(pa + kc * (kH * 128) + ks * 32),
                   smem_desc_mn_sw128(vb + ks * 16 * 128, kVStrideN, kVStrideK), kIdescO,
                   (kc | ks) ? 1u : 0u);
        mma_commit(&v_empty[st]);
        if (kc == kK / kVKeys - 1) mma_commit(o_ready);
      }
      // every MMA has completed before TMEM is released (bounded, also after an abort)
      mbar_drain(s_ready, 0u);
      mbar_drain(o_ready, 1u);
    }
    __syncwarp();
  } else {
    // ---------------- softmax and output: lane quadrant warp % 4, key half g
    const int g = warp >= kSoftmax1 ? 1 : 0;
    const int quad = warp & 3;
    const int h = quad * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    float* red = reinterpret_cast<float*>(smem + kOffRed);  // [stat][g][h]
    auto softmax_sync = [] { asm volatile("bar.sync 1, %0;" ::"n"(kSoftmaxThreads) : "memory"); };
    float m = -__int_as_float(0x7f800000), l = 0.f;
    bool ok = mbar_wait_warp(s_ready, 0u, s_abort, err);
    tc_fence_after();
    constexpr int kHalfChunks = kK / 32 / 2;  // 8 chunks of 32 keys per key half
    const int i0 = g * kHalfChunks;
    if (ok) {
      // Two passes over this thread's half of S, each reading 32-column chunks with the next
      // chunk's load in flight; the two halves combine their max and sum in shared memory.
      uint32_t rb[2][32];
      tmem_ld32(tmem + lane_base + 32 * i0, rb[0]);
      tmem_wait_ld();
      float mx = -__int_as_float(0x7f800000);
#pragma unroll 2
      for (int i = 0; i < kHalfChunks; ++i) {
        if (i + 1 < kHalfChunks) tmem_ld32(tmem + lane_base + 32 * (i0 + i + 1), rb[(i + 1) & 1]);
        const uint32_t* r = rb[i & 1];
        const uint32_t vm = s_mask[i0 + i];
#pragma unroll
        for (int j = 0; j < 32; ++j)
          mx = fmaxf(mx, ((vm >> j) & 1u) ? __uint_as_float(r[j]) : -__int_as_float(0x7f800000));
        tmem_wait_ld();
      }
      red[g * kH + h] = mx * p.scale_log2;  // scale > 0: the max of the scaled scores
    }
    softmax_sync();  // every softmax warp reaches it, also after an abort
    if (ok) {
      uint32_t rb[2][32];
      m = fmaxf(red[h], red[kH + h]);
      const float mm = m == -__int_as_float(0x7f800000) ? 0.f : m;
      tmem_ld32(tmem + lane_base + 32 * i0, rb[0]);
      tmem_wait_ld();
      float ls = 0.f;
#pragma unroll 2
      for (int i = 0; i < kHalfChunks; ++i) {
        if (i + 1 < kHalfChunks) tmem_ld32(tmem + lane_base + 32 * (i0 + i + 1), rb[(i + 1) & 1]);
        const uint32_t* r = rb[i & 1];
        const uint32_t vm = s_mask[i0 + i];
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float p0 = ((vm >> j) & 1u) ? exp2f(__uint_as_float(r[j]) * p.scale_log2 - mm) : 0.f;
          const float p1 = ((vm >> (j + 1)) & 1u) ? exp2f(__uint_as_float(r[j + 1]) * p.scale_log2 - mm) : 0.f;
          ls += p0 + p1;
          pk[j / 2] = pack_bf16x2(p0, p1);
        }
        // keys 32(i0+i)..+31 of head h: block (i0+i)/2, 16-byte chunks ((i0+i)%2)*4 .. +3 of row h
        const int ci = i0 + i;
        uint8_t* row = smem + kOffP + (ci >> 1) * (kH * 128) + h * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int cc = (ci & 1) * 4 + u;
          *reinterpret_cast<uint4*>(row + ((cc ^ (h & 7)) * 16)) =
              make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
        tmem_wait_ld();
      }
      red[2 * kH + g * kH + h] = ls;
    }
    fence_proxy_async_smem();  // P (generic writes) before the MMAs that read it
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(p_ready);
    softmax_sync();  // both halves' sums are in shared memory
    if (ok) l = red[2 * kH + h] + red[3 * kH + h];
    if (p.lse && g == 0)
      p.lse[t * kH + h] = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -__int_as_float(0x7f800000);
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint16_t* orow = p.out + (t * kH + h) * kDv;
    const uint64_t pass = policy_evict_first();
    for (int half = 0; ok && half < 2; ++half) {
      if (!(ok = mbar_wait_warp(o_ready, static_cast<uint32_t>(half), s_abort, err))) break;
      tc_fence_after();
      // this warp stores value dims 256 half + 128 g .. + 127
      uint32_t rb[2][32];
      const uint32_t ocol = tmem + lane_base + 256 * half + 128 * g;
      tmem_ld32(ocol, rb[0]);
      tmem_wait_ld();
      for (int i = 0; i < 4; ++i) {
        if (i + 1 < 4) tmem_ld32(ocol + 32 * (i + 1), rb[(i + 1) & 1]);
        const uint32_t* r = rb[i & 1];
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2)
          pk[j / 2] = pack_bf16x2(__uint_as_float(r[j]) * inv, __uint_as_float(r[j + 1]) * inv);
        uint4* dst = reinterpret_cast<uint4*>(orow + half * 256 + 128 * g + 32 * i);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          st_global_v4(dst + u, make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]), pass);
        tmem_wait_ld();
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_enc = nullptr;
std::once_flag g_enc_once;

bool encode(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  std::call_once(g_enc_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDqk), rows};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDqk) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kChunk), box_rows};
  cuuint32_t es[2] = {1u, 1u};
  return g_enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace ds4a

extern "C" int ds4idx_sparse_attention(const void* q, const void* kv, int64_t kv_rows,
                                       const int32_t* idx, const int64_t* kv_row0, int64_t T,
                                       int32_t n_heads, int32_t d_qk, int32_t d_v, int32_t topk,
                                       float sm_scale, void* out, float* lse, void* stream) {
  using namespace ds4a;
  if (n_heads != kH || d_qk != kDqk || d_v != kDv || topk != kK) return DS4IDX_ERR_UNSUPPORTED;
  if (T < 0 || kv_rows < 1 || kv_rows > 0x7FFFFFFF || T * kH > 0x7FFFFFFF) return DS4IDX_ERR_INVALID_ARG;
  if (T == 0) return DS4IDX_OK;
  auto al = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
  if (!q || !kv || !idx || !out || !al(q, 16) || !al(kv, 16) || !al(idx, 4) || !al(out, 16) ||
      (lse && !al(lse, 4)) || (kv_row0 && !al(kv_row0, 8)) || !(sm_scale > 0.f))
    return DS4IDX_ERR_INVALID_ARG;
  CUtensorMap tq;
  if (!encode(&tq, q, static_cast<uint64_t>(T) * kH, kH)) return DS4IDX_ERR_INVALID_ARG;
  SAParams p{};
  p.idx = idx;
  p.row0 = kv_row0;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.T = T;
  p.kv_rows = kv_rows;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  if (cudaFuncSetAttribute(sparse_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes) != cudaSuccess)
    return DS4IDX_ERR_CUDA;
  sparse_attn_kernel<<<static_cast<unsigned>(T), kThreads, kSmemBytes,
                       static_cast<cudaStream_t>(stream)>>>(tq, static_cast<const uint16_t*>(kv), p);
  if (cudaGetLastError() != cudaSuccess) return DS4IDX_ERR_LAUNCH;
  ds4w::launch_counter()->fetch_add(1, std::memory_order_relaxed);
  return DS4IDX_OK;
}

extern "C" int ds4idx_sparse_attention_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DS4IDX_ERR_CUDA;
  uint32_t e = 0;
  if (cudaMemcpyFromSymbol(&e, ds4a::g_err, sizeof e) != cudaSuccess) return DS4IDX_ERR_CUDA;
  if (e) {
    const uint32_t z = 0;
    cudaMemcpyToSymbol(ds4a::g_err, &z, sizeof z);
    return DS4IDX_ERR_DEVICE_TIMEOUT;
  }
  return DS4IDX_OK;
}
