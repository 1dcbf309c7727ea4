// The Lightning Indexer kernel for sm_103a: tcgen05 scorer with a fused epilogue and a
// streaming per-query Top-512.
//
// What it computes ("DeepSeek V4 Flash 추론을 1.6초로 줄인 ds4 최적화", 섹션별 상세 / 용어 해설:
// the indexer scores every visible key of a query and a Top-512 selection keeps the best):
//     I[t,s] = kscale[s] * sum_j w[t,j] * max(0, q[t,j,:] . k[s,:]),  s <= pos_offset + t,
// keeping per query the 512 largest (score, lower-index-first) pairs.
//
// One CTA owns NQ consecutive queries of one sequence (and, when the key range is split, one
// slice of their keys). Its warps:
//   epilogue     4 or 8 warps; warp e reads TMEM lanes 32(e%4)..32(e%4)+31, i.e. one key per
//                thread, for its group of queries, and reduces the 64 head columns of each
//                query thread-locally (ReLU, * w, sum) with packed fp32x2 FMAs, so the T x S
//                score matrix never leaves the SM; two warps per lane quadrant hide TMEM latency;
//   TMA          Q block once, then 128-key K tiles into a ring of stages;
//   MMA          TMEM owner and MMA issuer: per key tile, D[128 keys, NQ*64 (query, head)]
//                = K_tile . Q_block^T on tcgen05 into one of two TMEM accumulators;
//   selectors    one warp per query: filters the tile's scores against the running threshold
//                into an unsorted pool and radix-selects it back to exactly 512 when it fills.
// Keys are the MMA M dimension (128 = all TMEM lanes) and (query, head) pairs the N dimension,
// which is what makes the head reduction free of shuffles. The design on the page (a
// threadgroup-tiled scorer, then a register-blocked K-resident scorer, then a streaming
// Top-512, on Apple GPUs) is prior art; this layout follows from TMEM's lane/column shape.
#pragma once
#include <cstdint>
#include <cuda.h>

#include "ptx.cuh"
#include "topk.cuh"

namespace ds4 {

constexpr int kHeads = 64;       // H_I
constexpr int kDim = 128;        // d_I
constexpr int kTopK = 512;
constexpr int kTileKeys = 128;   // MMA M
constexpr int kMaxBatch = 64;
constexpr int kDtBf16 = 0;
constexpr int kDtFp8 = 1;

struct KParams {
  const float* w;        // [B, T, 64]
  const float* kscale;   // [B, S] (FP8) or null
  int32_t* out_idx;      // [B, T, 512]
  float* out_score;      // [B, T, 512] or null
  uint64_t* partial;     // [B, T, n_splits, 512] packed lists when n_splits > 1
  uint32_t* counters;    // [B * n_qb] split tickets (zero between calls) when n_splits > 1
  float* dense;          // [T, S] scores (debug variant)
  uint32_t* err;         // device error word
  int64_t T, S;
  int32_t B, n_qb, n_splits, tiles_per_split;
  int64_t pos[kMaxBatch];
};

template <int DT, int NQ, bool DENSE>
struct KCfg {
  static constexpr int kRowBytes = DT == kDtBf16 ? 2 * kDim : kDim;  // one 128-dim row
  static constexpr int kHalves = kRowBytes / 128;                    // 128-byte swizzle columns
  static constexpr int kN = kHeads * NQ;                             // MMA N
  static constexpr int kQBytes = kN * kRowBytes;
  static constexpr int kKBytes = kTileKeys * kRowBytes;
  static constexpr int kStages = DT == kDtBf16 ? (NQ == 4 ? 3 : 5) : (NQ == 4 ? 6 : 8);
  static constexpr int kKSteps = DT == kDtBf16 ? kDim / 16 : kDim / 32;
  static constexpr int kStepBytes = 32;                              // K bytes per MMA step
  // Depth of the epilogue -> selector score ring: it lets selectors fall behind by that many
  // tiles while they radix-select, without stalling the MMA pipeline.
  static constexpr int kScoreBufs = NQ == 1 ? 16 : 12;
  // TMEM accumulators: all 512 columns, so a narrow (one-query) MMA can run up to 8 tiles
  // ahead of the epilogue instead of waiting on a round trip per tile.
  static constexpr int kAccBufs = 512 / kN;
  // Candidate pool per selector warp (its kept 512 plus new candidates).
  static constexpr int kPool = 1024;
  // Epilogue: two warps per TMEM lane quadrant. With several queries the two groups split the
  // queries; with one query they take alternate tiles.
  static constexpr bool kEpiAltTiles = NQ == 1;
  static constexpr int kEpiWarps = 8;
  static constexpr int kEpiPerTile = kEpiAltTiles ? 4 : 8;  // epilogue warps that handle a tile
  static constexpr int kQPerGroup = kEpiAltTiles ? 1 : NQ / 2;
  // Selectors: one warp per query, or four for a single query (each filters one 32-key group of
  // every tile into its own pool), which keeps a one-query CTA's selection at HBM pace.
  static constexpr int kSelPerQuery = NQ == 1 ? 4 : 1;
  static constexpr int kSelectors = DENSE ? 0 : NQ * kSelPerQuery;
  static constexpr int kGroupsPerSel = (kTileKeys / 32) / kSelPerQuery;
  static constexpr int kTmaWarp = kEpiWarps;
  static constexpr int kMmaWarp = kEpiWarps + 1;
  static constexpr int kSelWarp0 = kEpiWarps + 2;
  static constexpr int kWarps = kEpiWarps + 2 + kSelectors;
  static constexpr int kThreads = 32 * kWarps;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kAccBufs * kN == 512 && kAccBufs >= 2, "accumulators tile the TMEM columns");
  static constexpr uint32_t kIdesc =
      DT == kDtBf16 ? instr_desc(1u, 1u, kTileKeys, kN) : instr_desc(0u, 0u, kTileKeys, kN);
  // shared memory layout (offsets from a 1024-byte aligned base)
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffW = kOffK + kStages * kKBytes;
  static constexpr int kOffHist = kOffW + NQ * kHeads * 4;
  static constexpr int kOffRing = kOffHist + (DENSE ? 0 : kSelectors * 256 * 4);
  static constexpr int kOffPool = kOffRing + (DENSE ? 0 : kScoreBufs * NQ * kTileKeys * 4);
  static constexpr int kOffSelEnd = kOffPool + (DENSE ? 0 : kSelectors * kPool * 8);
  static constexpr int kNumBars = 2 * kStages + 2 * kAccBufs + 2 * kScoreBufs + 1;
  // Buffered selection (one-query CTAs whose key split fits): the epilogue stores every fp32
  // score of the split here and one CTA-wide select runs at the end. The buffer overlays the
  // ring and the pools, which that mode leaves unused, plus whatever shared memory is left.
  static constexpr int kBufTiles =
      (NQ == 1 && !DENSE) ? (232448 - 1024 - 96 - kNumBars * 8 - kOffRing) / (kTileKeys * 4) : 0;
  static constexpr int kOffBar = kOffSelEnd > kOffRing + kBufTiles * kTileKeys * 4
                                     ? kOffSelEnd : kOffRing + kBufTiles * kTileKeys * 4;
  static_assert(4 * kTopK * 8 <= kStages * kKBytes, "split merge reuses the K stages");
  static_assert((kStages * kKBytes / 8 - 2 * kTopK) / kTopK >= 2, "split merge needs two lists per round");
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 96 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kQBytes % 1024 == 0 && kKBytes % 1024 == 0, "swizzle atoms need 1 KiB alignment");
};

template <int R>
__device__ __forceinline__ void write_output(const KParams& p, int64_t row,
                                             const uint64_t (&v)[R], int lane) {
  int32_t* oi = p.out_idx + row * kTopK + lane * R;
#pragma unroll
  for (int r = 0; r < R; ++r) oi[r] = v[r] ? key_index(v[r]) : -1;
  if (p.out_score) {
    float* os = p.out_score + row * kTopK + lane * R;
#pragma unroll
    for (int r = 0; r < R; ++r) os[r] = v[r] ? key_score(v[r]) : -__int_as_float(0x7f800000);
  }
}

// CTA-wide finish (split plans, and one-query CTAs whose two selector warps keep separate
// pools): for each query, the unused tails of its pools are zeroed (a CTA-wide select ignores
// zero words), the 512 best words are radix-selected with all warps, and then either published
// unordered as this split's list or sorted once and written as the output row.
// Buffered-mode words: the fp32 score of key key0 + i, packed, or 0 when the query cannot see it.
struct ScoreWords {
  const float* s;
  int64_t key0, vis_end;
  __device__ __forceinline__ uint64_t operator()(int i) const {
    const int64_t key = key0 + i;
    return key < vis_end ? pack_key(s[i], static_cast<uint32_t>(key)) : 0ull;
  }
};

template <class C>
__device__ void finish_cta_select(const KParams& p, int b, int64_t t0, int split,
                                  uint64_t* pools, const uint32_t* pool_n, uint64_t* stage,
                                  uint32_t* hist, uint32_t* scratch, int warp, int lane,
                                  const float* sbuf, int buffered_keys, int64_t key0,
                                  int64_t pos_b) {
  constexpr int R = kTopK / 32;
  constexpr int kWords = C::kSelPerQuery * C::kPool;
  for (int q = 0; q < C::kN / kHeads; ++q) {
    const int64_t t = t0 + q;
    if (t >= p.T) break;
    int cnt;
    if (buffered_keys > 0) {
      const int64_t pt = pos_b + t;
      const int64_t vis_end = (pt < p.S - 1 ? pt : p.S - 1) + 1;
      constexpr int kStageWords = C::kStages * C::kKBytes / 8;
      cnt = cta_select_sampled<kTopK, C::kThreads>(ScoreWords{sbuf, key0, vis_end}, buffered_keys,
                                                   stage, stage + kTopK, kStageWords - kTopK,
                                                   hist, scratch);
    } else {
      uint64_t* base = pools + q * kWords;
      for (int sw = 0; sw < C::kSelPerQuery; ++sw) {
        const int used = static_cast<int>(pool_n[q * C::kSelPerQuery + sw]);
        for (int i = used + threadIdx.x; i < C::kPool; i += C::kThreads)
          base[sw * C::kPool + i] = 0ull;
      }
      __syncthreads();
      cnt = cta_select<kTopK, C::kThreads>(base, kWords, stage, hist, scratch);
    }
    const int64_t row = static_cast<int64_t>(b) * p.T + t;
    if (p.n_splits > 1) {
      uint64_t* dst = p.partial + (row * p.n_splits + split) * kTopK;
      for (int i = threadIdx.x; i < kTopK; i += C::kThreads) dst[i] = i < cnt ? stage[i] : 0ull;
    } else if (warp == 0) {
      uint64_t v[R];
#pragma unroll
      for (int r = 0; r < R; ++r) v[r] = lane * R + r < cnt ? stage[lane * R + r] : 0ull;
      warp_sort_desc<R>(v, lane);
      write_output<R>(p, row, v, lane);
    }
    __syncthreads();
  }
  if (p.n_splits > 1) __threadfence();  // lists visible GPU-wide before the ticket is taken
}

// Split plans, part 2 (the CTA that takes a block's last ticket): copy every split's list of
// each query into shared memory with independent wide loads, radix-select the 512 best, sort
// them once in registers and write the output row. Lists that do not fit at once are folded in
// rounds (the 512 survivors of a round stay at the front of the gather area).
template <class C>
__device__ void merge_split_lists(const KParams& p, int b, int64_t t0, uint64_t* stage,
                                  uint32_t* hist, uint32_t* scratch, int warp, int lane) {
  constexpr int kStageWords = C::kStages * C::kKBytes / 8;
  constexpr int kCap = kStageWords - kTopK;  // gather area; the last 512 words receive selects
  constexpr int kListsPerRound = (kCap - kTopK) / kTopK;
  uint64_t* sel = stage + kCap;
  for (int q = 0; q < C::kN / kHeads; ++q) {
    const int64_t t = t0 + q;
    if (t >= p.T) break;
    const int64_t row = static_cast<int64_t>(b) * p.T + t;
    const uint64_t* lists = p.partial + row * p.n_splits * kTopK;
    int n = 0;  // words already in the gather area (survivors of earlier rounds)
    for (int sp0 = 0; sp0 < p.n_splits; sp0 += kListsPerRound) {
      const int nl = p.n_splits - sp0 < kListsPerRound ? p.n_splits - sp0 : kListsPerRound;
      const uint4* src = reinterpret_cast<const uint4*>(lists + static_cast<int64_t>(sp0) * kTopK);
      uint4* dst = reinterpret_cast<uint4*>(stage + n);
      const int n4 = nl * kTopK / 2;
#pragma unroll 8
      for (int i = threadIdx.x; i < n4; i += C::kThreads) dst[i] = src[i];
      __syncthreads();
      n += nl * kTopK;
      if (sp0 + nl < p.n_splits) {  // another round follows: keep only the 512 best
        const int kept = cta_select<kTopK, C::kThreads>(stage, n, sel, hist, scratch);
        // zero-padded to exactly 512 words, so the next round's copy stays 16-byte aligned
        for (int i = threadIdx.x; i < kTopK; i += C::kThreads) stage[i] = i < kept ? sel[i] : 0ull;
        __syncthreads();
        n = kTopK;
      }
    }
    // survivors of the sampled pre-filter go to the free words between the gather and `sel`
    const int cnt = cta_select_sampled<kTopK, C::kThreads>(ArrayWords{stage}, n, sel, stage + n,
                                                           kCap - n, hist, scratch);
    // one CTA-wide sort of the 512 winners (zero-padded), then a coalesced store of the row
    for (int i = cnt + threadIdx.x; i < kTopK; i += C::kThreads) sel[i] = 0ull;
    __syncthreads();
    cta_sort_desc<kTopK, C::kThreads>(sel);
    for (int i = threadIdx.x; i < kTopK; i += C::kThreads) {
      const uint64_t u = sel[i];
      p.out_idx[row * kTopK + i] = u ? key_index(u) : -1;
      if (p.out_score) p.out_score[row * kTopK + i] = u ? key_score(u) : -__int_as_float(0x7f800000);
    }
    __syncthreads();
  }
}

template <int DT, int NQ, bool DENSE>
__global__ void __launch_bounds__(KCfg<DT, NQ, DENSE>::kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ KParams p) {
  using C = KCfg<DT, NQ, DENSE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sK = smem + C::kOffK;
  float* sW = reinterpret_cast<float*>(smem + C::kOffW);
  float* sScore = reinterpret_cast<float*>(smem + C::kOffRing);
  float* sBuf = reinterpret_cast<float*>(smem + C::kOffRing);  // buffered mode only
  uint64_t* sPool = reinterpret_cast<uint64_t*>(smem + C::kOffPool);
  uint32_t* sHist = reinterpret_cast<uint32_t*>(smem + C::kOffHist);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full = bars;                         // [kStages]  TMA -> MMA
  uint64_t* empty = full + C::kStages;           // [kStages]  MMA -> TMA
  uint64_t* tfull = empty + C::kStages;          // [kAccBufs] MMA -> epilogue
  uint64_t* tempty = tfull + C::kAccBufs;        // [kAccBufs] epilogue -> MMA
  uint64_t* sfull = tempty + C::kAccBufs;        // [C::kScoreBufs] epilogue -> selectors
  uint64_t* sempty = sfull + C::kScoreBufs;         // [C::kScoreBufs] selectors -> epilogue
  uint64_t* qfull = sempty + C::kScoreBufs;         // Q block landed
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile uint32_t* s_abort = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 4);
  volatile uint32_t* s_last = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 8);
  uint32_t* s_scratch = reinterpret_cast<uint32_t*>(smem + C::kOffMisc + 16);  // 8 words
  uint32_t* s_pool_n = reinterpret_cast<uint32_t*>(smem + C::kOffMisc + 48);   // [selectors]
  // Running threshold published by each selector warp (only rises): a query's warps filter
  // against the largest of them, which is still at most the CTA's exact 512th best.
  volatile uint64_t* s_theta = reinterpret_cast<volatile uint64_t*>(smem + C::kOffMisc + 64);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: longest query blocks first; batches and key splits innermost
  const int wid = blockIdx.x;
  const int b = wid % p.B;
  const int rest = wid / p.B;
  const int split = rest % p.n_splits;
  const int qb = p.n_qb - 1 - rest / p.n_splits;
  const int64_t t0 = static_cast<int64_t>(qb) * NQ;
  const int64_t t_last = (t0 + NQ < p.T ? t0 + NQ : p.T) - 1;
  const int64_t pos_b = p.pos[b];
  int tile_lo, n_tiles;
  if (DENSE) {
    tile_lo = 0;
    n_tiles = static_cast<int>((p.S + kTileKeys - 1) / kTileKeys);
  } else {
    const int64_t p_last = pos_b + t_last;
    const int64_t vis_end = (p_last < p.S - 1 ? p_last : p.S - 1) + 1;
    const int tiles_total = static_cast<int>((vis_end + kTileKeys - 1) / kTileKeys);
    tile_lo = split * p.tiles_per_split;
    const int hi = tile_lo + p.tiles_per_split < tiles_total ? tile_lo + p.tiles_per_split
                                                              : tiles_total;
    n_tiles = hi > tile_lo ? hi - tile_lo : 0;
  }

  const bool buffered = C::kBufTiles > 0 && n_tiles <= C::kBufTiles;

  // ---- setup
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < C::kAccBufs; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], C::kEpiPerTile);
    }
    for (int i = 0; i < C::kScoreBufs; ++i) {
      mbar_init(&sfull[i], C::kEpiPerTile);
      mbar_init(&sempty[i], C::kSelectors > 0 ? C::kSelectors : 1);  // unused without selectors
    }
    mbar_init(qfull, 1);
    *s_abort = 0u;
    for (int i = 0; i < C::kSelectors; ++i) s_theta[i] = 0ull;
    fence_mbar_init();
  }
  if (warp == C::kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tmap_q);
    tma_prefetch_desc(&tmap_k);
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(s_tmem, C::kTmemCols);
    tmem_relinquish();
  }
  for (int i = threadIdx.x; i < NQ * kHeads; i += C::kThreads) {
    const int64_t t = t0 + i / kHeads;
    sW[i] = t < p.T ? p.w[(static_cast<int64_t>(b) * p.T + t) * kHeads + (i % kHeads)] : 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == C::kTmaWarp) {
    // ================= TMA producer
    if (lane == 0 && n_tiles > 0) {
      mbar_arrive_expect_tx(qfull, C::kQBytes);
      for (int h = 0; h < C::kHalves; ++h)
        tma_load_3d(sQ + h * (C::kN * 128), &tmap_q, qfull, h * 64 * (DT == kDtBf16 ? 1 : 2),
                    static_cast<int32_t>(t0 * kHeads), b);
      int it = 0;
      for (; it < n_tiles; ++it) {
        const int st = it % C::kStages;
        const uint32_t ph = (it / C::kStages) & 1;
        if (!mbar_wait(&empty[st], ph ^ 1u, s_abort, p.err)) break;
        mbar_arrive_expect_tx(&full[st], C::kKBytes);
        uint8_t* dst = sK + st * C::kKBytes;
        const int32_t key0 = (tile_lo + it) * kTileKeys;
        for (int h = 0; h < C::kHalves; ++h)
          tma_load_3d(dst + h * (kTileKeys * 128), &tmap_k, &full[st],
                      h * 64 * (DT == kDtBf16 ? 1 : 2), key0, b);
      }
      // Never leave the CTA with copies in flight: wait (bounded) for the last load of each
      // stage and for the Q block. After a normal run these have long completed.
      const int issued = it;
      for (int j = issued - C::kStages > 0 ? issued - C::kStages : 0; j < issued; ++j)
        mbar_wait(&full[j % C::kStages], (j / C::kStages) & 1, s_abort, p.err);
      mbar_wait(qfull, 0, s_abort, p.err);
    }
  } else if (warp == C::kMmaWarp) {
    // ================= MMA issuer (one thread)
    if (lane == 0 && n_tiles > 0) {
      int it = 0;
      bool ok = mbar_wait(qfull, 0, s_abort, p.err);
      for (; ok && it < n_tiles; ++it) {
        const int st = it % C::kStages;
        const uint32_t sph = (it / C::kStages) & 1;
        const int acc = it % C::kAccBufs;
        const uint32_t aph = (it / C::kAccBufs) & 1;
        if (!mbar_wait(&full[st], sph, s_abort, p.err)) break;
        if (!mbar_wait(&tempty[acc], aph ^ 1u, s_abort, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(acc * C::kN);
        const uint32_t a_base = smem_u32(sK + st * C::kKBytes);
        const uint32_t b_base = smem_u32(sQ);
#pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks) {
          const int half = ks / (128 / C::kStepBytes);
          const int koff = (ks % (128 / C::kStepBytes)) * C::kStepBytes;
          const uint64_t a_desc = smem_desc_sw128(a_base + half * (kTileKeys * 128) + koff);
          const uint64_t b_desc = smem_desc_sw128(b_base + half * (C::kN * 128) + koff);
          if (DT == kDtBf16)
            mma_bf16(d, a_desc, b_desc, C::kIdesc, ks > 0 ? 1u : 0u);
          else
            mma_fp8(d, a_desc, b_desc, C::kIdesc, ks > 0 ? 1u : 0u);
        }
        mma_commit(&empty[st]);
        mma_commit(&tfull[acc]);
      }
      // Before TMEM is released every issued MMA must have completed: wait for the commit of
      // the last tile issued (the epilogue waits on the same phase).
      if (it > 0) {
        const int last = it - 1;
        mbar_wait(&tfull[last % C::kAccBufs], (last / C::kAccBufs) & 1, s_abort, p.err);
      }
    }
    __syncwarp();
  } else if (warp < C::kEpiWarps) {
    // ================= epilogue: TMEM -> ReLU . w -> per-key score
    const int quad = warp & 3;
    const int grp = warp >> 2;
    const int q0 = C::kEpiAltTiles ? 0 : grp * C::kQPerGroup;
    const int it0 = C::kEpiAltTiles ? grp : 0;   // first tile of this warp
    const int step = C::kEpiAltTiles ? 2 : 1;    // tiles between this warp's tiles
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    // FP8 key scales are read two tiles ahead so their global-memory latency stays hidden
    // (decode streams the cache once, so these reads miss in L2).
    const float* kscale_b = DT == kDtFp8 ? p.kscale + static_cast<int64_t>(b) * p.S : nullptr;
    auto load_scale = [&](int tile) -> float {
      const int64_t k = static_cast<int64_t>(tile_lo + tile) * kTileKeys + quad * 32 + lane;
      return (tile < n_tiles && k < p.S) ? __ldg(kscale_b + k) : 0.f;
    };
    float ks_next0 = 1.f, ks_next1 = 1.f;
    if (DT == kDtFp8) {
      ks_next0 = load_scale(it0);
      ks_next1 = load_scale(it0 + step);
    }
    for (int it = it0; it < n_tiles; it += step) {
      const int acc = it % C::kAccBufs;
      const uint32_t aph = (it / C::kAccBufs) & 1;
      const int sb = it % C::kScoreBufs;
      const uint32_t sph = (it / C::kScoreBufs) & 1;
      const int64_t key = static_cast<int64_t>(tile_lo + it) * kTileKeys + quad * 32 + lane;
      float ks = 1.f;
      if (DT == kDtFp8) {
        ks = ks_next0;
        ks_next0 = ks_next1;
        ks_next1 = load_scale(it + 2 * step);
      }
      if (!mbar_wait_warp(&tfull[acc], aph, s_abort, p.err)) break;
      tc_fence_after();
      if (!DENSE && !buffered) {
        if (!mbar_wait_warp(&sempty[sb], sph ^ 1u, s_abort, p.err)) break;
      }
      // The warp's TMEM reads are 2 * kQPerGroup chunks of 32 head columns. Chunk c+1 is
      // requested before chunk c is reduced, so each load's latency hides behind arithmetic
      // (tcgen05.wait::ld waits for all outstanding loads; two 32-register buffers suffice).
      constexpr int kChunks = 2 * C::kQPerGroup;
      const uint32_t col0 = tmem + lane_base + static_cast<uint32_t>(acc * C::kN + q0 * kHeads);
      uint32_t rb[2][32];
      tmem_ld32(col0, rb[0]);
      tmem_wait_ld();
      uint64_t acc01 = 0ull, acc23 = 0ull;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        if (c + 1 < kChunks) tmem_ld32(col0 + 32 * (c + 1), rb[(c + 1) & 1]);
        const int q = q0 + c / 2;
        // Four accumulator chains (heads = 0, 1, 2, 3 mod 4), two per packed fp32x2 FMA.
        const float4* w4 = reinterpret_cast<const float4*>(sW + q * kHeads + (c & 1) * 32);
        const uint32_t* r = rb[c & 1];
#pragma unroll
        for (int h4 = 0; h4 < 8; ++h4) {
          const float4 wv = w4[h4];
          const float x0 = fmaxf(__uint_as_float(r[4 * h4 + 0]), 0.f);
          const float x1 = fmaxf(__uint_as_float(r[4 * h4 + 1]), 0.f);
          const float x2 = fmaxf(__uint_as_float(r[4 * h4 + 2]), 0.f);
          const float x3 = fmaxf(__uint_as_float(r[4 * h4 + 3]), 0.f);
          acc01 = fma_f32x2(pack_f32x2(x0, x1), pack_f32x2(wv.x, wv.y), acc01);
          acc23 = fma_f32x2(pack_f32x2(x2, x3), pack_f32x2(wv.z, wv.w), acc23);
        }
        if (c & 1) {  // both halves of query q reduced
          float a0, a1, a2, a3;
          unpack_f32x2(acc01, a0, a1);
          unpack_f32x2(acc23, a2, a3);
          acc01 = 0ull;
          acc23 = 0ull;
          float score = (a0 + a1) + (a2 + a3);
          if (DT == kDtFp8) score *= ks;
          if (DENSE) {
            const int64_t t = t0 + q;
            if (t < p.T && key < p.S) {
              const bool vis = key <= pos_b + t;
              p.dense[t * p.S + key] = vis ? score : -__int_as_float(0x7f800000);
            }
          } else if (buffered) {
            sBuf[it * kTileKeys + quad * 32 + lane] = score;
          } else {
            sScore[(sb * NQ + q) * kTileKeys + quad * 32 + lane] = score;
          }
        }
        if (c + 1 < kChunks) tmem_wait_ld();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&tempty[acc]);
        if (!DENSE && !buffered) mbar_arrive(&sfull[sb]);
      }
    }
  } else if (!DENSE) {
    // ================= selectors
    const int sidx = warp - C::kSelWarp0;
    const int q = sidx / C::kSelPerQuery;
    const int g0 = (sidx % C::kSelPerQuery) * C::kGroupsPerSel;  // first 32-key group it filters
    uint64_t* pool = sPool + sidx * C::kPool;
    uint32_t* hist = sHist + sidx * 256;
    const int64_t t = t0 + q;
    const bool valid = t < p.T;
    const int64_t pt = pos_b + t;
    const int64_t vis_end = valid ? (pt < p.S - 1 ? pt : p.S - 1) + 1 : 0;
    const uint32_t lt_mask = (1u << lane) - 1u;
    uint64_t theta = 0ull;  // exact 512th best word this warp has seen (0 until 512 were seen)
    int n = 0;              // words in the pool
    for (int it = 0; it < (buffered ? 0 : n_tiles); ++it) {
      const int sb = it % C::kScoreBufs;
      const uint32_t sph = (it / C::kScoreBufs) & 1;
      if (!mbar_wait_warp(&sfull[sb], sph, s_abort, p.err)) break;
      uint64_t th = theta;
#pragma unroll
      for (int o = 0; o < C::kSelPerQuery; ++o) th = umax64(th, s_theta[q * C::kSelPerQuery + o]);
      const int64_t key0 = static_cast<int64_t>(tile_lo + it) * kTileKeys;
      const float* sc = sScore + (sb * NQ + q) * kTileKeys;
      uint64_t u[C::kGroupsPerSel];
      uint32_t m[C::kGroupsPerSel];
#pragma unroll
      for (int r = 0; r < C::kGroupsPerSel; ++r) {  // independent 32-key groups
        const int g = g0 + r;
        const int64_t key = key0 + g * 32 + lane;
        u[r] = key < vis_end ? pack_key(sc[g * 32 + lane], static_cast<uint32_t>(key)) : 0ull;
        m[r] = __ballot_sync(0xffffffffu, u[r] > th);
      }
#pragma unroll
      for (int r = 0; r < C::kGroupsPerSel; ++r) {
        if (u[r] > th) pool[n + __popc(m[r] & lt_mask)] = u[r];
        n += __popc(m[r]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sempty[sb]);
      if (n > C::kPool - C::kGroupsPerSel * 32) {
        theta = select_compact<kTopK>(pool, n, hist, lane);
        n = kTopK;
        if (lane == 0) s_theta[sidx] = theta;
      }
    }
    if (C::kSelPerQuery > 1 || p.n_splits > 1) {
      // Finished with a CTA-wide select after the role loops (every warp helps).
      if (lane == 0) s_pool_n[sidx] = static_cast<uint32_t>(n);
    } else {
      if (n > kTopK) n = (select_compact<kTopK>(pool, n, hist, lane), kTopK);
      __syncwarp();
      // Final order: sort the (at most 512) survivors in registers, best first.
      constexpr int R = kTopK / 32;
      uint64_t v[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int i = lane * R + r;
        v[r] = i < n ? pool[i] : 0ull;
      }
      warp_sort_desc<R>(v, lane);
      if (valid && !*s_abort) write_output<R>(p, static_cast<int64_t>(b) * p.T + t, v, lane);
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (!DENSE && (C::kSelPerQuery > 1 || p.n_splits > 1) && !*s_abort)
    finish_cta_select<C>(p, b, t0, split, sPool, s_pool_n, reinterpret_cast<uint64_t*>(sK), sHist,
                         s_scratch, warp, lane, sBuf, buffered ? n_tiles * kTileKeys : 0,
                         static_cast<int64_t>(tile_lo) * kTileKeys, pos_b);
  if (!DENSE && p.n_splits > 1) {
    // Split plans: every CTA of a query block takes a ticket after publishing its lists; the
    // CTA that takes the last ticket merges them (nothing ever waits on another CTA).
    uint32_t* ticket = p.counters + static_cast<int64_t>(b) * p.n_qb + qb;
    if (threadIdx.x == 0) {
      __threadfence();
      *s_last = atomicAdd(ticket, 1u) == static_cast<uint32_t>(p.n_splits - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (*s_last) {
      __threadfence();
      if (!*s_abort)
        merge_split_lists<C>(p, b, t0, reinterpret_cast<uint64_t*>(sK), sHist, s_scratch, warp,
                             lane);
      if (threadIdx.x == 0) *ticket = 0u;  // ready for the next call
    }
  }
}

}  // namespace ds4
