// The Lightning Indexer kernel for sm_103a: tcgen05 scorer with a fused epilogue and a
// streaming per-query Top-512.
//
// What it computes ("DeepSeek V4 Flash 추론을 1.6초로 줄인 ds4 최적화", 섹션별 상세 / 용어 해설:
// the indexer scores every visible key of a query and a Top-512 selection keeps the best):
//     I[t,s] = kscale[s] * sum_j w[t,j] * max(0, q[t,j,:] . k[s,:]),  s <= pos_offset + t,
// keeping per query the 512 largest (score, lower-index-first) pairs.
//
// One CTA owns NQ (4, or 1 for decode) consecutive queries of one sequence (and, when the key
// range is split, one slice of their keys). Its warps:
//   epilogue     8 warps; warp e reads TMEM lanes 32(e%4)..32(e%4)+31, i.e. one key per
//                thread, for its queries, and reduces the 64 head columns of each query
//                thread-locally (ReLU, * w, sum) with packed fp32x2 FMAs, so the T x S score
//                matrix never leaves the SM; two warps per lane quadrant hide TMEM latency
//                (they split the queries, or take alternate tiles when NQ = 1). With NQ = 4
//                the CTA is four warpgroups and the two epilogue warpgroups hold their queries'
//                head weights in registers (setmaxnreg moves registers to them);
//   TMA          Q block once, then 128-key K tiles into a ring of stages;
//   MMA          TMEM owner and MMA issuer: per key tile, D[128 keys, NQ*64 (query, head)]
//                = K_tile . Q_block^T on tcgen05 into one of the TMEM accumulators (all 512
//                columns: 2 for NQ = 4, 8 for NQ = 1);
//   selectors    one warp per query (four for NQ = 1): filter the tile's scores against the
//                running threshold into an unsorted pool and radix-select it back to exactly
//                512 when it fills.
// One-query CTAs whose key split fits shared memory (decode) leave the selectors idle: the
// epilogue keeps every score and a running cut bin with per-bin counts (histsel.cuh), and the
// exact selection happens once, at the end (finish_hist, merge_hist_slots).
// Keys are the MMA M dimension (128 = all TMEM lanes) and (query, head) pairs the N dimension,
// which is what makes the head reduction free of shuffles. The design on the page (a
// threadgroup-tiled scorer, then a register-blocked K-resident scorer, then a streaming
// Top-512, on Apple GPUs) is prior art; this layout follows from TMEM's lane/column shape.
#pragma once
#include <cstdint>
#include <cuda.h>

#include "histsel.cuh"
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

// ---- one-query split plans: slot format of a split's published list
// A split publishes, in a slot of kSlotWords words:
//   word 0        count m | window start lo << 32 | window width nb << 48
//   words 2..129  a window of 256 32-bit counts of the published words per bin (histsel.cuh),
//                 bins lo .. lo + nb - 1; bins below the window may go uncounted (an undercount
//                 can only lower the merge's cut bin, never drop a winner)
//   words 130..   the m published words (m <= kSlotListCap), grouped by bin: the window's bins
//                 from the highest down, each bin's words in any order, then every word below
//                 the window; so the words at or above any bin of the window form a prefix
// A split publishes every word of its keys whose bin is at or above a bin that at least 512 of
// its words reach: a superset of its 512 best, hence of every global winner among its keys.
constexpr int kSlotHdrWords = 2;
constexpr int kSlotHistBins = 256;
constexpr int kSlotListOff = kSlotHdrWords + kSlotHistBins / 2;
constexpr int kSlotWords = 1152;
// Per split query block in `counters`: its merge ticket, then one word per split (up to 64) in
// which one-query splits publish a bin their k-th best key reaches, k = ceil(512 / splits). All
// zero between calls (the merging CTA clears its block's words).
constexpr int kCounterWords = 1 + 64;
constexpr int kSlotListCap = kSlotWords - kSlotListOff;
constexpr int kSurvCap = 2048;   // words the bin-ranked final selection takes at most
constexpr int kRankBins = 2048;  // bins (and refined buckets) it spans at most
constexpr int kRecut = 64;       // a warp's own candidates between its raises of the cut bin

// Shared-memory scratch of the bin-ranked final selection and of the slot merge.
struct RankArea {
  static constexpr int kBytes = 2 * kSurvCap * 8 + 3 * kRankBins * 4 + 256 * 4 + 512 * 4;
  uint64_t* sv;      // [kSurvCap] words to rank
  uint64_t* sorted;  // [kSurvCap] the same words grouped by bin, best bin first
  uint32_t* cnt;     // [kRankBins] words per bin
  uint32_t* off;     // [kRankBins] first position of each bin
  uint32_t* cur;     // [kRankBins] scatter cursors
  uint32_t* rhist;   // [256] radix-select scratch
  uint32_t* hdr;     // [512] merge headers
  __device__ explicit RankArea(uint8_t* base)
      : sv(reinterpret_cast<uint64_t*>(base)),
        sorted(reinterpret_cast<uint64_t*>(base) + kSurvCap),
        cnt(reinterpret_cast<uint32_t*>(base + 2 * kSurvCap * 8)),
        off(cnt + kRankBins),
        cur(off + kRankBins),
        rhist(cur + kRankBins),
        hdr(rhist + 256) {}
};

// One sequence of a call: its queries, its keys, its position and its share of the grid.
struct SeqDesc {
  int64_t T;          // queries
  int64_t S;          // keys in its cache
  int64_t pos;        // position of query 0 (query t sits at pos + t)
  int64_t q_row0;     // row of query 0 in the packed q [*, 64, 128], w, out_idx and out_score
  int64_t k_row0;     // row of key 0 in the key pool (contiguous caches)
  int64_t list0;      // first word of its split lists in `partial`
  int32_t n_qb;       // query blocks of NQ queries
  int32_t n_splits;   // key splits per query block
  int32_t tiles_per_split;
  int32_t cta0;       // first CTA of its work (calls that are not uniform)
  int32_t ticket0;    // first of its split tickets in `counters`
  int32_t pt_row;     // its row of the page table (paged caches)
};

struct KParams {
  const float* w;        // [rows, 64]
  const float* kscale;   // [pool rows] (FP8) or null
  int32_t* out_idx;      // [rows, 512]
  float* out_score;      // [rows, 512] or null
  uint64_t* partial;     // per-split lists of split plans: per query 512 words per split, or one
                         // slot of kSlotWords per split for one-query CTAs
  uint32_t* counters;    // split tickets (zero between calls)
  float* dense;          // [T, S] scores (debug variant, one sequence)
  uint32_t* err;         // device error word
  const int32_t* page_table;  // [*, pt_stride] page ids (paged key pool), or null (contiguous)
  int64_t pool_rows;     // rows of the key pool
  uint64_t wait_ns;      // limit of one bounded mbarrier wait (kWaitLimitNs)
  int32_t withhold;      // test only: CTA 0's first selector withholds its first ring release
  int32_t B;
  int32_t uniform;       // every sequence has the same plan: CTA i serves sequence i % B
  int32_t page_size;     // keys per page (a multiple of 64) when paged
  int32_t pt_stride;     // page-table entries per sequence
  SeqDesc seq[kMaxBatch];
};

// Pool row of key `key` (< sd.S) of a sequence. A page id outside the pool (the caller's
// mistake) gives pool_rows, a row past the pool: TMA loads it as zeros and the scale reads skip
// it, so a bad page table yields wrong scores, never an out-of-bounds access.
__device__ __forceinline__ int64_t key_row(const KParams& p, const SeqDesc& sd, int64_t key) {
  if (p.page_table == nullptr) return sd.k_row0 + key;
  const int64_t page = __ldg(p.page_table + static_cast<int64_t>(sd.pt_row) * p.pt_stride +
                             key / p.page_size);
  const int64_t row = page * p.page_size + key % p.page_size;
  return (page >= 0 && row < p.pool_rows) ? row : p.pool_rows;
}

template <int DT, int NQ, bool DENSE>
struct KCfg {
  static constexpr int kRowBytes = DT == kDtBf16 ? 2 * kDim : kDim;  // one 128-dim row
  static constexpr int kHalves = kRowBytes / 128;                    // 128-byte swizzle columns
  static constexpr int kN = kHeads * NQ;                             // MMA N
  static constexpr int kQBytes = kN * kRowBytes;
  static constexpr int kKBytes = kTileKeys * kRowBytes;
  static constexpr int kStages = DT == kDtBf16 ? (NQ == 4 ? 2 : 4) : (NQ == 4 ? 6 : 8);
  static constexpr int kKSteps = DT == kDtBf16 ? kDim / 16 : kDim / 32;
  static constexpr int kStepBytes = 32;                              // K bytes per MMA step
  // Depth of the epilogue -> selector score ring: it lets selectors fall behind by that many
  // tiles while they radix-select, without stalling the MMA pipeline. Selections cluster at the
  // start of each query block, while the threshold is still low, so a deep ring pays more than
  // a deep K pipeline: four-query bf16 CTAs keep two K stages (keys come from L2) and 28 ring
  // tiles.
  static constexpr int kScoreBufs = NQ == 1 ? 16 : (DT == kDtFp8 ? 30 : 28);
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
  // Four-query scoring CTAs keep the head weights of their two queries in registers (128 per
  // epilogue thread), so the hot loop issues no shared-memory loads beside the tensor core's
  // operand reads. The CTA is 4 whole warpgroups (two idle warps complete the last one) launched
  // at kRegLaunch registers per thread; after set-up the two epilogue warpgroups take kRegEpi
  // and the other two give up to kRegOther (setmaxnreg; 2 * kRegLaunch = kRegEpi + kRegOther, so
  // the exchange always completes), and before the end-of-kernel selection all return to
  // kRegLaunch. The debug export keeps the shared-memory weights: it runs the same arithmetic.
  static constexpr bool kRegW = NQ == 4 && !DENSE;
  static constexpr int kRegLaunch = 128, kRegEpi = 168, kRegOther = 88;
  static_assert(kRegEpi + kRegOther == 2 * kRegLaunch, "register exchange is balanced");
  static constexpr int kWarps = kRegW ? 16 : kEpiWarps + 2 + kSelectors;
  static_assert(!kRegW || kWarps >= kEpiWarps + 2 + kSelectors, "every role has a warp");
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
  static constexpr int kNumBars = 2 * kStages + 2 * kAccBufs + 2 * kScoreBufs + 2;
  static constexpr int kMiscBytes = 160;
  // mbarrier waits of one-query CTAs suspend (most warps wait while the epilogue works).
  static constexpr uint32_t kWaitHint = NQ == 1 ? 20000u : 0u;
  // Buffered selection (one-query CTAs whose key split fits): the epilogue keeps every fp32
  // score of the split, counts the keys that reach a running cut bin per bin (16-bit counters)
  // and lists their offsets and bins (one list per epilogue warp), while a selector warp raises
  // the cut; the final selection reads them back (finish_hist). These overlay the selector
  // histograms, the ring and the pools, which that mode leaves unused, plus whatever shared
  // memory is left.
  static constexpr bool kHistSel = NQ == 1 && !DENSE;
  static constexpr int kBinsBytes = kHBins * 2 + (kHBins / 32) * 4;  // bins, then 32-bin groups
  // Candidates per epilogue warp: each entry holds the key's offset in the split (low 16 bits)
  // and its bin (high 16 bits), so the final filter by the exact cut reads nothing else.
  static constexpr int kCandSeg = 512;
  static constexpr int kCandBytes = kHistSel ? kEpiWarps * kCandSeg * 4 : 0;
  static constexpr int kBufTiles =
      kHistSel ? (232448 - 1024 - kMiscBytes - kNumBars * 8 - kOffHist - kBinsBytes - kCandBytes) /
                     (kTileKeys * 4)
               : 0;
  static_assert(kBufTiles * kTileKeys <= 65536, "16-bit candidate offsets");
  static constexpr int kOffBins = kOffHist;
  static constexpr int kOffCand = kOffBins + kBinsBytes;
  static constexpr int kOffBuf = kOffCand + kCandBytes;
  static constexpr int kBufEnd = kHistSel ? kOffBuf + kBufTiles * kTileKeys * 4 : 0;
  static constexpr int kOffBar = kOffSelEnd > kBufEnd ? kOffSelEnd : kBufEnd;
  static_assert(!kHistSel || kOffBar - kOffHist >= RankArea::kBytes, "slot merge area");
  static_assert(!kHistSel || kStages * kKBytes >= RankArea::kBytes, "final ranking area");
  static_assert(4 * kTopK * 8 <= kStages * kKBytes, "split merge reuses the K stages");
  static_assert((kStages * kKBytes / 8 - 2 * kTopK) / kTopK >= 2, "split merge needs two lists per round");
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;  // + alignment slack
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

// The weighted head sum of one query for one key, sum_j w_j * max(0, x_j), accumulated four
// heads at a time in packed fp32x2 FMAs. FP8 scoring applies the ReLU directly (a max per head on
// the ALU pipe beside a packed FMA per two heads). bf16 scoring, whose epilogue runs beside a
// tensor core that is busier per key, uses max(0, x) = (x + |x|) / 2 and accumulates w.x and
// w.|x| separately, all on the FMA pipe: the same value up to fp32 rounding of the two sums.
// Every kernel of a dtype (Top-k and dense debug) uses the same helper, so their scores agree
// bit for bit.
template <int DT>
struct HeadSum {
  uint64_t a = 0ull, b = 0ull, c = 0ull, d = 0ull;
  __device__ __forceinline__ void add4(const uint32_t* r, float w0, float w1, float w2, float w3) {
    const float x0 = __uint_as_float(r[0]), x1 = __uint_as_float(r[1]);
    const float x2 = __uint_as_float(r[2]), x3 = __uint_as_float(r[3]);
    const uint64_t w01 = pack_f32x2(w0, w1), w23 = pack_f32x2(w2, w3);
    if constexpr (DT == kDtFp8) {
      a = fma_f32x2(pack_f32x2(fmaxf(x0, 0.f), fmaxf(x1, 0.f)), w01, a);
      b = fma_f32x2(pack_f32x2(fmaxf(x2, 0.f), fmaxf(x3, 0.f)), w23, b);
    } else {
      a = fma_f32x2(pack_f32x2(x0, x1), w01, a);
      b = fma_f32x2(pack_f32x2(fabsf(x0), fabsf(x1)), w01, b);
      c = fma_f32x2(pack_f32x2(x2, x3), w23, c);
      d = fma_f32x2(pack_f32x2(fabsf(x2), fabsf(x3)), w23, d);
    }
  }
  // The sum, and the accumulators cleared for the next query.
  __device__ __forceinline__ float take() {
    float a0, a1, b0, b1;
    unpack_f32x2(a, a0, a1);
    unpack_f32x2(b, b0, b1);
    float s = (a0 + a1) + (b0 + b1);
    if constexpr (DT != kDtFp8) {
      float c0, c1, d0, d1;
      unpack_f32x2(c, c0, c1);
      unpack_f32x2(d, d0, d1);
      s = 0.5f * (s + ((c0 + c1) + (d0 + d1)));
    }
    a = b = c = d = 0ull;
    return s;
  }
};

// Bucket positions for a bin-grouped slot list (one warp): bucket r < nb holds bin whi - r, the
// last bucket (r = nb) every word below the window. cur[r] receives the number of words in
// buckets before r; cnt(bin) gives the exact count of each window bin.
template <class Cnt>
__device__ __forceinline__ void slot_bucket_starts(const Cnt cnt, uint32_t whi, int nb,
                                                   uint32_t* cur, int lane) {
  uint32_t acc = 0u;
  for (int r0 = 0; r0 < nb; r0 += 32) {
    const int r = r0 + lane;
    const uint32_t c = r < nb ? cnt(whi - static_cast<uint32_t>(r)) : 0u;
    uint32_t s = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += v;
    }
    if (r < nb) cur[r] = acc + s - c;
    acc += __shfl_sync(0xffffffffu, s, 31);
  }
  if (lane == 0) cur[nb] = acc;
}

// Publishes cnt (<= 512) words as a one-query split's slot, grouped by bin, with a histogram
// window counted from the words themselves (the 256 bins up to the highest bin present).
// `tmp`: 2 * 257 words of shared scratch.
template <int NT>
__device__ void publish_slot(uint64_t* slot, const uint64_t* words, int cnt, uint32_t* tmp,
                             uint32_t* scratch, int warp, int lane) {
  uint32_t* counts = tmp;        // [256]
  uint32_t* cur = tmp + 257;     // [257]
  if (threadIdx.x == 0) scratch[0] = 0u;
  for (int i = threadIdx.x; i < kSlotHistBins; i += NT) counts[i] = 0u;
  __syncthreads();
  uint32_t mb = 0u;
  for (int i = threadIdx.x; i < cnt; i += NT) mb = max(mb, hbin(words[i]));
  mb = __reduce_max_sync(0xffffffffu, mb);
  if (lane == 0 && mb) atomicMax(&scratch[0], mb);
  __syncthreads();
  const uint32_t hi = scratch[0];
  const uint32_t lo = hi >= kSlotHistBins - 1 ? hi - (kSlotHistBins - 1) : 0u;
  const int nb = cnt > 0 ? static_cast<int>(hi - lo) + 1 : 0;
  for (int i = threadIdx.x; i < cnt; i += NT) {
    const uint32_t bn = hbin(words[i]);
    if (bn >= lo) atomicAdd(&counts[bn - lo], 1u);
  }
  __syncthreads();
  if (warp == 0) slot_bucket_starts(Hist32{counts}, hi - lo, nb, cur, lane);  // bins as offsets
  __syncthreads();
  for (int i = threadIdx.x; i < cnt; i += NT) {
    const uint64_t u = words[i];
    const uint32_t bn = hbin(u);
    const int r = bn >= lo ? static_cast<int>(hi - bn) : nb;
    slot[kSlotListOff + atomicAdd(&cur[r], 1u)] = u;
  }
  uint32_t* sh = reinterpret_cast<uint32_t*>(slot + kSlotHdrWords);
  for (int i = threadIdx.x; i < nb; i += NT) sh[i] = counts[i];
  if (threadIdx.x == 0)
    slot[0] = static_cast<uint64_t>(cnt) | (static_cast<uint64_t>(lo) << 32) |
              (static_cast<uint64_t>(nb) << 48);
  __syncthreads();
}

// CTA-wide finish (split plans, and one-query CTAs whose selector warps keep separate pools):
// for each query, the unused tails of its pools are zeroed (a CTA-wide select ignores zero
// words), the 512 best words are radix-selected with all warps, and then either published
// unordered as this split's list or sorted once and written as the output row.
template <class C>
__device__ void finish_cta_select(const KParams& p, const SeqDesc& sd, int64_t t0, int split,
                                  uint64_t* pools, const uint32_t* pool_n, uint64_t* stage,
                                  uint32_t* hist, uint32_t* scratch, int warp, int lane) {
  constexpr int R = kTopK / 32;
  constexpr int kWords = C::kSelPerQuery * C::kPool;
  for (int q = 0; q < C::kN / kHeads; ++q) {
    const int64_t t = t0 + q;
    if (t >= sd.T) break;
    uint64_t* base = pools + q * kWords;
    for (int sw = 0; sw < C::kSelPerQuery; ++sw) {
      const int used = static_cast<int>(pool_n[q * C::kSelPerQuery + sw]);
      for (int i = used + threadIdx.x; i < C::kPool; i += C::kThreads) base[sw * C::kPool + i] = 0ull;
    }
    __syncthreads();
    const int cnt = cta_select<kTopK, C::kThreads>(base, kWords, stage, hist, scratch);
    const int64_t row = sd.q_row0 + t;
    if (sd.n_splits > 1) {
      if constexpr (C::kHistSel) {
        publish_slot<C::kThreads>(p.partial + sd.list0 + (t * sd.n_splits + split) * kSlotWords,
                                  stage, cnt, hist, scratch, warp, lane);
      } else {
        uint64_t* dst = p.partial + sd.list0 + (t * sd.n_splits + split) * kTopK;
        for (int i = threadIdx.x; i < kTopK; i += C::kThreads) dst[i] = i < cnt ? stage[i] : 0ull;
      }
    } else if (warp == 0) {
      uint64_t v[R];
#pragma unroll
      for (int r = 0; r < R; ++r) v[r] = lane * R + r < cnt ? stage[lane * R + r] : 0ull;
      warp_sort_desc<R>(v, lane);
      write_output<R>(p, row, v, lane);
    }
    __syncthreads();
  }
  // Lists are made visible GPU-wide by the ticket's fence (thread 0, after a CTA barrier);
  // this orders the generic-proxy writes before the bulk copies that will read them.
  if (sd.n_splits > 1) fence_proxy_async_global();
}

// Writes the (up to) 512 best of the distinct words in ra.sv[0..n) (n <= kSurvCap) whose bins lie
// in [lo, hi] (others, such as zero padding, are skipped) as output row `row`, best first; hi - lo
// < kRankBins. Words are bucketed by their bin refined with e more bits of the code (e as large as
// kRankBins buckets allow); a counting sort over the buckets (best first, CTA-wide suffix scan)
// gives each bucket its range of positions, and a word's final position is its bucket's first
// position plus the number of larger words in the same bucket (buckets hold a few words). Buckets
// that start at or after position 512 are not ranked.
template <int NT>
__device__ void rank_write(const KParams& p, int64_t row, const RankArea& ra, int n, uint32_t lo,
                           uint32_t hi, int warp, int lane) {
  constexpr int kWarps = NT / 32;
  static_assert(kWarps + 1 <= 256 && kWarps <= 32,
                "per-warp sums fit the radix scratch and one warp");
  int e = 0;
  while (e < 20 && ((static_cast<int>(hi - lo) + 1) << (e + 1)) <= kRankBins) ++e;
  const int range = (static_cast<int>(hi - lo) + 1) << e;
  const int shift = 52 - e;
  const uint64_t base = static_cast<uint64_t>(lo) << e;
  auto in_range = [&](uint64_t u) {
    const uint32_t bn = hbin(u);
    return u != 0ull && bn >= lo && bn <= hi;
  };
  auto bucket = [&](uint64_t u) { return static_cast<int>((u >> shift) - base); };
  for (int i = threadIdx.x; i < range; i += NT) ra.cnt[i] = 0u;
  __syncthreads();
  // Counting also hands each word its slot within its bucket (kept in registers for the
  // scatter below).
  constexpr int kIter = (kSurvCap + NT - 1) / NT;
  uint32_t slot_in[kIter];
#pragma unroll
  for (int j = 0; j < kIter; ++j) {
    const int i = static_cast<int>(threadIdx.x) + j * NT;
    slot_in[j] = 0u;
    if (i < n) {
      const uint64_t u = ra.sv[i];
      if (in_range(u)) slot_in[j] = atomicAdd(&ra.cnt[bucket(u)], 1u);
    }
  }
  __syncthreads();
  // off[r] = words in buckets above r. Thread t owns the buckets v = t*per .. t*per+per-1 counted
  // from the top (r = range-1-v); a block-wide exclusive prefix of the per-thread sums follows.
  const int per = (range + NT - 1) / NT;
  const int v0 = static_cast<int>(threadIdx.x) * per;
  uint32_t own = 0u;
  for (int v = v0; v < v0 + per && v < range; ++v) own += ra.cnt[range - 1 - v];
  uint32_t s = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, s, o);
    if (lane >= o) s += x;
  }
  if (lane == 31) ra.rhist[warp] = s;
  __syncthreads();
  uint32_t run = s - own + __reduce_add_sync(0xffffffffu, lane < warp ? ra.rhist[lane] : 0u);
  for (int v = v0; v < v0 + per && v < range; ++v) {
    const int r = range - 1 - v;
    ra.off[r] = run;
    run += ra.cnt[r];
  }
  if (threadIdx.x == NT - 1) ra.rhist[kWarps] = run;  // words in range
  __syncthreads();
  const int nv = static_cast<int>(ra.rhist[kWarps]);
#pragma unroll
  for (int j = 0; j < kIter; ++j) {
    const int i = static_cast<int>(threadIdx.x) + j * NT;
    if (i < n) {
      const uint64_t u = ra.sv[i];
      if (in_range(u)) ra.sorted[ra.off[bucket(u)] + slot_in[j]] = u;
    }
  }
  __syncthreads();
  int32_t* oi = p.out_idx + row * kTopK;
  float* os = p.out_score ? p.out_score + row * kTopK : nullptr;
  for (int i = threadIdx.x; i < nv; i += NT) {
    const uint64_t u = ra.sorted[i];
    const int r = bucket(u);
    const int o = static_cast<int>(ra.off[r]);
    if (o < kTopK) {
      const int end = o + static_cast<int>(ra.cnt[r]);
      int pos = o;
      for (int j = o; j < end; ++j) pos += ra.sorted[j] > u ? 1 : 0;
      if (pos < kTopK) {
        oi[pos] = key_index(u);
        if (os) os[pos] = key_score(u);
      }
    }
  }
  for (int i = nv + threadIdx.x; i < kTopK; i += NT) {
    oi[i] = -1;
    if (os) os[i] = -__int_as_float(0x7f800000);
  }
  __syncthreads();
}

// Buffered-mode words: the fp32 score of key key0 + i, packed, or 0 when the query cannot see it.
struct ScoreWords {
  const float* s;
  int64_t key0, vis_end;
  __device__ __forceinline__ uint64_t operator()(int i) const {
    const int64_t key = key0 + i;
    return key < vis_end ? pack_key(s[i], static_cast<uint32_t>(key)) : 0ull;
  }
};

// Finish of a one-query CTA in buffered mode. During the stream the epilogue kept each key's fp32
// score (sbuf) and listed, per epilogue warp, the offsets and bins of the keys whose bin reached
// the running cut bin at the time (cand, ncand) and counted them per bin (bins). Counts at or above
// the final running cut are exact, so one scan finds the exact bin b* of the 512th best word, and
// the listed keys with bin >= b* (at least 512 of them unless fewer are visible, the CTA's 512 best
// among them) are read back. A split publishes them with its count window; otherwise they are
// ranked and written. A full candidate list, or too many keys at b* (exact ties, a very flat score
// distribution), fall back to a radix select over all buffered scores.
template <class C>
__device__ void finish_hist(const KParams& p, const SeqDesc& sd, int64_t t0, int split, uint32_t* bins,
                            const uint32_t* cand, const uint32_t* ncand, const float* sbuf,
                            int n_tiles, int64_t key0, int64_t vis_end, uint32_t floor_bin,
                            uint32_t maxbin, uint64_t* stage, uint32_t* scratch, int warp,
                            int lane) {
  constexpr int NT = C::kThreads;
  constexpr int kWarps = NT / 32;
  constexpr int kSegs = C::kEpiWarps;
  const int64_t row = sd.q_row0 + t0;
  bool listed = true;
#pragma unroll
  for (int s = 0; s < kSegs; ++s) listed = listed && ncand[s] <= static_cast<uint32_t>(C::kCandSeg);
  const bool split_plan = sd.n_splits > 1;
  RankArea ra(reinterpret_cast<uint8_t*>(stage));
  // The bucket window of a published slot (from the top bin down; see below).
  auto slot_window = [&](uint32_t bs, int mm, uint32_t* wlo_out) -> int {
    const uint32_t wlo = maxbin - bs >= static_cast<uint32_t>(kSlotHistBins)
                             ? maxbin - (kSlotHistBins - 1) : bs;
    *wlo_out = wlo;
    return mm > 0 ? static_cast<int>(maxbin - wlo) + 1 : 0;
  };
  if (warp == 0) {
    uint32_t m;
    const uint32_t bs =
        warp_find_cut_grouped(kTopK, bins, bins + kHBins / 2, floor_bin, maxbin, &m, lane);
    if (lane == 0) {
      scratch[0] = bs;
      scratch[1] = m;
    }
    if (split_plan && listed && m <= static_cast<uint32_t>(kSlotListCap)) {
      // the slot's bucket starts right away (the fast split path below uses them)
      uint32_t wlo;
      const int nb = slot_window(bs, static_cast<int>(m), &wlo);
      slot_bucket_starts(Hist16{bins}, maxbin, nb, ra.cur, lane);
    }
  }
  __syncthreads();
  const uint32_t bstar = scratch[0];
  const int m = static_cast<int>(scratch[1]);
  uint64_t* slot =
      split_plan ? p.partial + sd.list0 + (t0 * sd.n_splits + split) * kSlotWords : nullptr;
  const bool fast = listed && (split_plan ? m <= kSlotListCap
                                          : (m <= kSurvCap && maxbin - bstar < kRankBins));
  // A list entry's word, or 0 when its bin lies below the exact cut.
  auto listed_word = [&](uint32_t e) -> uint64_t {
    if ((e >> 16) < bstar) return 0ull;
    const int k = static_cast<int>(e & 0xFFFFu);
    return pack_key(sbuf[k], static_cast<uint32_t>(key0 + k));
  };
  if (fast) {
    // The lists side by side: position i is entry i % kCandSeg of list i / kCandSeg.
    constexpr int kSpan = kSegs * C::kCandSeg;
    auto word_at = [&](int i) -> uint64_t {
      const int s = i / C::kCandSeg;
      if (static_cast<uint32_t>(i - s * C::kCandSeg) >= ncand[s]) return 0ull;
      return listed_word(cand[i]);
    };
    if (split_plan) {
      // Grouped by bin (window bins from the top, then the rest) straight into the slot.
      uint32_t wlo;
      const int nb = slot_window(bstar, m, &wlo);  // (bucket starts: set before the barrier)
      uint64_t* dst = slot + kSlotListOff;
      // Thread t takes entry t (then t + NT) of every list: the lists' candidates are read and
      // filtered first, then all of a thread's slot claims (shared-memory atomics) are made
      // before any is used, then the words are stored.
      uint32_t nc[kSegs];
#pragma unroll
      for (int j = 0; j < kSegs; ++j) nc[j] = min(ncand[j], static_cast<uint32_t>(C::kCandSeg));
      for (int e = threadIdx.x; e < C::kCandSeg; e += NT) {
        uint64_t u[kSegs];
        uint32_t pos[kSegs];
#pragma unroll
        for (int j = 0; j < kSegs; ++j)
          u[j] = static_cast<uint32_t>(e) < nc[j] ? listed_word(cand[j * C::kCandSeg + e]) : 0ull;
#pragma unroll
        for (int j = 0; j < kSegs; ++j) {
          pos[j] = 0u;
          if (u[j]) {
            const uint32_t bn = hbin(u[j]);
            pos[j] = atomicAdd(&ra.cur[bn >= wlo ? static_cast<int>(maxbin - bn) : nb], 1u);
          }
        }
#pragma unroll
        for (int j = 0; j < kSegs; ++j)
          if (u[j] && pos[j] < static_cast<uint32_t>(kSlotListCap)) dst[pos[j]] = u[j];  // m fits
      }
      uint32_t* sh = reinterpret_cast<uint32_t*>(slot + kSlotHdrWords);
      for (int i = threadIdx.x; i < nb; i += NT) sh[i] = Hist16{bins}(wlo + i);
      if (threadIdx.x == 0)
        slot[0] = static_cast<uint64_t>(m) | (static_cast<uint64_t>(wlo) << 32) |
                  (static_cast<uint64_t>(nb) << 48);
      __syncthreads();
    } else {
      // Two passes over a stripe per warp (count, then write at the warp's offset) into sv.
      constexpr int kPerWarp = (kSpan + kWarps - 1) / kWarps;
      const int lo = warp * kPerWarp, hi = lo + kPerWarp < kSpan ? lo + kPerWarp : kSpan;
      const uint32_t lt_mask = (1u << lane) - 1u;
      uint32_t cnt = 0u;
      for (int x = lo; x < hi; x += 32) {
        const uint64_t u = x + lane < hi ? word_at(x + lane) : 0ull;
        cnt += __popc(__ballot_sync(0xffffffffu, u != 0ull));
      }
      uint32_t* wcnt = ra.rhist;  // not part of sv
      if (lane == 0) wcnt[warp] = cnt;
      __syncthreads();
      uint32_t at = 0u;
      for (int w = 0; w < warp; ++w) at += wcnt[w];
      for (int x = lo; x < hi; x += 32) {
        const uint64_t u = x + lane < hi ? word_at(x + lane) : 0ull;
        const uint32_t km = __ballot_sync(0xffffffffu, u != 0ull);
        const uint32_t pos = at + __popc(km & lt_mask);
        if (u && pos < static_cast<uint32_t>(kSurvCap)) ra.sv[pos] = u;  // m <= kSurvCap words
        at += __popc(km);
      }
      __syncthreads();
      rank_write<NT>(p, row, ra, m, bstar, maxbin, warp, lane);
    }
  } else {
    constexpr int kStageWords = C::kStages * C::kKBytes / 8;
    uint32_t* hist = bins;  // the counts are no longer needed
    const int cnt = cta_select_sampled<kTopK, NT>(ScoreWords{sbuf, key0, vis_end},
                                                  n_tiles * kTileKeys, stage, stage + kTopK,
                                                  kStageWords - kTopK, hist, scratch);
    if (split_plan) {
      publish_slot<NT>(slot, stage, cnt, hist, scratch, warp, lane);
    } else {
      constexpr int R = kTopK / 32;
      if (warp == 0) {
        uint64_t v[R];
#pragma unroll
        for (int r = 0; r < R; ++r) v[r] = lane * R + r < cnt ? stage[lane * R + r] : 0ull;
        warp_sort_desc<R>(v, lane);
        write_output<R>(p, row, v, lane);
      }
      __syncthreads();
    }
  }
  // The slot is made visible GPU-wide by the ticket's fence (thread 0, after a CTA barrier);
  // this orders the generic-proxy writes before the bulk copies that will read them.
  if (split_plan) fence_proxy_async_global();
}

// One-query split plans, part 2 (the CTA that takes the last ticket). One bulk copy per split
// brings its header and count window into shared memory; the windows are summed into one
// histogram, whose scan gives the highest bin G that at least 512 published words reach (the
// 512th best word overall lies in G or above). Each list is grouped by bin, so its words at or
// above G are a prefix whose length its window gives (a whole list when G lies below its
// window). The first round also brought each list's first words, which usually hold those
// prefixes; otherwise a second round of bulk copies brings them. rank_write orders the words
// with bin >= G. More of them than the ranking takes fall back to a radix select over all
// lists and one CTA-wide sort.
template <class C>
__device__ void merge_hist_slots(const KParams& p, const SeqDesc& sd, int64_t t0, uint64_t* buf,
                                 uint8_t* area, uint64_t* gbar, volatile uint32_t* abort_flag,
                                 uint32_t* scratch, int warp, int lane) {
  constexpr int NT = C::kThreads;
  constexpr int kWarps = NT / 32;
  constexpr int kCap = C::kStages * C::kKBytes / 8;  // words of the gather area
  constexpr int kHead = kSlotListOff;                // header + window words of a slot
  // The first round of copies also brings the first kPre words of each list: when every
  // list's words at or above the cut are among them (the usual case), no second round is needed.
  constexpr int kPre = 64;
  constexpr int kRound1 = kHead + kPre;
  static_assert(64 * kRound1 <= kCap && kRound1 <= kSlotWords && kRound1 % 2 == 0,
                "every split's header, window and first words fit at once");
  static_assert(kWarps <= 32, "one lane per warp in the slice scan");
  const RankArea ra(area);
  uint32_t* mh = ra.cnt;      // summed window counts of bins top, top - 1, .. (cnt, off, cur)
  static_assert(3 * kRankBins >= kHBins, "summed windows fit");
  uint32_t* hm = ra.hdr;      // [64] list sizes
  uint32_t* hlo = hm + 64;    // [64] window starts
  uint32_t* hnb = hlo + 64;   // [64] window widths
  uint32_t* hn = hnb + 64;    // [64] words to take from each list
  uint32_t* hpre = hn + 64;   // [65] their offsets in sv (rounded up to even)
  const int ns = sd.n_splits;
  const int64_t row = sd.q_row0 + t0;
  const uint64_t* slots = p.partial + sd.list0 + t0 * ns * kSlotWords;
  fence_proxy_async_smem();  // earlier generic accesses to the copy targets precede the copies
  __syncthreads();
  if (warp == 0) {
    if (lane == 0) mbar_arrive_expect_tx(gbar, static_cast<uint32_t>(ns * kRound1 * 8));
    __syncwarp();
    fence_proxy_async_global();  // the slots published by other CTAs, seen by the copies
    for (int i = lane; i < ns; i += 32)
      bulk_load(buf + i * kRound1, slots + static_cast<int64_t>(i) * kSlotWords, kRound1 * 8, gbar);
  }
  // CTA-uniform outcome: a thread may see the copies land while another gives up.
  if (!__syncthreads_and(mbar_wait(gbar, 0u, abort_flag, p.err, p.wait_ns))) {
    mbar_drain(gbar, 0u);  // never exit with copies in flight
    return;
  }
  for (int i = threadIdx.x; i < ns; i += NT) {
    const uint64_t h = buf[i * kRound1];
    const uint32_t m = static_cast<uint32_t>(h);
    const uint32_t lo = static_cast<uint32_t>(h >> 32) & 0xFFFFu;
    const uint32_t nb = static_cast<uint32_t>(h >> 48);
    hm[i] = m < static_cast<uint32_t>(kSlotListCap) ? m : static_cast<uint32_t>(kSlotListCap);
    hlo[i] = lo;
    hnb[i] = (nb <= static_cast<uint32_t>(kSlotHistBins) && lo + nb <= static_cast<uint32_t>(kHBins)) ? nb : 0u;
  }
  __syncthreads();
  // The counted range [bottom, top] (every warp finds it). Thread t sums the windows over its
  // slice of `per` bins from the top down (no atomics); a CTA-wide scan of the slice totals
  // then shows the slice, and the bin, where the count from the top first reaches 512.
  uint32_t top = 0u, bottom = kHBins - 1;
  for (int i = lane; i < ns; i += 32)
    if (hnb[i]) {
      top = max(top, hlo[i] + hnb[i] - 1u);
      bottom = min(bottom, hlo[i]);
    }
  top = __reduce_max_sync(0xffffffffu, top);
  bottom = __reduce_min_sync(0xffffffffu, bottom);
  bottom = bottom < top ? bottom : top;  // lowest counted bin (top itself when nothing counted)
  const int per = (static_cast<int>(top - bottom) + NT) / NT;
  const int r0 = static_cast<int>(threadIdx.x) * per;  // offsets below top: bins top - r
  const int r1 = min(r0 + per, static_cast<int>(top - bottom) + 1);
  uint32_t own = 0u;
  for (int r = r0; r < r1; ++r) {
    const uint32_t bin = top - static_cast<uint32_t>(r);
    uint32_t c = 0u;
#pragma unroll 4
    for (int i = 0; i < ns; ++i) {
      const uint32_t k = bin - hlo[i];  // wraps above hnb when bin < hlo
      if (k < hnb[i]) c += reinterpret_cast<const uint32_t*>(buf + i * kRound1 + kSlotHdrWords)[k];
    }
    mh[r] = c;
    own += c;
  }
  uint32_t incl = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  uint32_t* wsum = ra.rhist;  // [kWarps] slice totals per warp
  if (lane == 31) wsum[warp] = incl;
  if (threadIdx.x == 0) {
    scratch[0] = 0u;  // G = 0 (every published word stays) unless some bin reaches 512
    scratch[1] = top;
  }
  __syncthreads();
  const uint32_t above =
      incl - own + __reduce_add_sync(0xffffffffu, lane < warp ? wsum[lane] : 0u);
  if (above < static_cast<uint32_t>(kTopK) && above + own >= static_cast<uint32_t>(kTopK)) {
    uint32_t run = above;  // exactly one thread crosses 512 inside its slice
    for (int r = r0; r < r1; ++r) {
      run += mh[r];
      if (run >= static_cast<uint32_t>(kTopK)) {
        scratch[0] = top - static_cast<uint32_t>(r);
        break;
      }
    }
  }
  __syncthreads();
  const uint32_t G = scratch[0], H = scratch[1];
  // Words of list i at or above G: the window's counts from G up (a prefix of the list), or
  // the whole list when G lies at or below the window's start.
  for (int i = warp; i < ns; i += kWarps) {
    uint32_t n;
    if (G <= hlo[i]) {
      n = hm[i];
    } else {
      const uint32_t* win = reinterpret_cast<const uint32_t*>(buf + i * kRound1 + kSlotHdrWords);
      uint32_t s = 0u;
      for (int k = static_cast<int>(G - hlo[i]) + lane; k < static_cast<int>(hnb[i]); k += 32) s += win[k];
      n = __reduce_add_sync(0xffffffffu, s);
      n = n < hm[i] ? n : hm[i];
    }
    if (lane == 0) hn[i] = n;
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t acc = 0u;
    bool fits = true;  // every list's words at or above G came with the first round
    for (int i0 = 0; i0 < ns; i0 += 32) {
      const int i = i0 + lane;
      fits = __all_sync(0xffffffffu, i >= ns || hn[i] <= static_cast<uint32_t>(kPre)) && fits;
      const uint32_t sz = i < ns ? (hn[i] + 1u) & ~1u : 0u;
      uint32_t s = sz;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += v;
      }
      if (i < ns) hpre[i] = acc + s - sz;
      acc += __shfl_sync(0xffffffffu, s, 31);
    }
    if (lane == 0) {
      hpre[ns] = acc;
      scratch[2] = fits ? 1u : 0u;
    }
  }
  __syncthreads();  // sv took no generic accesses since the fence above: no second fence
  const int total = static_cast<int>(hpre[ns]);
  if (total <= kSurvCap && H - G < static_cast<uint32_t>(kRankBins) && scratch[2]) {
    for (int i = warp; i < ns; i += kWarps) {  // the prefixes, from the first round's copies
      const uint64_t* src = buf + i * kRound1 + kHead;
      const uint32_t n = hn[i], sz = (n + 1u) & ~1u;
      for (uint32_t k = lane; k < sz; k += 32) ra.sv[hpre[i] + k] = k < n ? src[k] : 0ull;
    }
    __syncthreads();
    rank_write<NT>(p, row, ra, total, G, H, warp, lane);
    return;
  }
  if (total <= kSurvCap && H - G < static_cast<uint32_t>(kRankBins)) {
    if (warp == 0) {
      if (lane == 0) mbar_arrive_expect_tx(gbar, static_cast<uint32_t>(total) * 8u);
      __syncwarp();
      for (int i = lane; i < ns; i += 32) {
        const uint32_t sz = (hn[i] + 1u) & ~1u;
        if (sz)
          bulk_load(ra.sv + hpre[i], slots + static_cast<int64_t>(i) * kSlotWords + kSlotListOff,
                    sz * 8u, gbar);
      }
    }
    if (!__syncthreads_and(mbar_wait(gbar, 1u, abort_flag, p.err, p.wait_ns))) {
      mbar_drain(gbar, 1u);
      return;
    }
    for (int i = threadIdx.x; i < ns; i += NT)
      if (hn[i] & 1u) ra.sv[hpre[i] + hn[i]] = 0ull;  // an odd prefix's padding word
    __syncthreads();
    rank_write<NT>(p, row, ra, total, G, H, warp, lane);
    return;
  }
  // Rare: too many published words at the cut bin. Exact radix selection over every list,
  // folded whenever the gather area would overflow, then one CTA-wide sort.
  uint64_t* sel = ra.sorted;
  int n = 0;
  for (int i = 0; i < ns; ++i) {
    if (n + kSlotListCap > kCap) {
      const int k = cta_select<kTopK, NT>(buf, n, sel, ra.rhist, scratch);
      for (int x = threadIdx.x; x < k; x += NT) buf[x] = sel[x];
      __syncthreads();
      n = k;
    }
    const uint64_t* src = slots + static_cast<int64_t>(i) * kSlotWords + kSlotListOff;
    for (int x = threadIdx.x; x < static_cast<int>(hm[i]); x += NT) buf[n + x] = src[x];
    __syncthreads();
    n += static_cast<int>(hm[i]);
  }
  const int cnt = cta_select<kTopK, NT>(buf, n, sel, ra.rhist, scratch);
  for (int x = cnt + threadIdx.x; x < kTopK; x += NT) sel[x] = 0ull;
  __syncthreads();
  cta_sort_desc<kTopK, NT>(sel);
  for (int i = threadIdx.x; i < kTopK; i += NT) {
    const uint64_t u = sel[i];
    p.out_idx[row * kTopK + i] = u ? key_index(u) : -1;
    if (p.out_score) p.out_score[row * kTopK + i] = u ? key_score(u) : -__int_as_float(0x7f800000);
  }
  __syncthreads();
}

// Split plans, part 2 (the CTA that takes a block's last ticket): copy every split's list of
// each query into shared memory with independent wide loads, radix-select the 512 best, sort
// them once in registers and write the output row. Lists that do not fit at once are folded in
// rounds (the 512 survivors of a round stay at the front of the gather area).
template <class C>
__device__ void merge_split_lists(const KParams& p, const SeqDesc& sd, int64_t t0, uint64_t* stage,
                                  uint32_t* hist, uint32_t* scratch, int warp, int lane) {
  constexpr int kStageWords = C::kStages * C::kKBytes / 8;
  constexpr int kCap = kStageWords - kTopK;  // gather area; the last 512 words receive selects
  constexpr int kListsPerRound = (kCap - kTopK) / kTopK;
  uint64_t* sel = stage + kCap;
  for (int q = 0; q < C::kN / kHeads; ++q) {
    const int64_t t = t0 + q;
    if (t >= sd.T) break;
    const int64_t row = sd.q_row0 + t;
    const uint64_t* lists = p.partial + sd.list0 + t * sd.n_splits * kTopK;
    int n = 0;  // words already in the gather area (survivors of earlier rounds)
    for (int sp0 = 0; sp0 < sd.n_splits; sp0 += kListsPerRound) {
      const int nl = sd.n_splits - sp0 < kListsPerRound ? sd.n_splits - sp0 : kListsPerRound;
      const uint4* src = reinterpret_cast<const uint4*>(lists + static_cast<int64_t>(sp0) * kTopK);
      uint4* dst = reinterpret_cast<uint4*>(stage + n);
      const int n4 = nl * kTopK / 2;
#pragma unroll 8
      for (int i = threadIdx.x; i < n4; i += C::kThreads) dst[i] = src[i];
      __syncthreads();
      n += nl * kTopK;
      if (sp0 + nl < sd.n_splits) {  // another round follows: keep only the 512 best
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
  // buffered mode only: scores, candidate offsets, per-bin counts
  float* sBuf = reinterpret_cast<float*>(smem + C::kOffBuf);
  uint32_t* s_cand = reinterpret_cast<uint32_t*>(smem + C::kOffCand);
  uint32_t* s_bins = reinterpret_cast<uint32_t*>(smem + C::kOffBins);
  uint32_t* s_grp = s_bins + kHBins / 2;  // 32-bin group counts
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
  uint64_t* gbar = qfull + 1;                       // slot merge: bulk copies landed
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile uint32_t* s_abort = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 4);
  volatile uint32_t* s_last = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 8);
  uint32_t* s_scratch = reinterpret_cast<uint32_t*>(smem + C::kOffMisc + 16);  // 8 words
  uint32_t* s_pool_n = reinterpret_cast<uint32_t*>(smem + C::kOffMisc + 48);   // [selectors]
  // Running threshold published by each selector warp (only rises): a query's warps filter
  // against the largest of them, which is still at most the CTA's exact 512th best.
  volatile uint64_t* s_theta = reinterpret_cast<volatile uint64_t*>(smem + C::kOffMisc + 64);
  // Buffered mode: running cut bin (only rises), the highest candidate bin, and the number of
  // candidates each epilogue warp listed.
  uint32_t* s_cut = reinterpret_cast<uint32_t*>(smem + C::kOffMisc + 96);
  uint32_t* s_maxbin = reinterpret_cast<uint32_t*>(smem + C::kOffMisc + 100);
  uint32_t* s_ncand = reinterpret_cast<uint32_t*>(smem + C::kOffMisc + 104);  // [kEpiWarps]
  // The cut as a score threshold (bin_floor_score of the cut bin, or lower while it catches up).
  float* s_cutf = reinterpret_cast<float*>(smem + C::kOffMisc + 136);
  // Set by the TMA producer once it has issued its last tile (the shared-cut loop stops).
  volatile uint32_t* s_stream_done = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 140);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: longest query blocks first, key splits innermost. Uniform calls interleave
  // the sequences (CTA i serves sequence i % B); otherwise each sequence owns a CTA range.
  const int wid = blockIdx.x;
  int b, rest;
  if (p.uniform) {
    b = wid % p.B;
    rest = wid / p.B;
  } else {
    b = 0;
    while (b + 1 < p.B && p.seq[b + 1].cta0 <= wid) ++b;
    rest = wid - p.seq[b].cta0;
  }
  const SeqDesc sd = p.seq[b];  // this sequence's fields, in registers
  const bool paged = p.page_table != nullptr;
  const int split = rest % sd.n_splits;
  const int qb = sd.n_qb - 1 - rest / sd.n_splits;
  const int64_t t0 = static_cast<int64_t>(qb) * NQ;
  const int64_t t_last = (t0 + NQ < sd.T ? t0 + NQ : sd.T) - 1;
  const int64_t pos_b = sd.pos;
  const int64_t S_b = sd.S;
  int tile_lo, n_tiles;
  if (DENSE) {
    tile_lo = 0;
    n_tiles = static_cast<int>((S_b + kTileKeys - 1) / kTileKeys);
  } else {
    const int64_t p_last = pos_b + t_last;
    const int64_t vis_end = (p_last < S_b - 1 ? p_last : S_b - 1) + 1;
    const int tiles_total = static_cast<int>((vis_end + kTileKeys - 1) / kTileKeys);
    tile_lo = split * sd.tiles_per_split;
    const int hi = tile_lo + sd.tiles_per_split < tiles_total ? tile_lo + sd.tiles_per_split
                                                               : tiles_total;
    n_tiles = hi > tile_lo ? hi - tile_lo : 0;
  }

  const bool buffered = C::kBufTiles > 0 && n_tiles <= C::kBufTiles;
  // Keys a one-query CTA's query can see: [0, vis_q).
  const int64_t vis_q = (pos_b + t0 < S_b - 1 ? pos_b + t0 : S_b - 1) + 1;

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
    mbar_init(gbar, 1);
    *s_abort = 0u;
    for (int i = 0; i < C::kSelectors; ++i) s_theta[i] = 0ull;
    *s_cut = 0u;
    *s_cutf = bin_floor_score(0u);
    *s_maxbin = 0u;
    *s_stream_done = 0u;
    fence_mbar_init();
  }
  if (buffered)
    for (int i = threadIdx.x; i < C::kBinsBytes / 4; i += C::kThreads) s_bins[i] = 0u;
  if (warp == C::kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tmap_q);
    tma_prefetch_desc(&tmap_k);
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(s_tmem, C::kTmemCols);
    tmem_relinquish();
  }
  // Everything above touches only this CTA's resources; global memory waits for the previous
  // kernel in the stream (a no-op unless launched as its programmatic dependent).
  griddep_wait();
  for (int i = threadIdx.x; i < NQ * kHeads; i += C::kThreads) {
    const int64_t t = t0 + i / kHeads;
    sW[i] = t < sd.T ? p.w[(sd.q_row0 + t) * kHeads + (i % kHeads)] : 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  // ---- warp roles
  auto tma_role = [&]() {
    // ================= TMA producer
    if (lane == 0 && n_tiles > 0) {
      mbar_arrive_expect_tx(qfull, C::kQBytes);
      for (int h = 0; h < C::kHalves; ++h)
        tma_load_3d(sQ + h * (C::kN * 128), &tmap_q, qfull, h * 64 * (DT == kDtBf16 ? 1 : 2),
                    static_cast<int32_t>((sd.q_row0 + t0) * kHeads), 0);
      int it = 0;
      for (; it < n_tiles; ++it) {
        const int st = it % C::kStages;
        const uint32_t ph = (it / C::kStages) & 1;
        if (!mbar_wait<C::kWaitHint>(&empty[st], ph ^ 1u, s_abort, p.err, p.wait_ns)) break;
        mbar_arrive_expect_tx(&full[st], C::kKBytes);
        uint8_t* dst = sK + st * C::kKBytes;
        const int64_t key0 = static_cast<int64_t>(tile_lo + it) * kTileKeys;
        if (!paged) {
          // contiguous pool: one 128-row box per swizzle column (rows past the pool read 0)
          const int32_t row = static_cast<int32_t>(sd.k_row0 + key0);
          for (int h = 0; h < C::kHalves; ++h)
            tma_load_3d(dst + h * (kTileKeys * 128), &tmap_k, &full[st],
                        h * 64 * (DT == kDtBf16 ? 1 : 2), row, 0);
        } else {
          // paged pool: two 64-row boxes (a page holds a multiple of 64 keys); a box past the
          // sequence's keys reads rows past the pool, which load as zeros
          for (int sub = 0; sub < 2; ++sub) {
            const int64_t key = key0 + sub * 64;
            const int32_t row = static_cast<int32_t>(key < S_b ? key_row(p, sd, key) : p.pool_rows);
            for (int h = 0; h < C::kHalves; ++h)
              tma_load_3d(dst + h * (kTileKeys * 128) + sub * (64 * 128), &tmap_k, &full[st],
                          h * 64 * (DT == kDtBf16 ? 1 : 2), row, 0);
          }
        }
      }
      // Never leave the CTA with copies in flight: wait for the last load of each stage and
      // for the Q block, also after an abort (the waits ignore the abort flag; the copies
      // complete on their own, the limit only bounds the wait). After a normal run these have
      // long completed.
      const int issued = it;
      for (int j = issued - C::kStages > 0 ? issued - C::kStages : 0; j < issued; ++j)
        mbar_drain(&full[j % C::kStages], (j / C::kStages) & 1);
      mbar_drain(qfull, 0);
    }
    if (lane == 0) *s_stream_done = 1u;  // (also when this CTA had no tile to stream)
  };
  auto mma_role = [&]() {
    // ================= MMA issuer (one thread)
    if (lane == 0 && n_tiles > 0) {
      int it = 0;
      bool ok = mbar_wait<C::kWaitHint>(qfull, 0, s_abort, p.err, p.wait_ns);
      for (; ok && it < n_tiles; ++it) {
        const int st = it % C::kStages;
        const uint32_t sph = (it / C::kStages) & 1;
        const int acc = it % C::kAccBufs;
        const uint32_t aph = (it / C::kAccBufs) & 1;
        if (!mbar_wait<C::kWaitHint>(&full[st], sph, s_abort, p.err, p.wait_ns)) break;
        if (!mbar_wait<C::kWaitHint>(&tempty[acc], aph ^ 1u, s_abort, p.err, p.wait_ns)) break;
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
      // the last tile issued (the epilogue waits on the same phase), also after an abort.
      if (it > 0) {
        const int last = it - 1;
        mbar_drain(&tfull[last % C::kAccBufs], (last / C::kAccBufs) & 1);
      }
    }
    __syncwarp();
  };
  auto epi_role = [&]() {
    // ================= epilogue: TMEM -> ReLU . w -> per-key score
    const int quad = warp & 3;
    const int grp = warp >> 2;
    const int q0 = C::kEpiAltTiles ? 0 : grp * C::kQPerGroup;
    const int it0 = C::kEpiAltTiles ? grp : 0;   // first tile of this warp
    const int step = C::kEpiAltTiles ? 2 : 1;    // tiles between this warp's tiles
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    // FP8 key scales are read two tiles ahead so their global-memory latency stays hidden
    // (decode streams the cache once, so these reads miss in L2).
    const float* kscale_c = DT == kDtFp8 && !paged ? p.kscale + sd.k_row0 : nullptr;
    auto load_scale = [&](int tile) -> float {
      const int64_t k = static_cast<int64_t>(tile_lo + tile) * kTileKeys + quad * 32 + lane;
      if (tile >= n_tiles || k >= S_b) return 0.f;
      if (!paged) return __ldg(kscale_c + k);
      const int64_t row = key_row(p, sd, k);
      return row < p.pool_rows ? __ldg(p.kscale + row) : 0.f;
    };
    float ks_next0 = 1.f, ks_next1 = 1.f;
    float wr[C::kRegW ? C::kQPerGroup * kHeads : 1];        // the group's head weights
    if constexpr (C::kRegW) {
#pragma unroll
      for (int i = 0; i < C::kQPerGroup * kHeads; ++i) wr[i] = sW[q0 * kHeads + i];
    }
    uint32_t own_cand = 0u;                                  // buffered mode: keys listed
    uint32_t* own_list = s_cand + warp * C::kCandSeg;        // buffered mode: offsets and bins
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
      if (!mbar_wait_warp<C::kWaitHint>(&tfull[acc], aph, s_abort, p.err, p.wait_ns)) break;
      tc_fence_after();
      if (!DENSE && !buffered) {
        if (!mbar_wait_warp<C::kWaitHint>(&sempty[sb], sph ^ 1u, s_abort, p.err, p.wait_ns)) break;
      }
      if constexpr (C::kRegW) {
        // Weights in registers: 16-column TMEM chunks (8 per tile), double-buffered.
        constexpr int kChunks16 = 4 * C::kQPerGroup;
        const uint32_t col0 = tmem + lane_base + static_cast<uint32_t>(acc * C::kN + q0 * kHeads);
        uint32_t rb[2][16];
        tmem_ld16(col0, rb[0]);
        tmem_wait_ld();
        HeadSum<DT> hs;
#pragma unroll
        for (int c = 0; c < kChunks16; ++c) {
          if (c + 1 < kChunks16) tmem_ld16(col0 + 16 * (c + 1), rb[(c + 1) & 1]);
          const int lq = c / 4;  // query of the group
          const uint32_t* r = rb[c & 1];
#pragma unroll
          for (int h4 = 0; h4 < 4; ++h4) {
            const int wi = lq * kHeads + (c % 4) * 16 + 4 * h4;
            hs.add4(r + 4 * h4, wr[wi], wr[wi + 1], wr[wi + 2], wr[wi + 3]);
          }
          if (c % 4 == 3) {  // all 64 heads of query q0 + lq reduced
            float score = hs.take();
            if (DT == kDtFp8) score *= ks;
            sScore[(sb * NQ + q0 + lq) * kTileKeys + quad * 32 + lane] = score;
          }
          if (c + 1 < kChunks16) tmem_wait_ld();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&tempty[acc]);
          mbar_arrive(&sfull[sb]);
        }
        continue;
      }
      // The warp's TMEM reads are 2 * kQPerGroup chunks of 32 head columns. Chunk c+1 is
      // requested before chunk c is reduced, so each load's latency hides behind arithmetic
      // (tcgen05.wait::ld waits for all outstanding loads; two 32-register buffers suffice).
      constexpr int kChunks = 2 * C::kQPerGroup;
      const uint32_t col0 = tmem + lane_base + static_cast<uint32_t>(acc * C::kN + q0 * kHeads);
      uint32_t rb[2][32];
      tmem_ld32(col0, rb[0]);
      tmem_wait_ld();
      HeadSum<DT> hs;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        if (c + 1 < kChunks) tmem_ld32(col0 + 32 * (c + 1), rb[(c + 1) & 1]);
        const int q = q0 + c / 2;
        const float4* w4 = reinterpret_cast<const float4*>(sW + q * kHeads + (c & 1) * 32);
        const uint32_t* r = rb[c & 1];
#pragma unroll
        for (int h4 = 0; h4 < 8; ++h4) {
          const float4 wv = w4[h4];
          hs.add4(r + 4 * h4, wv.x, wv.y, wv.z, wv.w);
        }
        if (c & 1) {  // both halves of query q reduced
          float score = hs.take();
          if (DT == kDtFp8) score *= ks;
          if (DENSE) {
            const int64_t t = t0 + q;
            if (t < sd.T && key < S_b) {
              const bool vis = key <= pos_b + t;
              p.dense[t * S_b + key] = vis ? score : -__int_as_float(0x7f800000);
            }
          } else if (buffered) {
            // Running cut: a key is a candidate when its bin reaches the cut bin, which some
            // 512 candidates already reach (so the cut never passes the bin of the CTA's 512th
            // best). Candidates are counted per bin and listed; after every kRecut candidates
            // of its own a warp raises the cut from the counts (which only grow, so any value
            // read is a lower bound and the cut stays valid).
            // The test runs on the score against the cut's threshold; only kept keys are packed.
            const int k = it * kTileKeys + quad * 32 + lane;
            sBuf[k] = score;
            const bool keep = key < vis_q && score >= *reinterpret_cast<volatile float*>(s_cutf);
            const uint32_t km = __ballot_sync(0xffffffffu, keep);
            if (km) {
              const uint32_t bn = keep ? hbin(pack_key(score, static_cast<uint32_t>(key))) : 0u;
              if (keep) {
                hist16_inc(s_bins, bn);
                atomicAdd(&s_grp[bn >> 5], 1u);
                const uint32_t pos = own_cand + __popc(km & ((1u << lane) - 1u));
                if (pos < static_cast<uint32_t>(C::kCandSeg))
                  own_list[pos] = static_cast<uint32_t>(k) | (bn << 16);
              }
              const uint32_t before = own_cand;
              own_cand += static_cast<uint32_t>(__popc(km));
              const uint32_t mb = __reduce_max_sync(0xffffffffu, keep ? bn : 0u);
              if (lane == 0) atomicMax(s_maxbin, mb);
              if (own_cand / kRecut != before / kRecut) {
                __syncwarp();
                uint32_t lo = 0u, hi = 0u, cnt;
                if (lane == 0) {
                  lo = *reinterpret_cast<volatile uint32_t*>(s_cut);
                  hi = *reinterpret_cast<volatile uint32_t*>(s_maxbin);
                }
                lo = __shfl_sync(0xffffffffu, lo, 0);
                hi = __shfl_sync(0xffffffffu, hi, 0);
                const uint32_t nb =
                    warp_find_cut_grouped(kTopK, s_bins, s_grp, lo, hi >= lo ? hi : lo, &cnt, lane);
                if (lane == 0 && cnt >= static_cast<uint32_t>(kTopK) && nb > lo) {
                  const uint32_t prev = atomicMax(s_cut, nb);
                  *reinterpret_cast<volatile float*>(s_cutf) = bin_floor_score(max(prev, nb));
                }
              }
            }
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
    if (buffered && lane == 0) s_ncand[warp] = own_cand;
  };
  // A selector warp's last step (one CTA, no key split): its pool back to exactly the 512 best,
  // sorted in registers, best first, and written as the query's output row.
  auto sel_finish = [&](int sidx, int n) {
    uint64_t* pool = sPool + sidx * C::kPool;
    const int64_t t = t0 + sidx / C::kSelPerQuery;
    if (n > kTopK) n = (select_compact<kTopK>(pool, n, sHist + sidx * 256, lane), kTopK);
    __syncwarp();
    constexpr int R = kTopK / 32;
    uint64_t v[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int i = lane * R + r;
      v[r] = i < n ? pool[i] : 0ull;
    }
    warp_sort_desc<R>(v, lane);
    if (t < sd.T && !*s_abort) write_output<R>(p, sd.q_row0 + t, v, lane);
  };
  auto shared_cut_role = [&]() {
    // ================= one-query split plans: a cut shared by the sequence's splits. Each split
    // publishes a bin its k-th best key reaches (k = ceil(512 / splits); the counts only grow,
    // so a bin read from them stays valid); once every split has published, the lowest of
    // those bins is reached by at least 512 keys of the sequence, so the sequence's 512th best
    // lies at or above it, and this split's running cut is raised to it: fewer keys are listed
    // and published. Counts at or above the final cut stay exact, which the merge relies on.
    const int ns = sd.n_splits;
    const uint32_t k = static_cast<uint32_t>((kTopK + ns - 1) / ns);
    uint32_t* pub = p.counters + kCounterWords * (sd.ticket0 + qb) + 1;  // [ns]: bin + 1, 0 = none
    uint32_t published = 0u;
    const uint64_t t_start = globaltimer_ns();
    // (bounded like every wait here: it also ends after the kernel's wait limit)
    while (!*s_stream_done && !*s_abort && globaltimer_ns() - t_start < p.wait_ns) {
      __nanosleep(1000);
      uint32_t lo = 0u, hi = 0u, cnt;
      if (lane == 0) {
        lo = *reinterpret_cast<volatile uint32_t*>(s_cut);
        hi = *reinterpret_cast<volatile uint32_t*>(s_maxbin);
      }
      lo = __shfl_sync(0xffffffffu, lo, 0);
      hi = __shfl_sync(0xffffffffu, hi, 0);
      const uint32_t b = warp_find_cut_grouped(k, s_bins, s_grp, lo, hi >= lo ? hi : lo, &cnt, lane);
      if (lane == 0 && cnt >= k && b + 1u > published) {
        published = b + 1u;
        *reinterpret_cast<volatile uint32_t*>(pub + split) = published;
      }
      uint32_t low = 0xFFFFFFFFu;
      for (int i = lane; i < ns; i += 32)
        low = min(low, *reinterpret_cast<volatile uint32_t*>(pub + i));
      low = __reduce_min_sync(0xffffffffu, low);
      if (lane == 0 && low > 0u && low - 1u > *reinterpret_cast<volatile uint32_t*>(s_cut)) {
        const uint32_t prev = atomicMax(s_cut, low - 1u);
        *reinterpret_cast<volatile float*>(s_cutf) = bin_floor_score(max(prev, low - 1u));
      }
    }
  };
  auto sel_role = [&]() {
    // ================= selectors
    if (buffered) {
      if (sd.n_splits > 1 && warp == C::kSelWarp0) shared_cut_role();
      return;
    }
    const int sidx = warp - C::kSelWarp0;
    const int q = sidx / C::kSelPerQuery;
    const int g0 = (sidx % C::kSelPerQuery) * C::kGroupsPerSel;  // first 32-key group it filters
    uint64_t* pool = sPool + sidx * C::kPool;
    uint32_t* hist = sHist + sidx * 256;
    const int64_t t = t0 + q;
    const bool valid = t < sd.T;
    const int64_t pt = pos_b + t;
    const int64_t vis_end = valid ? (pt < S_b - 1 ? pt : S_b - 1) + 1 : 0;
    const uint32_t lt_mask = (1u << lane) - 1u;
    uint64_t theta = 0ull;  // exact 512th best word this warp has seen (0 until 512 were seen)
    int n = 0;              // words in the pool
    for (int it = 0; it < (buffered ? 0 : n_tiles); ++it) {
      const int sb = it % C::kScoreBufs;
      const uint32_t sph = (it / C::kScoreBufs) & 1;
      if (!mbar_wait_warp<C::kWaitHint>(&sfull[sb], sph, s_abort, p.err, p.wait_ns)) break;
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
      // (p.withhold: a test makes the epilogue's bounded wait for this ring slot run out.)
      if (lane == 0 && !(p.withhold && blockIdx.x == 0 && sidx == 0 && it == 0))
        mbar_arrive(&sempty[sb]);
      if (n > C::kPool - C::kGroupsPerSel * 32) {
        theta = select_compact<kTopK>(pool, n, hist, lane);
        n = kTopK;
        if (lane == 0) s_theta[sidx] = theta;
      }
    }
    if (C::kSelPerQuery > 1 || sd.n_splits > 1) {
      // Finished with a CTA-wide select after the role loops (every warp helps).
      if (lane == 0) s_pool_n[sidx] = static_cast<uint32_t>(n);
    } else {
      sel_finish(sidx, n);
    }
  };
  if constexpr (C::kRegW) {
    // whole warpgroups change their register allocation at the top of their branch
    if (warp < C::kEpiWarps) {
      setmaxnreg_inc<C::kRegEpi>();
      epi_role();
      setmaxnreg_dec<C::kRegLaunch>();
    } else {
      setmaxnreg_dec<C::kRegOther>();
      if (warp == C::kTmaWarp) tma_role();
      else if (warp == C::kMmaWarp) mma_role();
      else if (warp < C::kSelWarp0 + C::kSelectors) sel_role();
      setmaxnreg_inc<C::kRegLaunch>();
    }
  } else {
    if (warp == C::kTmaWarp) tma_role();
    else if (warp == C::kMmaWarp) mma_role();
    else if (warp < C::kEpiWarps) epi_role();
    else if (!DENSE && warp < C::kSelWarp0 + C::kSelectors) sel_role();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  griddep_launch_dependents();  // the stream is done: the next kernel may start its setup
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (!DENSE && !*s_abort) {
    if (buffered)
      finish_hist<C>(p, sd, t0, split, s_bins, s_cand, s_ncand, sBuf, n_tiles,
                     static_cast<int64_t>(tile_lo) * kTileKeys, vis_q, *s_cut, *s_maxbin,
                     reinterpret_cast<uint64_t*>(sK), s_scratch, warp, lane);
    else if (C::kSelPerQuery > 1 || sd.n_splits > 1)
      finish_cta_select<C>(p, sd, t0, split, sPool, s_pool_n, reinterpret_cast<uint64_t*>(sK),
                           sHist, s_scratch, warp, lane);
  }
  if (!DENSE && sd.n_splits > 1) {
    // Split plans: every CTA of a query block takes a ticket after publishing its lists; the
    // CTA that takes the last ticket merges them (nothing ever waits on another CTA).
    uint32_t* ticket = p.counters + kCounterWords * (sd.ticket0 + qb);
    __syncthreads();  // every thread's list writes (and proxy fence) precede the ticket
    if (threadIdx.x == 0) {
      __threadfence();
      *s_last = atomicAdd(ticket, 1u) == static_cast<uint32_t>(sd.n_splits - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (*s_last) {
      __threadfence();
      if (!*s_abort) {
        if constexpr (C::kHistSel)
          merge_hist_slots<C>(p, sd, t0, reinterpret_cast<uint64_t*>(sK), smem + C::kOffHist,
                              gbar, s_abort, s_scratch, warp, lane);
        else
          merge_split_lists<C>(p, sd, t0, reinterpret_cast<uint64_t*>(sK), sHist, s_scratch,
                               warp, lane);
      }
      // ready for the next call: the ticket and (one-query splits) the published bins
      for (int i = threadIdx.x; i < (C::kHistSel ? 1 + sd.n_splits : 1); i += C::kThreads)
        ticket[i] = 0u;
    }
  }
}

}  // namespace ds4
