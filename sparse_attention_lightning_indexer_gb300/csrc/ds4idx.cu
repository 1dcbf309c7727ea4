// Host side of the ds4idx C ABI: argument validation, TMA descriptor encoding, work
// decomposition (query blocks x key splits) and kernel launches. Semantics of every entry point
// are documented in include/ds4idx.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>

#include "ds4idx.h"
#include "indexer_kernel.cuh"

using namespace ds4;

namespace {
std::atomic<uint64_t> g_launches{0};  // kernels this library has enqueued (process-wide)
}  // namespace

// Shared with the library's other translation units (their launches are counted too).
namespace ds4w {
std::atomic<uint64_t>* launch_counter() { return &g_launches; }
}  // namespace ds4w

struct ds4idx_handle {
  ds4idx_config cfg;
  int device = 0;
  int num_sms = 0;
  uint32_t* err = nullptr;        // device error word
  uint64_t* partial = nullptr;    // per-split Top-512 lists
  size_t partial_words = 0;
  uint32_t* counters = nullptr;   // per split query block: ticket and published bins, zero between calls
  size_t n_counters = 0;          // split query blocks the counters hold
  uint64_t wait_ns = 0;           // bounded-wait limit passed to the kernels
  int32_t withhold = 0;           // test hook (ds4idx_debug_wait_test)
};

namespace {

constexpr int kVersion = (1 << 16) | 1;
// Fixed scratch of the no-allocation entry point: 2^21 list words (16 MiB) and the counters
// (ticket and published bins) of up to 4096 split query blocks.
constexpr size_t kNoAllocListWords = static_cast<size_t>(1) << 21;
constexpr size_t kNoAllocTickets = 4096;
constexpr int kMaxSplits = 64;
constexpr int kMinTilesPerSplit = 4;


PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool load_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int queries_per_cta(int64_t T) { return T == 1 ? 1 : 4; }

// Work decomposition. Long sequences give plenty of CTAs from query blocks alone; short ones
// (decode, small chunks) also split the key range so every SM gets work, and a second kernel
// merges the per-split lists.
struct Plan {
  int nq = 4;
  int n_qb = 0;
  int n_splits = 1;
  int tiles_per_split = 0;
  int64_t grid = 0;
};

size_t plan_partial_words(const Plan& pl, int64_t B, int64_t T);
size_t plan_counters(const Plan& pl, int64_t B);

// max_words / max_counters cap the scratch a split plan may use (the fixed array of the
// no-allocation entry point): the split count steps down until the plan fits; one split needs
// no scratch at all.
Plan make_plan(int num_sms, int64_t B, int64_t T, int64_t max_vis,
               size_t max_words = SIZE_MAX, size_t max_counters = SIZE_MAX) {
  Plan pl;
  pl.nq = queries_per_cta(T);
  pl.n_qb = static_cast<int>((T + pl.nq - 1) / pl.nq);
  const int64_t tiles = (max_vis + kTileKeys - 1) / kTileKeys;
  const int64_t blocks = B * pl.n_qb;
  int64_t splits = 1;
  if (blocks < 4LL * num_sms) {
    // Few query blocks of similar size (decode, short chunks): split the key range so the CTAs
    // fill whole waves of SMs. Every split repeats the Top-512 warm-up and adds a list to merge,
    // so take the fewest splits whose wave occupancy is within 5% of the best achievable.
    const int64_t max_s = std::min<int64_t>(kMaxSplits, std::max<int64_t>(1, tiles / kMinTilesPerSplit));
    auto occupancy = [&](int64_t sp) {
      const int64_t ctas = blocks * sp;
      const int64_t waves = (ctas + num_sms - 1) / num_sms;
      return static_cast<double>(ctas) / static_cast<double>(waves * num_sms);
    };
    double best = 0.0;
    for (int64_t sp = 1; sp <= max_s; ++sp) best = std::max(best, occupancy(sp));
    for (int64_t sp = 1; sp <= max_s; ++sp) {
      if (occupancy(sp) >= best - 0.05) {
        splits = sp;
        break;
      }
    }
  }
  for (;; --splits) {
    pl.tiles_per_split = static_cast<int>(tiles > 0 ? (tiles + splits - 1) / splits : 0);
    pl.n_splits = pl.tiles_per_split > 0
                      ? static_cast<int>((tiles + pl.tiles_per_split - 1) / pl.tiles_per_split)
                      : 1;
    if (pl.n_splits < 1) pl.n_splits = 1;
    if (splits <= 1 || (plan_partial_words(pl, B, T) <= max_words &&
                        plan_counters(pl, B) <= max_counters))
      break;
  }
  pl.grid = blocks * pl.n_splits;
  return pl;
}

size_t plan_partial_words(const Plan& pl, int64_t B, int64_t T) {
  // one-query CTAs publish a slot per split (count window + candidates), others 512 words
  const size_t per_split = pl.nq == 1 ? static_cast<size_t>(kSlotWords) : static_cast<size_t>(kTopK);
  return pl.n_splits > 1 ? static_cast<size_t>(B * T) * pl.n_splits * per_split : 0;
}
size_t plan_counters(const Plan& pl, int64_t B) {
  return pl.n_splits > 1 ? static_cast<size_t>(B) * pl.n_qb : 0;
}

template <int DT, int NQ, bool DENSE>
cudaError_t set_smem_attr() {
  using C = KCfg<DT, NQ, DENSE>;
  if constexpr (C::kRegW) {
    // The kernel moves registers between its warpgroups (setmaxnreg); that exchange completes
    // only if each thread was launched with exactly kRegLaunch registers. Refuse to run a build
    // whose register count differs rather than risk a kernel that waits forever.
    cudaFuncAttributes fa{};
    const cudaError_t e = cudaFuncGetAttributes(&fa, indexer_kernel<DT, NQ, DENSE>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != C::kRegLaunch) return cudaErrorInvalidKernelImage;
  }
  return cudaFuncSetAttribute(indexer_kernel<DT, NQ, DENSE>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
}

// Tensor map over `rows` rows of 128 elements per batch entry: dims {128, rows, B}.
bool encode_rows(CUtensorMap* map, const void* base, int dtype, int64_t rows, int64_t B,
                 int box_rows) {
  const bool bf16 = dtype == DS4IDX_BF16;
  const cuuint64_t row_bytes = bf16 ? 256 : 128;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[2] = {row_bytes, row_bytes * static_cast<cuuint64_t>(rows)};
  cuuint32_t box[3] = {bf16 ? 64u : 128u, static_cast<cuuint32_t>(box_rows), 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                              3, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int DT, int NQ, bool DENSE>
cudaError_t launch(const CUtensorMap& tq, const CUtensorMap& tk, const KParams& kp, int64_t grid,
                   cudaStream_t stream) {
  using C = KCfg<DT, NQ, DENSE>;
  // Programmatic stream serialization: this launch may begin while the previous kernel in the
  // stream finishes (its CTAs set up shared memory and TMEM, then wait in griddep_wait before
  // touching global memory), hiding launch latency behind that kernel's tail.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, indexer_kernel<DT, NQ, DENSE>, tq, tk, kp);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
  return e;
}

template <int DT>
cudaError_t launch_dt(int nq, bool dense, const CUtensorMap& tq, const CUtensorMap& tk,
                      const KParams& kp, int64_t grid, cudaStream_t stream) {
  if (dense) return nq == 1 ? launch<DT, 1, true>(tq, tk, kp, grid, stream)
                            : launch<DT, 4, true>(tq, tk, kp, grid, stream);
  if (nq == 1) return launch<DT, 1, false>(tq, tk, kp, grid, stream);
  return launch<DT, 4, false>(tq, tk, kp, grid, stream);
}

// Scratch and limits one compute call runs with: a handle's workspace, or the fixed array of
// the no-allocation entry point.
struct Ctx {
  int32_t dtype = DS4IDX_BF16;
  int64_t max_T = 0, max_S = 0, max_batch = 0;
  int device = 0;
  int num_sms = 0;
  uint32_t* err = nullptr;
  uint64_t* partial = nullptr;
  size_t partial_words = 0;
  uint32_t* counters = nullptr;
  size_t n_counters = 0;
  bool cap_splits = false;  // fit the split count to the scratch instead of rejecting the call
  uint64_t wait_ns = kWaitLimitNs;
  int32_t withhold = 0;
};

Ctx handle_ctx(const ds4idx_handle* h) {
  Ctx c;
  c.dtype = h->cfg.dtype;
  c.max_T = h->cfg.max_T;
  c.max_S = h->cfg.max_S;
  c.max_batch = h->cfg.max_batch;
  c.device = h->device;
  c.num_sms = h->num_sms;
  c.err = h->err;
  c.partial = h->partial;
  c.partial_words = h->partial_words;
  c.counters = h->counters;
  c.n_counters = h->n_counters;
  c.wait_ns = h->wait_ns;
  c.withhold = h->withhold;
  return c;
}

// A validated call, ready to enqueue.
struct Call {
  int nq = 4;
  int64_t grid = 0;
  CUtensorMap tq, tk;
  KParams kp;
  bool dense = false;
  bool noop = false;  // no query at all
  int64_t n_blocks = 0;  // split query blocks (counters) the call uses
};

// One sequence of a call, as the caller describes it.
struct SeqSpec {
  int64_t T = 0, S = 0, pos = 0;
  int64_t q_row0 = 0;  // first row in the packed q / w / outputs
  int64_t k_row0 = 0;  // first row in the contiguous key pool (unused when paged)
};

// Everything a compute call passes, in one place.
struct CallSpec {
  int32_t B = 0;
  SeqSpec seq[kMaxBatch];
  bool uniform = true;       // every sequence has the same T, S (batched / single calls)
  int64_t q_rows = 0;        // rows of the packed queries (sum of T)
  int64_t pool_rows = 0;     // rows of the key pool
  const void* q = nullptr;
  const float* w = nullptr;
  const void* kcache = nullptr;
  const float* kscale = nullptr;
  const int32_t* page_table = nullptr;  // device [B, pt_stride], or null (contiguous)
  int32_t page_size = 0;
  int32_t pt_stride = 0;
  int32_t topk = kTopK;
  int32_t* out_idx = nullptr;
  float* out_score = nullptr;
  float* dense = nullptr;
};

// Split plan for sequences of different lengths: one key-tile count per split for all of them
// (a sequence gets ceil(its tiles / tps) splits), chosen like the uniform plan: the fewest
// splits whose estimated wave occupancy is within 5% of the best; then fewer splits until the
// lists and tickets fit the scratch.
void plan_varlen(int num_sms, const CallSpec& cs, int nq, size_t max_words, size_t max_tickets,
                 int32_t* n_qb, int32_t* n_splits, int32_t* tps_out) {
  int64_t blocks = 0, max_tiles = 1;
  int64_t tiles[kMaxBatch];
  for (int b = 0; b < cs.B; ++b) {
    const SeqSpec& q = cs.seq[b];
    n_qb[b] = static_cast<int32_t>((q.T + nq - 1) / nq);
    const int64_t vis = q.T > 0 ? std::min<int64_t>(q.pos + q.T, q.S) : 0;
    tiles[b] = (vis + kTileKeys - 1) / kTileKeys;
    blocks += n_qb[b];
    max_tiles = std::max<int64_t>(max_tiles, tiles[b]);
  }
  auto splits_of = [&](int b, int64_t tps) {
    return static_cast<int32_t>(std::max<int64_t>(1, (tiles[b] + tps - 1) / tps));
  };
  auto fits = [&](int64_t tps) {
    size_t words = 0, tickets = 0;
    const size_t per = nq == 1 ? static_cast<size_t>(kSlotWords) : static_cast<size_t>(kTopK);
    for (int b = 0; b < cs.B; ++b) {
      const int32_t sp = splits_of(b, tps);
      if (sp > 1) {
        words += static_cast<size_t>(cs.seq[b].T) * sp * per;
        tickets += static_cast<size_t>(n_qb[b]);
      }
    }
    return words <= max_words && tickets <= max_tickets;
  };
  int64_t tps = max_tiles;  // one split each
  if (blocks < 4LL * num_sms) {
    const int64_t max_s = std::min<int64_t>(kMaxSplits, std::max<int64_t>(1, max_tiles / kMinTilesPerSplit));
    auto occupancy = [&](int64_t t) {  // tile work over the tile slots of the waves it needs
      int64_t ctas = 0, work = 0;
      for (int b = 0; b < cs.B; ++b) {
        ctas += static_cast<int64_t>(n_qb[b]) * splits_of(b, t);
        work += static_cast<int64_t>(n_qb[b]) * tiles[b];
      }
      const int64_t waves = (ctas + num_sms - 1) / num_sms;
      return static_cast<double>(work) / static_cast<double>(waves * num_sms * t);
    };
    double best = 0.0;
    for (int64_t sp = 1; sp <= max_s; ++sp) best = std::max(best, occupancy((max_tiles + sp - 1) / sp));
    for (int64_t sp = 1; sp <= max_s; ++sp) {
      const int64_t t = (max_tiles + sp - 1) / sp;
      if (occupancy(t) >= best - 0.05) {
        tps = t;
        break;
      }
    }
  }
  while (tps < max_tiles && !fits(tps)) ++tps;
  for (int b = 0; b < cs.B; ++b) n_splits[b] = splits_of(b, tps);
  *tps_out = static_cast<int32_t>(tps);
}

// Validates a compute call and prepares its launch. Enqueues nothing and touches no device
// memory: every argument error is reported here, before any work is queued.
int prepare(const Ctx& c, const CallSpec& cs, Call* call) {
  const bool dense = cs.dense != nullptr;
  if (cs.B < 1 || cs.B > c.max_batch || cs.B > kMaxBatch) return DS4IDX_ERR_INVALID_ARG;
  if (!dense && cs.topk != kTopK) return DS4IDX_ERR_INVALID_ARG;
  int64_t total_T = 0;
  for (int b = 0; b < cs.B; ++b) {
    const SeqSpec& q = cs.seq[b];
    if (q.T < 0 || q.T > c.max_T || q.S < 1 || q.S > c.max_S) return DS4IDX_ERR_INVALID_ARG;
    if (q.pos < 0 || q.pos > (1LL << 40) || q.q_row0 < 0 || q.k_row0 < 0)
      return DS4IDX_ERR_INVALID_ARG;
    if (q.T > 0 && q.q_row0 + q.T > cs.q_rows) return DS4IDX_ERR_INVALID_ARG;
    if (!cs.page_table && q.k_row0 + q.S > cs.pool_rows) return DS4IDX_ERR_INVALID_ARG;
    if (cs.page_table && (q.S + cs.page_size - 1) / cs.page_size > cs.pt_stride)
      return DS4IDX_ERR_INVALID_ARG;
    total_T += q.T;
  }
  call->dense = dense;
  call->noop = total_T == 0;
  if (call->noop) return DS4IDX_OK;
  if (cs.q_rows * kHeads > (1LL << 31) - 1 || cs.pool_rows < 1 || cs.pool_rows > (1LL << 31) - 1)
    return DS4IDX_ERR_INVALID_ARG;
  if (cs.page_table && (cs.page_size < 64 || cs.page_size % 64 != 0 || cs.pt_stride < 1 ||
                        (reinterpret_cast<uintptr_t>(cs.page_table) & 3u)))
    return DS4IDX_ERR_INVALID_ARG;
  if (!cs.q || !cs.w || !cs.kcache || !aligned16(cs.q) || !aligned16(cs.w) || !aligned16(cs.kcache))
    return DS4IDX_ERR_INVALID_ARG;
  if (c.dtype == DS4IDX_FP8_E4M3) {
    if (!cs.kscale || (reinterpret_cast<uintptr_t>(cs.kscale) & 3u)) return DS4IDX_ERR_INVALID_ARG;
  } else if (cs.kscale) {
    return DS4IDX_ERR_INVALID_ARG;
  }
  if (dense) {
    if (!aligned16(cs.dense) || cs.B != 1) return DS4IDX_ERR_INVALID_ARG;
  } else {
    if (!cs.out_idx || !aligned16(cs.out_idx)) return DS4IDX_ERR_INVALID_ARG;
    if (cs.out_score && !aligned16(cs.out_score)) return DS4IDX_ERR_INVALID_ARG;
  }
  if (!load_encode()) return DS4IDX_ERR_CUDA;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != c.device) return DS4IDX_ERR_INVALID_ARG;

  // ---- work decomposition
  bool all_one = true;
  for (int b = 0; b < cs.B; ++b) all_one = all_one && cs.seq[b].T <= 1;
  const int nq = dense ? queries_per_cta(cs.seq[0].T) : (all_one ? 1 : 4);
  int32_t n_qb[kMaxBatch], n_splits[kMaxBatch];
  int32_t tps = 0;
  if (dense) {
    n_qb[0] = static_cast<int32_t>((cs.seq[0].T + nq - 1) / nq);
    n_splits[0] = 1;
    tps = static_cast<int32_t>((cs.seq[0].S + kTileKeys - 1) / kTileKeys);
  } else if (cs.uniform) {
    int64_t max_vis = 0;
    for (int b = 0; b < cs.B; ++b)
      max_vis = std::max<int64_t>(max_vis, std::min<int64_t>(cs.seq[b].pos + cs.seq[0].T, cs.seq[0].S));
    const Plan pl = c.cap_splits
                        ? make_plan(c.num_sms, cs.B, cs.seq[0].T, max_vis, c.partial_words, c.n_counters)
                        : make_plan(c.num_sms, cs.B, cs.seq[0].T, max_vis);
    if (plan_partial_words(pl, cs.B, cs.seq[0].T) > c.partial_words ||
        plan_counters(pl, cs.B) > c.n_counters)
      return c.cap_splits ? DS4IDX_ERR_SCRATCH_LIMIT : DS4IDX_ERR_INVALID_ARG;
    for (int b = 0; b < cs.B; ++b) {
      n_qb[b] = pl.n_qb;
      n_splits[b] = pl.n_splits;
    }
    tps = pl.tiles_per_split;
  } else {
    plan_varlen(c.num_sms, cs, nq, c.partial_words, c.n_counters, n_qb, n_splits, &tps);
  }

  KParams& kp = call->kp;
  std::memset(&kp, 0, sizeof kp);
  int64_t list = 0, tickets = 0, ctas = 0;
  const size_t per_split = nq == 1 ? static_cast<size_t>(kSlotWords) : static_cast<size_t>(kTopK);
  for (int b = 0; b < cs.B; ++b) {
    SeqDesc& d = kp.seq[b];
    const SeqSpec& q = cs.seq[b];
    d.T = q.T;
    d.S = q.S;
    d.pos = q.pos;
    d.q_row0 = q.q_row0;
    d.k_row0 = q.k_row0;
    d.n_qb = n_qb[b];
    d.n_splits = n_splits[b];
    d.tiles_per_split = tps;
    d.list0 = list;
    d.ticket0 = static_cast<int32_t>(tickets);
    d.cta0 = static_cast<int32_t>(ctas);
    d.pt_row = b;
    if (n_splits[b] > 1) {
      list += static_cast<int64_t>(q.T) * n_splits[b] * static_cast<int64_t>(per_split);
      tickets += n_qb[b];
    }
    ctas += static_cast<int64_t>(n_qb[b]) * n_splits[b];
  }
  call->n_blocks = tickets;
  if (static_cast<size_t>(list) > c.partial_words || static_cast<size_t>(tickets) > c.n_counters)
    return c.cap_splits ? DS4IDX_ERR_SCRATCH_LIMIT : DS4IDX_ERR_INVALID_ARG;
  if (ctas > 0x7FFFFFFF) return DS4IDX_ERR_INVALID_ARG;

  if (!encode_rows(&call->tq, cs.q, c.dtype, cs.q_rows * kHeads, 1, kHeads * nq))
    return DS4IDX_ERR_INVALID_ARG;
  if (!encode_rows(&call->tk, cs.kcache, c.dtype, cs.pool_rows, 1, cs.page_table ? 64 : kTileKeys))
    return DS4IDX_ERR_INVALID_ARG;
  kp.w = cs.w;
  kp.kscale = cs.kscale;
  kp.out_idx = cs.out_idx;
  kp.out_score = cs.out_score;
  kp.partial = c.partial;
  kp.counters = c.counters;
  kp.dense = cs.dense;
  kp.err = c.err;
  kp.page_table = cs.page_table;
  kp.pool_rows = cs.pool_rows;
  kp.wait_ns = c.wait_ns;
  kp.withhold = c.withhold;
  kp.B = cs.B;
  kp.uniform = cs.uniform ? 1 : 0;
  kp.page_size = cs.page_size;
  kp.pt_stride = cs.pt_stride;
  call->nq = nq;
  call->grid = ctas;
  if (ctas == 0) call->noop = true;
  return DS4IDX_OK;
}

// The spec of a uniform call: B sequences of T queries and S keys, stored densely one after
// another (q [B, T, 64, 128], kcache [B, S, 128]).
int uniform_spec(int32_t B, const void* q, const float* w, const void* kcache,
                 const float* kscale, int64_t T, int64_t S, const int64_t* pos_offsets,
                 int32_t topk, int32_t* out_idx, float* out_score, float* dense, CallSpec* cs) {
  if (B < 1 || B > kMaxBatch || !pos_offsets || T < 0 || S < 1) return DS4IDX_ERR_INVALID_ARG;
  cs->B = B;
  cs->uniform = true;
  for (int b = 0; b < B; ++b) {
    cs->seq[b].T = T;
    cs->seq[b].S = S;
    cs->seq[b].pos = pos_offsets[b];
    cs->seq[b].q_row0 = b * T;
    cs->seq[b].k_row0 = b * S;
  }
  cs->q_rows = B * T;
  cs->pool_rows = B * S;
  cs->q = q;
  cs->w = w;
  cs->kcache = kcache;
  cs->kscale = kscale;
  cs->topk = topk;
  cs->out_idx = out_idx;
  cs->out_score = out_score;
  cs->dense = dense;
  return DS4IDX_OK;
}

int enqueue(const Ctx& c, const Call& call, void* stream_ptr) {
  if (call.noop) return DS4IDX_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  cudaError_t e =
      c.dtype == DS4IDX_BF16
          ? launch_dt<kDtBf16>(call.nq, call.dense, call.tq, call.tk, call.kp, call.grid, stream)
          : launch_dt<kDtFp8>(call.nq, call.dense, call.tq, call.tk, call.kp, call.grid, stream);
  return e == cudaSuccess ? DS4IDX_OK : DS4IDX_ERR_LAUNCH;
}

// Shared implementation of the handle-based uniform compute entry points.
int run(ds4idx_t h, int32_t B, const void* q, const float* w, const void* kcache,
        const float* kscale, int64_t T, int64_t S, const int64_t* pos_offsets, int32_t topk,
        int32_t* out_idx, float* out_score, float* dense, void* stream_ptr) {
  if (!h) return DS4IDX_ERR_INVALID_ARG;
  const Ctx c = handle_ctx(h);
  CallSpec cs;
  int st = uniform_spec(B, q, w, kcache, kscale, T, S, pos_offsets, topk, out_idx, out_score,
                        dense, &cs);
  if (st != DS4IDX_OK) return st;
  Call call;
  st = prepare(c, cs, &call);
  if (st != DS4IDX_OK) return st;
  return enqueue(c, call, stream_ptr);
}

}  // namespace

extern "C" {

int ds4idx_version(void) { return kVersion; }

uint64_t ds4idx_kernels_launched(void) { return g_launches.load(std::memory_order_relaxed); }

const char* ds4idx_status_string(int status) {
  switch (status) {
    case DS4IDX_OK: return "ok";
    case DS4IDX_ERR_INVALID_ARG: return "invalid argument";
    case DS4IDX_ERR_UNSUPPORTED: return "unsupported shape, dtype or device";
    case DS4IDX_ERR_ALLOC: return "device workspace allocation failed";
    case DS4IDX_ERR_LAUNCH: return "kernel launch failed";
    case DS4IDX_ERR_DEVICE_TIMEOUT: return "a kernel gave up on a bounded device wait";
    case DS4IDX_ERR_CUDA: return "CUDA runtime or driver error";
    case DS4IDX_ERR_SCRATCH_LIMIT: return "request exceeds the fixed scratch of the no-allocation entry point";
    default: return "unknown status";
  }
}

int ds4idx_create(ds4idx_t* out, const ds4idx_config* cfg) {
  if (!out) return DS4IDX_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg) return DS4IDX_ERR_INVALID_ARG;
  if (cfg->dtype != DS4IDX_BF16 && cfg->dtype != DS4IDX_FP8_E4M3) return DS4IDX_ERR_INVALID_ARG;
  if (cfg->max_T < 1 || cfg->max_S < 1 || cfg->max_S > (1LL << 31) - 1 || cfg->max_batch < 1 ||
      cfg->max_batch > kMaxBatch)
    return DS4IDX_ERR_INVALID_ARG;
  if (cfg->n_heads != kHeads || cfg->head_dim != kDim || cfg->topk != kTopK)
    return DS4IDX_ERR_UNSUPPORTED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DS4IDX_ERR_CUDA;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return DS4IDX_ERR_CUDA;
  if (!(prop.major == 10 && prop.minor == 3)) return DS4IDX_ERR_UNSUPPORTED;
  if (!load_encode()) return DS4IDX_ERR_CUDA;

  if (set_smem_attr<kDtBf16, 4, false>() != cudaSuccess ||
      set_smem_attr<kDtBf16, 1, false>() != cudaSuccess ||
      set_smem_attr<kDtBf16, 4, true>() != cudaSuccess ||
      set_smem_attr<kDtBf16, 1, true>() != cudaSuccess ||
      set_smem_attr<kDtFp8, 1, true>() != cudaSuccess ||
      set_smem_attr<kDtFp8, 4, false>() != cudaSuccess ||
      set_smem_attr<kDtFp8, 1, false>() != cudaSuccess ||
      set_smem_attr<kDtFp8, 4, true>() != cudaSuccess)
    return DS4IDX_ERR_CUDA;

  ds4idx_handle* h = new (std::nothrow) ds4idx_handle();
  if (!h) return DS4IDX_ERR_ALLOC;
  h->cfg = *cfg;
  h->device = dev;
  h->num_sms = prop.multiProcessorCount;
  h->wait_ns = kWaitLimitNs;

  // Workspace for the largest per-split candidate set any admissible call can need.
  size_t words = 0, counters = 0;
  for (int64_t B = 1; B <= cfg->max_batch; ++B) {
    const int64_t t_hi = std::min<int64_t>(cfg->max_T, 16LL * h->num_sms);
    for (int64_t T = 1; T <= t_hi; ++T) {
      const Plan pl = make_plan(h->num_sms, B, T, cfg->max_S);
      words = std::max(words, plan_partial_words(pl, B, T));
      counters = std::max(counters, plan_counters(pl, B));
    }
  }
  h->partial_words = words;
  h->n_counters = counters;
  // err word at [0], split counters (ticket, published bins) from [64] (own cache lines), all
  // zeroed once here
  const size_t misc_bytes = 256 + counters * kCounterWords * sizeof(uint32_t);
  if (cudaMalloc(&h->err, misc_bytes) != cudaSuccess) {
    delete h;
    return DS4IDX_ERR_ALLOC;
  }
  h->counters = h->err + 64;
  if (words && cudaMalloc(&h->partial, words * sizeof(uint64_t)) != cudaSuccess) {
    cudaFree(h->err);
    delete h;
    return DS4IDX_ERR_ALLOC;
  }
  if (cudaMemset(h->err, 0, misc_bytes) != cudaSuccess) {
    cudaFree(h->partial);
    cudaFree(h->err);
    delete h;
    return DS4IDX_ERR_CUDA;
  }
  *out = h;
  return DS4IDX_OK;
}

int ds4idx_score_topk(ds4idx_t h, const void* q, const float* w, const void* kcache,
                      const float* kscale, int64_t T, int64_t S, int64_t pos_offset, int32_t topk,
                      int32_t* out_idx, float* out_score, void* stream) {
  return run(h, 1, q, w, kcache, kscale, T, S, &pos_offset, topk, out_idx, out_score, nullptr,
             stream);
}

int ds4idx_score_topk_batched(ds4idx_t h, int32_t B, const void* q, const float* w,
                              const void* kcache, const float* kscale, int64_t T, int64_t S,
                              const int64_t* pos_offsets, int32_t topk, int32_t* out_idx,
                              float* out_score, void* stream) {
  return run(h, B, q, w, kcache, kscale, T, S, pos_offsets, topk, out_idx, out_score, nullptr,
             stream);
}

int ds4idx_score_topk_varlen(ds4idx_t h, int32_t B, const void* q, const float* w,
                             const int64_t* cu_seqlens_q, const void* kcache, const float* kscale,
                             int64_t pool_rows, const int64_t* kv_start,
                             const int32_t* page_table, int32_t page_size, int32_t pages_per_seq,
                             const int64_t* seq_lens, const int64_t* pos_offsets, int32_t topk,
                             int32_t* out_idx, float* out_score, void* stream) {
  if (!h || B < 1 || B > kMaxBatch || !cu_seqlens_q || !seq_lens || !pos_offsets)
    return DS4IDX_ERR_INVALID_ARG;
  if ((kv_start == nullptr) == (page_table == nullptr)) return DS4IDX_ERR_INVALID_ARG;
  if (cu_seqlens_q[0] != 0) return DS4IDX_ERR_INVALID_ARG;
  CallSpec cs;
  cs.B = B;
  cs.uniform = false;
  for (int b = 0; b < B; ++b) {
    if (cu_seqlens_q[b + 1] < cu_seqlens_q[b]) return DS4IDX_ERR_INVALID_ARG;
    cs.seq[b].T = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
    cs.seq[b].S = seq_lens[b];
    cs.seq[b].pos = pos_offsets[b];
    cs.seq[b].q_row0 = cu_seqlens_q[b];
    cs.seq[b].k_row0 = kv_start ? kv_start[b] : 0;
  }
  cs.q_rows = cu_seqlens_q[B];
  cs.pool_rows = pool_rows;
  cs.q = q;
  cs.w = w;
  cs.kcache = kcache;
  cs.kscale = kscale;
  cs.page_table = page_table;
  cs.page_size = page_size;
  cs.pt_stride = pages_per_seq;
  cs.topk = topk;
  cs.out_idx = out_idx;
  cs.out_score = out_score;
  Ctx c = handle_ctx(h);
  c.cap_splits = true;  // split lists of mixed lengths are fitted to the handle's workspace
  Call call;
  const int st = prepare(c, cs, &call);
  if (st != DS4IDX_OK) return st;
  return enqueue(c, call, stream);
}

int ds4idx_score_dense_debug(ds4idx_t h, const void* q, const float* w, const void* kcache,
                             const float* kscale, int64_t T, int64_t S, int64_t pos_offset,
                             float* out_scores, void* stream) {
  if (!out_scores) return DS4IDX_ERR_INVALID_ARG;
  return run(h, 1, q, w, kcache, kscale, T, S, &pos_offset, 0, nullptr, nullptr, out_scores,
             stream);
}

int ds4idx_sync_status(ds4idx_t h, void* stream) {
  if (!h) return DS4IDX_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DS4IDX_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, h->err, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return DS4IDX_ERR_CUDA;
  if (word) {
    // A CTA that gave up may have left a split ticket half counted: start the next call clean.
    cudaMemset(h->err, 0, 256 + h->n_counters * kCounterWords * sizeof(uint32_t));
    return DS4IDX_ERR_DEVICE_TIMEOUT;
  }
  return DS4IDX_OK;
}

int ds4idx_debug_wait_test(ds4idx_t h, uint64_t wait_limit_ns, int32_t withhold) {
  if (!h || wait_limit_ns < 1000000ull || wait_limit_ns > kWaitLimitNs) return DS4IDX_ERR_INVALID_ARG;
  h->wait_ns = wait_limit_ns;
  h->withhold = withhold ? 1 : 0;
  return DS4IDX_OK;
}

int ds4idx_plan_query(int32_t num_sms, int32_t B, int64_t T, int64_t S,
                      const int64_t* pos_offsets, int32_t fixed_scratch, int64_t* out) {
  if (num_sms < 1 || B < 1 || B > kMaxBatch || T < 1 || S < 1 || !pos_offsets || !out)
    return DS4IDX_ERR_INVALID_ARG;
  int64_t max_vis = 0;
  for (int b = 0; b < B; ++b) {
    if (pos_offsets[b] < 0) return DS4IDX_ERR_INVALID_ARG;
    max_vis = std::max<int64_t>(max_vis, std::min<int64_t>(pos_offsets[b] + T, S));
  }
  const Plan pl = fixed_scratch ? make_plan(num_sms, B, T, max_vis, kNoAllocListWords,
                                            kNoAllocTickets)
                                : make_plan(num_sms, B, T, max_vis);
  out[0] = pl.nq;
  out[1] = pl.n_qb;
  out[2] = pl.n_splits;
  out[3] = pl.tiles_per_split;
  out[4] = pl.grid;
  out[5] = static_cast<int64_t>(plan_partial_words(pl, B, T));
  out[6] = static_cast<int64_t>(plan_counters(pl, B));
  return DS4IDX_OK;
}

int ds4idx_destroy(ds4idx_t h) {
  if (!h) return DS4IDX_OK;
  const cudaError_t e = cudaDeviceSynchronize();
  cudaFree(h->partial);
  cudaFree(h->err);
  delete h;
  return e == cudaSuccess ? DS4IDX_OK : DS4IDX_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------- no-allocation entry point
// For callers that cannot allocate device memory at call time (an engine that pre-reserved its
// HBM, an allocator that must account for every byte): the split-plan scratch lives in a fixed
// array compiled into the library instead of a handle's workspace. See the header for the rules.
namespace {

// [0, kNoAllocListWords): per-split candidate lists; then the error word (own 256-byte line);
// then the split counters (per split query block a ticket and the splits' published bins,
// 32-bit; the blocks a call uses are zeroed at its start together with the error word).
static __device__ __align__(256) uint64_t
    g_noalloc_scratch[kNoAllocListWords + 32 + kNoAllocTickets * kCounterWords / 2];

struct NoAllocDevice {
  std::once_flag once;
  int status = DS4IDX_OK;
  uint64_t* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int num_sms = 0;
};
constexpr int kNoAllocMaxDevices = 64;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];

// One-time set-up per device, run with that device current.
int noalloc_setup(int dev) {
  NoAllocDevice& d = g_noalloc_dev[dev];
  std::call_once(d.once, [&d, dev] {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      d.status = DS4IDX_ERR_CUDA;
      return;
    }
    if (!(major == 10 && minor == 3)) {
      d.status = DS4IDX_ERR_UNSUPPORTED;
      return;
    }
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      d.status = DS4IDX_ERR_CUDA;
      return;
    }
    if (!load_encode() || set_smem_attr<kDtBf16, 4, false>() != cudaSuccess ||
        set_smem_attr<kDtBf16, 1, false>() != cudaSuccess ||
        set_smem_attr<kDtFp8, 4, false>() != cudaSuccess ||
        set_smem_attr<kDtFp8, 1, false>() != cudaSuccess) {
      d.status = DS4IDX_ERR_CUDA;
      return;
    }
    d.scratch = static_cast<uint64_t*>(ptr);
    d.num_sms = sms;
    d.status = DS4IDX_OK;
  });
  return d.status;
}

}  // namespace

extern "C" int ds4idx_score_topk_batched_noalloc(int32_t dtype, int32_t B, const void* q,
                                                 const float* w, const void* kcache,
                                                 const float* kscale, int64_t T, int64_t S,
                                                 const int64_t* pos_offsets, int32_t topk,
                                                 int32_t* out_idx, float* out_score,
                                                 void* stream) {
  if (dtype != DS4IDX_BF16 && dtype != DS4IDX_FP8_E4M3) return DS4IDX_ERR_INVALID_ARG;
  if (B < 1 || B > kMaxBatch || T < 0 || S < 1 || S > (1LL << 31) - 1 || !pos_offsets)
    return DS4IDX_ERR_INVALID_ARG;
  if (topk != kTopK) return DS4IDX_ERR_INVALID_ARG;
  if (T == 0) return DS4IDX_OK;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return DS4IDX_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return DS4IDX_ERR_UNSUPPORTED;
  const int st = noalloc_setup(dev);
  if (st != DS4IDX_OK) return st;
  const NoAllocDevice& d = g_noalloc_dev[dev];

  // The shared launch path over the fixed scratch. Short sequences split their key range only
  // as far as the split lists fit the array (one split uses no list at all).
  Ctx c;
  c.dtype = dtype;
  c.max_T = T;
  c.max_S = S;
  c.max_batch = kMaxBatch;
  c.device = dev;
  c.num_sms = d.num_sms;
  c.partial = d.scratch;
  c.partial_words = kNoAllocListWords;
  c.err = reinterpret_cast<uint32_t*>(d.scratch + kNoAllocListWords);
  c.counters = reinterpret_cast<uint32_t*>(d.scratch + kNoAllocListWords + 32);
  c.n_counters = kNoAllocTickets;
  c.cap_splits = true;
  CallSpec cs;
  int vs = uniform_spec(B, q, w, kcache, kscale, T, S, pos_offsets, topk, out_idx, out_score,
                        nullptr, &cs);
  if (vs != DS4IDX_OK) return vs;
  Call call;
  vs = prepare(c, cs, &call);
  if (vs != DS4IDX_OK) return vs;
  // Valid call: the array keeps the previous call's contents, so clear the error word and the
  // tickets on the stream right before the launch.
  const size_t clear = 256 + static_cast<size_t>(call.n_blocks) * kCounterWords * sizeof(uint32_t);
  if (cudaMemsetAsync(c.err, 0, clear, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DS4IDX_ERR_LAUNCH;
  return enqueue(c, call, stream);
}
