/*
 * ds4idx — Lightning Indexer for DeepSeek-V4-style sparse attention on GB300 (sm_103a).
 *
 * The operation. "DeepSeek V4 Flash 추론을 1.6초로 줄인 ds4 최적화" (aitrends), sections
 * 섹션별 상세 and 용어 해설, describes the Lightning Indexer as the kernel that picks, for every
 * query token, the key positions sparse attention will read, with a Top-512 selection after a
 * scorer. The pages print no formula; the score computed here is the DeepSeek indexer score
 *
 *     I[t,s] = kscale[s] * sum_{j < H_I} w[t,j] * max(0, sum_{i < d_I} q[t,j,i] * k[s,i])
 *
 * over H_I = 64 index heads of width d_I = 128, for every causally visible key
 * s <= p(t) = pos_offset + t (a token sees itself), with kscale[s] = 1 for bf16 caches. For each
 * query the library returns the top-k (k = 512) keys ordered by score descending, ties going to
 * the lower key index; when fewer than k keys are visible, all of them are returned and the
 * remaining slots are (-1, -inf). "DeepSeek V4 Flash는 단일 AMD MI300X에서 실행됩니다", section
 * 두 가지 핵심 정확성 수정 사항 (FP8 형식 불일치), gives the FP8 E4M3 indexer key cache; here
 * it is OCP E4M3FN (largest finite 448) with one fp32 scale per key.
 *
 * Arithmetic: products of bf16 (or E4M3) operands accumulate in fp32 on the tensor cores; the
 * ReLU, the weighted head sum and the key scale are fp32. Scores match an fp64 evaluation within
 * 1e-4 * (1 + |I|) for bf16 inputs.
 *
 * Conventions for every entry point:
 *  - All tensor arguments are DEVICE pointers on the current CUDA device, row-major, dense,
 *    16-byte aligned, owned by the caller. Nothing is copied or retained after the call.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Calls are asynchronous: they
 *    enqueue kernels on `stream` and return; outputs are valid once the stream has reached that
 *    point. No entry point synchronises the host except ds4idx_sync_status and ds4idx_destroy.
 *    Kernels are launched as programmatic dependents of the previous kernel on `stream`: their
 *    blocks may start (shared memory and tensor-memory setup) while that kernel finishes, but
 *    touch no global memory before it has completed, so stream order holds as usual.
 *  - A handle is not thread-safe: use one handle per stream / host thread. The handle owns a
 *    small device workspace (error word, per-split candidate lists) allocated at create; the
 *    compute entry points allocate nothing.
 *  - Return value: DS4IDX_OK (0) or a negative ds4idx_status. Argument errors are detected on
 *    the host before anything is enqueued. Inputs must be finite (not checked on the device).
 */
#ifndef DS4IDX_H_
#define DS4IDX_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DS4IDX_OK = 0,
  DS4IDX_ERR_INVALID_ARG = -1,    /* null pointer, misalignment, size out of range, mismatch */
  DS4IDX_ERR_UNSUPPORTED = -2,    /* shape/dtype not built (H_I != 64, d_I != 128, k != 512),
                                     or the current device is not sm_103 */
  DS4IDX_ERR_ALLOC = -3,          /* workspace allocation failed at create */
  DS4IDX_ERR_LAUNCH = -4,         /* a kernel launch or an enqueue failed */
  DS4IDX_ERR_DEVICE_TIMEOUT = -5, /* a kernel gave up on a bounded device-side wait */
  DS4IDX_ERR_CUDA = -6,           /* another CUDA runtime or driver call failed */
  DS4IDX_ERR_SCRATCH_LIMIT = -7   /* request needs more than the fixed scratch of the
                                     no-allocation entry point */
} ds4idx_status;

/* Element types. q and kcache of the indexer are BF16 or FP8_E4M3 codes; F32 is accepted as the
 * input of the FP8 cache writer only. */
typedef enum { DS4IDX_BF16 = 0, DS4IDX_FP8_E4M3 = 1, DS4IDX_F32 = 2 } ds4idx_dtype;

typedef struct {
  int32_t n_heads;   /* H_I; must be 64 */
  int32_t head_dim;  /* d_I; must be 128 */
  int32_t topk;      /* k; must be 512 */
  int32_t dtype;     /* ds4idx_dtype of q and kcache */
  int64_t max_T;     /* largest query count per sequence passed to any call (>= 1) */
  int64_t max_S;     /* largest key count per sequence (>= 1, < 2^31) */
  int64_t max_batch; /* largest B for ds4idx_score_topk_batched (1..64) */
} ds4idx_config;

typedef struct ds4idx_handle* ds4idx_t;

/* Creates a handle for the current CUDA device and allocates its workspace.
 * Errors: INVALID_ARG (null out/cfg, ranges), UNSUPPORTED (shape or device), ALLOC, CUDA.
 * On error *out is set to NULL. */
int ds4idx_create(ds4idx_t* out, const ds4idx_config* cfg);

/* Scores and selects for one sequence.
 *  q         [T, 64, 128]  bf16, or E4M3 codes (uint8) for FP8 handles. For FP8 the per-token q
 *                          scale is folded into w by the caller (w[t,j] * qscale[t]); this is exact
 *                          because ReLU is positively homogeneous.
 *  w         [T, 64]       fp32 head weights.
 *  kcache    [S, 128]      bf16, or E4M3 codes for FP8 handles.
 *  kscale    [S]           fp32 per-key scale (>= 0) for FP8; must be NULL for bf16.
 *  T         number of query tokens (0 <= T <= max_T; T = 0 is a no-op).
 *  S         number of keys in the cache (1 <= S <= max_S).
 *  pos_offset position of query 0 (>= 0); query t sits at p(t) = pos_offset + t and sees keys
 *            0..min(p(t), S - 1). A well-formed prefill or decode call has pos_offset + T <= S
 *            (every query's own key is in the cache); positions past the cache see all S keys.
 *  topk      must equal the handle's topk (512).
 *  out_idx   [T, topk] int32, written: key indices, best first; -1 in unused slots.
 *  out_score [T, topk] fp32, written: the scores of out_idx (-inf in unused slots); may be NULL.
 */
int ds4idx_score_topk(ds4idx_t h, const void* q, const float* w, const void* kcache,
                      const float* kscale, int64_t T, int64_t S, int64_t pos_offset, int32_t topk,
                      int32_t* out_idx, float* out_score, void* stream);

/* B independent sequences in one launch (batched decode or chunked prefill). Every array gains
 * a leading [B] dimension with a dense stride: q [B, T, 64, 128], w [B, T, 64],
 * kcache [B, S, 128], kscale [B, S] (FP8), out_idx / out_score [B, T, topk].
 * pos_offsets is a HOST array of B positions (>= 0), one per sequence.
 * 1 <= B <= max_batch. Other arguments as in ds4idx_score_topk. */
int ds4idx_score_topk_batched(ds4idx_t h, int32_t B, const void* q, const float* w,
                              const void* kcache, const float* kscale, int64_t T, int64_t S,
                              const int64_t* pos_offsets, int32_t topk, int32_t* out_idx,
                              float* out_score, void* stream);

/* Variable-length, optionally paged batch: B independent sequences, each with its own number
 * of queries, its own key count and its own position, in one launch (continuous-batching decode
 * and mixed chunked prefill). The pages have no interface for this; the concurrency sweep and
 * the hybrid KV-cache rows of "DeepSeek V4 Flash는 단일 AMD MI300X에서 실행됩니다" (동시성 스윕,
 * 프로덕션 수준 튜닝 세부 사항) are the serving setting it is for.
 *  q, w          packed queries of all sequences: q [Q, 64, 128], w [Q, 64] fp32, where
 *                Q = cu_seqlens_q[B]; sequence b owns rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1
 *                (cu_seqlens_q: HOST int64 [B + 1], starting at 0, non-decreasing; a sequence
 *                may have no query).
 *  kcache        the key pool [pool_rows, 128] (bf16 or E4M3 codes), pool_rows < 2^31;
 *  kscale        [pool_rows] fp32 for FP8 handles, NULL for bf16.
 *  Keys of sequence b (S_b = seq_lens[b] >= 1, HOST int64 [B]) are found either
 *   - contiguously: kv_start (HOST int64 [B]) gives the pool row of its key 0, or
 *   - through a page table: page_table (DEVICE int32 [B, pages_per_seq], 4-byte aligned) lists
 *     the pages of sequence b in key order; page_size keys per page (a multiple of 64); key s
 *     lives in pool row page_table[b][s / page_size] * page_size + s % page_size. Page ids are
 *     not checked on the host: an id outside the pool reads as zero keys (wrong results, no
 *     out-of-bounds access).
 *    Exactly one of kv_start and page_table is given.
 *  pos_offsets   HOST int64 [B]: the position of each sequence's first query (as in
 *                ds4idx_score_topk: query t sees keys 0 .. min(pos + t, S_b - 1)).
 *  out_idx / out_score  [Q, topk], rows packed like q. Key indices are positions within the
 *                sequence (0 .. S_b - 1), not pool rows.
 * Limits: B <= max_batch, every T_b <= max_T and S_b <= max_S of the handle. Key-range splits of
 * short sequences are fitted to the handle's workspace. Errors: INVALID_ARG, LAUNCH, CUDA. */
int ds4idx_score_topk_varlen(ds4idx_t h, int32_t B, const void* q, const float* w,
                             const int64_t* cu_seqlens_q, const void* kcache, const float* kscale,
                             int64_t pool_rows, const int64_t* kv_start,
                             const int32_t* page_table, int32_t page_size, int32_t pages_per_seq,
                             const int64_t* seq_lens, const int64_t* pos_offsets, int32_t topk,
                             int32_t* out_idx, float* out_score, void* stream);

/* Debug/test entry: the fp32 scores the selection kernels see, before selection.
 * out_scores [T, S] fp32, written: I[t,s] for visible s, -inf for s > p(t). Same inputs and
 * rules as ds4idx_score_topk; it runs the same scoring code path. */
int ds4idx_score_dense_debug(ds4idx_t h, const void* q, const float* w, const void* kcache,
                             const float* kscale, int64_t T, int64_t S, int64_t pos_offset,
                             float* out_scores, void* stream);

/* Synchronises `stream`, then reads and clears the handle's device error word.
 * Returns DEVICE_TIMEOUT if any kernel since the last check gave up on a bounded wait
 * (its outputs are then undefined), CUDA if the synchronisation reported an error, else OK. */
int ds4idx_sync_status(ds4idx_t h, void* stream);

/* Synchronises the device, frees the workspace and the handle. NULL is accepted (no-op). */
int ds4idx_destroy(ds4idx_t h);

/* Static English text for a status code. Never NULL. */
const char* ds4idx_status_string(int status);

/* Library ABI version: (major << 16) | minor. */
int ds4idx_version(void);

/* Number of kernels this library has enqueued in this process (all handles and entry points).
 * Instrumentation for benchmarks: a successful compute call adds the launches it made. */
uint64_t ds4idx_kernels_launched(void);

/* No-allocation variant of ds4idx_score_topk_batched. The pages have no counterpart: this is an
 * integration aid for callers that cannot allocate device memory when they call the indexer.
 * Examples are a serving engine that reserved all free HBM for its own KV-cache pool at start-up,
 * and a host framework whose allocator must account for every device byte. Neither can let a
 * library call cudaMalloc behind its back, and it may not be able to hold a ds4idx handle
 * either, since a handle allocates its workspace at create.
 *
 * This entry point takes no handle and allocates nothing (no cudaMalloc, no cudaFree, no
 * allocating library call). Its scratch, the per-split candidate lists of short sequences plus
 * an error word and the split counters, lives in one fixed array (16 MiB of lists, 1 MiB of
 * counters) compiled into the library as file-scope __device__ storage. Every GPU that loads the
 * library holds that array until the process exits.
 *  - dtype is a ds4idx_dtype. All other arguments, layouts and rules are those of
 *    ds4idx_score_topk_batched, with 1 <= B <= 64, 0 <= T, 1 <= S < 2^31 and topk = 512.
 *  - Limit: the array holds 2^21 list words (16 MiB) and the split counters (merge ticket and the
 *    splits' published bins) of 4096 query blocks. Short sequences (decode, small chunks) split
 *    their key range over several CTAs, and each split publishes a list of 512 words per query
 *    (1152 per one-query sequence). Here the split count steps down from the one
 *    ds4idx_score_topk_batched would use until the lists fit (B * T * splits * 512 <= 2^21); one
 *    split needs no list, so every valid call runs, only with fewer CTAs where the handle path
 *    would split further. Outputs are the same as the handle path's. DS4IDX_ERR_SCRATCH_LIMIT is
 *    returned only if a plan still did not fit.
 *  - Set-up: the first call on each device looks up the array's device address and sets kernel
 *    attributes, with that device current. Make that first call before any stream capture.
 *  - Argument errors return INVALID_ARG before anything is enqueued or the array is touched.
 *  - Sharing: all calls use the same array, and it keeps the previous call's contents. The error
 *    word and the split counters the call uses are cleared on `stream` at the start of every
 *    valid call; the candidate lists are always fully written before they are read. Calls that
 *    can overlap on the GPU (different streams or host threads without ordering between them)
 *    race on the array and corrupt each other's outputs, so order them, for example on one
 *    stream.
 *  - A kernel that gives up on a bounded device wait records it in the array's error word. This
 *    entry point cannot report it; callers that need that status use a handle and
 *    ds4idx_sync_status. */
int ds4idx_score_topk_batched_noalloc(int32_t dtype, int32_t B, const void* q, const float* w,
                                      const void* kcache, const float* kscale, int64_t T,
                                      int64_t S, const int64_t* pos_offsets, int32_t topk,
                                      int32_t* out_idx, float* out_score, void* stream);

/* ---- FP8 index-cache writer: the step before an FP8 indexer call.
 * "DeepSeek V4 Flash는 단일 AMD MI300X에서 실행됩니다", section 두 가지 핵심 정확성 수정 사항
 * (FP8 형식 불일치): the indexer key cache is written as FP8 E4M3, and the format's largest
 * finite value sets the scale. Here the format is OCP E4M3FN (largest finite 448) with one fp32
 * scale per token row:
 *     scale = absmax(row) / 448,  code[i] = E4M3(clamp(x[i] / scale, -448, 448)),
 * each fp32 operation correctly rounded, the conversion round-to-nearest-even; a row whose
 * scale is 0 gets codes 0. The results are bit-exact functions of the inputs. Inputs must be
 * finite. Both calls are asynchronous on `stream` and allocate nothing. */

/* Quantises n new key rows k [n, 128] (in_dtype DS4IDX_F32 or DS4IDX_BF16, 16-byte aligned)
 * into the index cache: row i goes to cache row slots[i] when `slots` (device int64 [n]) is
 * given, else to dst_offset + i. kcache [cache_rows, 128] uint8 E4M3 codes (16-byte aligned),
 * kscale [cache_rows] fp32. Slots outside [0, cache_rows) (e.g. -1 for padding tokens) are
 * skipped. Errors: INVALID_ARG (dtype, null or misaligned pointer, n < 0, a contiguous range
 * past cache_rows), LAUNCH. n = 0 is a no-op. */
int ds4idx_quantize_keys(const void* k, int32_t in_dtype, int64_t n, const int64_t* slots,
                         int64_t dst_offset, uint8_t* kcache, float* kscale, int64_t cache_rows,
                         void* stream);

/* Quantises the queries of an FP8 indexer call: q [T, 64, 128] (DS4IDX_F32 or DS4IDX_BF16)
 * with one scale per token over all 64 x 128 values into q_codes [T, 64, 128] uint8, and folds
 * the scale into the head weights, w_out[t, j] = w[t, j] * qscale[t] (fp32, correctly rounded;
 * exact in the score because ReLU is positively homogeneous). w [T, 64] fp32; qscale [T] fp32
 * receives the scales and may be NULL. w_out may equal w (in place). Errors: INVALID_ARG,
 * LAUNCH. T = 0 is a no-op. */
int ds4idx_quantize_queries(const void* q, int32_t in_dtype, int64_t T, const float* w,
                            uint8_t* q_codes, float* w_out, float* qscale, void* stream);

/* ---- Merge of key-sharded Top-k lists (the exchange step of a key-range-sharded indexer).
 * When the keys of a sequence are split into disjoint ranges (shards) and each shard's Top-k is
 * computed on its own (ds4idx_score_topk on that range), the union of the shards' lists holds
 * the global Top-k: a key among the k best of all keys is also among the k best of its shard.
 * This call merges them: for every row it takes the k largest (score, key) pairs of all lists,
 * ordered by score descending with ties to the lower key, padded with (-1, -inf).
 *  in_idx, in_score  DEVICE [n_lists, rows, topk] int32 / fp32: each list's indices are local to
 *                    its shard (-1 = empty slot); 1 <= n_lists <= 16.
 *  idx_offsets       HOST int64 [n_lists]: the first key of each shard, added to its indices
 *                    (merged keys must stay below 2^31).
 *  row0              HOST int64 [n_lists] or NULL: list l has no entries for rows < row0[l]
 *                    (queries that see none of its keys); NULL = all rows.
 *  out_idx, out_score DEVICE [rows, topk] (out_score may be NULL). topk must be 512.
 * Shards must be disjoint (a key in two lists would be kept twice). Asynchronous on `stream`,
 * allocates nothing. Errors: INVALID_ARG, LAUNCH, CUDA. */
int ds4idx_merge_topk(int32_t n_lists, int64_t rows, const int32_t* in_idx,
                      const float* in_score, const int64_t* idx_offsets, const int64_t* row0,
                      int32_t topk, int32_t* out_idx, float* out_score, void* stream);

/* ---- Sparse attention over the selected keys: the step that consumes the indexer's output.
 * "DeepSeek V4 Flash 추론을 1.6초로 줄인 ds4 최적화", 용어 해설 (희소 어텐션, Lightning Indexer):
 * sparse attention computes only some token pairs, and the indexer picks the positions. For
 * query token t and head h over its selected positions J(t) (one row of out_idx; -1 = empty):
 *     s_j = sm_scale * q[t,h,:] . kv[j,:],   out[t,h,:] = sum_j softmax(s)_j * kv[j, 0:d_v],
 *     lse[t,h] = log sum_j exp(s_j)          (natural log; -inf and out = 0 if J(t) is empty)
 * with one latent row per position shared by all heads (the value is the row's first d_v dims).
 *  q       DEVICE [T, n_heads, d_qk] bf16, 16-byte aligned.
 *  kv      DEVICE [kv_rows, d_qk] bf16 (1 <= kv_rows < 2^31), 16-byte aligned.
 *  idx     DEVICE [T, topk] int32: selected positions; position s of token t is kv row
 *          kv_row0[t] + s (kv_row0: DEVICE int64 [T], or NULL for 0). Positions whose row falls
 *          outside [0, kv_rows) are treated as empty. Selected positions must be distinct.
 *  out     DEVICE [T, n_heads, d_v] bf16; lse DEVICE [T, n_heads] fp32 or NULL.
 * Built shape: n_heads = 128, d_qk = 576, d_v = 512, topk = 512 (else UNSUPPORTED); sm_scale > 0.
 * Arithmetic: bf16 products with fp32 accumulation on the tensor cores, fp32 softmax, the
 * probabilities rounded to bf16 for the value product, the output rounded to bf16.
 * Asynchronous on `stream`, allocates nothing. Bounded device waits that run out are recorded
 * for ds4idx_sparse_attention_status. Errors: INVALID_ARG, UNSUPPORTED, LAUNCH, CUDA. */
int ds4idx_sparse_attention(const void* q, const void* kv, int64_t kv_rows, const int32_t* idx,
                            const int64_t* kv_row0, int64_t T, int32_t n_heads, int32_t d_qk,
                            int32_t d_v, int32_t topk, float sm_scale, void* out, float* lse,
                            void* stream);

/* Synchronises `stream`, then reads and clears the sparse-attention error word: DEVICE_TIMEOUT if
 * a kernel gave up on a bounded wait since the last check (outputs undefined), CUDA if the
 * synchronisation failed, else OK. */
int ds4idx_sparse_attention_status(void* stream);

/* Test support for the bounded device waits (the pages have no counterpart). Every mbarrier
 * wait in the kernels gives up after a limit (2 s by default), records DS4IDX_ERR_DEVICE_TIMEOUT
 * for ds4idx_sync_status, waits for its own copies and tensor-core work to finish, frees its
 * tensor memory and returns, so a lost arrival turns into an error status instead of a hang.
 * This call sets the limit used by the handle's later calls (1e6 <= wait_limit_ns <= 2e9) and,
 * with withhold != 0, makes the next calls of a four-query (T > 1) plan without key splits
 * withhold one arrival of their first CTA's first selector warp, so that CTA's epilogue wait for
 * the score ring runs out once the ring wraps (more than 30 key tiles in that CTA). Every copy
 * and MMA already issued completes on its own. Reset with (2000000000, 0).
 * Errors: INVALID_ARG (null handle, limit out of range). */
int ds4idx_debug_wait_test(ds4idx_t h, uint64_t wait_limit_ns, int32_t withhold);

/* The work decomposition a call would use, computed on the host alone (no device access), for
 * tests and capacity planning. num_sms: the device's SM count; B, T, S, pos_offsets[B] as in
 * ds4idx_score_topk_batched; fixed_scratch != 0 gives the plan of
 * ds4idx_score_topk_batched_noalloc. out[7] receives: queries per CTA, query blocks per
 * sequence, key splits, key tiles per split, CTAs in the grid, split-list words, split tickets.
 * Errors: INVALID_ARG. */
int ds4idx_plan_query(int32_t num_sms, int32_t B, int64_t T, int64_t S,
                      const int64_t* pos_offsets, int32_t fixed_scratch, int64_t* out);

#ifdef __cplusplus
}
#endif

#endif /* DS4IDX_H_ */
