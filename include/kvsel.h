/*
 * kvsel.h -- C ABI of the query-aware sparse KV-block selection and sparse
 * decode-attention library (libkvsel.so), written for NVIDIA GB300 (sm_103a).
 *
 * The method is SparPR's decode-step loop ("SparPR KV cache recovery on a
 * consumer GPU", section "Three decisions rather than one compression
 * ratio"): every cached KV block is summarised by its mean key per KV head;
 * a query scores each block by the sum over heads of query.summary inner
 * products; Top-k picks the blocks; adjacent picks merge into spans; a cost
 * model (copy vs recompute) with a Minimum Keep Floor sets the keep ratio and
 * a Dense Fallback Threshold gamma switches back to full attention. Attention
 * then runs over the selected blocks only, with split partial results merged
 * by log-sum-exp (the flash-style merge of the DKV abstract).
 *
 * Conventions shared by every entry point
 *  - Return value: KVSEL_OK (0) or a KVSEL_ERR_* code. No entry point aborts,
 *    traps the device or allocates device memory. Host-side argument checks
 *    return KVSEL_ERR_INVALID_ARG / KVSEL_ERR_UNSUPPORTED before anything is
 *    enqueued. Launch failures return KVSEL_ERR_CUDA.
 *  - Data-dependent faults found by a kernel (an out-of-range block-table
 *    entry, page, selection index or count) are not fatal: the kernel skips
 *    the offending access, latches the first error code into a per-device
 *    error word and carries on. kvsel_get_error() reads and clears it.
 *  - Device entry points are asynchronous on the caller's stream; the caller
 *    owns every buffer. Scratch comes from a caller workspace whose size
 *    kvsel_workspace_size() returns. No workspace needs particular initial
 *    contents: every byte a call reads from its workspace, that call wrote
 *    first. Calls that share a workspace must not overlap on the GPU.
 *  - The library looks up the device addresses of its own device variables
 *    (the error word, the static scratch array) once per device and keeps
 *    them for the life of the process: do not keep using it on a device
 *    after cudaDeviceReset() on that device.
 *  - bf16 tensors are passed as kvsel_bf16 (the 16-bit pattern). Device
 *    pointers must be 16-byte aligned.
 *  - Supported shapes: head_dim in {64, 128}; block_size in {16, 32, 64};
 *    n_qheads a multiple of n_kvheads with n_qheads / n_kvheads <= 16;
 *    batch <= 4096; max_blocks <= 16384; n_kvheads * head_dim / 8 a power
 *    of two times a divisor of 32 whose quotient is at most 16.
 *
 * Layouts (row-major, innermost last)
 *  q            [batch][n_qheads][head_dim]                    bf16
 *  KV pages     [n_pages][n_kvheads][2][head_dim/64][block_size][64] bf16:
 *               for each (page, KV head) the K tile, then the V tile. A tile
 *               is "tiled": it keeps its block_size x head_dim values as
 *               head_dim/64 column halves of block_size rows x 64 channels,
 *               and inside every 128-byte row the 16-byte chunk c of token row
 *               t is stored at chunk position c ^ (t % 8). The K and V of a
 *               run of consecutive heads of a page are one contiguous range.
 *  block_table  [batch][max_blocks]                            int32 (page id)
 *  seq_lens     [batch]                                        int32 (T_b)
 *  summaries    [batch][max_blocks][n_kvheads][head_dim]       bf16
 *  open_acc     [batch][n_kvheads][head_dim]                   fp64
 *  sel_idx      [batch][k_max]  ascending block indices        int32
 *  spans        span_start / span_len [batch][k_max]           int32
 *  host tier    [batch][host_blocks][one KV page] bf16 (block n of sequence
 *               b is a copy of its page, so spans are contiguous)
 *  staging      [batch][staging_slots][one KV page] bf16
 *  out          [batch][n_qheads][head_dim] fp32; lse [batch][n_qheads] fp32
 * A sequence b holds T_b = seq_lens[b] tokens in N_b = ceil(T_b / block_size)
 * blocks; token t lives in page block_table[b][t / block_size], row
 * t % block_size. Channel c of token row t of the key (v = 0) or value
 * (v = 1) of KV head j in page p is element
 * (((p * n_kvheads + j) * 2 + v) * head_dim/64 + c/64) * block_size * 64 +
 * t * 64 + (((c % 64) / 8) ^ (t % 8)) * 8 + c % 8.
 */
#ifndef KVSEL_H_
#define KVSEL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVSEL_VERSION_STRING "kvsel 0.1.0 (sm_103a)"

#if defined(__GNUC__)
#define KVSEL_API __attribute__((visibility("default")))
#else
#define KVSEL_API
#endif

typedef uint16_t kvsel_bf16;               /* bf16 bit pattern */
typedef struct CUstream_st* kvsel_stream_t; /* a cudaStream_t; NULL = legacy default stream */

enum kvsel_status {
  KVSEL_OK = 0,
  KVSEL_ERR_INVALID_ARG = 1,  /* bad pointer, size, alignment or shape */
  KVSEL_ERR_CUDA = 2,         /* a CUDA runtime call or launch failed */
  KVSEL_ERR_BOUNDS = 3,       /* device-detected out-of-range index or count */
  KVSEL_ERR_TIMEOUT = 4,      /* a bounded device wait ran out */
  KVSEL_ERR_UNSUPPORTED = 5,  /* shape outside the compiled variants */
  KVSEL_ERR_WORKSPACE = 6     /* workspace missing or smaller than required */
};

/* Shape of one layer's decode step. */
typedef struct kvsel_problem {
  int32_t batch;       /* sequences in the batch */
  int32_t n_qheads;    /* query heads H_q */
  int32_t n_kvheads;   /* KV heads H_kv (GQA group G = H_q / H_kv) */
  int32_t head_dim;    /* d */
  int32_t block_size;  /* B, tokens per block (= per page) */
  int32_t max_blocks;  /* row stride of block_table and summaries (blocks per sequence capacity) */
  int32_t k_max;       /* row stride of sel_idx / span arrays (selection capacity) */
} kvsel_problem;

enum kvsel_summary_mode {
  KVSEL_SUMMARY_FULL = 0,   /* rebuild every block summary of every sequence */
  KVSEL_SUMMARY_APPEND = 1  /* fold one appended token per sequence into its open block */
};

/*
 * kvsel_build_summaries -- block summaries ("SparPR KV cache recovery on a
 * consumer GPU", paragraph "Query-Aware key-block selection": each block gets
 * a compact precomputed summary, the mean key; kept resident on the GPU).
 *
 * summaries[b][n][j][:] = bf16_rne( (sum over the block's tokens t < T_b of
 * K[t][j][:]) / count ), the sum taken in fp64 in token order from +0.0, the
 * division in fp64 and one round-to-nearest-even to bf16.
 *
 * FULL:   for every b and every block n < N_b. open_acc[b] receives the fp64
 *         sum of block N_b - 1 (the open block). new_k/new_v/append_pos unused.
 * APPEND: for every b with t = append_pos[b] >= 0 (others are skipped): if
 *         new_k != NULL, new_k[b][j][:] is first written to K row t (and new_v
 *         to V row t when new_v != NULL); then open_acc[b] becomes K_t when
 *         t % B == 0 (a new block) or open_acc[b] + K_t otherwise, and the
 *         summary of block t / B is rewritten from it over t % B + 1 tokens.
 *         The caller sets seq_lens[b] = t + 1 for the steps that follow.
 *
 * kv_pages: the paged cache (written only by APPEND with new_k / new_v).
 * block_table, seq_lens: device int32. append_pos: device [batch] int32.
 * new_k, new_v: device [batch][n_kvheads][head_dim] bf16 in natural channel
 * order, nullable; they are stored into the tiled page layout.
 * summaries: device output. open_acc: device [batch][n_kvheads][head_dim] fp64.
 * Errors: INVALID_ARG (null required pointer, bad shape), UNSUPPORTED, CUDA;
 * device BOUNDS when a block-table entry is negative or >= n_pages or
 * T_b > max_blocks * B (the access is skipped).
 */
KVSEL_API int kvsel_build_summaries(const kvsel_problem* p, int mode, kvsel_bf16* kv_pages,
                                    int64_t n_pages, const int32_t* block_table,
                                    const int32_t* seq_lens, const int32_t* append_pos,
                                    const kvsel_bf16* new_k, const kvsel_bf16* new_v,
                                    kvsel_bf16* summaries, double* open_acc,
                                    kvsel_stream_t stream);

/*
 * kvsel_score_topk -- query-aware block score, Top-k and span merge
 * ("SparPR KV cache recovery on a consumer GPU", paragraphs "Query-Aware
 * key-block selection" and "On-demand local recomputation with cost-aware
 * fallback"). Enqueues on `stream` either one kernel -- one thread-block
 * cluster per sequence scores the sequence's blocks and its leader CTA ranks
 * them, when every sequence's cluster fits on the device at once and
 * max_blocks <= 4096 -- or two (a score grid, then one Top-k CTA per
 * sequence); kvsel_score_path_for() tells which. Both give the same results
 * bit for bit. The first kernel is launched with programmatic stream
 * serialization: it may become resident while the kernel before it still
 * runs, but reads no input before that kernel has completed, so stream order
 * is kept.
 *
 * score[b][n] = sum over query heads h of <q[b][h], summaries[b][n][kv(h)]>,
 * kv(h) = h / G, accumulated in fp32 (q is first folded over each GQA group).
 * k_b = min(k_per_seq[b], N_b, k_max) blocks with the largest scores are
 * selected, ties to the lower block index; sel_idx[b][0..k_b) holds them in
 * ascending order and n_sel[b] = k_b. Runs of consecutive indices become
 * spans: span_start / span_len [b][0..n_spans[b]).
 * Dense fallback (gamma): dense_flag[b] = (n_spans * tau_rel + k_b >=
 * gamma * (tau_rel + N_b)), evaluated in fp64; tau_rel is the per-span
 * overhead in units of one block's recovery cost (0 gives k_b >= gamma*N_b).
 *
 * q: device [batch][n_qheads][head_dim] bf16. summaries: device.
 * k_per_seq: device [batch] int32 (k_per_seq[b] > k_max latches BOUNDS and
 * is clamped). scores_out: device [batch][max_blocks] fp32, nullable.
 * dense_flag: device [batch] uint8, nullable. ws: workspace of
 * kvsel_workspace_size(p, KVSEL_WS_SCORE_TOPK) bytes (no initial contents
 * required).
 */
KVSEL_API int kvsel_score_topk(const kvsel_problem* p, const kvsel_bf16* q, const kvsel_bf16* summaries,
                     const int32_t* seq_lens, const int32_t* k_per_seq, float gamma,
                     float tau_rel, int32_t* sel_idx, int32_t* n_sel, int32_t* span_start,
                     int32_t* span_len, int32_t* n_spans, uint8_t* dense_flag,
                     float* scores_out, void* ws, size_t ws_bytes, kvsel_stream_t stream);

/* Which form the score + Top-k calls take (kvsel_set_score_path). */
enum kvsel_score_path {
  KVSEL_SCORE_PATH_AUTO = 0,     /* one launch of clusters where the problem allows, else two grids */
  KVSEL_SCORE_PATH_TWO_GRID = 1, /* always the score grid + Top-k grid */
  KVSEL_SCORE_PATH_CLUSTER = 2   /* always the cluster launch; other problems fail with UNSUPPORTED */
};

/*
 * kvsel_set_score_path -- process-wide choice of the form every later
 * kvsel_score_topk, kvsel_append_score_topk, kvsel_score_topk_window and
 * kvsel_score_topk_noalloc call takes (default AUTO). The forms compute the
 * same results bit for bit; the choice exists for measurement and tests.
 * Returns the previous value, or -1 (and changes nothing) for an unknown one.
 * Not synchronised with calls running in other host threads.
 */
KVSEL_API int kvsel_set_score_path(int path);

/*
 * kvsel_score_path_for -- the form (KVSEL_SCORE_PATH_TWO_GRID or
 * KVSEL_SCORE_PATH_CLUSTER) a score + Top-k call on problem p takes on the
 * current device under the current setting, with (with_append != 0) or
 * without a folded append; *cluster_ctas (nullable) receives the CTAs per
 * sequence of the cluster form (0 for the two-grid form). Returns a negative
 * KVSEL_ERR_* code on an invalid problem.
 */
KVSEL_API int kvsel_score_path_for(const kvsel_problem* p, int with_append, int32_t* cluster_ctas);

/* The inputs of the APPEND mode of kvsel_build_summaries, for the fused call
 * below. Pointers are device pointers with the meaning, layout and alignment
 * given there; new_k and new_v are nullable (new_v needs new_k). */
typedef struct kvsel_append_in {
  kvsel_bf16* kv_pages;           /* paged cache; the new K/V row is written into it */
  int64_t n_pages;
  const int32_t* block_table;     /* [batch][max_blocks] */
  const int32_t* append_pos;      /* [batch]; t < 0 skips the sequence */
  const kvsel_bf16* new_k;        /* [batch][n_kvheads][head_dim] or NULL */
  const kvsel_bf16* new_v;        /* [batch][n_kvheads][head_dim] or NULL */
  kvsel_bf16* summaries;          /* the summary table: updated, then scored */
  double* open_acc;               /* [batch][n_kvheads][head_dim] fp64 */
} kvsel_append_in;

/*
 * kvsel_append_score_topk -- kvsel_build_summaries(APPEND) followed by
 * kvsel_score_topk on the updated table, in the kernel(s) of
 * kvsel_score_topk (the decode step of "SparPR KV cache recovery on a
 * consumer GPU", paragraph "Query-Aware key-block selection": the new token's
 * key updates its block's summary before the query scores the blocks).
 *
 * Every output (kv_pages, summaries, open_acc, scores, selection, spans,
 * dense_flag) equals, bit for bit, that of the two calls made in sequence on
 * the same stream. seq_lens must already count the appended token
 * (seq_lens[b] = append_pos[b] + 1 for an appending sequence). The append is
 * done by the CTA whose share of the score work holds the open block, so it
 * adds no kernel and no dependency step to the call.
 *
 * Arguments as kvsel_build_summaries (app) and kvsel_score_topk (the rest).
 * Errors: INVALID_ARG (NULL app or required pointer, misalignment, new_v
 * without new_k), UNSUPPORTED, WORKSPACE, CUDA; device BOUNDS as for the two
 * calls.
 */
KVSEL_API int kvsel_append_score_topk(const kvsel_problem* p, const kvsel_append_in* app,
                                      const kvsel_bf16* q, const int32_t* seq_lens,
                                      const int32_t* k_per_seq, float gamma, float tau_rel,
                                      int32_t* sel_idx, int32_t* n_sel, int32_t* span_start,
                                      int32_t* span_len, int32_t* n_spans, uint8_t* dense_flag,
                                      float* scores_out, void* ws, size_t ws_bytes,
                                      kvsel_stream_t stream);

/* Blocks attended whatever their score. */
typedef struct kvsel_window {
  int32_t n_sink;    /* the first n_sink blocks of every sequence */
  int32_t n_recent;  /* the last n_recent blocks of every sequence (the recency window) */
} kvsel_window;

/*
 * kvsel_score_topk_window -- kvsel_score_topk (or, with app != NULL,
 * kvsel_append_score_topk) with a forced block window: the recency window
 * that the DKV abstract ("DKV: Anchor + Low-Rank Differential KV-Cache
 * Compression") attends exactly beside its Top-k blocks, merging the two
 * parts by the flash-style log-sum-exp reduction. Here both parts go into one
 * selection, so the split-K decode of kvsel_sparse_decode performs that
 * merge. The leading n_sink blocks are the same rule at the start of the
 * sequence (position-based keeping; the pages describe only the recency
 * window).
 *
 * For sequence b with N_b blocks: the forced blocks are [0, lo) and [hi, N_b)
 * with lo = min(n_sink, N_b), hi = max(lo, N_b - n_recent); the Top-k runs
 * over the candidates [lo, hi) only, k_b = min(k_per_seq[b], hi - lo,
 * k_max - F_b) of them (F_b = N_b - (hi - lo) forced blocks), ties to the
 * lower index. sel_idx[b] holds the union in ascending order, n_sel[b] =
 * F_b + k_b; spans and the gamma decision are taken on that union. A window
 * of zero gives exactly the results of kvsel_score_topk.
 *
 * win: host pointer; n_sink >= 0, n_recent >= 0 and n_sink + n_recent <=
 * k_max, else INVALID_ARG. k_per_seq[b] > k_max - F_b latches BOUNDS and is
 * clamped. summaries: used when app == NULL; with app it must be NULL or
 * app->summaries. Everything else as kvsel_score_topk and
 * kvsel_append_score_topk, with the same errors.
 */
KVSEL_API int kvsel_score_topk_window(const kvsel_problem* p, const kvsel_window* win,
                                      const kvsel_append_in* app, const kvsel_bf16* q,
                                      const kvsel_bf16* summaries, const int32_t* seq_lens,
                                      const int32_t* k_per_seq, float gamma, float tau_rel,
                                      int32_t* sel_idx, int32_t* n_sel, int32_t* span_start,
                                      int32_t* span_len, int32_t* n_spans, uint8_t* dense_flag,
                                      float* scores_out, void* ws, size_t ws_bytes,
                                      kvsel_stream_t stream);

/*
 * kvsel_merge_spans -- span merge of an existing ascending selection ("SparPR
 * KV cache recovery on a consumer GPU", paragraph "On-demand local
 * recomputation with cost-aware fallback": adjacent blocks merge into
 * continuous spans). Indices that differ by exactly one join a span.
 * sel_idx [batch][k_max] with n_sel[b] entries (device); outputs as in
 * kvsel_score_topk. A selection that is not strictly ascending latches BOUNDS.
 */
KVSEL_API int kvsel_merge_spans(const kvsel_problem* p, const int32_t* sel_idx, const int32_t* n_sel,
                      int32_t* span_start, int32_t* span_len, int32_t* n_spans,
                      kvsel_stream_t stream);

/*
 * kvsel_select_scores -- the Top-k, span merge and dense flag of
 * kvsel_score_topk on score rows the caller already holds ("SparPR KV cache
 * recovery on a consumer GPU", paragraphs "Query-Aware key-block selection"
 * and "On-demand local recomputation with cost-aware fallback"), for example
 * the scores_out of an earlier kvsel_score_topk call: one CTA per sequence
 * on `stream`. Every output, rule and tie break is that of kvsel_score_topk
 * on the same scores; k_per_seq may differ from the k the scores were
 * selected with (a larger k gives a wider list, e.g. a prefetch prediction).
 * scores: device [batch][max_blocks] fp32 (entries from N_b on are not read).
 * No workspace. Errors as kvsel_score_topk.
 */
KVSEL_API int kvsel_select_scores(const kvsel_problem* p, const float* scores, const int32_t* seq_lens,
                                  const int32_t* k_per_seq, float gamma, float tau_rel,
                                  int32_t* sel_idx, int32_t* n_sel, int32_t* span_start,
                                  int32_t* span_len, int32_t* n_spans, uint8_t* dense_flag,
                                  kvsel_stream_t stream);

/*
 * kvsel_score_topk_noalloc -- kvsel_score_topk without a caller workspace.
 * The pages describe no such entry point; it exists for callers that cannot
 * allocate device memory: code embedded in a host framework that owns the
 * whole device-memory budget and forbids allocations outside its own
 * allocator, or a latency-critical path where the implicit synchronisation
 * of cudaMalloc/cudaFree is not acceptable.
 *
 * Same arguments, results and errors as kvsel_score_topk minus ws/ws_bytes.
 * Its scratch is a file-scope device array of kvsel_noalloc_scratch_bytes()
 * bytes (4 MiB) that every GPU which loads the library holds until the
 * process exits. A problem whose kvsel_workspace_size(p, KVSEL_WS_SCORE_TOPK)
 * exceeds it (roughly batch * max_blocks > 1M) is rejected with
 * KVSEL_ERR_WORKSPACE and nothing is enqueued; the limit applies whether or
 * not scores_out is given. The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress) with that device
 * current; make that first call before any stream capture. Nothing in the
 * array needs to start at zero, so no call clears it; no call allocates.
 * All calls on a device share the one array, so calls that can overlap on
 * the GPU (different streams without ordering between them) race.
 */
KVSEL_API int kvsel_score_topk_noalloc(const kvsel_problem* p, const kvsel_bf16* q,
                                       const kvsel_bf16* summaries, const int32_t* seq_lens,
                                       const int32_t* k_per_seq, float gamma, float tau_rel,
                                       int32_t* sel_idx, int32_t* n_sel, int32_t* span_start,
                                       int32_t* span_len, int32_t* n_spans, uint8_t* dense_flag,
                                       float* scores_out, kvsel_stream_t stream);

/* Bytes of the static scratch array behind kvsel_score_topk_noalloc. */
KVSEL_API size_t kvsel_noalloc_scratch_bytes(void);

enum kvsel_kv_kind {
  KVSEL_KV_PAGED = 0,  /* K/V pages in device memory + block table */
  KVSEL_KV_STAGED = 1, /* selected blocks already in a device staging buffer */
  KVSEL_KV_HOST = 2,   /* full K/V in pinned host memory: fetch the spans, then attend */
  KVSEL_KV_HOST_DIRECT = 3 /* full K/V in pinned host memory, read by the attention kernel itself */
};

/* Where the K/V of the attended blocks come from. */
typedef struct kvsel_kv_src {
  int32_t kind;                   /* enum kvsel_kv_kind */
  int32_t staging_slots;          /* STAGED/HOST: block slots per sequence in staging */
  const kvsel_bf16* kv_pages;     /* PAGED */
  const int32_t* block_table;     /* PAGED */
  int64_t n_pages;                /* PAGED: pages in kv_pages */
  kvsel_bf16* staging;            /* STAGED/HOST: device staging buffer */
  const kvsel_bf16* host_kv;      /* HOST, HOST_DIRECT: pinned host tier (device-mapped) */
  int32_t host_blocks;            /* HOST, HOST_DIRECT: block stride of the host tier per sequence */
  int32_t fetch_ctas;             /* HOST: CTAs of the gather kernel (0 = one per SM) */
} kvsel_kv_src;

/*
 * kvsel_sparse_decode -- attention over the selected blocks only ("SparPR KV
 * cache recovery on a consumer GPU", paragraph "On-demand local
 * recomputation with cost-aware fallback"; split partial results merged by
 * the flash-style log-sum-exp reduction of the DKV abstract).
 *
 * For every b and query head h: out[b][h] = sum_t softmax_t(scale * q.K_t) V_t
 * over the tokens t < T_b of the blocks sel_idx[b][0..n_sel[b]) -- or of all
 * N_b blocks when dense_flag != NULL and dense_flag[b] != 0 -- using KV head
 * h / G. lse[b][h] = ln sum_t exp(scale * q.K_t). A sequence with no attended
 * token gets out = 0 and lse = -inf. Math in fp32 (bf16 tensor-core products,
 * fp32 accumulation).
 *
 * kv: see kvsel_kv_src. STAGED: the o-th attended block of b is staging slot
 * o (block n when dense). HOST: the selected spans (or all blocks when dense)
 * are first gathered from host_kv into staging on `stream` (see
 * kvsel_fetch_spans), then treated as STAGED. HOST_DIRECT: the attention
 * kernel reads each attended block straight from host_kv (block n of b at
 * [b][n] of the host tier) through unified virtual addressing with 16-byte
 * asynchronous copies into shared memory, so no staging buffer and no
 * second pass over device memory is needed ("KV cache offloading", sections
 * "NOSA" and "SparDA": kernels that read host memory directly); a block
 * index >= host_blocks latches BOUNDS and is skipped.
 * out: device fp32 output; out_bf16: optional bf16 copy; lse: device fp32.
 * ws: kvsel_workspace_size(p, KVSEL_WS_SPARSE_DECODE) bytes (no initial
 * contents required). Two kernels: the attention grid and a row merge grid
 * launched as its programmatic dependent.
 * Errors: UNSUPPORTED when batch * n_kvheads * max_blocks >= 2^31 (the tile
 * list is counted in int32).
 */
KVSEL_API int kvsel_sparse_decode(const kvsel_problem* p, const kvsel_bf16* q, const kvsel_kv_src* kv,
                        const int32_t* seq_lens, const int32_t* sel_idx, const int32_t* n_sel,
                        const int32_t* span_start, const int32_t* span_len,
                        const int32_t* n_spans, const uint8_t* dense_flag, float softmax_scale,
                        float* out, kvsel_bf16* out_bf16, float* lse, void* ws,
                        size_t ws_bytes, kvsel_stream_t stream);

/*
 * kvsel_fetch_spans -- the offload tier's recovery copy: full K/V stays in
 * pinned host memory and only the selected spans cross the host link ("KV
 * cache offloading", sections "Fetching a sparse subset per step" and "NOSA":
 * a kernel that reads host memory directly through unified virtual
 * addressing). A gather kernel of kv->fetch_ctas CTAs reads each span's
 * contiguous blocks from kv->host_kv and writes them to consecutive staging
 * slots; with dense_flag[b] set it copies all N_b blocks. No host round trip.
 * Requires kind == KVSEL_KV_HOST. Returns INVALID_ARG when host_kv is not
 * device-accessible.
 */
KVSEL_API int kvsel_fetch_spans(const kvsel_problem* p, const kvsel_kv_src* kv, const int32_t* seq_lens,
                      const int32_t* span_start, const int32_t* span_len,
                      const int32_t* n_spans, const uint8_t* dense_flag,
                      kvsel_stream_t stream);

/* A GPU-resident cache of host-tier blocks: `slots` pool pages per sequence
 * and the state that maps blocks to them. Every pointer is a device pointer
 * owned by the caller. */
typedef struct kvsel_block_cache {
  int32_t slots;        /* pool pages per sequence; k_max <= slots <= 4096 */
  kvsel_bf16* pool;     /* [batch][slots][one KV page] bf16 (page b * slots + s) */
  int32_t* page_of;     /* [batch][max_blocks]: pool page holding block n, or -1 */
  int32_t* block_in;    /* [batch][slots]: block held by slot s, or -1 */
  int32_t* last_use;    /* [batch][slots]: last step slot s was selected, -1 = empty */
} kvsel_block_cache;

/*
 * kvsel_cache_reset -- empties the cache: every page_of, block_in and
 * last_use entry becomes -1 (three cudaMemsetAsync on `stream`). Call it once
 * before the first kvsel_cache_fetch, and whenever the host tier is replaced.
 */
KVSEL_API int kvsel_cache_reset(const kvsel_problem* p, const kvsel_block_cache* cache,
                                kvsel_stream_t stream);

/*
 * kvsel_cache_fetch -- the offload tier's recovery copy with cross-step reuse
 * ("KV cache offloading", section "NOSA": block selection is local across
 * consecutive decode steps, so blocks fetched in one step are kept on the GPU
 * and reused in the next, and an eviction policy bounds the blocks fetched
 * from host memory). Two kernels on `stream`:
 *  - per sequence b, every selected block sel_idx[b][0..n_sel[b]) that the
 *    cache holds is a hit and its slot is stamped with `step`; the misses, in
 *    ascending block order, take the slots not selected in this step with the
 *    smallest (last_use, slot) -- least recently selected first, empty slots
 *    before any -- evicting the blocks they held;
 *  - every miss is copied from host_kv (pinned, device-mapped; layout of the
 *    host tier) into its pool page, and so is the block holding the last
 *    token (N_b - 1) when it was a hit, since appends change it.
 * n_fetched[b] (nullable, device int32) receives the number of blocks copied.
 * Afterwards every selected block is resident: attend with
 * kvsel_sparse_decode on kind KVSEL_KV_PAGED with kv_pages = cache->pool,
 * block_table = cache->page_of, n_pages = batch * slots, and dense_flag =
 * NULL (a sequence whose gamma flag is set needs every block: serve it with
 * KVSEL_KV_HOST instead; the cache is not updated for it).
 *
 * step: >= 0 and different from the step of the previous call on this cache
 * (a step counter). slots >= k_max guarantees a free slot for every miss.
 * ws: kvsel_workspace_size(p, KVSEL_WS_CACHE_FETCH) bytes (job lists; no
 * initial contents required). fetch_ctas: CTAs of the copy kernel (0 = eight
 * per SM). Errors: INVALID_ARG (NULL or misaligned pointer, slots outside
 * [k_max, 4096], step < 0, host_kv not device-mapped pinned memory),
 * WORKSPACE, UNSUPPORTED, CUDA; device BOUNDS for a selection that is not
 * strictly ascending, an index outside [0, min(N_b, host_blocks)) (not
 * served) or an inconsistent cache state (the block is fetched again).
 */
KVSEL_API int kvsel_cache_fetch(const kvsel_problem* p, const kvsel_block_cache* cache,
                                const kvsel_bf16* host_kv, int32_t host_blocks,
                                const int32_t* seq_lens, const int32_t* sel_idx,
                                const int32_t* n_sel, int32_t step, int32_t* n_fetched,
                                int32_t fetch_ctas, void* ws, size_t ws_bytes,
                                kvsel_stream_t stream);

/*
 * kvsel_cache_prefetch -- loads a predicted block list into the cache ahead
 * of the selection that may ask for it ("KV cache offloading": the Hugging
 * Face Transformers paragraph, the next layer's cache fetched while the
 * current one is computed; section "SparDA", the blocks the next layer will
 * select fetched from pinned host memory on a dedicated stream while the
 * layer before it runs). The kernels of kvsel_cache_fetch, on `stream`, with
 * pred_idx / n_pred in place of the selection and three differences:
 *  - a predicted block that is resident stays in its slot, stamp unchanged;
 *  - the other predicted blocks, ascending, take the slots that hold no
 *    predicted block, smallest (last_use, slot) first, and get last_use -1
 *    (never selected): a wrong prediction is evicted before any block that
 *    a step selected;
 *  - the block holding the last token (N_b - 1) is not prefetched (appends
 *    change it; a selection of it fetches it).
 * n_fetched[b] (nullable) receives the number of blocks copied. The copy
 * kernel's CTAs have half the threads of a fetch's and default to one per SM
 * (fetch_ctas = 0), so that a prefetch on another stream leaves room on each
 * SM for the score and decode kernels. A later
 * kvsel_cache_fetch on the same cache must be ordered after this call (same
 * stream, or an event): both update the cache state and share `ws` if the
 * caller passes the same one. Calls on different caches may overlap.
 * pred_idx: device [batch][k_max] int32, strictly ascending per sequence,
 * n_pred[b] <= k_max entries. Other arguments and errors as
 * kvsel_cache_fetch (no step).
 */
KVSEL_API int kvsel_cache_prefetch(const kvsel_problem* p, const kvsel_block_cache* cache,
                                   const kvsel_bf16* host_kv, int32_t host_blocks,
                                   const int32_t* seq_lens, const int32_t* pred_idx,
                                   const int32_t* n_pred, int32_t* n_fetched, int32_t fetch_ctas,
                                   void* ws, size_t ws_bytes, kvsel_stream_t stream);

/* Budget inputs ("SparPR KV cache recovery on a consumer GPU", paragraph
 * "Dynamic budget control"). */
typedef struct kvsel_budget_in {
  int32_t block_size, kv_heads, head_dim, elem_bytes; /* one block of one layer */
  int64_t hidden;                /* model hidden size */
  int64_t n_blocks;              /* candidate blocks N */
  double h2d_bytes_per_s;        /* bandwidth the blocks are recovered over */
  double recompute_flop_per_s;   /* throughput of the recompute path */
  double kappa;                  /* flops per multiply-add of the recompute (2) */
  double keep_floor;             /* Minimum Keep Floor */
  double gamma;                  /* Dense Fallback Threshold */
  double tau_s;                  /* per-span recovery overhead, seconds */
  double keep_override;          /* >= 0: use this ratio instead of the model's */
} kvsel_budget_in;

typedef struct kvsel_budget_out {
  double c_copy_s;   /* 2 * S_blk / BW, S_blk = B * H_kv * d * elem_bytes */
  double c_rec_s;    /* kappa * B * hidden^2 / F */
  double r_model;    /* c_rec / c_copy */
  double r;          /* min(1, max(keep_floor, keep_override >= 0 ? keep_override : r_model)) */
  int64_t k;         /* clamp(floor(r * N + 1/2), 1, N); 0 when N = 0 */
  double tau_rel;    /* tau_s / c_copy */
  int32_t dense;     /* 1 if even a single-span sparse recovery is not clearly cheaper */
} kvsel_budget_out;

/*
 * kvsel_budget -- host-only, pure. The per-block copy cost is data volume over
 * host-to-device bandwidth with a factor 2 for K and V; the recompute cost
 * grows with block length and the square of the hidden size; their ratio
 * maps to the keep ratio, bounded below by the Minimum Keep Floor ("SparPR KV
 * cache recovery on a consumer GPU", paragraph "Dynamic budget control").
 * The dense decision uses the gamma rule of kvsel_score_topk with one span.
 * Errors: INVALID_ARG for null pointers, non-positive sizes or bandwidths.
 */
KVSEL_API int kvsel_budget(const kvsel_budget_in* in, kvsel_budget_out* out);

enum kvsel_ws_kind { KVSEL_WS_SCORE_TOPK = 0, KVSEL_WS_SPARSE_DECODE = 1, KVSEL_WS_CACHE_FETCH = 2 };

/* Workspace bytes an entry point needs for problem p (0 on bad input). */
KVSEL_API size_t kvsel_workspace_size(const kvsel_problem* p, int which);

/* KV bytes per cached token: 2 * layers * kv_heads * head_dim * elem_bytes
 * ("KV cache offloading", section "Why the cache leaves the GPU"). -1 on
 * negative input. */
KVSEL_API int64_t kvsel_kv_bytes_per_token(int32_t layers, int32_t kv_heads, int32_t head_dim,
                                 int32_t elem_bytes);

/* Reads and clears the current device's latched error word after draining
 * `stream` (a synchronising call). Returns KVSEL_OK or the first device error. */
KVSEL_API int kvsel_get_error(kvsel_stream_t stream);

/*
 * kvsel_selftest_wait_timeout -- exercises, on the current device, the path
 * that every bounded device wait of the library takes when it runs out: one
 * thread waits on an mbarrier phase that nothing completes; after the wait
 * limit (2 s) the wait gives up, the kernel latches KVSEL_ERR_TIMEOUT into
 * the error word and returns, and the context stays usable. The pages
 * describe no such call; it lets a deployment check its failure detection
 * without faulting or hanging the GPU. Enqueued on `stream`; the next
 * kvsel_get_error() returns KVSEL_ERR_TIMEOUT (and clears it).
 */
KVSEL_API int kvsel_selftest_wait_timeout(kvsel_stream_t stream);

/*
 * kvsel_selftest_divide -- applies, on the device, the division with which
 * the summary kernels form a block mean (an fp64 key sum over a token count:
 * one correctly rounded reciprocal, the product, its exact residual and one
 * correction step, in place of an fp64 division per channel) to n given
 * pairs: out[i] = x[i] / count[i] as those kernels compute it, before the
 * rounding to bf16. The pages describe no such call; it lets a test check
 * that division against IEEE division (the summaries are bit-exact only if
 * it is correctly rounded). x, out: device fp64 [n], 8-byte aligned; count:
 * device int32 [n], each >= 1. Enqueued on `stream`. Errors: INVALID_ARG for
 * n < 0, NULL or misaligned pointers; CUDA.
 */
KVSEL_API int kvsel_selftest_divide(const double* x, const int32_t* count, double* out, int64_t n,
                                    kvsel_stream_t stream);

/* Kernel launches made by this library since load (host-side counter). */
KVSEL_API uint64_t kvsel_launch_count(void);

/* Human-readable text of the last host-side error in this thread. */
KVSEL_API const char* kvsel_last_error(void);

KVSEL_API const char* kvsel_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KVSEL_H_ */
