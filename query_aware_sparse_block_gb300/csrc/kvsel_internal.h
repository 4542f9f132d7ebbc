// Host-side launchers shared between the C-ABI layer (api.cu) and the kernel
// translation units. Arguments are validated by the caller before a launcher
// runs; launchers only size grids and enqueue work.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kvsel.h"

namespace kvsel {

// Per-device error word (device address) and launch counter.
int* device_error_word();
void count_launch(int n = 1);
int sm_count();
int max_smem_optin();
// Raises the kernel's dynamic shared-memory limit to at least `bytes`, calling
// the runtime only the first time a larger size is needed on this device.
cudaError_t ensure_smem(const void* kernel, int bytes);
void set_last_error(const char* fmt, ...);

// ---- summaries (summaries.cu) ----
cudaError_t launch_build_summaries(const kvsel_problem& p, int mode, kvsel_bf16* kv_pages,
                                   int64_t n_pages, const int32_t* block_table,
                                   const int32_t* seq_lens, const int32_t* append_pos,
                                   const kvsel_bf16* new_k, const kvsel_bf16* new_v,
                                   kvsel_bf16* summaries, double* open_acc, int* err,
                                   cudaStream_t s);

// The block-mean division of the summary kernels on given (sum, count) pairs
// (summaries.cu), for kvsel_selftest_divide.
cudaError_t launch_selftest_divide(const double* x, const int32_t* cnt, double* out, int64_t n,
                                   cudaStream_t s);

// ---- score + Top-k + spans (score_topk.cu); app != nullptr folds the
// APPEND summary update into the score grid; the first n_sink and the last
// n_recent blocks of every sequence are selected whatever their score ----
size_t score_topk_ws_bytes(const kvsel_problem& p);
cudaError_t launch_score_topk(const kvsel_problem& p, const kvsel_bf16* q,
                              const kvsel_bf16* summaries, const int32_t* seq_lens,
                              const int32_t* k_per_seq, float gamma, float tau_rel,
                              int32_t* sel_idx, int32_t* n_sel, int32_t* span_start,
                              int32_t* span_len, int32_t* n_spans, uint8_t* dense_flag,
                              float* scores_out, void* ws, const kvsel_append_in* app,
                              int n_sink, int n_recent, int* err, cudaStream_t s);
// The one-launch form of launch_score_topk (score_cluster.cu): one
// thread-block cluster per sequence. *launched = false (and nothing enqueued)
// when the problem is outside that form; launch_score_topk then uses its
// two grids.
cudaError_t launch_score_topk_cluster(const kvsel_problem& p, const kvsel_bf16* q,
                                      const kvsel_bf16* summaries, const int32_t* seq_lens,
                                      const int32_t* k_per_seq, float gamma, float tau_rel,
                                      int32_t* sel_idx, int32_t* n_sel, int32_t* span_start,
                                      int32_t* span_len, int32_t* n_spans, uint8_t* dense_flag,
                                      float* scores_out, const kvsel_append_in* app, int n_sink,
                                      int n_recent, int* err, cudaStream_t s, bool* launched);
// CTAs per cluster the one-launch form takes for p on the current device (0:
// outside it).
int score_cluster_size(const kvsel_problem& p, bool app);
// Process-wide choice between the forms (KVSEL_SCORE_PATH_*).
void set_score_path(int path);
int score_path();
cudaError_t launch_select_scores(const kvsel_problem& p, const float* scores,
                                 const int32_t* seq_lens, const int32_t* k_per_seq, float gamma,
                                 float tau_rel, int32_t* sel_idx, int32_t* n_sel,
                                 int32_t* span_start, int32_t* span_len, int32_t* n_spans,
                                 uint8_t* dense_flag, int* err, cudaStream_t s);
cudaError_t launch_merge_spans(const kvsel_problem& p, const int32_t* sel_idx,
                               const int32_t* n_sel, int32_t* span_start, int32_t* span_len,
                               int32_t* n_spans, int* err, cudaStream_t s);

// ---- sparse decode (sparse_decode.cu) ----
size_t sparse_decode_ws_bytes(const kvsel_problem& p);
cudaError_t launch_sparse_decode(const kvsel_problem& p, const kvsel_bf16* q,
                                 const kvsel_kv_src& kv, const int32_t* seq_lens,
                                 const int32_t* sel_idx, const int32_t* n_sel,
                                 const uint8_t* dense_flag, float softmax_scale, float* out,
                                 kvsel_bf16* out_bf16, float* lse, void* ws, int* err,
                                 cudaStream_t s);

// ---- offload tier (offload.cu) ----
cudaError_t launch_fetch_spans(const kvsel_problem& p, const kvsel_kv_src& kv,
                               const int32_t* seq_lens, const int32_t* span_start,
                               const int32_t* span_len, const int32_t* n_spans,
                               const uint8_t* dense_flag, int* err, cudaStream_t s);

// ---- GPU-resident block cache of the host tier (block_cache.cu) ----
size_t cache_fetch_ws_bytes(const kvsel_problem& p);
size_t cache_update_smem_bytes(const kvsel_problem& p, int slots);
cudaError_t launch_cache_fetch(const kvsel_problem& p, const kvsel_block_cache& c,
                               const kvsel_bf16* host_kv, int host_blocks,
                               const int32_t* seq_lens, const int32_t* sel_idx,
                               const int32_t* n_sel, int step, bool prefetch, int32_t* n_fetched,
                               void* ws, int fetch_ctas, int* err, cudaStream_t s);

}  // namespace kvsel
