// C ABI of libkvsel: argument checks, workspace sizing, the host-side budget
// model and the per-device error word. Kernels live in summaries.cu,
// score_topk.cu, sparse_decode.cu and offload.cu.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "kvsel_common.cuh"
#include "kvsel_internal.h"

namespace kvsel {

namespace {
__device__ int g_error_word;   // latched first device error (0 = none)

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
int g_smem_optin[kMaxDevices] = {};
struct SmemEntry { int dev; const void* fn; int bytes; };
SmemEntry g_smem_set[256];
int g_smem_n = 0;
std::atomic<uint64_t> g_launches{0};
thread_local char g_msg[512] = "";

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return d;
}
}  // namespace

void set_last_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
}

int* device_error_word() {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[d] = static_cast<int*>(p);
  }
  return g_err_ptr[d];
}

int sm_count() {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[d]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
    g_sms[d] = n > 0 ? n : 1;
  }
  return g_sms[d];
}

int max_smem_optin() {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_smem_optin[d]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
    g_smem_optin[d] = n;
  }
  return g_smem_optin[d];
}

cudaError_t ensure_smem(const void* kernel, int bytes) {
  const int d = current_device();
  std::lock_guard<std::mutex> lk(g_mu);
  for (int i = 0; i < g_smem_n; ++i) {
    SmemEntry& e = g_smem_set[i];
    if (e.dev == d && e.fn == kernel) {
      if (e.bytes >= bytes) return cudaSuccess;
      const cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      if (r == cudaSuccess) e.bytes = bytes;
      return r;
    }
  }
  const cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (r == cudaSuccess && g_smem_n < 256) g_smem_set[g_smem_n++] = SmemEntry{d, kernel, bytes};
  return r;
}

void count_launch(int n) { g_launches.fetch_add(uint64_t(n), std::memory_order_relaxed); }

}  // namespace kvsel

using namespace kvsel;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int fail(int code, const char* what) {
  set_last_error("%s", what);
  return code;
}

int check_problem(const kvsel_problem* p) {
  if (!p) return fail(KVSEL_ERR_INVALID_ARG, "problem is NULL");
  if (p->batch < 0 || p->batch > 4096) return fail(KVSEL_ERR_INVALID_ARG, "batch must be in [0, 4096]");
  if (p->n_qheads <= 0 || p->n_kvheads <= 0 || p->n_qheads % p->n_kvheads)
    return fail(KVSEL_ERR_INVALID_ARG, "n_qheads must be a positive multiple of n_kvheads");
  if (p->n_qheads / p->n_kvheads > 16)
    return fail(KVSEL_ERR_UNSUPPORTED, "GQA group larger than 16 query heads");
  if (p->head_dim != 64 && p->head_dim != 128)
    return fail(KVSEL_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (p->block_size != 16 && p->block_size != 32 && p->block_size != 64)
    return fail(KVSEL_ERR_UNSUPPORTED, "block_size must be 16, 32 or 64");
  if (p->max_blocks <= 0 || p->max_blocks > 16384)
    return fail(KVSEL_ERR_INVALID_ARG, "max_blocks must be in [1, 16384]");
  if (p->k_max <= 0 || p->k_max > p->max_blocks)
    return fail(KVSEL_ERR_INVALID_ARG, "k_max must be in [1, max_blocks]");
  const int nv = p->n_kvheads * p->head_dim / 8;
  int lpb = 32;
  while (nv % lpb) lpb >>= 1;
  const int vpl = nv / lpb;
  if (vpl != 1 && vpl != 2 && vpl != 4 && vpl != 8 && vpl != 16)
    return fail(KVSEL_ERR_UNSUPPORTED, "n_kvheads * head_dim not supported by the scoring kernel");
  return KVSEL_OK;
}

// An NVTX range around one entry-point call, named like the entry point, so
// that a profiler attached to the process (ncu --nvtx, nsys) groups each
// call's kernels; with no profiler attached, push and pop return at once.
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};

int cuda_status(cudaError_t e, const char* where) {
  if (e == cudaSuccess) return KVSEL_OK;
  set_last_error("%s: %s", where, cudaGetErrorString(e));
  return KVSEL_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* kvsel_version(void) { return KVSEL_VERSION_STRING; }

const char* kvsel_last_error(void) { return g_msg; }

uint64_t kvsel_launch_count(void) { return g_launches.load(); }

int64_t kvsel_kv_bytes_per_token(int32_t layers, int32_t kv_heads, int32_t head_dim,
                                 int32_t elem_bytes) {
  if (layers < 0 || kv_heads < 0 || head_dim < 0 || elem_bytes < 0) return -1;
  return int64_t(2) * layers * kv_heads * head_dim * elem_bytes;
}

size_t kvsel_workspace_size(const kvsel_problem* p, int which) {
  if (check_problem(p) != KVSEL_OK) return 0;
  if (which == KVSEL_WS_SCORE_TOPK) return score_topk_ws_bytes(*p);
  if (which == KVSEL_WS_SPARSE_DECODE) return sparse_decode_ws_bytes(*p);
  if (which == KVSEL_WS_CACHE_FETCH) return cache_fetch_ws_bytes(*p);
  return 0;
}

int kvsel_budget(const kvsel_budget_in* in, kvsel_budget_out* out) {
  if (!in || !out) return fail(KVSEL_ERR_INVALID_ARG, "budget: NULL argument");
  if (in->block_size <= 0 || in->kv_heads <= 0 || in->head_dim <= 0 || in->elem_bytes <= 0 ||
      in->hidden <= 0 || in->n_blocks < 0 || !(in->h2d_bytes_per_s > 0) ||
      !(in->recompute_flop_per_s > 0) || !(in->kappa > 0))
    return fail(KVSEL_ERR_INVALID_ARG, "budget: sizes and rates must be positive");
  const double s_blk = double(in->block_size) * in->kv_heads * in->head_dim * in->elem_bytes;
  const double c_copy = 2.0 * s_blk / in->h2d_bytes_per_s;
  const double c_rec = in->kappa * double(in->block_size) * double(in->hidden) *
                       double(in->hidden) / in->recompute_flop_per_s;
  const double r_model = c_rec / c_copy;
  const double r_src = in->keep_override >= 0.0 ? in->keep_override : r_model;
  const double r = std::fmin(1.0, std::fmax(in->keep_floor, r_src));
  int64_t k = 0;
  const int64_t N = in->n_blocks;
  if (N > 0) {
    k = int64_t(std::floor(r * double(N) + 0.5));
    k = k < 1 ? 1 : (k > N ? N : k);
  }
  const double tau_rel = in->tau_s / c_copy;
  int dense = 0;
  if (N > 0) {
    const double lhs = 1.0 * tau_rel + double(k);
    const double rhs = in->gamma * (tau_rel + double(N));
    dense = lhs >= rhs ? 1 : 0;
  }
  out->c_copy_s = c_copy;
  out->c_rec_s = c_rec;
  out->r_model = r_model;
  out->r = r;
  out->k = k;
  out->tau_rel = tau_rel;
  out->dense = dense;
  return KVSEL_OK;
}

}  // extern "C"

namespace kvsel {
namespace {
// One thread waits, with the library's bounded wait, on a barrier phase that
// nothing completes: the wait must give up and the kernel report it.
__global__ void wait_selftest_kernel(int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    if (!mbar_wait_bounded(&bar, 0u)) latch_error(err, KVSEL_ERR_TIMEOUT);
  }
}
}  // namespace
}  // namespace kvsel

extern "C" {

int kvsel_selftest_wait_timeout(kvsel_stream_t stream) {
  CallRange range("kvsel_selftest_wait_timeout");
  int* ew = device_error_word();
  if (!ew) return fail(KVSEL_ERR_CUDA, "selftest_wait_timeout: no CUDA device");
  wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(ew);
  count_launch();
  return cuda_status(cudaGetLastError(), "selftest_wait_timeout launch");
}

int kvsel_selftest_divide(const double* x, const int32_t* count, double* out, int64_t n,
                          kvsel_stream_t stream) {
  CallRange range("kvsel_selftest_divide");
  if (n < 0) return fail(KVSEL_ERR_INVALID_ARG, "selftest_divide: n must be >= 0");
  if (n == 0) return KVSEL_OK;
  if (!x || !count || !out) return fail(KVSEL_ERR_INVALID_ARG, "selftest_divide: NULL pointer");
  if ((reinterpret_cast<uintptr_t>(x) & 7u) || (reinterpret_cast<uintptr_t>(out) & 7u) || !aligned4(count))
    return fail(KVSEL_ERR_INVALID_ARG, "selftest_divide: misaligned pointer");
  return cuda_status(launch_selftest_divide(x, count, out, n, reinterpret_cast<cudaStream_t>(stream)),
                     "selftest_divide launch");
}

int kvsel_get_error(kvsel_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int r = cuda_status(cudaStreamSynchronize(s), "kvsel_get_error: stream sync");
  if (r) return r;
  int* ew = device_error_word();
  if (!ew) return fail(KVSEL_ERR_CUDA, "kvsel_get_error: no error word on this device");
  int h = 0;
  r = cuda_status(cudaMemcpy(&h, ew, sizeof(int), cudaMemcpyDeviceToHost), "kvsel_get_error: read");
  if (r) return r;
  r = cuda_status(cudaMemset(ew, 0, sizeof(int)), "kvsel_get_error: clear");
  if (r) return r;
  return h;
}

int kvsel_build_summaries(const kvsel_problem* p, int mode, kvsel_bf16* kv_pages, int64_t n_pages,
                          const int32_t* block_table, const int32_t* seq_lens,
                          const int32_t* append_pos, const kvsel_bf16* new_k,
                          const kvsel_bf16* new_v, kvsel_bf16* summaries, double* open_acc,
                          kvsel_stream_t stream) {
  CallRange range("kvsel_build_summaries");
  int r = check_problem(p);
  if (r) return r;
  if (mode != KVSEL_SUMMARY_FULL && mode != KVSEL_SUMMARY_APPEND)
    return fail(KVSEL_ERR_INVALID_ARG, "build_summaries: mode must be FULL or APPEND");
  if (p->batch == 0) return KVSEL_OK;
  if (!kv_pages || !block_table || !summaries || !open_acc || n_pages <= 0)
    return fail(KVSEL_ERR_INVALID_ARG, "build_summaries: NULL pointer or no pages");
  if (!aligned16(kv_pages) || !aligned16(summaries) || !aligned16(open_acc) || !aligned4(block_table))
    return fail(KVSEL_ERR_INVALID_ARG, "build_summaries: misaligned pointer");
  if (n_pages * p->n_kvheads * 2 * p->block_size >= (int64_t(1) << 31))
    return fail(KVSEL_ERR_UNSUPPORTED, "build_summaries: more than 2^31 cache rows");
  if (mode == KVSEL_SUMMARY_FULL && !seq_lens)
    return fail(KVSEL_ERR_INVALID_ARG, "build_summaries: FULL needs seq_lens");
  if (mode == KVSEL_SUMMARY_APPEND) {
    if (!append_pos) return fail(KVSEL_ERR_INVALID_ARG, "build_summaries: APPEND needs append_pos");
    if ((new_k && !aligned16(new_k)) || (new_v && !aligned16(new_v)))
      return fail(KVSEL_ERR_INVALID_ARG, "build_summaries: misaligned new_k/new_v");
    if (new_v && !new_k)
      return fail(KVSEL_ERR_INVALID_ARG, "build_summaries: new_v needs new_k");
  }
  int* ew = device_error_word();
  if (!ew) return fail(KVSEL_ERR_CUDA, "build_summaries: no CUDA device");
  return cuda_status(launch_build_summaries(*p, mode, kv_pages, n_pages, block_table, seq_lens,
                                            append_pos, new_k, new_v, summaries, open_acc, ew,
                                            reinterpret_cast<cudaStream_t>(stream)),
                     "build_summaries launch");
}

static int score_topk_impl(const char* who, const kvsel_problem* p, const kvsel_bf16* q,
                           const kvsel_bf16* summaries, const int32_t* seq_lens,
                           const int32_t* k_per_seq, float gamma, float tau_rel, int32_t* sel_idx,
                           int32_t* n_sel, int32_t* span_start, int32_t* span_len,
                           int32_t* n_spans, uint8_t* dense_flag, float* scores_out, void* ws,
                           size_t ws_bytes, const kvsel_append_in* app, int n_sink, int n_recent,
                           kvsel_stream_t stream) {
  char msg[160];
  if (!q || !summaries || !seq_lens || !k_per_seq || !sel_idx || !n_sel || !span_start ||
      !span_len || !n_spans) {
    std::snprintf(msg, sizeof msg, "%s: NULL pointer", who);
    return fail(KVSEL_ERR_INVALID_ARG, msg);
  }
  if (!aligned16(q) || !aligned16(summaries) || !aligned4(seq_lens) || !aligned4(k_per_seq) ||
      !aligned4(sel_idx) || !aligned4(n_sel) || !aligned4(span_start) || !aligned4(span_len) ||
      !aligned4(n_spans) || (scores_out && !aligned4(scores_out))) {
    std::snprintf(msg, sizeof msg, "%s: misaligned pointer", who);
    return fail(KVSEL_ERR_INVALID_ARG, msg);
  }
  if (!std::isfinite(gamma) || !std::isfinite(tau_rel) || tau_rel < 0) {
    std::snprintf(msg, sizeof msg, "%s: gamma and tau_rel must be finite, tau_rel >= 0", who);
    return fail(KVSEL_ERR_INVALID_ARG, msg);
  }
  if (!ws || ws_bytes < score_topk_ws_bytes(*p) || !aligned16(ws)) {
    std::snprintf(msg, sizeof msg, "%s: workspace missing, small or misaligned", who);
    return fail(KVSEL_ERR_WORKSPACE, msg);
  }
  int* ew = device_error_word();
  if (!ew) {
    std::snprintf(msg, sizeof msg, "%s: no CUDA device", who);
    return fail(KVSEL_ERR_CUDA, msg);
  }
  if (score_path() == KVSEL_SCORE_PATH_CLUSTER && score_cluster_size(*p, app != nullptr) == 0) {
    std::snprintf(msg, sizeof msg, "%s: the cluster form was requested but does not fit this problem", who);
    return fail(KVSEL_ERR_UNSUPPORTED, msg);
  }
  std::snprintf(msg, sizeof msg, "%s launch", who);
  return cuda_status(launch_score_topk(*p, q, summaries, seq_lens, k_per_seq, gamma, tau_rel,
                                       sel_idx, n_sel, span_start, span_len, n_spans, dense_flag,
                                       scores_out, ws, app, n_sink, n_recent, ew,
                                       reinterpret_cast<cudaStream_t>(stream)),
                     msg);
}

int kvsel_score_topk(const kvsel_problem* p, const kvsel_bf16* q, const kvsel_bf16* summaries,
                     const int32_t* seq_lens, const int32_t* k_per_seq, float gamma,
                     float tau_rel, int32_t* sel_idx, int32_t* n_sel, int32_t* span_start,
                     int32_t* span_len, int32_t* n_spans, uint8_t* dense_flag,
                     float* scores_out, void* ws, size_t ws_bytes, kvsel_stream_t stream) {
  CallRange range("kvsel_score_topk");
  int r = check_problem(p);
  if (r) return r;
  if (p->batch == 0) return KVSEL_OK;
  return score_topk_impl("score_topk", p, q, summaries, seq_lens, k_per_seq, gamma, tau_rel,
                         sel_idx, n_sel, span_start, span_len, n_spans, dense_flag, scores_out,
                         ws, ws_bytes, nullptr, 0, 0, stream);
}

// Checks the inputs of a folded append; returns 0 or the failure code.
static int check_append(const char* who, const kvsel_problem* p, const kvsel_append_in* app) {
  char msg[160];
  if (!app->kv_pages || !app->block_table || !app->append_pos || !app->summaries ||
      !app->open_acc || app->n_pages <= 0) {
    std::snprintf(msg, sizeof msg, "%s: NULL append pointer or no pages", who);
    return fail(KVSEL_ERR_INVALID_ARG, msg);
  }
  if (!aligned16(app->kv_pages) || !aligned16(app->summaries) || !aligned16(app->open_acc) ||
      !aligned4(app->block_table) || !aligned4(app->append_pos) ||
      (app->new_k && !aligned16(app->new_k)) || (app->new_v && !aligned16(app->new_v))) {
    std::snprintf(msg, sizeof msg, "%s: misaligned append pointer", who);
    return fail(KVSEL_ERR_INVALID_ARG, msg);
  }
  if (app->new_v && !app->new_k) {
    std::snprintf(msg, sizeof msg, "%s: new_v needs new_k", who);
    return fail(KVSEL_ERR_INVALID_ARG, msg);
  }
  if (app->n_pages * p->n_kvheads * 2 * p->block_size >= (int64_t(1) << 31)) {
    std::snprintf(msg, sizeof msg, "%s: more than 2^31 cache rows", who);
    return fail(KVSEL_ERR_UNSUPPORTED, msg);
  }
  return KVSEL_OK;
}

int kvsel_append_score_topk(const kvsel_problem* p, const kvsel_append_in* app,
                            const kvsel_bf16* q, const int32_t* seq_lens,
                            const int32_t* k_per_seq, float gamma, float tau_rel,
                            int32_t* sel_idx, int32_t* n_sel, int32_t* span_start,
                            int32_t* span_len, int32_t* n_spans, uint8_t* dense_flag,
                            float* scores_out, void* ws, size_t ws_bytes,
                            kvsel_stream_t stream) {
  CallRange range("kvsel_append_score_topk");
  int r = check_problem(p);
  if (r) return r;
  if (!app) return fail(KVSEL_ERR_INVALID_ARG, "append_score_topk: NULL append inputs");
  if (p->batch == 0) return KVSEL_OK;
  r = check_append("append_score_topk", p, app);
  if (r) return r;
  return score_topk_impl("append_score_topk", p, q, app->summaries, seq_lens, k_per_seq, gamma,
                         tau_rel, sel_idx, n_sel, span_start, span_len, n_spans, dense_flag,
                         scores_out, ws, ws_bytes, app, 0, 0, stream);
}

int kvsel_score_topk_window(const kvsel_problem* p, const kvsel_window* win,
                            const kvsel_append_in* app, const kvsel_bf16* q,
                            const kvsel_bf16* summaries, const int32_t* seq_lens,
                            const int32_t* k_per_seq, float gamma, float tau_rel,
                            int32_t* sel_idx, int32_t* n_sel, int32_t* span_start,
                            int32_t* span_len, int32_t* n_spans, uint8_t* dense_flag,
                            float* scores_out, void* ws, size_t ws_bytes,
                            kvsel_stream_t stream) {
  CallRange range("kvsel_score_topk_window");
  int r = check_problem(p);
  if (r) return r;
  if (!win) return fail(KVSEL_ERR_INVALID_ARG, "score_topk_window: NULL window");
  if (win->n_sink < 0 || win->n_recent < 0 ||
      int64_t(win->n_sink) + win->n_recent > int64_t(p->k_max))
    return fail(KVSEL_ERR_INVALID_ARG,
                "score_topk_window: need n_sink >= 0, n_recent >= 0, n_sink + n_recent <= k_max");
  if (p->batch == 0) return KVSEL_OK;
  if (app) {
    r = check_append("score_topk_window", p, app);
    if (r) return r;
    if (summaries && summaries != app->summaries)
      return fail(KVSEL_ERR_INVALID_ARG,
                  "score_topk_window: with an append, summaries must be NULL or app->summaries");
    summaries = app->summaries;
  }
  return score_topk_impl("score_topk_window", p, q, summaries, seq_lens, k_per_seq, gamma,
                         tau_rel, sel_idx, n_sel, span_start, span_len, n_spans, dense_flag,
                         scores_out, ws, ws_bytes, app, win->n_sink, win->n_recent, stream);
}

int kvsel_set_score_path(int path) {
  if (path != KVSEL_SCORE_PATH_AUTO && path != KVSEL_SCORE_PATH_TWO_GRID &&
      path != KVSEL_SCORE_PATH_CLUSTER)
    return -1;
  const int prev = score_path();
  set_score_path(path);
  return prev;
}

int kvsel_score_path_for(const kvsel_problem* p, int with_append, int32_t* cluster_ctas) {
  int r = check_problem(p);
  if (r) return -r;
  const int C = score_path() == KVSEL_SCORE_PATH_TWO_GRID ? 0 : score_cluster_size(*p, with_append != 0);
  if (cluster_ctas) *cluster_ctas = C;
  return C > 0 ? KVSEL_SCORE_PATH_CLUSTER : KVSEL_SCORE_PATH_TWO_GRID;
}

int kvsel_merge_spans(const kvsel_problem* p, const int32_t* sel_idx, const int32_t* n_sel,
                      int32_t* span_start, int32_t* span_len, int32_t* n_spans,
                      kvsel_stream_t stream) {
  CallRange range("kvsel_merge_spans");
  int r = check_problem(p);
  if (r) return r;
  if (p->batch == 0) return KVSEL_OK;
  if (!sel_idx || !n_sel || !span_start || !span_len || !n_spans)
    return fail(KVSEL_ERR_INVALID_ARG, "merge_spans: NULL pointer");
  int* ew = device_error_word();
  if (!ew) return fail(KVSEL_ERR_CUDA, "merge_spans: no CUDA device");
  return cuda_status(launch_merge_spans(*p, sel_idx, n_sel, span_start, span_len, n_spans, ew,
                                        reinterpret_cast<cudaStream_t>(stream)),
                     "merge_spans launch");
}

static int check_host_kv(const kvsel_problem* p, const kvsel_kv_src* kv, const void** dev_ptr) {
  if (!kv->host_kv || !kv->staging || kv->staging_slots <= 0 || kv->host_blocks <= 0)
    return fail(KVSEL_ERR_INVALID_ARG, "host tier: host_kv, staging, slots and host_blocks required");
  if (!aligned16(kv->host_kv) || !aligned16(kv->staging))
    return fail(KVSEL_ERR_INVALID_ARG, "host tier: misaligned pointer");
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, kv->host_kv) != cudaSuccess) {
    cudaGetLastError();
    return fail(KVSEL_ERR_INVALID_ARG, "host tier: host_kv is not known to CUDA (pin it)");
  }
  if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr)
    return fail(KVSEL_ERR_INVALID_ARG, "host tier: host_kv is not device-mapped pinned memory");
  *dev_ptr = at.devicePointer;
  const int64_t rows = int64_t(p->batch) * kv->staging_slots * p->n_kvheads * 2 * p->block_size;
  if (rows >= (int64_t(1) << 31))
    return fail(KVSEL_ERR_UNSUPPORTED, "host tier: staging larger than 2^31 rows");
  return KVSEL_OK;
}

static int check_cache(const char* who, const kvsel_problem* p, const kvsel_block_cache* c) {
  char msg[200];
  if (!c || !c->pool || !c->page_of || !c->block_in || !c->last_use) {
    std::snprintf(msg, sizeof msg, "%s: cache and its pool, page_of, block_in, last_use required", who);
    return fail(KVSEL_ERR_INVALID_ARG, msg);
  }
  if (c->slots < p->k_max || c->slots > 4096) {
    std::snprintf(msg, sizeof msg, "%s: slots must be in [k_max, 4096]", who);
    return fail(KVSEL_ERR_INVALID_ARG, msg);
  }
  if (!aligned16(c->pool) || !aligned4(c->page_of) || !aligned4(c->block_in) || !aligned4(c->last_use)) {
    std::snprintf(msg, sizeof msg, "%s: misaligned cache pointer", who);
    return fail(KVSEL_ERR_INVALID_ARG, msg);
  }
  if (int64_t(p->batch) * c->slots * p->n_kvheads * 2 * p->block_size >= (int64_t(1) << 31)) {
    std::snprintf(msg, sizeof msg, "%s: pool larger than 2^31 rows", who);
    return fail(KVSEL_ERR_UNSUPPORTED, msg);
  }
  return KVSEL_OK;
}

int kvsel_cache_reset(const kvsel_problem* p, const kvsel_block_cache* c, kvsel_stream_t stream) {
  CallRange range("kvsel_cache_reset");
  int r = check_problem(p);
  if (r) return r;
  r = check_cache("cache_reset", p, c);
  if (r) return r;
  if (p->batch == 0) return KVSEL_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // all-ones bytes are -1 in every int32 entry: no block cached, every slot empty
  cudaError_t e = cudaMemsetAsync(c->page_of, 0xFF, size_t(p->batch) * p->max_blocks * 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->block_in, 0xFF, size_t(p->batch) * c->slots * 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->last_use, 0xFF, size_t(p->batch) * c->slots * 4, s);
  return cuda_status(e, "cache_reset");
}

// kvsel_cache_fetch and kvsel_cache_prefetch: the same checks and kernels,
// on a selection (stamped with `step`) or on a prediction.
static int cache_fetch_impl(const char* who, const kvsel_problem* p, const kvsel_block_cache* c,
                            const kvsel_bf16* host_kv, int32_t host_blocks, const int32_t* seq_lens,
                            const int32_t* idx, const int32_t* n_idx, int32_t step, bool prefetch,
                            int32_t* n_fetched, int32_t fetch_ctas, void* ws, size_t ws_bytes,
                            kvsel_stream_t stream) {
  char msg[160];
  int r = check_problem(p);
  if (r) return r;
  r = check_cache(who, p, c);
  if (r) return r;
  if (p->batch == 0) return KVSEL_OK;
  if (!host_kv || host_blocks <= 0 || !seq_lens || !idx || !n_idx) {
    std::snprintf(msg, sizeof msg, "%s: host_kv, host_blocks, seq_lens and the block list required", who);
    return fail(KVSEL_ERR_INVALID_ARG, msg);
  }
  if (step < 0) {
    std::snprintf(msg, sizeof msg, "%s: step must be >= 0", who);
    return fail(KVSEL_ERR_INVALID_ARG, msg);
  }
  if (!aligned16(host_kv) || !aligned4(seq_lens) || !aligned4(idx) || !aligned4(n_idx) ||
      (n_fetched && !aligned4(n_fetched))) {
    std::snprintf(msg, sizeof msg, "%s: misaligned pointer", who);
    return fail(KVSEL_ERR_INVALID_ARG, msg);
  }
  if (!ws || ws_bytes < cache_fetch_ws_bytes(*p) || !aligned16(ws)) {
    std::snprintf(msg, sizeof msg, "%s: workspace missing, small or misaligned", who);
    return fail(KVSEL_ERR_WORKSPACE, msg);
  }
  if (cache_update_smem_bytes(*p, c->slots) > size_t(max_smem_optin())) {
    std::snprintf(msg, sizeof msg, "%s: slots and k_max exceed shared memory", who);
    return fail(KVSEL_ERR_UNSUPPORTED, msg);
  }
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, host_kv) != cudaSuccess) {
    cudaGetLastError();
    std::snprintf(msg, sizeof msg, "%s: host_kv is not known to CUDA (pin it)", who);
    return fail(KVSEL_ERR_INVALID_ARG, msg);
  }
  if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) {
    std::snprintf(msg, sizeof msg, "%s: host_kv is not device-mapped pinned memory", who);
    return fail(KVSEL_ERR_INVALID_ARG, msg);
  }
  int* ew = device_error_word();
  if (!ew) {
    std::snprintf(msg, sizeof msg, "%s: no CUDA device", who);
    return fail(KVSEL_ERR_CUDA, msg);
  }
  std::snprintf(msg, sizeof msg, "%s launch", who);
  return cuda_status(launch_cache_fetch(*p, *c, static_cast<const kvsel_bf16*>(at.devicePointer),
                                        host_blocks, seq_lens, idx, n_idx, step, prefetch, n_fetched,
                                        ws, fetch_ctas, ew, reinterpret_cast<cudaStream_t>(stream)),
                     msg);
}

int kvsel_cache_fetch(const kvsel_problem* p, const kvsel_block_cache* c, const kvsel_bf16* host_kv,
                      int32_t host_blocks, const int32_t* seq_lens, const int32_t* sel_idx,
                      const int32_t* n_sel, int32_t step, int32_t* n_fetched, int32_t fetch_ctas,
                      void* ws, size_t ws_bytes, kvsel_stream_t stream) {
  CallRange range("kvsel_cache_fetch");
  return cache_fetch_impl("cache_fetch", p, c, host_kv, host_blocks, seq_lens, sel_idx, n_sel, step,
                          false, n_fetched, fetch_ctas, ws, ws_bytes, stream);
}

int kvsel_cache_prefetch(const kvsel_problem* p, const kvsel_block_cache* c,
                         const kvsel_bf16* host_kv, int32_t host_blocks, const int32_t* seq_lens,
                         const int32_t* pred_idx, const int32_t* n_pred, int32_t* n_fetched,
                         int32_t fetch_ctas, void* ws, size_t ws_bytes, kvsel_stream_t stream) {
  CallRange range("kvsel_cache_prefetch");
  return cache_fetch_impl("cache_prefetch", p, c, host_kv, host_blocks, seq_lens, pred_idx, n_pred,
                          0, true, n_fetched, fetch_ctas, ws, ws_bytes, stream);
}

int kvsel_select_scores(const kvsel_problem* p, const float* scores, const int32_t* seq_lens,
                        const int32_t* k_per_seq, float gamma, float tau_rel, int32_t* sel_idx,
                        int32_t* n_sel, int32_t* span_start, int32_t* span_len, int32_t* n_spans,
                        uint8_t* dense_flag, kvsel_stream_t stream) {
  CallRange range("kvsel_select_scores");
  int r = check_problem(p);
  if (r) return r;
  if (p->batch == 0) return KVSEL_OK;
  if (!scores || !seq_lens || !k_per_seq || !sel_idx || !n_sel || !span_start || !span_len ||
      !n_spans)
    return fail(KVSEL_ERR_INVALID_ARG, "select_scores: NULL pointer");
  if (!aligned4(scores) || !aligned4(seq_lens) || !aligned4(k_per_seq) || !aligned4(sel_idx) ||
      !aligned4(n_sel) || !aligned4(span_start) || !aligned4(span_len) || !aligned4(n_spans))
    return fail(KVSEL_ERR_INVALID_ARG, "select_scores: misaligned pointer");
  if (!std::isfinite(gamma) || !std::isfinite(tau_rel) || tau_rel < 0)
    return fail(KVSEL_ERR_INVALID_ARG, "select_scores: gamma and tau_rel must be finite, tau_rel >= 0");
  int* ew = device_error_word();
  if (!ew) return fail(KVSEL_ERR_CUDA, "select_scores: no CUDA device");
  return cuda_status(launch_select_scores(*p, scores, seq_lens, k_per_seq, gamma, tau_rel, sel_idx,
                                          n_sel, span_start, span_len, n_spans, dense_flag, ew,
                                          reinterpret_cast<cudaStream_t>(stream)),
                     "select_scores launch");
}

int kvsel_fetch_spans(const kvsel_problem* p, const kvsel_kv_src* kv, const int32_t* seq_lens,
                      const int32_t* span_start, const int32_t* span_len,
                      const int32_t* n_spans, const uint8_t* dense_flag,
                      kvsel_stream_t stream) {
  CallRange range("kvsel_fetch_spans");
  int r = check_problem(p);
  if (r) return r;
  if (!kv || kv->kind != KVSEL_KV_HOST)
    return fail(KVSEL_ERR_INVALID_ARG, "fetch_spans: kv source must be KVSEL_KV_HOST");
  if (p->batch == 0) return KVSEL_OK;
  if (!seq_lens || !span_start || !span_len || !n_spans)
    return fail(KVSEL_ERR_INVALID_ARG, "fetch_spans: NULL pointer");
  const void* dev_host = nullptr;
  r = check_host_kv(p, kv, &dev_host);
  if (r) return r;
  kvsel_kv_src k2 = *kv;
  k2.host_kv = static_cast<const kvsel_bf16*>(dev_host);
  int* ew = device_error_word();
  if (!ew) return fail(KVSEL_ERR_CUDA, "fetch_spans: no CUDA device");
  return cuda_status(launch_fetch_spans(*p, k2, seq_lens, span_start, span_len, n_spans,
                                        dense_flag, ew, reinterpret_cast<cudaStream_t>(stream)),
                     "fetch_spans launch");
}

int kvsel_sparse_decode(const kvsel_problem* p, const kvsel_bf16* q, const kvsel_kv_src* kv,
                        const int32_t* seq_lens, const int32_t* sel_idx, const int32_t* n_sel,
                        const int32_t* span_start, const int32_t* span_len,
                        const int32_t* n_spans, const uint8_t* dense_flag, float softmax_scale,
                        float* out, kvsel_bf16* out_bf16, float* lse, void* ws,
                        size_t ws_bytes, kvsel_stream_t stream) {
  CallRange range("kvsel_sparse_decode");
  int r = check_problem(p);
  if (r) return r;
  if (!kv) return fail(KVSEL_ERR_INVALID_ARG, "sparse_decode: kv is NULL");
  if (p->batch == 0) return KVSEL_OK;
  if (!q || !seq_lens || !sel_idx || !n_sel || !out || !lse)
    return fail(KVSEL_ERR_INVALID_ARG, "sparse_decode: NULL pointer");
  if (!aligned16(q) || !aligned16(out) || !aligned4(lse) || !aligned4(sel_idx) ||
      !aligned4(n_sel) || !aligned4(seq_lens) || (out_bf16 && !aligned16(out_bf16)))
    return fail(KVSEL_ERR_INVALID_ARG, "sparse_decode: misaligned pointer");
  if (!std::isfinite(softmax_scale))
    return fail(KVSEL_ERR_INVALID_ARG, "sparse_decode: softmax_scale must be finite");
  // the tile list is counted in int32 (every block of every sequence, dense, per KV head)
  if (int64_t(p->batch) * p->n_kvheads * p->max_blocks >= (int64_t(1) << 31))
    return fail(KVSEL_ERR_UNSUPPORTED, "sparse_decode: batch * n_kvheads * max_blocks must be below 2^31");
  if (!ws || ws_bytes < sparse_decode_ws_bytes(*p) || !aligned16(ws))
    return fail(KVSEL_ERR_WORKSPACE, "sparse_decode: workspace missing, small or misaligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* ew = device_error_word();
  if (!ew) return fail(KVSEL_ERR_CUDA, "sparse_decode: no CUDA device");
  kvsel_kv_src src = *kv;
  if (kv->kind == KVSEL_KV_PAGED) {
    if (!kv->kv_pages || !kv->block_table || kv->n_pages <= 0)
      return fail(KVSEL_ERR_INVALID_ARG, "sparse_decode: paged source needs pages and a block table");
    if (!aligned16(kv->kv_pages))
      return fail(KVSEL_ERR_INVALID_ARG, "sparse_decode: misaligned pages");
    if (kv->n_pages * p->n_kvheads * 2 * p->block_size >= (int64_t(1) << 31))
      return fail(KVSEL_ERR_UNSUPPORTED, "sparse_decode: more than 2^31 cache rows");
  } else if (kv->kind == KVSEL_KV_STAGED || kv->kind == KVSEL_KV_HOST) {
    if (kv->kind == KVSEL_KV_HOST) {
      if (!span_start || !span_len || !n_spans)
        return fail(KVSEL_ERR_INVALID_ARG, "sparse_decode: host source needs the spans");
      const void* dev_host = nullptr;
      r = check_host_kv(p, kv, &dev_host);
      if (r) return r;
      src.host_kv = static_cast<const kvsel_bf16*>(dev_host);
      r = cuda_status(launch_fetch_spans(*p, src, seq_lens, span_start, span_len, n_spans,
                                         dense_flag, ew, s),
                      "sparse_decode fetch launch");
      if (r) return r;
    }
    if (!kv->staging || kv->staging_slots <= 0 || !aligned16(kv->staging))
      return fail(KVSEL_ERR_INVALID_ARG, "sparse_decode: staging buffer and slots required");
    if (int64_t(p->batch) * kv->staging_slots * 2 * p->n_kvheads * p->block_size >= (int64_t(1) << 31))
      return fail(KVSEL_ERR_UNSUPPORTED, "sparse_decode: staging larger than 2^31 rows");
    src.kind = KVSEL_KV_STAGED;
  } else if (kv->kind == KVSEL_KV_HOST_DIRECT) {
    if (!kv->host_kv || kv->host_blocks <= 0 || !aligned16(kv->host_kv))
      return fail(KVSEL_ERR_INVALID_ARG, "sparse_decode: host_direct needs an aligned host_kv and host_blocks");
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, kv->host_kv) != cudaSuccess) {
      cudaGetLastError();
      return fail(KVSEL_ERR_INVALID_ARG, "sparse_decode: host_kv is not known to CUDA (pin it)");
    }
    if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr)
      return fail(KVSEL_ERR_INVALID_ARG, "sparse_decode: host_kv is not device-mapped pinned memory");
    if (!aligned16(at.devicePointer))
      return fail(KVSEL_ERR_INVALID_ARG, "sparse_decode: misaligned host_kv mapping");
    if (int64_t(p->batch) * kv->host_blocks * p->n_kvheads >= (int64_t(1) << 31))
      return fail(KVSEL_ERR_UNSUPPORTED, "sparse_decode: host tier larger than 2^31 tiles");
    src.host_kv = static_cast<const kvsel_bf16*>(at.devicePointer);
  } else {
    return fail(KVSEL_ERR_INVALID_ARG, "sparse_decode: unknown kv kind");
  }
  return cuda_status(launch_sparse_decode(*p, q, src, seq_lens, sel_idx, n_sel, dense_flag,
                                          softmax_scale, out, out_bf16, lse, ws, ew, s),
                     "sparse_decode launch");
}

}  // extern "C"
