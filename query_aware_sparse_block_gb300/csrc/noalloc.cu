// kvsel_score_topk_noalloc: the score + Top-k + span entry point for callers
// that cannot allocate device memory themselves. Its scratch (the fp32 score
// row of every sequence) lives in a fixed file-scope device array of this
// library instead of a caller workspace. Every score is written before it is
// read within one call, so nothing in the array has to start at zero.
//
// The array is a device symbol: host code cannot use its name as an address.
// Its device address is looked up once per device with cudaGetSymbolAddress,
// with that device current, on the first call made on that device.
#include <mutex>

#include "kvsel_common.cuh"
#include "kvsel_internal.h"

namespace kvsel {
namespace {

// 4 MiB: scores for batch * max_blocks <= about one million blocks.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDev] = {};

cudaError_t scratch_address(void** out) {
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  if (d < 0 || d >= kMaxDev) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[d]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[d] = p;
  }
  *out = g_scratch_ptr[d];
  return cudaSuccess;
}

}  // namespace
}  // namespace kvsel

extern "C" {

KVSEL_API size_t kvsel_noalloc_scratch_bytes(void) { return kvsel::kNoAllocScratchBytes; }

KVSEL_API int kvsel_score_topk_noalloc(const kvsel_problem* p, const kvsel_bf16* q,
                                       const kvsel_bf16* summaries, const int32_t* seq_lens,
                                       const int32_t* k_per_seq, float gamma, float tau_rel,
                                       int32_t* sel_idx, int32_t* n_sel, int32_t* span_start,
                                       int32_t* span_len, int32_t* n_spans, uint8_t* dense_flag,
                                       float* scores_out, kvsel_stream_t stream) {
  const size_t need = kvsel_workspace_size(p, KVSEL_WS_SCORE_TOPK);
  if (need == 0)  // invalid problem: the regular entry point reports why
    return kvsel_score_topk(p, q, summaries, seq_lens, k_per_seq, gamma, tau_rel, sel_idx, n_sel,
                            span_start, span_len, n_spans, dense_flag, scores_out, nullptr, 0,
                            stream);
  if (need > kvsel::kNoAllocScratchBytes) {
    kvsel::set_last_error(
        "score_topk_noalloc: this problem needs %zu bytes of scratch; the static array holds %zu "
        "(batch * max_blocks too large); use kvsel_score_topk with a workspace",
        need, kvsel::kNoAllocScratchBytes);
    return KVSEL_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  cudaError_t e = kvsel::scratch_address(&scratch);
  if (e != cudaSuccess) {
    kvsel::set_last_error("score_topk_noalloc: scratch address: %s", cudaGetErrorString(e));
    return KVSEL_ERR_CUDA;
  }
  return kvsel_score_topk(p, q, summaries, seq_lens, k_per_seq, gamma, tau_rel, sel_idx, n_sel,
                          span_start, span_len, n_spans, dense_flag, scores_out, scratch,
                          kvsel::kNoAllocScratchBytes, stream);
}

}  // extern "C"
