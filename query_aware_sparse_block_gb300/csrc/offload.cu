// Offload tier: full K/V stays in pinned host memory, only the selected spans
// cross the host link ("SparPR KV cache recovery on a consumer GPU",
// paragraph "Query-Aware key-block selection": scoring touches only the
// GPU-resident summaries, never the offloaded blocks; "KV cache offloading",
// sections "Fetching a sparse subset per step" and "NOSA": the GPU reads host
// memory directly through unified virtual addressing).
//
// The gather kernel copies, for every sequence, the blocks of its spans (or
// all blocks when the dense fallback fired) from the host tier
// [b][host_blocks][one KV page] into consecutive staging slots
// [b][slots][one KV page]; a page is copied opaquely. Each CTA owns one sequence row of the grid and a
// share of that sequence's blocks; within a block the CTA streams 16-byte
// host reads with several requests in flight per thread. The span list never
// leaves the GPU, so there is no host round trip between selection and fetch.
#include "kvsel_common.cuh"
#include "kvsel_internal.h"

namespace kvsel {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;

__global__ void __launch_bounds__(kThreads) fetch_spans_kernel(
    const kvsel_bf16* __restrict__ host_kv, kvsel_bf16* __restrict__ staging,
    const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ span_start,
    const int32_t* __restrict__ span_len, const int32_t* __restrict__ n_spans,
    const uint8_t* __restrict__ dense_flag, int host_blocks, int slots, int B, int max_blocks,
    int k_max, int64_t block_vec, int* err) {
  extern __shared__ int pref_s[];     // [k_max + 1] prefix of span lengths
  const int b = blockIdx.y;
  const int tid = threadIdx.x;
  int T = seq_lens[b];
  T = T < 0 ? 0 : min(T, max_blocks * B);
  const int N = (T + B - 1) / B;
  const bool dense = dense_flag && dense_flag[b];
  int ns = 0, total = 0;
  if (dense) {
    total = N;
  } else {
    ns = n_spans[b];
    if (ns < 0 || ns > k_max) {
      if (tid == 0 && blockIdx.x == 0) latch_error(err, KVSEL_ERR_BOUNDS);
      ns = ns < 0 ? 0 : k_max;
    }
    // serial prefix (span lists are short) by thread 0, then shared
    if (tid == 0) {
      int acc = 0;
      pref_s[0] = 0;
      for (int s = 0; s < ns; ++s) {
        int l = span_len[int64_t(b) * k_max + s];
        l = l < 0 ? 0 : l;
        acc += l;
        pref_s[s + 1] = acc;
      }
    }
    __syncthreads();
    total = pref_s[ns];
  }
  if (total > slots) {
    if (tid == 0 && blockIdx.x == 0) latch_error(err, KVSEL_ERR_BOUNDS);
    total = slots;
  }
  const int per = (total + gridDim.x - 1) / gridDim.x;
  const int o0 = blockIdx.x * per, o1 = min(total, o0 + per);
  for (int o = o0; o < o1; ++o) {
    int n;
    if (dense) {
      n = o;
    } else {
      int lo = 0, hi = ns - 1;          // span s with pref[s] <= o < pref[s+1]
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pref_s[mid] <= o) lo = mid; else hi = mid - 1;
      }
      n = span_start[int64_t(b) * k_max + lo] + (o - pref_s[lo]);
    }
    if (n < 0 || n >= N || n >= host_blocks) {
      if (tid == 0) latch_error(err, KVSEL_ERR_BOUNDS);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(host_kv) + (int64_t(b) * host_blocks + n) * block_vec;
    uint4* dst = reinterpret_cast<uint4*>(staging) + (int64_t(b) * slots + o) * block_vec;
    int64_t v = tid;
    for (; v + (kUnroll - 1) * kThreads < block_vec; v += kUnroll * kThreads) {
      uint4 r[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) r[u] = ld_sys_v4(src + v + u * kThreads);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) stg_stream(dst + v + u * kThreads, r[u]);
    }
    for (; v < block_vec; v += kThreads) stg_stream(dst + v, ld_sys_v4(src + v));
  }
}

}  // namespace

cudaError_t launch_fetch_spans(const kvsel_problem& p, const kvsel_kv_src& kv,
                               const int32_t* seq_lens, const int32_t* span_start,
                               const int32_t* span_len, const int32_t* n_spans,
                               const uint8_t* dense_flag, int* err, cudaStream_t s) {
  if (p.batch == 0) return cudaSuccess;
  const int64_t block_vec = int64_t(2) * p.n_kvheads * p.block_size * p.head_dim * 2 / 16;
  const int64_t ctas = kv.fetch_ctas > 0 ? kv.fetch_ctas : sm_count();
  const int per_seq = int(std::min<int64_t>(std::max<int64_t>(1, (ctas + p.batch - 1) / p.batch),
                                            std::max(1, kv.staging_slots)));
  dim3 grid(per_seq, p.batch);
  const size_t smem = (size_t(p.k_max) + 1) * 4;
  if (smem > 48 * 1024) {
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(fetch_spans_kernel), int(smem));
    if (e != cudaSuccess) return e;
  }
  fetch_spans_kernel<<<grid, kThreads, smem, s>>>(kv.host_kv, kv.staging, seq_lens, span_start,
                                                 span_len, n_spans, dense_flag, kv.host_blocks,
                                                 kv.staging_slots, p.block_size, p.max_blocks,
                                                 p.k_max, block_vec, err);
  count_launch();
  return cudaGetLastError();
}

}  // namespace kvsel
