// Block summaries: the mean key of every KV block, one vector per KV head
// ("SparPR KV cache recovery on a consumer GPU", paragraph "Query-Aware
// key-block selection": a compact precomputed summary per block, resident on
// the GPU), plus the incremental update as decode appends tokens.
//
// Arithmetic (summary_math.cuh): each summary element is the fp64 sum of the
// block's keys in token order, divided by the token count and rounded once to
// bf16.
#include "kvsel_common.cuh"
#include "kvsel_internal.h"
#include "summary_math.cuh"

namespace kvsel {
namespace {

constexpr int kThreads = 128;

// A CTA takes `bpc` consecutive blocks of sequence b (as many as its threads
// cover: one thread per 8-channel column vector of one KV head, so a block of
// few heads shares the CTA with its neighbours). Each thread walks its
// column's tokens in order (pages in the tiled layout).
__global__ void __launch_bounds__(kThreads) summaries_full_kernel(
    const kvsel_bf16* __restrict__ kv_pages, int64_t n_pages, const int32_t* __restrict__ block_table,
    const int32_t* __restrict__ seq_lens, kvsel_bf16* __restrict__ summaries,
    double* __restrict__ open_acc, int H, int d, int B, int max_blocks, int* err) {
  // a kernel launched after this one with programmatic serialization may
  // become resident now; it waits for this grid's completion before reading
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int vec_per_head = d / 8;
  const int n_vec = H * vec_per_head;
  const int bpc = n_vec >= kThreads ? 1 : kThreads / n_vec;     // blocks per CTA
  const int sub = n_vec >= kThreads ? 0 : int(threadIdx.x) / n_vec;
  if (sub >= bpc) return;                                        // threads past the last block
  const int lt = n_vec >= kThreads ? int(threadIdx.x) : int(threadIdx.x) % n_vec;
  const int step = n_vec >= kThreads ? kThreads : n_vec;
  const int n = blockIdx.x * bpc + sub;
  const int b = blockIdx.y;
  int T = seq_lens[b];
  if (T < 0 || T > max_blocks * B) {
    if (n == 0 && lt == 0) latch_error(err, KVSEL_ERR_BOUNDS);
    T = T < 0 ? 0 : max_blocks * B;
  }
  const int N = (T + B - 1) / B;
  if (N == 0) {
    if (n == 0)
      for (int i = lt; i < H * d; i += step) open_acc[int64_t(b) * H * d + i] = 0.0;
    return;
  }
  if (n >= N) return;
  const int64_t page = block_table[int64_t(b) * max_blocks + n];
  if (page < 0 || page >= n_pages) {
    if (lt == 0) latch_error(err, KVSEL_ERR_BOUNDS);
    return;
  }
  const int cnt = min(B, T - n * B);
  for (int v = lt; v < n_vec; v += step) {
    const int j = v / vec_per_head;
    const int c0 = (v % vec_per_head) * 8;
    const kvsel_bf16* tile = kv_pages + (page * H + j) * 2 * int64_t(B) * d;
    // the exact sum on the integer pipe (equal to the sequential fp64 sum when
    // the column's exponents lie within 39 of each other), else the fp64 sum
    ExactSum es[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) exact_init(es[i]);
    {
      int t = 0;
      for (; t + 8 <= cnt; t += 8) {
        uint4 r[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) r[u] = ldg_stream(tile + tiled_off(t + u, c0, B));
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t w[4] = {r[u].x, r[u].y, r[u].z, r[u].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            exact_add(es[2 * i], w[i] & 0xFFFFu);
            exact_add(es[2 * i + 1], w[i] >> 16);
          }
        }
      }
      for (; t < cnt; ++t) {
        const uint4 r = ldg_stream(tile + tiled_off(t, c0, B));
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          exact_add(es[2 * i], w[i] & 0xFFFFu);
          exact_add(es[2 * i + 1], w[i] >> 16);
        }
      }
    }
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) bad = bad || es[i].bad;
    double acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = exact_result(es[i]);
    if (bad) {
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0;
    int t = 0;
    for (; t + 8 <= cnt; t += 8) {
      uint4 r[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) r[u] = ldg_stream(tile + tiled_off(t + u, c0, B));
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        double x[8];
        unpack8(r[u], x);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += x[i];
      }
    }
    for (; t < cnt; ++t) {
      double x[8];
      unpack8(ldg_stream(tile + tiled_off(t, c0, B)), x);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += x[i];
    }
    }
    const int64_t so = ((int64_t(b) * max_blocks + n) * H + j) * d + c0;
    *reinterpret_cast<uint4*>(summaries + so) = mean_to_bf16x8(acc, cnt);
    if (n == N - 1) {
      double* oa = open_acc + (int64_t(b) * H + j) * d + c0;
#pragma unroll
      for (int i = 0; i < 8; ++i) oa[i] = acc[i];
    }
  }
}

// One CTA per sequence: write the new token (optional), fold it into the open
// block's fp64 accumulator and rewrite that block's summary.
__global__ void __launch_bounds__(kThreads) summaries_append_kernel(
    kvsel_bf16* __restrict__ kv_pages, int64_t n_pages,
    const int32_t* __restrict__ block_table, const int32_t* __restrict__ append_pos,
    const kvsel_bf16* __restrict__ new_k, const kvsel_bf16* __restrict__ new_v,
    kvsel_bf16* __restrict__ summaries, double* __restrict__ open_acc, int H, int d, int B,
    int max_blocks, int* err) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int b = blockIdx.x;
  const int t = append_pos[b];
  if (t < 0) return;
  if (t >= max_blocks * B) {
    if (threadIdx.x == 0) latch_error(err, KVSEL_ERR_BOUNDS);
    return;
  }
  const int n = t / B;
  const int row = t % B;
  const int64_t page = block_table[int64_t(b) * max_blocks + n];
  if (page < 0 || page >= n_pages) {
    if (threadIdx.x == 0) latch_error(err, KVSEL_ERR_BOUNDS);
    return;
  }
  const int vec_per_head = d / 8;
  const int n_vec = H * vec_per_head;
  for (int v = threadIdx.x; v < n_vec; v += blockDim.x) {
    const int j = v / vec_per_head;
    const int c0 = (v % vec_per_head) * 8;
    const int64_t k_off = (page * H + j) * 2 * int64_t(B) * d + tiled_off(row, c0, B);
    const int64_t v_off = k_off + int64_t(B) * d;
    const int64_t tok_off = (int64_t(b) * H + j) * d + c0;
    uint4 kv;
    if (new_k) {
      kv = *reinterpret_cast<const uint4*>(new_k + tok_off);
      *reinterpret_cast<uint4*>(kv_pages + k_off) = kv;
      if (new_v)
        *reinterpret_cast<uint4*>(kv_pages + v_off) = *reinterpret_cast<const uint4*>(new_v + tok_off);
    } else {
      kv = *reinterpret_cast<const uint4*>(kv_pages + k_off);
    }
    double x[8];
    unpack8(kv, x);
    double* oa = open_acc + tok_off;
    double acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      acc[i] = (row == 0 ? 0.0 : oa[i]) + x[i];
      oa[i] = acc[i];
    }
    const int64_t so = ((int64_t(b) * max_blocks + n) * H + j) * d + c0;
    *reinterpret_cast<uint4*>(summaries + so) = mean_to_bf16x8(acc, row + 1);
  }
}

// The division of a block mean, applied to given (sum, count) pairs: the
// same reciprocal and correction step as mean_to_bf16x8, without the final
// rounding to bf16.
__global__ void selftest_divide_kernel(const double* __restrict__ x, const int32_t* __restrict__ cnt,
                                       double* __restrict__ out, int64_t n) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
    const double c = static_cast<double>(cnt[i]);
    out[i] = div_by_count(x[i], c, 1.0 / c);
  }
}

}  // namespace

cudaError_t launch_build_summaries(const kvsel_problem& p, int mode, kvsel_bf16* kv_pages,
                                   int64_t n_pages, const int32_t* block_table,
                                   const int32_t* seq_lens, const int32_t* append_pos,
                                   const kvsel_bf16* new_k, const kvsel_bf16* new_v,
                                   kvsel_bf16* summaries, double* open_acc, int* err,
                                   cudaStream_t s) {
  if (p.batch == 0) return cudaSuccess;
  if (mode == KVSEL_SUMMARY_FULL) {
    const int n_vec = p.n_kvheads * p.head_dim / 8;
    const int bpc = n_vec >= kThreads ? 1 : kThreads / n_vec;
    dim3 grid((p.max_blocks + bpc - 1) / bpc, p.batch);
    summaries_full_kernel<<<grid, kThreads, 0, s>>>(kv_pages, n_pages, block_table, seq_lens,
                                                    summaries, open_acc, p.n_kvheads, p.head_dim,
                                                    p.block_size, p.max_blocks, err);
  } else {
    summaries_append_kernel<<<p.batch, kThreads, 0, s>>>(
        kv_pages, n_pages, block_table, append_pos, new_k, new_v, summaries, open_acc, p.n_kvheads,
        p.head_dim, p.block_size, p.max_blocks, err);
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_selftest_divide(const double* x, const int32_t* cnt, double* out, int64_t n,
                                   cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>(int64_t(sm_count()) * 8, (n + 255) / 256);
  selftest_divide_kernel<<<unsigned(blocks), 256, 0, s>>>(x, cnt, out, n);
  count_launch();
  return cudaGetLastError();
}

}  // namespace kvsel
