// GPU-resident cache of host-tier blocks ("KV cache offloading", section
// "NOSA": block selection is local across consecutive decode steps, so the
// blocks fetched in one step are kept on the GPU and reused in the next, and
// an eviction policy bounds the blocks fetched from host memory).
//
// Every sequence owns `slots` pages of a device pool. The state is three
// int32 arrays: page_of[b][n] (the pool page holding block n, or -1),
// block_in[b][s] (the block in slot s, or -1) and last_use[b][s] (the last
// step in which slot s was selected, -1 while empty). A step:
//   1. cache_update_kernel, one CTA per sequence: a selected block that is
//      resident is a hit and its slot is stamped with the step; the misses,
//      in ascending block order, take the slots not stamped this step in the
//      order of (last_use, slot) -- least recently selected first, empty
//      slots before any -- found by a bitonic sort of those keys in shared
//      memory. The evicted blocks' page_of entries are cleared, the new ones
//      set, and a job list (block, pool page) is written: the misses, then
//      the block holding the last token if it was a hit (appends change that
//      block, so its copy is fetched again).
//   2. cache_copy_kernel: every job copies one block from pinned host memory
//      (read through unified virtual addressing) into its pool page.
// The decode then reads the pool as a paged cache with page_of as its block
// table, so only the misses cross the host link.
//
// A prefetch ("KV cache offloading": the Hugging Face Transformers paragraph,
// the next layer's cache fetched ahead of its use; section "SparDA", the
// blocks a layer will select fetched on a dedicated stream while the layer
// before it runs) is the same two kernels on a predicted block list, with
// three differences in step 1: a resident predicted block is left as it is
// (no stamp); the victims are the slots holding no predicted block; a filled
// slot gets the stamp -1 (never selected), so that a wrong prediction is the
// first to go. The block holding the last token is not prefetched.
#include "kvsel_common.cuh"
#include "kvsel_internal.h"

namespace kvsel {
namespace {

constexpr int kUpdThreads = 512;
constexpr int kUpdWarps = kUpdThreads / 32;
constexpr int kCopyThreads = 256;
constexpr int kUnroll = 8;

struct CacheArgs {
  const int32_t* seq_lens;
  const int32_t* sel_idx;
  const int32_t* n_sel;
  int32_t* page_of;      // [batch][max_blocks]
  int32_t* block_in;     // [batch][slots]
  int32_t* last_use;     // [batch][slots]
  int2* jobs;            // [batch][k_max + 1] (block, pool page)
  int32_t* n_jobs;       // [batch]
  int32_t* n_fetched;    // [batch], nullable
  int slots, pow2, max_blocks, k_max, B, host_blocks, step;
  int prefetch;          // 1: the list is a prediction (see above)
  int* err;
};

__global__ void __launch_bounds__(kUpdThreads) cache_update_kernel(CacheArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned long long* key_s = reinterpret_cast<unsigned long long*>(smem_raw);   // [pow2]
  int* use_s = reinterpret_cast<int*>(key_s + a.pow2);                          // [slots]
  int* blk_s = use_s + a.slots;                                                  // [slots]
  int* miss_s = blk_s + a.slots;                                                 // [k_max]
  int* scan_s = miss_s + a.k_max;                                                // [kUpdWarps + 4]
  unsigned char* pin_s = reinterpret_cast<unsigned char*>(scan_s + kUpdWarps + 4);  // [slots]
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = a.slots;
  int T = a.seq_lens[b];
  T = T < 0 ? 0 : min(T, a.max_blocks * a.B);
  const int N = (T + a.B - 1) / a.B;
  int n = a.n_sel[b];
  if (n < 0 || n > a.k_max) {
    if (tid == 0) latch_error(a.err, KVSEL_ERR_BOUNDS);
    n = n < 0 ? 0 : a.k_max;
  }
  int32_t* page_row = a.page_of + int64_t(b) * a.max_blocks;
  const int32_t* sel = a.sel_idx + int64_t(b) * a.k_max;
  for (int s = tid; s < C; s += kUpdThreads) {
    use_s[s] = a.last_use[int64_t(b) * C + s];
    blk_s[s] = a.block_in[int64_t(b) * C + s];
    pin_s[s] = 0;
  }
  if (tid == 0) scan_s[kUpdWarps] = -1;          // refresh job: pool page, or -1
  __syncthreads();

  // ---- hits and misses, selection entries in contiguous per-thread ranges ----
  const int per = (n + kUpdThreads - 1) / kUpdThreads;
  const int i0 = min(n, tid * per), i1 = min(n, i0 + per);
  int n_miss = 0;
  for (int i = i0; i < i1; ++i) {
    const int blk = sel[i];
    if (blk < 0 || blk >= N || blk >= a.host_blocks || (i > 0 && sel[i - 1] >= blk)) {
      latch_error(a.err, KVSEL_ERR_BOUNDS);      // not ascending or out of range: not served
      continue;
    }
    const int pg = page_row[blk];
    const int s = pg - b * C;
    if (pg >= 0 && s >= 0 && s < C && blk_s[s] == blk) {
      if (a.prefetch) {
        pin_s[s] = 1;                            // stays; no stamp
      } else {
        use_s[s] = a.step;
        if (blk == N - 1) scan_s[kUpdWarps] = pg;  // the open block: fetch its copy again
      }
    } else {
      if (pg >= 0) latch_error(a.err, KVSEL_ERR_BOUNDS);   // inconsistent state: refetch
      if (!a.prefetch || blk != N - 1) ++n_miss;
    }
  }
  // exclusive scan of the miss counts gives each miss its rank in block order
  int x = n_miss;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) scan_s[warp] = x;
  __syncthreads();
  int base = 0, m = 0;
  for (int w = 0; w < kUpdWarps; ++w) {
    const int v = scan_s[w];
    if (w < warp) base += v;
    m += v;
  }
  int r = base + x - n_miss;
  for (int i = i0; i < i1; ++i) {
    const int blk = sel[i];
    if (blk < 0 || blk >= N || blk >= a.host_blocks || (i > 0 && sel[i - 1] >= blk)) continue;
    const int pg = page_row[blk];
    const int s = pg - b * C;
    if (!(pg >= 0 && s >= 0 && s < C && blk_s[s] == blk) && (!a.prefetch || blk != N - 1))
      miss_s[r++] = blk;
  }
  // ---- victims: slots not stamped this step (a prefetch: holding no
  // predicted block), ordered by (last_use, slot) ----
  for (int s = tid; s < a.pow2; s += kUpdThreads) {
    unsigned long long key = ~0ull;
    if (s < C && (a.prefetch ? pin_s[s] == 0 : use_s[s] != a.step))
      key = (static_cast<unsigned long long>(static_cast<uint32_t>(use_s[s] + 1)) << 32) | uint32_t(s);
    key_s[s] = key;
  }
  __syncthreads();
  for (int size = 2; size <= a.pow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = tid; t < (a.pow2 >> 1); t += kUpdThreads) {
        const int lo = 2 * t - (t & (stride - 1));   // pair (lo, lo + stride)
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const unsigned long long u = key_s[lo], v = key_s[hi];
        if ((u > v) == up) {
          key_s[lo] = v;
          key_s[hi] = u;
        }
      }
      __syncthreads();
    }
  }
  // ---- the r-th miss goes to the r-th victim ----
  int2* jobs = a.jobs + int64_t(b) * (a.k_max + 1);
  for (int q = tid; q < m; q += kUpdThreads) {
    const unsigned long long key = key_s[q];
    if (key == ~0ull) {                      // fewer free slots than misses (cannot happen
      latch_error(a.err, KVSEL_ERR_BOUNDS);  // when slots >= k_max)
      jobs[q] = make_int2(-1, -1);
      continue;
    }
    const int s = int(key & 0xFFFFFFFFull);
    const int blk = miss_s[q];
    const int old = blk_s[s];
    if (old >= 0 && old < a.max_blocks) page_row[old] = -1;
    page_row[blk] = b * C + s;
    blk_s[s] = blk;
    use_s[s] = a.prefetch ? -1 : a.step;
    jobs[q] = make_int2(blk, b * C + s);
  }
  __syncthreads();
  for (int s = tid; s < C; s += kUpdThreads) {
    a.last_use[int64_t(b) * C + s] = use_s[s];
    a.block_in[int64_t(b) * C + s] = blk_s[s];
  }
  if (tid == 0) {
    const int refresh = scan_s[kUpdWarps];
    int nj = m;
    if (refresh >= 0) jobs[nj++] = make_int2(N - 1, refresh);
    a.n_jobs[b] = nj;
    if (a.n_fetched) a.n_fetched[b] = nj;
  }
}

// Copies every job's block (one KV page, `block_vec` 16-byte vectors) from
// the host tier [b][host_blocks][page] to its pool page. Grid (per_seq,
// batch): the CTAs of a sequence split its job list. blockDim.x is
// kCopyThreads, or half of it for a prefetch.
__global__ void __launch_bounds__(kCopyThreads) cache_copy_kernel(
    const kvsel_bf16* __restrict__ host_kv, kvsel_bf16* __restrict__ pool,
    const int2* __restrict__ jobs, const int32_t* __restrict__ n_jobs, int host_blocks,
    int k_max, int64_t block_vec, int* err) {
  const int b = blockIdx.y, tid = threadIdx.x, nt = blockDim.x;
  const int nj = n_jobs[b];
  const int per = (nj + gridDim.x - 1) / gridDim.x;
  const int j0 = blockIdx.x * per, j1 = min(nj, j0 + per);
  for (int j = j0; j < j1; ++j) {
    const int2 job = jobs[int64_t(b) * (k_max + 1) + j];
    if (job.x < 0 || job.x >= host_blocks || job.y < 0) {
      if (tid == 0) latch_error(err, KVSEL_ERR_BOUNDS);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(host_kv) + (int64_t(b) * host_blocks + job.x) * block_vec;
    uint4* dst = reinterpret_cast<uint4*>(pool) + int64_t(job.y) * block_vec;
    int64_t v = tid;
    for (; v + (kUnroll - 1) * nt < block_vec; v += kUnroll * nt) {
      uint4 r[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) r[u] = ld_sys_v4(src + v + u * nt);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) stg_stream(dst + v + u * nt, r[u]);
    }
    for (; v < block_vec; v += nt) stg_stream(dst + v, ld_sys_v4(src + v));
  }
}

}  // namespace

size_t cache_fetch_ws_bytes(const kvsel_problem& p) {
  const size_t jobs = size_t(p.batch) * (size_t(p.k_max) + 1) * sizeof(int2);
  return (jobs + 255) / 256 * 256 + size_t(p.batch) * 4;
}

size_t cache_update_smem_bytes(const kvsel_problem& p, int slots) {
  int pow2 = 1;
  while (pow2 < slots) pow2 <<= 1;
  return size_t(pow2) * 8 + size_t(slots) * 8 + size_t(p.k_max) * 4 + (kUpdWarps + 4) * 4 +
         size_t(slots);
}

cudaError_t launch_cache_fetch(const kvsel_problem& p, const kvsel_block_cache& c,
                               const kvsel_bf16* host_kv, int host_blocks,
                               const int32_t* seq_lens, const int32_t* sel_idx,
                               const int32_t* n_sel, int step, bool prefetch, int32_t* n_fetched,
                               void* ws, int fetch_ctas, int* err, cudaStream_t s) {
  if (p.batch == 0) return cudaSuccess;
  CacheArgs a;
  a.seq_lens = seq_lens; a.sel_idx = sel_idx; a.n_sel = n_sel;
  a.page_of = c.page_of; a.block_in = c.block_in; a.last_use = c.last_use;
  char* w = static_cast<char*>(ws);
  a.jobs = reinterpret_cast<int2*>(w);
  const size_t jobs = size_t(p.batch) * (size_t(p.k_max) + 1) * sizeof(int2);
  a.n_jobs = reinterpret_cast<int32_t*>(w + (jobs + 255) / 256 * 256);
  a.n_fetched = n_fetched;
  a.slots = c.slots;
  int pow2 = 1;
  while (pow2 < c.slots) pow2 <<= 1;
  a.pow2 = pow2;
  a.max_blocks = p.max_blocks; a.k_max = p.k_max; a.B = p.block_size;
  a.host_blocks = host_blocks; a.step = step; a.err = err;
  a.prefetch = prefetch ? 1 : 0;
  const size_t smem = cache_update_smem_bytes(p, c.slots);
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(cache_update_kernel), int(smem));
  if (e != cudaSuccess) return e;
  cache_update_kernel<<<p.batch, kUpdThreads, smem, s>>>(a);
  e = cudaGetLastError();
  count_launch();
  if (e != cudaSuccess) return e;
  const int64_t block_vec = int64_t(2) * p.n_kvheads * p.block_size * p.head_dim * 2 / 16;
  // default for a fetch: eight CTAs per SM, so that a sequence with many misses spreads
  // them over many CTAs (64 sequences of 64 KiB blocks: 190-200 GB/s with one CTA per
  // SM, 201-202 GB/s with four to sixteen per SM). A prefetch runs beside the other
  // stream's kernels: one CTA of half the threads per SM, so that it fits on an SM
  // beside a CTA of the score or decode kernels (registers: 128 x 40 beside 512 x 112
  // or 256 x 168 of the 65 536)
  const int64_t ctas = fetch_ctas > 0 ? fetch_ctas : (prefetch ? 1 : 8) * sm_count();
  const int threads = prefetch ? kCopyThreads / 2 : kCopyThreads;
  const int per_seq = int(std::min<int64_t>(std::max<int64_t>(1, (ctas + p.batch - 1) / p.batch),
                                            int64_t(p.k_max) + 1));
  cache_copy_kernel<<<dim3(per_seq, p.batch), threads, 0, s>>>(
      host_kv, c.pool, a.jobs, a.n_jobs, host_blocks, p.k_max, block_vec, err);
  count_launch();
  return cudaGetLastError();
}

}  // namespace kvsel
