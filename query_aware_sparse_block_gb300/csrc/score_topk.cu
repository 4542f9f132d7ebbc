// Query-aware block scoring, Top-k selection and span merge in one launch
// ("SparPR KV cache recovery on a consumer GPU": paragraph "Query-Aware
// key-block selection" for the score and Top-k, paragraph "On-demand local
// recomputation with cost-aware fallback" for spans and the Dense Fallback
// Threshold gamma).
//
// Design (GB300): the summary table is the only large input, so the kernel is
// a balanced stream over it. The flattened list of (sequence, block) pairs is
// cut into equal contiguous ranges, one per CTA of a grid sized to the SM
// count; each warp streams whole block summaries with 16-byte loads and
// reduces the dot product with shuffles. The last CTA to finish a sequence
// (an atomic ticket per sequence; no CTA ever waits for another) runs the
// Top-k on that sequence's scores: a 4-pass 8-bit radix select finds the
// k-th largest key, ties at that key are taken in index order, and two
// block-wide scans emit the ascending selection, the spans and the gamma
// decision. Tickets are reset by their last user, so the workspace stays
// zero-filled between calls.
#include "kvsel_common.cuh"
#include "kvsel_internal.h"

namespace kvsel {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxBatchSmem = 4096;   // sequences whose prefix fits the static smem table

struct ScoreArgs {
  const kvsel_bf16* q;
  const kvsel_bf16* summaries;
  const int32_t* seq_lens;
  const int32_t* k_per_seq;
  float gamma, tau_rel;
  int32_t* sel_idx;
  int32_t* n_sel;
  int32_t* span_start;
  int32_t* span_len;
  int32_t* n_spans;
  uint8_t* dense_flag;
  float* scores;       // [batch][max_blocks]
  uint32_t* tickets;   // [batch]
  int* err;
  int batch, Hq, Hkv, d, B, max_blocks, k_max;
  int NV, LPB;         // 16-byte vectors per block summary; lanes per block
};

__device__ __forceinline__ int seq_blocks(const ScoreArgs& a, int b) {
  int T = a.seq_lens[b];
  T = T < 0 ? 0 : (T > a.max_blocks * a.B ? a.max_blocks * a.B : T);
  return (T + a.B - 1) / a.B;
}

// Order-preserving map of fp32 to uint32 (larger float -> larger key); -0 is
// folded onto +0 first so that equal scores compare equal.
__device__ __forceinline__ uint32_t order_key(float s) {
  uint32_t u = __float_as_uint(s + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Scores blocks [lo, hi) of sequence b. qf_s: folded query [Hkv][d] fp32 in smem.
template <int VPL>
__device__ void score_blocks(const ScoreArgs& a, int b, int lo, int hi, const float* qf_s) {
  constexpr int U = VPL >= 8 ? 1 : 8 / VPL;    // warp steps in flight
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int LPB = a.LPB, BPW = 32 / LPB;
  const int sub = lane / LPB, li = lane % LPB;
  const int NV = a.NV;
  const kvsel_bf16* base = a.summaries + int64_t(b) * a.max_blocks * NV * 8;
  float* out = a.scores + int64_t(b) * a.max_blocks;

  float qreg[VPL <= 4 ? VPL : 1][8];
  if constexpr (VPL <= 4) {
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const float4* src = reinterpret_cast<const float4*>(qf_s + (li + LPB * i) * 8);
      float4 x = src[0], y = src[1];
      qreg[i][0] = x.x; qreg[i][1] = x.y; qreg[i][2] = x.z; qreg[i][3] = x.w;
      qreg[i][4] = y.x; qreg[i][5] = y.y; qreg[i][6] = y.z; qreg[i][7] = y.w;
    }
  }
  const int step = kWarps * BPW * U;
  for (int n0 = lo + warp * BPW * U; n0 < hi; n0 += step) {
    uint4 r[U][VPL];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int n = n0 + u * BPW + sub;
      if (n < hi) {
        const kvsel_bf16* src = base + (int64_t(n) * NV + li) * 8;
#pragma unroll
        for (int i = 0; i < VPL; ++i) r[u][i] = ldg_stream(src + i * LPB * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int n = n0 + u * BPW + sub;
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        float qv[8];
        if constexpr (VPL <= 4) {
#pragma unroll
          for (int e = 0; e < 8; ++e) qv[e] = qreg[i][e];
        } else {
          const float4* src = reinterpret_cast<const float4*>(qf_s + (li + LPB * i) * 8);
          float4 x = src[0], y = src[1];
          qv[0] = x.x; qv[1] = x.y; qv[2] = x.z; qv[3] = x.w;
          qv[4] = y.x; qv[5] = y.y; qv[6] = y.z; qv[7] = y.w;
        }
        const uint4 v = r[u][i];
        acc = fmaf(qv[0], bf16lo(v.x), acc);
        acc = fmaf(qv[1], bf16hi(v.x), acc);
        acc = fmaf(qv[2], bf16lo(v.y), acc);
        acc = fmaf(qv[3], bf16hi(v.y), acc);
        acc = fmaf(qv[4], bf16lo(v.z), acc);
        acc = fmaf(qv[5], bf16hi(v.z), acc);
        acc = fmaf(qv[6], bf16lo(v.w), acc);
        acc = fmaf(qv[7], bf16hi(v.w), acc);
      }
      for (int off = LPB >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (li == 0 && n < hi) out[n] = acc;
    }
  }
}

// Block-wide exclusive scan of one int per thread; returns the prefix, and
// the block total through *total. Uses smem scratch of kWarps ints.
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  int wsum = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int s = scratch[w];
    if (w < warp) wsum += s;
    all += s;
  }
  __syncthreads();
  *total = all;
  return wsum + x - v;
}

// Top-k + spans + gamma decision for sequence b (whole CTA). keys_s holds
// max_blocks + 2 uint32, flags_s max_blocks bytes.
__device__ void select_sequence(const ScoreArgs& a, int b, uint32_t* keys_s, uint8_t* flags_s,
                                int* hist_s, int* scratch_s, int* bcast_s) {
  const int tid = threadIdx.x;
  const int N = seq_blocks(a, b);
  int kreq = a.k_per_seq[b];
  if (kreq > a.k_max && tid == 0) latch_error(a.err, KVSEL_ERR_BOUNDS);
  int k = kreq < 0 ? 0 : kreq;
  k = min(k, min(N, a.k_max));
  const float* sc = a.scores + int64_t(b) * a.max_blocks;

  for (int i = tid; i < N; i += kThreads) keys_s[i] = order_key(__ldcg(sc + i));
  __syncthreads();

  // ---- radix select: threshold key K* and how many ties at K* to take ----
  uint32_t prefix = 0, mask = 0;
  int k_rem = k;
  if (k > 0 && k < N) {
    for (int shift = 24; shift >= 0; shift -= 8) {
      hist_s[tid] = 0;
      __syncthreads();
      for (int i = tid; i < N; i += kThreads) {
        const uint32_t key = keys_s[i];
        if ((key & mask) == prefix) atomicAdd(&hist_s[(key >> shift) & 255u], 1);
      }
      __syncthreads();
      // inclusive suffix sum over the 256 bins: bin t -> sum_{u >= t} hist[u]
      const int h = hist_s[tid];
      int tot;
      const int excl = block_exclusive_scan(h, scratch_s, &tot);   // sum_{u < t}
      const int suffix_incl = tot - excl;                          // sum_{u >= t}
      const int above = suffix_incl - h;                           // sum_{u > t}
      if (above < k_rem && suffix_incl >= k_rem) {
        bcast_s[0] = tid;
        bcast_s[1] = k_rem - above;
      }
      __syncthreads();
      prefix |= uint32_t(bcast_s[0]) << shift;
      mask |= 255u << shift;
      k_rem = bcast_s[1];
      __syncthreads();
    }
  }
  const bool take_all = (k >= N);
  const uint32_t kstar = prefix;
  const int need_eq = k_rem;

  // ---- pass A: selection flags in index order (ties -> lower index) ----
  const int chunk = (N + kThreads - 1) / kThreads;
  const int c0 = min(N, tid * chunk), c1 = min(N, c0 + chunk);
  int eq_cnt = 0;
  if (k > 0 && !take_all)
    for (int i = c0; i < c1; ++i) eq_cnt += (keys_s[i] == kstar);
  int eq_tot;
  int eq_rank = block_exclusive_scan(eq_cnt, scratch_s, &eq_tot);
  for (int i = c0; i < c1; ++i) {
    bool s;
    if (k == 0) s = false;
    else if (take_all) s = true;
    else {
      const uint32_t key = keys_s[i];
      s = key > kstar;
      if (key == kstar) { s = eq_rank < need_eq; ++eq_rank; }
    }
    flags_s[i] = s ? 1 : 0;
  }
  __syncthreads();

  // ---- pass B: positions, span starts and ends ----
  int nsel_c = 0, nstart_c = 0;
  for (int i = c0; i < c1; ++i) {
    if (flags_s[i]) {
      ++nsel_c;
      if (i == 0 || !flags_s[i - 1]) ++nstart_c;
    }
  }
  int sel_tot, start_tot;
  int pos = block_exclusive_scan(nsel_c, scratch_s, &sel_tot);
  int sidx = block_exclusive_scan(nstart_c, scratch_s, &start_tot);
  int32_t* sel_out = a.sel_idx + int64_t(b) * a.k_max;
  int32_t* st_out = a.span_start + int64_t(b) * a.k_max;
  uint32_t* starts_s = keys_s;                          // keys are no longer needed
  uint32_t* ends_s = keys_s + (N + 1) / 2 + 1;
  __syncthreads();
  for (int i = c0; i < c1; ++i) {
    if (!flags_s[i]) continue;
    sel_out[pos++] = i;
    if (i == 0 || !flags_s[i - 1]) {
      st_out[sidx] = i;
      starts_s[sidx] = i;
      ++sidx;
    }
    if (i == N - 1 || !flags_s[i + 1]) ends_s[sidx - 1] = i;
  }
  __syncthreads();
  int32_t* len_out = a.span_len + int64_t(b) * a.k_max;
  for (int s = tid; s < start_tot; s += kThreads) len_out[s] = int(ends_s[s] - starts_s[s]) + 1;
  if (tid == 0) {
    a.n_sel[b] = sel_tot;
    a.n_spans[b] = start_tot;
    if (a.dense_flag) {
      const double lhs = double(start_tot) * double(a.tau_rel) + double(sel_tot);
      const double rhs = double(a.gamma) * (double(a.tau_rel) + double(N));
      a.dense_flag[b] = (N > 0 && lhs >= rhs) ? 1 : 0;
    }
  }
  __syncthreads();
}

template <int VPL>
__global__ void __launch_bounds__(kThreads) score_topk_kernel(ScoreArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int base_s[kMaxBatchSmem + 1];
  __shared__ int hist_s[256];
  __shared__ int scratch_s[kWarps];
  __shared__ int bcast_s[4];
  __shared__ int last_s[2];
  float* qf_s = reinterpret_cast<float*>(smem);                              // Hkv*d floats
  uint32_t* keys_s = reinterpret_cast<uint32_t*>(smem + size_t(a.Hkv) * a.d * 4);
  uint8_t* flags_s = reinterpret_cast<uint8_t*>(keys_s + a.max_blocks + 2);

  const int tid = threadIdx.x;
  // exclusive prefix of blocks over sequences
  int carry = 0;
  for (int b0 = 0; b0 < a.batch; b0 += kThreads) {
    const int b = b0 + tid;
    const int nb = b < a.batch ? seq_blocks(a, b) : 0;
    int tot;
    const int ex = block_exclusive_scan(nb, scratch_s, &tot);
    if (b < a.batch) base_s[b] = carry + ex;
    carry += tot;
  }
  if (tid == 0) base_s[a.batch] = carry;
  __syncthreads();
  const int64_t total = carry;

  // sequences with no block never see a ticket: finish them here
  for (int b = blockIdx.x * kThreads + tid; b < a.batch; b += gridDim.x * kThreads) {
    if (base_s[b + 1] == base_s[b]) {
      a.n_sel[b] = 0;
      a.n_spans[b] = 0;
      if (a.dense_flag) a.dense_flag[b] = 0;
      if (a.k_per_seq[b] > a.k_max) latch_error(a.err, KVSEL_ERR_BOUNDS);
    }
  }
  const int64_t g0 = total * blockIdx.x / gridDim.x;
  const int64_t g1 = total * (blockIdx.x + 1) / gridDim.x;
  if (g0 >= g1) return;

  // first sequence of the range
  int bfirst = 0;
  {
    int lo = 0, hi = a.batch - 1;
    while (lo < hi) {           // largest b with base_s[b] <= g0
      const int mid = (lo + hi + 1) >> 1;
      if (base_s[mid] <= g0) lo = mid; else hi = mid - 1;
    }
    bfirst = lo;
  }
  int blast = bfirst;
  for (int b = bfirst; b < a.batch && base_s[b] < g1; ++b) {
    blast = b;
    const int64_t s0 = max(int64_t(g0), int64_t(base_s[b]));
    const int64_t s1 = min(int64_t(g1), int64_t(base_s[b + 1]));
    if (s0 >= s1) continue;
    // fold q over each GQA group: qf[j][c] = sum_r q[b][j*G + r][c]
    const int G = a.Hq / a.Hkv;
    for (int e = tid; e < a.Hkv * a.d; e += kThreads) {
      const int j = e / a.d, c = e % a.d;
      const kvsel_bf16* qb = a.q + (int64_t(b) * a.Hq + int64_t(j) * G) * a.d + c;
      float acc = 0.f;
      for (int r = 0; r < G; ++r) acc += __uint_as_float(uint32_t(qb[int64_t(r) * a.d]) << 16);
      qf_s[e] = acc;
    }
    __syncthreads();
    score_blocks<VPL>(a, b, int(s0 - base_s[b]), int(s1 - base_s[b]), qf_s);
    __syncthreads();
  }

  // publish scores, take tickets for the first and last sequence touched
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    last_s[0] = last_s[1] = -1;
    const int cand[2] = {bfirst, blast};
    for (int c = 0; c < 2; ++c) {
      const int b = cand[c];
      if (c == 1 && blast == bfirst) break;
      const int64_t s0 = max(int64_t(g0), int64_t(base_s[b]));
      const int64_t s1 = min(int64_t(g1), int64_t(base_s[b + 1]));
      const uint32_t mine = uint32_t(s1 - s0);
      const uint32_t nb = uint32_t(base_s[b + 1] - base_s[b]);
      const uint32_t before = atomicAdd(&a.tickets[b], mine);
      if (before + mine == nb) last_s[c] = b;
    }
    // sequences strictly inside the range are owned entirely by this CTA
    __threadfence();
  }
  __syncthreads();
  for (int b = bfirst; b <= blast; ++b) {
    const bool inner = (b != bfirst && b != blast);
    const bool mine = inner || (b == bfirst && last_s[0] == b) || (b == blast && last_s[1] == b);
    if (!mine) continue;
    if (inner && base_s[b + 1] == base_s[b]) continue;
    select_sequence(a, b, keys_s, flags_s, hist_s, scratch_s, bcast_s);
    if (tid == 0 && !inner) a.tickets[b] = 0;
  }
}

__global__ void merge_spans_kernel(const int32_t* __restrict__ sel_idx, const int32_t* __restrict__ n_sel,
                                   int32_t* __restrict__ span_start, int32_t* __restrict__ span_len,
                                   int32_t* __restrict__ n_spans, int k_max, int* err) {
  // one warp per sequence; serial walk in lane 0 keeps it obviously ordered
  const int b = blockIdx.x;
  if (threadIdx.x != 0) return;
  int n = n_sel[b];
  if (n < 0 || n > k_max) {
    latch_error(err, KVSEL_ERR_BOUNDS);
    n = n < 0 ? 0 : k_max;
  }
  const int32_t* s = sel_idx + int64_t(b) * k_max;
  int32_t* st = span_start + int64_t(b) * k_max;
  int32_t* ln = span_len + int64_t(b) * k_max;
  int ns = 0;
  for (int i = 0; i < n; ++i) {
    const int v = s[i];
    if (i > 0 && v <= s[i - 1]) latch_error(err, KVSEL_ERR_BOUNDS);
    if (i > 0 && v == s[i - 1] + 1) {
      ++ln[ns - 1];
    } else {
      st[ns] = v;
      ln[ns] = 1;
      ++ns;
    }
  }
  n_spans[b] = ns;
}

}  // namespace

size_t score_topk_ws_bytes(const kvsel_problem& p) {
  const size_t tickets = (size_t(p.batch) * 4 + 255) / 256 * 256;
  const size_t scores = size_t(p.batch) * p.max_blocks * 4;
  return tickets + scores;
}

cudaError_t launch_score_topk(const kvsel_problem& p, const kvsel_bf16* q,
                              const kvsel_bf16* summaries, const int32_t* seq_lens,
                              const int32_t* k_per_seq, float gamma, float tau_rel,
                              int32_t* sel_idx, int32_t* n_sel, int32_t* span_start,
                              int32_t* span_len, int32_t* n_spans, uint8_t* dense_flag,
                              float* scores_out, void* ws, int* err, cudaStream_t s) {
  if (p.batch == 0) return cudaSuccess;
  ScoreArgs a;
  a.q = q; a.summaries = summaries; a.seq_lens = seq_lens; a.k_per_seq = k_per_seq;
  a.gamma = gamma; a.tau_rel = tau_rel;
  a.sel_idx = sel_idx; a.n_sel = n_sel; a.span_start = span_start; a.span_len = span_len;
  a.n_spans = n_spans; a.dense_flag = dense_flag;
  char* w = static_cast<char*>(ws);
  a.tickets = reinterpret_cast<uint32_t*>(w);
  a.scores = scores_out ? scores_out
                        : reinterpret_cast<float*>(w + (size_t(p.batch) * 4 + 255) / 256 * 256);
  a.err = err;
  a.batch = p.batch; a.Hq = p.n_qheads; a.Hkv = p.n_kvheads; a.d = p.head_dim;
  a.B = p.block_size; a.max_blocks = p.max_blocks; a.k_max = p.k_max;
  a.NV = p.n_kvheads * p.head_dim / 8;
  int lpb = 32;
  while (a.NV % lpb) lpb >>= 1;
  a.LPB = lpb;
  const int vpl = a.NV / lpb;
  const size_t smem = size_t(p.n_kvheads) * p.head_dim * 4 + (size_t(p.max_blocks) + 2) * 4 +
                      size_t(p.max_blocks) + 16;
  const int64_t upper = int64_t(p.batch) * p.max_blocks;
  int grid = int(std::min<int64_t>(int64_t(2) * sm_count(), std::max<int64_t>(1, upper / 16)));
  cudaError_t e = cudaSuccess;
#define KVSEL_SCORE_CASE(V)                                                                  \
  case V: {                                                                                  \
    auto kfn = score_topk_kernel<V>;                                                         \
    e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));   \
    if (e != cudaSuccess) return e;                                                          \
    kfn<<<grid, kThreads, smem, s>>>(a);                                                     \
    break;                                                                                   \
  }
  switch (vpl) {
    KVSEL_SCORE_CASE(1)
    KVSEL_SCORE_CASE(2)
    KVSEL_SCORE_CASE(4)
    KVSEL_SCORE_CASE(8)
    KVSEL_SCORE_CASE(16)
    default:
      return cudaErrorInvalidValue;
  }
#undef KVSEL_SCORE_CASE
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_merge_spans(const kvsel_problem& p, const int32_t* sel_idx,
                               const int32_t* n_sel, int32_t* span_start, int32_t* span_len,
                               int32_t* n_spans, int* err, cudaStream_t s) {
  if (p.batch == 0) return cudaSuccess;
  merge_spans_kernel<<<p.batch, 32, 0, s>>>(sel_idx, n_sel, span_start, span_len, n_spans,
                                            p.k_max, err);
  count_launch();
  return cudaGetLastError();
}

}  // namespace kvsel
