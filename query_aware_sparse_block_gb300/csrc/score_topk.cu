// Query-aware block scoring, Top-k selection and span merge in one launch
// ("SparPR KV cache recovery on a consumer GPU": paragraph "Query-Aware
// key-block selection" for the score and Top-k, paragraph "On-demand local
// recomputation with cost-aware fallback" for spans and the Dense Fallback
// Threshold gamma).
//
// Design (GB300): the summary table is the only large input, so the kernel is
// a balanced stream over it. The flattened list of (sequence, block) pairs is
// cut into equal contiguous ranges, one per CTA (one CTA per SM). A CTA's
// range is cut into chunks of whole blocks of one sequence (contiguous in
// memory); one thread moves each chunk into shared memory with a 1-D bulk
// (TMA) copy, S chunks ahead, completions counted on mbarriers. Warps read
// block summaries from shared memory, multiply by the query folded over its
// GQA group (fp32, kept in registers) and reduce with shuffles. The last CTA
// to finish a sequence (an atomic ticket per sequence; no CTA ever waits for
// another) runs the Top-k on that sequence's scores: a 4-pass 8-bit radix
// select (shared-memory histograms) finds the k-th largest key, ties at
// that key are taken in index order, and block-wide scans emit the ascending
// selection, the spans and the gamma decision. Tickets are reset by their
// last user, so the workspace stays zero-filled between calls.
#include "kvsel_common.cuh"
#include "kvsel_internal.h"

namespace kvsel {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kStageBytes = 32 * 1024;
constexpr int kMaxStages = 4;

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
  int chunk_blocks;    // blocks per bulk copy
  int stages;
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

// Block-wide exclusive scan of one int per thread; returns the prefix and the
// block total through *total. scratch: kWarps ints.
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
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
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = seq_blocks(a, b);
  const int kreq = a.k_per_seq[b];
  if (kreq > a.k_max && tid == 0) latch_error(a.err, KVSEL_ERR_BOUNDS);
  int k = kreq < 0 ? 0 : kreq;
  k = min(k, min(N, a.k_max));
  const float* sc = a.scores + int64_t(b) * a.max_blocks;
  const int KPT = (N + kThreads - 1) / kThreads;     // keys per thread, index order
  const int c0 = min(N, tid * KPT), c1 = min(N, c0 + KPT);

  for (int i = tid; i < N; i += kThreads) keys_s[i] = order_key(__ldcg(sc + i));
  __syncthreads();

  // ---- radix select: threshold key K* and how many ties at K* to take ----
  uint32_t prefix = 0, mask = 0;
  int k_rem = k;
  const bool take_all = (k >= N);
  if (k > 0 && !take_all) {
    for (int shift = 24; shift >= 0; shift -= 8) {
      if (tid < 256) hist_s[tid] = 0;
      __syncthreads();
      for (int i = 0; i < KPT; ++i) {
        const int idx = c0 + i;
        const uint32_t key = idx < c1 ? keys_s[idx] : 0u;
        const bool valid = idx < c1 && (key & mask) == prefix;
        if (valid) atomicAdd(&hist_s[(key >> shift) & 255u], 1);
      }
      __syncthreads();
      // suffix sums over the 256 bins: warp w < 8 owns bins [32w, 32w + 32)
      int h = 0, x = 0;
      if (warp < 8) {
        h = hist_s[warp * 32 + lane];
        x = h;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int y = __shfl_down_sync(0xffffffffu, x, off);
          if (lane + off < 32) x += y;
        }
        if (lane == 0) scratch_s[warp] = x;
      }
      __syncthreads();
      if (warp < 8) {
        int higher = 0;
        for (int w = warp + 1; w < 8; ++w) higher += scratch_s[w];
        const int suffix_incl = x + higher;          // sum_{u >= bin}
        const int above = suffix_incl - h;           // sum_{u > bin}
        if (above < k_rem && suffix_incl >= k_rem) {
          bcast_s[0] = warp * 32 + lane;
          bcast_s[1] = k_rem - above;
        }
      }
      __syncthreads();
      prefix |= uint32_t(bcast_s[0]) << shift;
      mask |= 255u << shift;
      k_rem = bcast_s[1];
    }
  }
  const uint32_t kstar = prefix;
  const int need_eq = k_rem;

  // ---- pass A: selection flags in index order (ties -> lower index) ----
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

  // ---- pass B: positions and span starts (one packed scan), then ends ----
  int nsel_c = 0, nstart_c = 0;
  for (int i = c0; i < c1; ++i) {
    if (flags_s[i]) {
      ++nsel_c;
      if (i == 0 || !flags_s[i - 1]) ++nstart_c;
    }
  }
  int packed_tot;
  const int packed = block_exclusive_scan(nsel_c | (nstart_c << 16), scratch_s, &packed_tot);
  int pos = packed & 0xFFFF, sidx = packed >> 16;
  const int sel_tot = packed_tot & 0xFFFF, start_tot = packed_tot >> 16;
  int32_t* sel_out = a.sel_idx + int64_t(b) * a.k_max;
  int32_t* st_out = a.span_start + int64_t(b) * a.k_max;
  uint32_t* starts_s = keys_s;                          // keys are no longer needed
  uint32_t* ends_s = keys_s + (N + 1) / 2 + 1;
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
__global__ void __launch_bounds__(kThreads, 1) score_topk_kernel(ScoreArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int hist_s[256];
  __shared__ int scratch_s[kWarps];
  __shared__ int bcast_s[4];
  __shared__ int last_s[2];
  const int S = a.stages;
  unsigned char* stage = smem;                                               // [S][kStageBytes]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + size_t(S) * kStageBytes);
  float* qf_s = reinterpret_cast<float*>(bars + kMaxStages);                 // Hkv*d floats
  int* base_s = reinterpret_cast<int*>(qf_s + a.Hkv * a.d);                  // batch + 1
  uint32_t* keys_s = reinterpret_cast<uint32_t*>(base_s + a.batch + 1);      // max_blocks + 2
  uint8_t* flags_s = reinterpret_cast<uint8_t*>(keys_s + a.max_blocks + 2);  // max_blocks

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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

  auto find_seq = [&](int64_t g) {
    int lo = 0, hi = a.batch - 1;
    while (lo < hi) {             // largest b with base_s[b] <= g
      const int mid = (lo + hi + 1) >> 1;
      if (base_s[mid] <= g) lo = mid; else hi = mid - 1;
    }
    return lo;
  };
  const int bfirst = find_seq(g0);
  const int blast = find_seq(g1 - 1);
  const int NV = a.NV;
  const int block_bytes = NV * 16;
  const int CH = a.chunk_blocks;

  // chunks of the range never cross a sequence end or the range end
  auto chunk_at = [&](int64_t g, int& b, int& n0, int& nblk) {
    b = find_seq(g);
    n0 = int(g - base_s[b]);
    const int64_t seq_end = base_s[b + 1];
    nblk = int(min(int64_t(CH), min(seq_end, g1) - g));
  };
  if (tid == 0) {
    for (int i = 0; i < S; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
  }
  __syncthreads();
  // producer (thread 0): the next chunk to copy starts at prod_g
  int64_t prod_g = g0;
  int n_issued = 0;
  auto issue_next = [&]() {
    if (prod_g >= g1) return;
    int b, n0, nblk;
    chunk_at(prod_g, b, n0, nblk);
    uint64_t* bar = &bars[n_issued % S];
    const uint32_t bytes = uint32_t(nblk) * block_bytes;
    mbar_arrive_expect_tx(bar, bytes);
    bulk_load(stage + size_t(n_issued % S) * kStageBytes,
              a.summaries + (int64_t(b) * a.max_blocks + n0) * NV * 8, bytes, bar);
    prod_g += nblk;
    ++n_issued;
  };
  if (tid == 0)
    for (int i = 0; i < S; ++i) issue_next();

  const int LPB = a.LPB, BPW = 32 / LPB;
  const int sub = lane / LPB, li = lane % LPB;
  const int G = a.Hq / a.Hkv;
  float qreg[VPL <= 4 ? VPL : 1][8];
  int cur_b = -1;
  bool dead = false;
  int c = 0;
  for (int64_t g = g0; g < g1; ++c) {
    int b, n0, nblk;
    chunk_at(g, b, n0, nblk);
    if (b != cur_b) {
      cur_b = b;
      const kvsel_bf16* qb = a.q + int64_t(b) * a.Hq * a.d;
      if constexpr (VPL <= 4) {
        // fold q over the GQA group for this lane's vectors, straight from global
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          const int e0 = (li + LPB * i) * 8;
          const int j = e0 / a.d, cc = e0 % a.d;
#pragma unroll
          for (int e = 0; e < 8; ++e) qreg[i][e] = 0.f;
          for (int r = 0; r < G; ++r) {
            const uint4 v = *reinterpret_cast<const uint4*>(qb + int64_t(j * G + r) * a.d + cc);
            qreg[i][0] += bf16lo(v.x); qreg[i][1] += bf16hi(v.x);
            qreg[i][2] += bf16lo(v.y); qreg[i][3] += bf16hi(v.y);
            qreg[i][4] += bf16lo(v.z); qreg[i][5] += bf16hi(v.z);
            qreg[i][6] += bf16lo(v.w); qreg[i][7] += bf16hi(v.w);
          }
        }
      } else {
        for (int e = tid; e < a.Hkv * a.d; e += kThreads) {
          const int j = e / a.d, cc = e % a.d;
          float acc = 0.f;
          for (int r = 0; r < G; ++r)
            acc += __uint_as_float(uint32_t(qb[int64_t(j * G + r) * a.d + cc]) << 16);
          qf_s[e] = acc;
        }
        __syncthreads();
      }
    }
    if (!dead && !mbar_wait_bounded(&bars[c % S], uint32_t((c / S) & 1))) {
      dead = true;
      if (tid == 0) latch_error(a.err, KVSEL_ERR_TIMEOUT);
    }
    if (!dead) {
      const unsigned char* st = stage + size_t(c % S) * kStageBytes;
      float* out = a.scores + int64_t(b) * a.max_blocks + n0;
      const int steps = (nblk + BPW - 1) / BPW;
      for (int s = warp; s < steps; s += kWarps) {
        const int r = s * BPW + sub;
        float acc = 0.f;
        if (r < nblk) {
#pragma unroll
          for (int i = 0; i < VPL; ++i) {
            const uint4 v = *reinterpret_cast<const uint4*>(st + (size_t(r) * NV + li + LPB * i) * 16);
            float qv[8];
            if constexpr (VPL <= 4) {
#pragma unroll
              for (int e = 0; e < 8; ++e) qv[e] = qreg[i][e];
            } else {
              const float4* src = reinterpret_cast<const float4*>(qf_s + (li + LPB * i) * 8);
              const float4 x0 = src[0], x1 = src[1];
              qv[0] = x0.x; qv[1] = x0.y; qv[2] = x0.z; qv[3] = x0.w;
              qv[4] = x1.x; qv[5] = x1.y; qv[6] = x1.z; qv[7] = x1.w;
            }
            acc = fmaf(qv[0], bf16lo(v.x), acc);
            acc = fmaf(qv[1], bf16hi(v.x), acc);
            acc = fmaf(qv[2], bf16lo(v.y), acc);
            acc = fmaf(qv[3], bf16hi(v.y), acc);
            acc = fmaf(qv[4], bf16lo(v.z), acc);
            acc = fmaf(qv[5], bf16hi(v.z), acc);
            acc = fmaf(qv[6], bf16lo(v.w), acc);
            acc = fmaf(qv[7], bf16hi(v.w), acc);
          }
        }
        for (int off = LPB >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (li == 0 && r < nblk) out[r] = acc;
      }
    }
    __syncthreads();                  // every warp is done with this stage
    if (tid == 0 && !dead) {
      fence_proxy_async();
      issue_next();
    }
    g += nblk;
  }
  // no copy may land after the CTA exits: drain what a timeout left in flight
  if (dead && tid == 0)
    for (int i = c; i < n_issued; ++i) (void)mbar_wait_bounded(&bars[i % S], uint32_t((i / S) & 1));

  // publish scores, take tickets for the first and last sequence touched
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    last_s[0] = last_s[1] = -1;
    const int cand[2] = {bfirst, blast};
    for (int cI = 0; cI < 2; ++cI) {
      const int b = cand[cI];
      if (cI == 1 && blast == bfirst) break;
      const int64_t s0 = max(int64_t(g0), int64_t(base_s[b]));
      const int64_t s1 = min(int64_t(g1), int64_t(base_s[b + 1]));
      const uint32_t mine = uint32_t(s1 - s0);
      const uint32_t nb = uint32_t(base_s[b + 1] - base_s[b]);
      const uint32_t before = atomicAdd(&a.tickets[b], mine);
      if (before + mine == nb) last_s[cI] = b;
    }
    __threadfence();
  }
  __syncthreads();
  // sequences strictly inside the range are owned entirely by this CTA
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
  // one thread per sequence walks the selection in order
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
  const int block_bytes = a.NV * 16;
  a.chunk_blocks = std::max(1, kStageBytes / block_bytes);
  const size_t tail = size_t(kMaxStages) * 8 + size_t(p.n_kvheads) * p.head_dim * 4 +
                      (size_t(p.batch) + 1) * 4 + (size_t(p.max_blocks) + 2) * 4 +
                      size_t(p.max_blocks) + 256;
  const int max_optin = max_smem_optin();
  const int static_smem = 256 * 4 + kWarps * 4 + 32 + 64;
  int stages = int((int64_t(max_optin) - static_smem - int64_t(tail)) / kStageBytes);
  stages = std::min(kMaxStages, stages);
  if (stages < 1) return cudaErrorInvalidConfiguration;
  a.stages = stages;
  const size_t smem = size_t(stages) * kStageBytes + tail;
  const int64_t upper = int64_t(p.batch) * p.max_blocks;
  const int grid = int(std::min<int64_t>(sm_count(), std::max<int64_t>(1, upper / 8)));
  cudaError_t e = cudaSuccess;
#define KVSEL_SCORE_CASE(V)                                                                  \
  case V: {                                                                                  \
    auto kfn = score_topk_kernel<V>;                                                         \
    e = ensure_smem(reinterpret_cast<const void*>(kfn), int(smem));                          \
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
