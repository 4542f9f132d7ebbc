// Device code shared by the two forms of the query-aware score + Top-k call
// ("SparPR KV cache recovery on a consumer GPU", paragraph "Query-Aware
// key-block selection" for the score and Top-k, paragraph "On-demand local
// recomputation with cost-aware fallback" for spans and the Dense Fallback
// Threshold gamma): the call's arguments, the per-block score arithmetic
// helpers, the order keys of fp32 scores, the CTA-wide Top-k + span + gamma
// core, and the APPEND summary update folded into the score work.
//
// score_topk.cu holds the two-grid form (a score grid, then one Top-k CTA per
// sequence); score_cluster.cu the one-launch form (one thread-block cluster
// per sequence). Both compute every score with the same fp32 operations in
// the same order, so their scores, and with them their selections, are equal
// bit for bit.
#pragma once

#include "kvsel_common.cuh"
#include "summary_math.cuh"

namespace kvsel {
namespace {
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kConsumerWarps = 8;        // score grid: warps that reduce summaries
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kAppendWarp0 = kConsumerWarps + 1;   // first of the append warps
constexpr int kAppendWarps = 4;
constexpr int kAppendThreads = kAppendWarps * 32;
constexpr int kBins = 2048;               // histogram bins of the Top-k threshold search
constexpr int kBinsPerThread = kBins / kThreads;
constexpr int kCand = 128;                // bin size ranked exactly instead of refined
static_assert(kBins % kThreads == 0, "bins per thread");

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
  int* err;
  // the APPEND summary update folded into the call (append_pos == nullptr: none)
  kvsel_bf16* kv_pages;
  int64_t n_pages;
  const int32_t* block_table;
  const int32_t* append_pos;
  const kvsel_bf16* new_k;
  const kvsel_bf16* new_v;
  kvsel_bf16* summaries_out;   // the table behind `summaries`
  double* open_acc;
  int batch, Hq, Hkv, d, B, max_blocks, k_max;
  int n_sink, n_recent;  // forced leading / trailing blocks of every sequence
  int NV, LPB;         // 16-byte vectors per block summary; lanes per block
  int chunk_blocks;    // blocks per bulk copy
  int stages;
  int stage_bytes;     // bytes of one stage
  int csize;           // one-launch form: CTAs per cluster (one cluster per sequence)
};

// fp32 pairs for the packed FMA (fma.rn.f32x2: two IEEE fp32 FMAs, each
// rounded as fmaf rounds). A block's score sums, per lane, its even channels
// and its odd channels in two chains, adds them, and combines the lanes by the
// xor tree; the consumers and the append warps both follow this order.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f32x2_sum(uint64_t v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return lo + hi;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// the two bf16 of a 32-bit word as an fp32 pair, the lower channel first
__device__ __forceinline__ uint64_t bf16x2_f32x2(uint32_t w) { return f32x2(bf16lo(w), bf16hi(w)); }

// Key blocks of a sequence of T tokens in a row of max_blocks: ceil(T / B), T clamped.
__device__ __forceinline__ int blocks_of_len(const ScoreArgs& a, int T) {
  T = T < 0 ? 0 : (T > a.max_blocks * a.B ? a.max_blocks * a.B : T);
  return (T + a.B - 1) / a.B;
}

__device__ __forceinline__ int seq_blocks(const ScoreArgs& a, int b) {
  return blocks_of_len(a, a.seq_lens[b]);
}

// Order-preserving map of fp32 to uint32 (larger float -> larger key); -0 is
// folded onto +0 first so that equal scores compare equal, and a NaN score
// (from non-finite keys) takes the lowest key, below -inf, whatever its sign
// bit: it is chosen after every number, ties by index, as the Top-k's sort
// order has it.
__device__ __forceinline__ uint32_t order_key(float s) {
  if (s != s) return 0u;
  uint32_t u = __float_as_uint(s + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inverse of order_key (-0 comes back as +0).
__device__ __forceinline__ float key_float(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
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

struct SelectSmem {
  uint32_t* keys;     // [max_blocks + 2] order keys (later: span starts / ends)
  uint8_t* flags;     // [max_blocks] selection flags
  int* hist;          // [kBins], all zero between uses
  uint32_t* cand;     // [kCand] keys of the threshold bin
  int* scratch;       // [kWarps] scan partials
  uint32_t* mm;       // [2 * kWarps] min / max partials
  int* bcast;         // [8]; bcast[7] is a gather counter, zero between uses
  uint32_t* binkey;   // [kBins] a key that fell in each bin of the value histogram
};

// After a histogram of the candidates' bins: the bin holding the r-th largest
// candidate (bcast[0]), how many candidates lie in higher bins (bcast[1]) and
// in that bin (bcast[2]). Clears the histogram. Two barriers.
__device__ __forceinline__ void locate_bin(const SelectSmem& sm, int r) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int h[kBinsPerThread];
  int tot = 0;
#pragma unroll
  for (int j = 0; j < kBinsPerThread; ++j) {
    h[j] = sm.hist[tid * kBinsPerThread + j];
    sm.hist[tid * kBinsPerThread + j] = 0;
    tot += h[j];
  }
  int x = tot;                                // suffix sum over this warp's threads
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_down_sync(0xffffffffu, x, off);
    if (lane + off < 32) x += y;
  }
  if (lane == 0) sm.scratch[warp] = x;
  __syncthreads();
  int above = x - tot;                        // candidates in higher bins
  for (int w = warp + 1; w < kWarps; ++w) above += sm.scratch[w];
#pragma unroll
  for (int j = kBinsPerThread - 1; j >= 0; --j) {
    if (above < r && above + h[j] >= r) {
      sm.bcast[0] = tid * kBinsPerThread + j;
      sm.bcast[1] = above;
      sm.bcast[2] = h[j];
    }
    above += h[j];
  }
  __syncthreads();
}

// Rank the m (<= kCand) gathered candidates exactly: the r-th largest key
// (bcast[4]), how many candidates exceed it (bcast[5]) and equal it
// (bcast[6]). Resets the gather counter. One barrier after the gather's.
__device__ __forceinline__ void rank_candidates(const SelectSmem& sm, int m, int r) {
  const int tid = threadIdx.x;
  if (tid < m) {
    const uint32_t c = sm.cand[tid];
    int g = 0, e = 0;
    for (int j = 0; j < m; ++j) {
      const uint32_t o = sm.cand[j];
      g += o > c;
      e += o == c;
    }
    if (g < r && r <= g + e) {
      sm.bcast[4] = int(c);
      sm.bcast[5] = g;
      sm.bcast[6] = e;
    }
  }
  __syncthreads();
  if (tid == 0) sm.bcast[7] = 0;
}

// Bin of a score on a linear scale over [smin, smin + 2048 / scale]; the
// rounded steps are non-decreasing in s (no contraction), so a larger score
// never lands in a lower bin and equal scores share a bin.
__device__ __forceinline__ int value_bin(float s, float smin, float scale) {
  // every candidate key lies in [smin, smax], so the lower clamp never acts; it
  // keeps a shared-memory index in range should that ever not hold
  return max(0, min(kBins - 1, __float2int_rz(__fmul_rn(__fsub_rn(s, smin), scale))));
}

// Top-k + spans + gamma decision for sequence b (whole CTA of kThreads).
// On entry keys[0, N) hold the order keys of the sequence's N blocks, kmin /
// kmax (the same in every thread) the smallest and largest key of the
// candidates, hist is all zero and bcast[7] is zero; kreq is k_per_seq[b].
//
// Forced blocks: the first n_sink and the last n_recent blocks of the
// sequence are selected whatever their score (the recency window that the
// DKV abstract attends exactly beside the Top-k blocks). The Top-k runs over
// the candidate blocks [lo, hi) between them; with no window lo = 0, hi = N.
//
// Threshold: the k-th largest order key K* (with n_gt keys above it and n_eq
// equal to it). Fast path: a histogram with 2048 bins linear in the score
// value between the row's minimum and maximum finds the bin holding the k-th
// score; when it holds at most kCand scores they are gathered and ranked
// exactly. Otherwise (clustered or tied scores) the search runs over the key
// space: a window that starts as [min key, max key] narrows, 2048 bins at a
// time, to the bin holding the k-th key, until that bin holds at most kCand
// keys (ranked exactly) or a single key value. Equal keys always share a bin,
// so n_eq counts every key equal to K*. The selection is every key > K* plus
// the (k - n_gt) lowest-index keys equal to K*.
__device__ void select_core(const ScoreArgs& a, int b, const SelectSmem& sm, int N, int kreq,
                            uint32_t kmin, uint32_t kmax) {
  const int tid = threadIdx.x;
  uint32_t* keys_s = sm.keys;
  uint8_t* flags_s = sm.flags;
  const int lo = min(a.n_sink, N), hi = max(lo, N - a.n_recent);   // candidates [lo, hi)
  const int M = hi - lo, F = N - M;                                  // candidates, forced
  if (kreq > a.k_max - F && tid == 0) latch_error(a.err, KVSEL_ERR_BOUNDS);
  int k = kreq < 0 ? 0 : kreq;
  k = min(k, min(M, a.k_max - F));
  const int KPT = (N + kThreads - 1) / kThreads;     // keys per thread, index order
  const int c0 = min(N, tid * KPT), c1 = min(N, c0 + KPT);
  const bool partial = k > 0 && k < M;

  uint32_t kstar = 0;
  int n_gt = 0, n_eq = 0;
  if (partial && kmin == kmax) {
    kstar = kmin;                            // one value: take the lowest indices
    n_eq = M;
  } else if (partial) {
    bool done = false, single = false;
    if (M <= kCand) {
      // few keys: rank them all
      for (int i = tid; i < M; i += kThreads) sm.cand[i] = keys_s[lo + i];
      __syncthreads();
      rank_candidates(sm, M, k);
      done = true;
    } else {
      const float smin = key_float(kmin), smax = key_float(kmax);
      const float span = __fsub_rn(smax, smin);
      const float scale = __fdiv_rn(float(kBins), span);
      if (isfinite(smin) && isfinite(span) && span > 0.f && isfinite(scale) && scale > 0.f) {
        for (int i = lo + tid; i < hi; i += kThreads) {
          const uint32_t key = keys_s[i];
          const int bin = value_bin(key_float(key), smin, scale);
          atomicAdd(&sm.hist[bin], 1);
          sm.binkey[bin] = key;                // one of the bin's keys (the only one if m == 1)
        }
        __syncthreads();
        locate_bin(sm, k);
        const int bin = sm.bcast[0], above = sm.bcast[1], m = sm.bcast[2];
        if (m == 1) {
          // a bin of one score: it is the k-th largest
          kstar = sm.binkey[bin];
          n_gt = above;
          n_eq = 1;
          single = true;
        } else if (m <= kCand) {
          for (int i = lo + tid; i < hi; i += kThreads) {
            const uint32_t key = keys_s[i];
            if (value_bin(key_float(key), smin, scale) == bin) sm.cand[atomicAdd(&sm.bcast[7], 1)] = key;
          }
          __syncthreads();
          rank_candidates(sm, m, k - above);
          n_gt = above;
          done = true;
        }
      }
    }
    if (single) {
      // K* known: the one score of its bin
    } else if (done) {
      kstar = uint32_t(sm.bcast[4]);
      n_gt += sm.bcast[5];
      n_eq = sm.bcast[6];
    } else {
      uint32_t klo = kmin;    // key window: klo <= key, (key - klo) < 2^wbits (wbits 32: no upper bound)
      int wbits = 32;
      int r = k;              // rank of K* from the top among the window's keys
      int m = M;              // keys in the window
      int shift = max(0, (32 - __clz(int(kmax - kmin))) - 11);
      while (true) {
        for (int i = lo + tid; i < hi; i += kThreads) {
          const uint32_t key = keys_s[i];
          const uint32_t dl = key - klo;
          if (key >= klo && (wbits == 32 || (dl >> wbits) == 0u)) atomicAdd(&sm.hist[dl >> shift], 1);
        }
        __syncthreads();
        locate_bin(sm, r);
        const int bin = sm.bcast[0];
        r -= sm.bcast[1];
        n_gt += sm.bcast[1];
        m = sm.bcast[2];
        klo += uint32_t(bin) << shift;
        wbits = shift;
        if (shift == 0 || m <= kCand) break;
        shift = max(0, shift - 11);
      }
      if (wbits == 0) {
        kstar = klo;                         // the bin is one key value
        n_eq = m;
      } else {
        for (int i = lo + tid; i < hi; i += kThreads) {
          const uint32_t key = keys_s[i];
          if (key >= klo && ((key - klo) >> wbits) == 0u) sm.cand[atomicAdd(&sm.bcast[7], 1)] = key;
        }
        __syncthreads();
        rank_candidates(sm, m, r);
        kstar = uint32_t(sm.bcast[4]);
        n_gt += sm.bcast[5];
        n_eq = sm.bcast[6];
      }
    }
  }
  const int need_eq = k - n_gt;              // keys equal to K* to take, lowest index first

  // ---- selection flags in index order ----
  if (partial && need_eq < n_eq) {
    int eq_cnt = 0;
    for (int i = max(c0, lo); i < min(c1, hi); ++i) eq_cnt += (keys_s[i] == kstar);
    int eq_tot;
    int eq_rank = block_exclusive_scan(eq_cnt, sm.scratch, &eq_tot);
    for (int i = c0; i < c1; ++i) {
      const uint32_t key = keys_s[i];
      bool s = true;                                    // forced blocks take no equal-key rank
      if (i >= lo && i < hi) {
        s = key > kstar;
        if (key == kstar) { s = eq_rank < need_eq; ++eq_rank; }
      }
      flags_s[i] = s ? 1 : 0;
    }
  } else {
    for (int i = c0; i < c1; ++i)
      flags_s[i] = (i < lo || i >= hi || (k > 0 && (!partial || keys_s[i] >= kstar))) ? 1 : 0;
  }
  __syncthreads();

  // ---- positions and span starts (one packed scan), then span ends ----
  int nsel_c = 0, nstart_c = 0;
  for (int i = c0; i < c1; ++i) {
    if (flags_s[i]) {
      ++nsel_c;
      if (i == 0 || !flags_s[i - 1]) ++nstart_c;
    }
  }
  int packed_tot;
  const int packed = block_exclusive_scan(nsel_c | (nstart_c << 16), sm.scratch, &packed_tot);
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
}

// select_core on the score row the score grid wrote to global memory: the
// whole row is read in the same round trip as the sequence length and k
// (entries past N are never used); the candidates' min and max keys are taken
// on the way.
__device__ void select_sequence(const ScoreArgs& a, int b, const SelectSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kreq = a.k_per_seq[b];
  const float* sc = a.scores + int64_t(b) * a.max_blocks;
  const int N = seq_blocks(a, b);
  const int lo = min(a.n_sink, N), hi = max(lo, N - a.n_recent);
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll 4
  for (int i = tid; i < a.max_blocks; i += kThreads) {
    const uint32_t key = order_key(__ldcg(sc + i));
    sm.keys[i] = key;
    if (i >= lo && i < hi) {
      kmin = min(kmin, key);
      kmax = max(kmax, key);
    }
  }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) {
    sm.mm[warp] = kmin;
    sm.mm[kWarps + warp] = kmax;
  }
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    kmin = min(kmin, sm.mm[w]);
    kmax = max(kmax, sm.mm[kWarps + w]);
  }
  select_core(a, b, sm, N, kreq, kmin, kmax);
}

// Append warps only.
__device__ __forceinline__ void append_sync() {
  asm volatile("bar.sync 2, %0;" ::"n"(kAppendThreads) : "memory");
}

// The APPEND summary update folded into the score grid, for the sequences
// whose open block lies in this CTA's share of slots: the new K/V row goes
// into its page, the block's fp64 key sum and summary are updated exactly as
// the summary kernels do, and the block's score is computed from the new
// summary. Run by the kAppendWarps append warps, one 8-channel vector per
// thread, with every load issued before the page check so that the update
// costs about two global round trips; it overlaps the first copies of the
// share. The score then follows the consumers' arithmetic exactly: the lanes
// li < LPB of the first append warp take the vectors li + LPB*i in order i
// (the summary and the query folded in the consumers' order, from shared
// scratch) and the shuffle tree is theirs, so the score equals, bit for bit,
// the one a consumer computes from the updated summary; the consumers skip
// that block. The bulk copy of the open block may carry either version of its
// summary; the score computed from that copy is not stored. emit(b, n, score)
// stores the open block's score (lane 0 of the first append warp).
template <int VPL, class Emit>
__device__ void append_open_blocks(const ScoreArgs& a, int64_t g0, int64_t g1, uint4* sum_scr,
                                   float* qf_scr, Emit emit) {
  const int at = threadIdx.x - kAppendWarp0 * 32;   // 0 .. kAppendThreads-1
  const int lane = at & 31;
  const int NV = a.NV, LPB = a.LPB;
  const int G = a.Hq / a.Hkv;
  const int vec_per_head = a.d / 8;
  const int b_first = int(g0 / a.max_blocks), b_last = int((g1 - 1) / a.max_blocks);
  for (int b = b_first; b <= b_last; ++b) {
    const int t = a.append_pos[b];
    if (t < 0) continue;
    if (t >= a.max_blocks * a.B) {
      // reported once, by the CTA that holds the sequence's first slot
      if (at == 0 && int64_t(b) * a.max_blocks >= g0) latch_error(a.err, KVSEL_ERR_BOUNDS);
      continue;
    }
    const int n = t / a.B, row = t % a.B;
    const int64_t gs = int64_t(b) * a.max_blocks + n;   // slot of the open block
    if (gs < g0 || gs >= g1) continue;                   // another CTA's slot
    const int64_t page = a.block_table[gs];
    const bool scored = n < seq_blocks(a, b);           // the score call covers the block
    const int64_t so = gs * a.Hkv * a.d;                 // the block's summary row
    for (int v = at; v < NV; v += kAppendThreads) {
      const int j = v / vec_per_head, c0 = (v % vec_per_head) * 8;
      const int64_t tok_off = (int64_t(b) * a.Hkv + j) * a.d + c0;
      // loads that do not need the page
      uint4 kn = make_uint4(0, 0, 0, 0), vn = make_uint4(0, 0, 0, 0);
      if (a.new_k) kn = *reinterpret_cast<const uint4*>(a.new_k + tok_off);
      if (a.new_v) vn = *reinterpret_cast<const uint4*>(a.new_v + tok_off);
      double* oa = a.open_acc + tok_off;
      double prev[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) prev[e] = row == 0 ? 0.0 : oa[e];
      float qf[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) qf[e] = 0.f;
      for (int r = 0; r < G; ++r) {
        const uint4 x = *reinterpret_cast<const uint4*>(a.q + (int64_t(b) * a.Hq + j * G + r) * a.d + c0);
        qf[0] += bf16lo(x.x); qf[1] += bf16hi(x.x);
        qf[2] += bf16lo(x.y); qf[3] += bf16hi(x.y);
        qf[4] += bf16lo(x.z); qf[5] += bf16hi(x.z);
        qf[6] += bf16lo(x.w); qf[7] += bf16hi(x.w);
      }
      uint4 sv;
      if (page >= 0 && page < a.n_pages) {
        const int64_t k_off = (page * a.Hkv + j) * 2 * int64_t(a.B) * a.d + tiled_off(row, c0, a.B);
        if (a.new_k) {
          *reinterpret_cast<uint4*>(a.kv_pages + k_off) = kn;
          if (a.new_v) *reinterpret_cast<uint4*>(a.kv_pages + k_off + int64_t(a.B) * a.d) = vn;
        } else {
          kn = *reinterpret_cast<const uint4*>(a.kv_pages + k_off);
        }
        double x[8], sum[8];
        unpack8(kn, x);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          sum[e] = prev[e] + x[e];
          oa[e] = sum[e];
        }
        sv = mean_to_bf16x8(sum, row + 1);
        *reinterpret_cast<uint4*>(a.summaries_out + so + v * 8) = sv;
      } else {
        if (at == 0 && v == 0) latch_error(a.err, KVSEL_ERR_BOUNDS);
        sv = *reinterpret_cast<const uint4*>(a.summaries + so + v * 8);   // left unchanged
      }
      sum_scr[v] = sv;
      float4* q4 = reinterpret_cast<float4*>(qf_scr + v * 8);
      q4[0] = make_float4(qf[0], qf[1], qf[2], qf[3]);
      q4[1] = make_float4(qf[4], qf[5], qf[6], qf[7]);
    }
    append_sync();
    if (at < 32) {
      float acc = 0.f;
      if (lane < LPB) {
        float ev = 0.f, od = 0.f;      // even and odd channels, as the consumers' pairs
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          const int v = lane + LPB * i;
          const uint4 sv = sum_scr[v];
          const float4 x0 = reinterpret_cast<const float4*>(qf_scr + v * 8)[0];
          const float4 x1 = reinterpret_cast<const float4*>(qf_scr + v * 8)[1];
          ev = fmaf(x0.x, bf16lo(sv.x), ev);
          od = fmaf(x0.y, bf16hi(sv.x), od);
          ev = fmaf(x0.z, bf16lo(sv.y), ev);
          od = fmaf(x0.w, bf16hi(sv.y), od);
          ev = fmaf(x1.x, bf16lo(sv.z), ev);
          od = fmaf(x1.y, bf16hi(sv.z), od);
          ev = fmaf(x1.z, bf16lo(sv.w), ev);
          od = fmaf(x1.w, bf16hi(sv.w), od);
        }
        acc = ev + od;
      }
      for (int off = LPB >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (lane == 0 && scored) emit(b, n, acc);
    }
    append_sync();                    // the scratch is free for the next open block
  }
}

// The arguments of one call, common to both forms; scores is the fp32 score
// row output (nullable in the one-launch form). Stage geometry is left to the
// launcher.
inline ScoreArgs make_score_args(const kvsel_problem& p, const kvsel_bf16* q,
                                 const kvsel_bf16* summaries, const int32_t* seq_lens,
                                 const int32_t* k_per_seq, float gamma, float tau_rel,
                                 int32_t* sel_idx, int32_t* n_sel, int32_t* span_start,
                                 int32_t* span_len, int32_t* n_spans, uint8_t* dense_flag,
                                 float* scores, const kvsel_append_in* app, int n_sink,
                                 int n_recent, int* err) {
  ScoreArgs a{};
  a.n_sink = n_sink; a.n_recent = n_recent;
  a.q = q; a.summaries = summaries; a.seq_lens = seq_lens; a.k_per_seq = k_per_seq;
  a.kv_pages = app ? app->kv_pages : nullptr;
  a.n_pages = app ? app->n_pages : 0;
  a.block_table = app ? app->block_table : nullptr;
  a.append_pos = app ? app->append_pos : nullptr;
  a.new_k = app ? app->new_k : nullptr;
  a.new_v = app ? app->new_v : nullptr;
  a.summaries_out = app ? app->summaries : nullptr;
  a.open_acc = app ? app->open_acc : nullptr;
  a.gamma = gamma; a.tau_rel = tau_rel;
  a.sel_idx = sel_idx; a.n_sel = n_sel; a.span_start = span_start; a.span_len = span_len;
  a.n_spans = n_spans; a.dense_flag = dense_flag;
  a.scores = scores;
  a.err = err;
  a.batch = p.batch; a.Hq = p.n_qheads; a.Hkv = p.n_kvheads; a.d = p.head_dim;
  a.B = p.block_size; a.max_blocks = p.max_blocks; a.k_max = p.k_max;
  a.NV = p.n_kvheads * p.head_dim / 8;
  int lpb = 32;
  while (a.NV % lpb) lpb >>= 1;
  a.LPB = lpb;
  return a;
}

}  // namespace
}  // namespace kvsel
