// Query-aware block scoring, Top-k selection and span merge
// ("SparPR KV cache recovery on a consumer GPU": paragraph "Query-Aware
// key-block selection" for the score and Top-k, paragraph "On-demand local
// recomputation with cost-aware fallback" for spans and the Dense Fallback
// Threshold gamma).
//
// Design (GB300): two grids per call. The score grid is launched with
// programmatic stream serialization (resident while the kernel before it
// finishes; it reads no input before griddepcontrol.wait); the Top-k grid is
// an ordinary launch after it.
//
// score_kernel streams the summary table, the only large input. The padded
// list of (sequence, block) slots, max_blocks per sequence, is cut into equal
// contiguous shares, one per CTA (one CTA per SM). No input decides the cut,
// so the first copies leave right after the wait on the previous kernel. A
// share is walked in chunks of up to 32 KiB of whole block summaries of one
// sequence. A producer warp moves each chunk into shared memory with one 1-D
// bulk (TMA) copy, S stages ahead: full / empty mbarrier pairs let it refill a
// stage as soon as every consumer warp has released it, so the refill never
// waits on a CTA-wide barrier. The first S chunks are copied before the
// sequence lengths are read; later chunks stop at a sequence's last key block.
// The query rows of a sequence ride with the first chunk of that sequence in
// the same stage. Eight consumer warps fold q over its GQA group once per
// sequence (shared memory, then registers), each warp reduces two block
// summaries per pass against it (fp32 FMA, independent accumulators, shuffle
// tree) and writes one fp32 score per block.
//
// select_kernel runs one CTA per sequence on those scores: a 2048-bin
// histogram linear in the score value locates the bin holding the k-th
// largest score and the few scores of that bin are ranked exactly (tied or
// clustered rows fall back to a histogram search over the order keys), ties
// at the k-th key are taken in index order, and block-wide scans emit the
// ascending selection, the spans and the gamma decision.
#include <type_traits>

#include "kvsel_internal.h"
#include "score_common.cuh"

namespace kvsel {
namespace {

constexpr int kScoreThreads = (kConsumerWarps + 1 + kAppendWarps) * 32;
constexpr int kStageBytes = 32 * 1024;   // summary bytes per stage (query rows follow)
constexpr int kMaxStages = 5;

// Consumer warps only (the producer warp is not counted).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

template <int VPL>
__global__ void __launch_bounds__(kScoreThreads, 1) score_kernel(ScoreArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int S = a.stages;
  const int SB = a.stage_bytes;
  unsigned char* stage = smem;                                               // [S][SB]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(S) * SB);       // copy landed
  uint64_t* empty = full + kMaxStages;                                       // stage read
  int* flag_s = reinterpret_cast<int*>(empty + kMaxStages);                  // [0] failure
  float* qf_s = reinterpret_cast<float*>(flag_s + 4);                        // Hkv*d floats
  // append scratch (only with an append): NV summary vectors, NV*8 folded q
  uint4* app_sum = reinterpret_cast<uint4*>(qf_s + a.Hkv * a.d);
  float* app_qf = reinterpret_cast<float*>(app_sum + a.NV);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // Static share of the padded (sequence, block) slots. No input decides it,
  // so it is known before the wait on the previous kernel and the first
  // copies leave right after that wait. Chunks run from g0 in steps of CH
  // blocks and stop at each row end.
  const int64_t total = int64_t(a.batch) * a.max_blocks;
  const int64_t g0 = total * blockIdx.x / gridDim.x;
  const int64_t g1 = total * (blockIdx.x + 1) / gridDim.x;
  if (g0 >= g1) return;
  const int b_first = int(g0 / a.max_blocks);
  const int n_first = int(g0 - int64_t(b_first) * a.max_blocks);
  const int CH = a.chunk_blocks;
  auto chunk_len = [&](int64_t g, int n0) {
    return min(int(min(int64_t(CH), g1 - g)), a.max_blocks - n0);
  };
  // key blocks of sequence b from the token counts of the share's first 32
  // sequences, one per lane (whole warp, b uniform)
  int T_lane = 0;
  auto n_of = [&](int b) {
    const int i = b - b_first;
    const int T = __shfl_sync(0xffffffffu, T_lane, i & 31);
    return i < 32 ? blocks_of_len(a, T) : seq_blocks(a, b);
  };
  const int NV = a.NV;
  const uint32_t block_bytes = uint32_t(NV) * 16;
  const uint32_t q_bytes = uint32_t(a.Hq) * a.d * 2;

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    flag_s[0] = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // every input may still be being written by an earlier kernel of the stream
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp >= kAppendWarp0) {
    if (a.append_pos)
      append_open_blocks<VPL>(a, g0, g1, app_sum, app_qf, [&](int b, int n, float score) {
        a.scores[int64_t(b) * a.max_blocks + n] = score;
      });
    return;
  }

  if (warp == kProducerWarp) {
    // ---- producer warp: lane 0 refills a stage as soon as every consumer
    // warp has released it. The first S chunks are copied whole before the
    // sequence lengths are known (rows are max_blocks long, so the reads stay
    // inside the table); later chunks stop at the last key block, and a chunk
    // without one completes its stage with no copy. The query rows of a
    // sequence ride with its first copied chunk. ----
    const uint64_t pol = l2_evict_first_policy();   // summaries are read once per step
    int q_b = -1;
    int c = 0;
    bool failed = false;
    int b = b_first, n0 = n_first;
    int nb_b = -1, nb = 0;            // key blocks of sequence nb_b
    int slot = 0, round = 0;          // c = round * S + slot
    for (int64_t g = g0; g < g1; ++c) {
      const int nblk = chunk_len(g, n0);
      int nc = nblk;
      if (round > 0) {
        if (c == S) T_lane = b_first + lane < a.batch ? a.seq_lens[b_first + lane] : 0;
        if (!mbar_wait_bounded(&empty[slot], uint32_t((round - 1) & 1))) {
          if (lane == 0) latch_error(a.err, KVSEL_ERR_TIMEOUT);
          failed = true;
        }
        failed = __any_sync(0xffffffffu, failed) || *reinterpret_cast<volatile int*>(flag_s) != 0;
        if (failed) break;
        if (b != nb_b) {
          nb = n_of(b);
          nb_b = b;
        }
        nc = max(0, min(nblk, nb - n0));
      }
      if (lane == 0) {
        if (nc > 0) {
          const bool with_q = b != q_b;
          const uint32_t bytes = uint32_t(nc) * block_bytes;
          unsigned char* dst = stage + size_t(slot) * SB;
          mbar_arrive_expect_tx(&full[slot], bytes + (with_q ? q_bytes : 0u));
          bulk_load_hint(dst, a.summaries + (int64_t(b) * a.max_blocks + n0) * NV * 8, bytes,
                         &full[slot], pol);
          if (with_q) bulk_load(dst + kStageBytes, a.q + int64_t(b) * a.Hq * a.d, q_bytes, &full[slot]);
        } else {
          mbar_arrive(&full[slot]);
        }
      }
      if (nc > 0) q_b = b;
      g += nblk;
      n0 += nblk;
      if (n0 == a.max_blocks) { n0 = 0; ++b; }
      if (++slot == S) { slot = 0; ++round; }
    }
    // no copy may land after the CTA exits: after a failure, wait for the
    // stages still in flight (the latest phase of each slot)
    if (failed && lane == 0)
      for (int i = max(0, c - S); i < c; ++i) (void)mbar_wait_bounded(&full[i % S], uint32_t((i / S) & 1));
    return;
  }

  // ---- consumer warps: block summaries against the query folded over its
  // GQA group (fp32); a warp takes two blocks per pass with independent
  // accumulators ----
  const int LPB = a.LPB, BPW = 32 / LPB;
  const int lg_bpw = __ffs(BPW) - 1;
  const int sub = lane / LPB, li = lane % LPB;
  const int G = a.Hq / a.Hkv;
  const int HD = a.Hkv * a.d;
  uint64_t qreg[VPL <= 4 ? VPL : 1][4];     // folded q, channel pairs
  int cur_b = -1, N_cur = 0;
  int n_open = -1;                    // block of cur_b whose score the append warp writes
  bool dead = false;
  int b = b_first, n0 = n_first;
  T_lane = b_first + lane < a.batch ? a.seq_lens[b_first + lane] : 0;
  const int P_lane = a.append_pos && b_first + lane < a.batch ? a.append_pos[b_first + lane] : -1;
  int slot = 0, round = 0;            // of the chunk in hand: round * S + slot
  for (int64_t g = g0; g < g1;) {
    const int nblk = chunk_len(g, n0);
    if (!dead && !mbar_wait_bounded(&full[slot], uint32_t(round & 1))) {
      dead = true;
      *reinterpret_cast<volatile int*>(flag_s) = 1;
      if (lane == 0) latch_error(a.err, KVSEL_ERR_TIMEOUT);
    }
    const unsigned char* st = stage + size_t(slot) * SB;
    if (b != cur_b) {
      // a new sequence, whose query rows came with this chunk: fold them over
      // the GQA group once for the CTA, 8 channels per thread
      cur_b = b;
      N_cur = n_of(b);
      if (a.append_pos) {
        const int i = b - b_first;
        int t = __shfl_sync(0xffffffffu, P_lane, i & 31);
        if (i >= 32) t = a.append_pos[b];
        n_open = t >= 0 && t < a.max_blocks * a.B ? t / a.B : -1;
      }
      const kvsel_bf16* qs = reinterpret_cast<const kvsel_bf16*>(st + kStageBytes);
      consumer_sync();                // no warp still reads the previous fold
      for (int v = tid; v < HD / 8; v += kConsumerWarps * 32) {
        const int j = (v * 8) / a.d, cc = (v * 8) % a.d;
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = 0.f;
        for (int r = 0; r < G; ++r) {
          const uint4 x = *reinterpret_cast<const uint4*>(qs + (j * G + r) * a.d + cc);
          f[0] += bf16lo(x.x); f[1] += bf16hi(x.x);
          f[2] += bf16lo(x.y); f[3] += bf16hi(x.y);
          f[4] += bf16lo(x.z); f[5] += bf16hi(x.z);
          f[6] += bf16lo(x.w); f[7] += bf16hi(x.w);
        }
        float4* dq = reinterpret_cast<float4*>(qf_s + v * 8);
        dq[0] = make_float4(f[0], f[1], f[2], f[3]);
        dq[1] = make_float4(f[4], f[5], f[6], f[7]);
      }
      consumer_sync();
      if constexpr (VPL <= 4) {
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          const float4* src = reinterpret_cast<const float4*>(qf_s + (li + LPB * i) * 8);
          const float4 x0 = src[0], x1 = src[1];
          qreg[i][0] = f32x2(x0.x, x0.y);
          qreg[i][1] = f32x2(x0.z, x0.w);
          qreg[i][2] = f32x2(x1.x, x1.y);
          qreg[i][3] = f32x2(x1.z, x1.w);
        }
      }
    }
    const int nv = min(nblk, N_cur - n0);   // blocks of this chunk that hold keys
    if (!dead && nv > 0) {
      float* out = a.scores + int64_t(b) * a.max_blocks + n0;
      const int steps = (nv + BPW - 1) >> lg_bpw;
      for (int s0 = warp; s0 < steps; s0 += 2 * kConsumerWarps) {
        const int r0 = s0 * BPW + sub;
        const int r1 = r0 + kConsumerWarps * BPW;
        // rows past nv read stage bytes that are never stored
        const unsigned char* p0 = st + size_t(r0 < nv ? r0 : 0) * NV * 16;
        const unsigned char* p1 = st + size_t(r1 < nv ? r1 : 0) * NV * 16;
        uint64_t acc0 = f32x2(0.f, 0.f), acc1 = f32x2(0.f, 0.f);   // (even, odd) channel sums
        constexpr int kUnroll = VPL <= 4 ? VPL : 4;
#pragma unroll kUnroll
        for (int i = 0; i < VPL; ++i) {
          const uint4 v0 = *reinterpret_cast<const uint4*>(p0 + (li + LPB * i) * 16);
          const uint4 v1 = *reinterpret_cast<const uint4*>(p1 + (li + LPB * i) * 16);
          uint64_t qv[4];
          if constexpr (VPL <= 4) {
#pragma unroll
            for (int e = 0; e < 4; ++e) qv[e] = qreg[i][e];
          } else {
            const float4* src = reinterpret_cast<const float4*>(qf_s + (li + LPB * i) * 8);
            const float4 x0 = src[0], x1 = src[1];
            qv[0] = f32x2(x0.x, x0.y);
            qv[1] = f32x2(x0.z, x0.w);
            qv[2] = f32x2(x1.x, x1.y);
            qv[3] = f32x2(x1.z, x1.w);
          }
          acc0 = ffma2(qv[0], bf16x2_f32x2(v0.x), acc0);
          acc1 = ffma2(qv[0], bf16x2_f32x2(v1.x), acc1);
          acc0 = ffma2(qv[1], bf16x2_f32x2(v0.y), acc0);
          acc1 = ffma2(qv[1], bf16x2_f32x2(v1.y), acc1);
          acc0 = ffma2(qv[2], bf16x2_f32x2(v0.z), acc0);
          acc1 = ffma2(qv[2], bf16x2_f32x2(v1.z), acc1);
          acc0 = ffma2(qv[3], bf16x2_f32x2(v0.w), acc0);
          acc1 = ffma2(qv[3], bf16x2_f32x2(v1.w), acc1);
        }
        // The xor tree of both blocks at once: at the first level the lanes
        // with the LPB/2 bit keep block r1 and hand block r0 to their partner,
        // the others the reverse; each later level works on one value. The
        // sums are those of two separate trees.
        const float sum0 = f32x2_sum(acc0), sum1 = f32x2_sum(acc1);
        const int half = LPB >> 1;
        const bool upper = (li & half) != 0;
        float v = (upper ? sum1 : sum0) + __shfl_xor_sync(0xffffffffu, upper ? sum0 : sum1, half);
        for (int off = half >> 1; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (li == 0 && r0 < nv && n0 + r0 != n_open) out[r0] = v;
        if (li == half && r1 < nv && n0 + r1 != n_open) out[r1] = v;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);   // this warp is done with the stage
    g += nblk;
    n0 += nblk;
    if (n0 == a.max_blocks) { n0 = 0; ++b; }
    if (++slot == S) { slot = 0; ++round; }
  }
}

// One CTA per sequence: Top-k, spans and the gamma decision on the scores the
// score grid wrote. Launched as a programmatic dependent of that grid.
__global__ void __launch_bounds__(kThreads, 1) select_kernel(ScoreArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int hist_s[kBins];
  __shared__ uint32_t binkey_s[kBins];
  __shared__ uint32_t cand_s[kCand];
  __shared__ int scratch_s[kWarps];
  __shared__ uint32_t mm_s[2 * kWarps];
  __shared__ int bcast_s[8];
  // the decode grid may be scheduled now; it waits for this grid's completion
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x;
  for (int i = tid; i < kBins; i += kThreads) hist_s[i] = 0;
  if (tid < 8) bcast_s[tid] = 0;
  SelectSmem sel;
  sel.keys = reinterpret_cast<uint32_t*>(smem);                              // max_blocks + 2
  sel.flags = reinterpret_cast<uint8_t*>(sel.keys + a.max_blocks + 2);       // max_blocks
  sel.hist = hist_s;
  sel.cand = cand_s;
  sel.scratch = scratch_s;
  sel.mm = mm_s;
  sel.bcast = bcast_s;
  sel.binkey = binkey_s;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __syncthreads();
  select_sequence(a, blockIdx.x, sel);
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
  // a reserved word per sequence (never read or written), then the fp32
  // score rows; nothing in it needs initial contents
  const size_t reserved = (size_t(p.batch) * 4 + 255) / 256 * 256;
  const size_t scores = size_t(p.batch) * p.max_blocks * 4;
  return reserved + scores;
}


cudaError_t launch_score_topk(const kvsel_problem& p, const kvsel_bf16* q,
                              const kvsel_bf16* summaries, const int32_t* seq_lens,
                              const int32_t* k_per_seq, float gamma, float tau_rel,
                              int32_t* sel_idx, int32_t* n_sel, int32_t* span_start,
                              int32_t* span_len, int32_t* n_spans, uint8_t* dense_flag,
                              float* scores_out, void* ws, const kvsel_append_in* app,
                              int n_sink, int n_recent, int* err, cudaStream_t s) {
  if (p.batch == 0) return cudaSuccess;
  if (score_path() != KVSEL_SCORE_PATH_TWO_GRID) {
    bool launched = false;
    const cudaError_t e = launch_score_topk_cluster(p, q, summaries, seq_lens, k_per_seq, gamma,
                                                    tau_rel, sel_idx, n_sel, span_start, span_len,
                                                    n_spans, dense_flag, scores_out, app, n_sink,
                                                    n_recent, err, s, &launched);
    if (e != cudaSuccess || launched) return e;
    if (score_path() == KVSEL_SCORE_PATH_CLUSTER) return cudaErrorNotSupported;
  }
  char* w = static_cast<char*>(ws);
  float* scores = scores_out ? scores_out
                             : reinterpret_cast<float*>(w + (size_t(p.batch) * 4 + 255) / 256 * 256);
  ScoreArgs a = make_score_args(p, q, summaries, seq_lens, k_per_seq, gamma, tau_rel, sel_idx, n_sel,
                                span_start, span_len, n_spans, dense_flag, scores, app, n_sink,
                                n_recent, err);
  const int vpl = a.NV / a.LPB;
  const int block_bytes = a.NV * 16;
  a.chunk_blocks = std::max(1, kStageBytes / block_bytes);
  const size_t q_bytes = size_t(p.n_qheads) * p.head_dim * 2;
  a.stage_bytes = int((kStageBytes + q_bytes + 127) / 128 * 128);
  // after the stages: full and empty barriers, a failure flag, folded q
  const size_t tail = size_t(kMaxStages) * 16 + 16 + size_t(p.n_kvheads) * p.head_dim * 4 +
                      (app ? size_t(a.NV) * 48 : 0);
  const int max_optin = max_smem_optin();
  const size_t static_smem = 256;
  int stages = 0;
  for (int st = kMaxStages; st >= 1; --st)
    if (size_t(st) * a.stage_bytes + tail + static_smem <= size_t(max_optin)) {
      stages = st;
      break;
    }
  if (stages < 1) return cudaErrorInvalidConfiguration;
  a.stages = stages;
  const size_t smem = size_t(stages) * a.stage_bytes + tail;
  const int64_t upper = int64_t(p.batch) * p.max_blocks;
  const int grid = int(std::min<int64_t>(sm_count(), std::max<int64_t>(1, upper / 8)));
  cudaError_t e = cudaSuccess;
#define KVSEL_SCORE_CASE(V)                                                                  \
  case V: {                                                                                  \
    auto kfn = score_kernel<V>;                                                              \
    e = ensure_smem(reinterpret_cast<const void*>(kfn), int(smem));                          \
    if (e != cudaSuccess) return e;                                                          \
    e = launch_pdl(kfn, dim3(grid), dim3(kScoreThreads), smem, s, a);                        \
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
  if (e != cudaSuccess) return e;
  const size_t sel_smem = ((size_t(p.max_blocks) + 2) * 4 + size_t(p.max_blocks) + 127) / 128 * 128;
  e = ensure_smem(reinterpret_cast<const void*>(select_kernel), int(sel_smem));
  if (e != cudaSuccess) return e;
  // An ordinary launch: made resident early, the Top-k CTAs would wait on SMs
  // that still stream scores and slow that stream (measured: 0.9 us later end).
  select_kernel<<<p.batch, kThreads, sel_smem, s>>>(a);
  e = cudaGetLastError();
  count_launch();
  return e;
}

cudaError_t launch_select_scores(const kvsel_problem& p, const float* scores,
                                 const int32_t* seq_lens, const int32_t* k_per_seq, float gamma,
                                 float tau_rel, int32_t* sel_idx, int32_t* n_sel,
                                 int32_t* span_start, int32_t* span_len, int32_t* n_spans,
                                 uint8_t* dense_flag, int* err, cudaStream_t s) {
  if (p.batch == 0) return cudaSuccess;
  // the select grid of the two-grid form on the caller's rows (it only reads them)
  ScoreArgs a = make_score_args(p, nullptr, nullptr, seq_lens, k_per_seq, gamma, tau_rel, sel_idx,
                                n_sel, span_start, span_len, n_spans, dense_flag,
                                const_cast<float*>(scores), nullptr, 0, 0, err);
  const size_t sel_smem = ((size_t(p.max_blocks) + 2) * 4 + size_t(p.max_blocks) + 127) / 128 * 128;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(select_kernel), int(sel_smem));
  if (e != cudaSuccess) return e;
  select_kernel<<<p.batch, kThreads, sel_smem, s>>>(a);
  e = cudaGetLastError();
  count_launch();
  return e;
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
