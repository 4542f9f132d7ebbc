// Query-aware block scoring, Top-k selection and span merge in one launch
// ("SparPR KV cache recovery on a consumer GPU": paragraph "Query-Aware
// key-block selection" for the score and Top-k, paragraph "On-demand local
// recomputation with cost-aware fallback" for spans and the Dense Fallback
// Threshold gamma).
//
// Design (GB300): one thread-block cluster of C CTAs per sequence, all
// clusters resident at once (C is the largest cluster size for which the
// batch fits in one wave). Nothing but the selection leaves the cluster: no
// score row goes through global memory and no second grid is launched.
//  * CTA r of the cluster owns the blocks [r*M/C, (r+1)*M/C) of the
//    sequence's summary row (M = max_blocks; a static cut, so the first
//    copies leave right after the wait on the previous kernel). The range is
//    walked in chunks of whole block summaries, each moved into shared memory
//    by one 1-D bulk (TMA) copy onto its own mbarrier. One warp issues the
//    query rows and the first round of S chunks; after that each of the eight
//    consumer warps owns S/8 stages: it waits for its chunk, scores it and
//    refills the same stage with its next chunk, so a stage is only ever
//    refilled by the warp that has just drained it and no stage needs an
//    "empty" barrier.
//  * A consumer warp scores four rows of blocks per pass with independent
//    accumulators (fp32 FMA on channel pairs, against the query folded over
//    its GQA group once per CTA) and one transposing shuffle tree; every score
//    is computed with the operations, in the order, of the two-grid form, so
//    the two forms agree bit for bit. The order key of each score goes
//    straight into the leader CTA's key row through distributed shared
//    memory, and the smallest and largest candidate keys into two leader words
//    by cluster-scope atomics.
//  * With an APPEND folded in, the four append warps of the CTA owning the
//    open block update it exactly as the two-grid form does and emit its key.
//  * After one cluster barrier (release by every thread, acquire by the
//    leader) the leader CTA runs the shared Top-k + span + gamma core on the
//    key row in its own shared memory. The other CTAs exit at the barrier.
// Every wait on a copy is bounded (KVSEL_ERR_TIMEOUT); the cluster barriers
// are reached by every thread on every path, after those bounded waits.
#include <mutex>

#include "kvsel_internal.h"
#include "score_common.cuh"

namespace kvsel {
namespace {

constexpr int kCW = 8;                   // consumer warps
constexpr int kIssueWarp = kCW;          // issues the query rows and the first round of chunks
constexpr int kInfoWarp = kAppendWarp0 + kAppendWarps;   // reads N and k for the leader's Top-k
static_assert(kAppendWarp0 == kCW + 1, "warp roles");
static_assert(kInfoWarp < kWarps, "warp roles");
constexpr int kMaxCluster = 16;
constexpr int kMaxClusterBlocks = 4096;  // key row held in the leader's shared memory
constexpr int kMinCtaBytes = 8 * 1024;   // fewest summary bytes worth a CTA of its own

// Select-phase scratch of the leader, carved from its drained stage area.
constexpr int kSelBinkey = 0;                          // kBins keys
constexpr int kSelCand = kSelBinkey + kBins * 4;       // kCand keys
constexpr int kSelScratch = kSelCand + kCand * 4;      // kWarps ints
constexpr int kSelBcast = kSelScratch + kWarps * 4;    // 8 ints
constexpr int kSelFlags = kSelBcast + 32;              // max_blocks bytes

__host__ __device__ constexpr uint32_t up16(uint32_t x) { return (x + 15u) & ~15u; }

// Dynamic shared-memory layout, computed the same way on host and device.
struct Layout {
  uint32_t q, qf, keys, hist, bars, misc, app_sum, app_qf, total;
  __host__ __device__ Layout(int S, int SB, int Hq, int Hkv, int d, int max_blocks, int NV,
                             bool app) {
    uint32_t o = uint32_t(S) * uint32_t(SB);           // stages
    q = o;     o = up16(o + uint32_t(Hq) * d * 2);     // raw query rows (bf16)
    qf = o;    o = up16(o + uint32_t(Hkv) * d * 4);    // query folded over each GQA group
    keys = o;  o = up16(o + uint32_t(max_blocks + 2) * 4);
    hist = o;  o = o + kBins * 4;
    bars = o;  o = up16(o + uint32_t(S + 1) * 8);      // full[S], query barrier
    misc = o;  o = o + 16;                             // min key, max key, T, k
    app_sum = o; o = o + (app ? uint32_t(NV) * 16 : 0u);
    app_qf = o;  o = o + (app ? uint32_t(NV) * 32 : 0u);
    total = o;
  }
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void red_cluster_min(uint32_t addr, uint32_t v) {
  asm volatile("red.relaxed.cluster.shared::cluster.min.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void red_cluster_max(uint32_t addr, uint32_t v) {
  asm volatile("red.relaxed.cluster.shared::cluster.max.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// Cluster barrier, whole warps: arrival releases this thread's earlier
// writes; the wait acquires every arrived thread's.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Consumer warps only.
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kCW * 32) : "memory");
}

template <int VPL>
__global__ void __launch_bounds__(kThreads, 1) score_topk_cluster_kernel(ScoreArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = a.stages, SB = a.stage_bytes, CHB = a.chunk_blocks, C = a.csize;
  const int NV = a.NV;
  const uint32_t block_bytes = uint32_t(NV) * 16;
  const Layout L(S, SB, a.Hq, a.Hkv, a.d, a.max_blocks, NV, a.append_pos != nullptr);
  unsigned char* stage = smem;
  const kvsel_bf16* q_s = reinterpret_cast<const kvsel_bf16*>(smem + L.q);
  float* qf_s = reinterpret_cast<float*>(smem + L.qf);
  uint32_t* keys_s = reinterpret_cast<uint32_t*>(smem + L.keys);
  int* hist_s = reinterpret_cast<int*>(smem + L.hist);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* qbar = full + S;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L.misc);   // [0] min key, [1] max key, [2] T, [3] k

  const uint32_t rank = cluster_rank();
  const int b = int(cluster_index());
  const int n_lo = int(int64_t(a.max_blocks) * rank / C);
  const int n_hi = int(int64_t(a.max_blocks) * (rank + 1) / C);
  const int nch = (n_hi - n_lo + CHB - 1) / CHB;

  if (tid == 0) {
    for (int i = 0; i <= S; ++i) mbar_init(&full[i], 1);   // full[S] is the query barrier
    misc[0] = 0xFFFFFFFFu;
    misc[1] = 0u;
    fence_barrier_init();
  }
  for (int i = tid; i < kBins; i += kThreads) hist_s[i] = 0;
  __syncthreads();
  // this CTA's shared memory is set up: peers may write into it once they
  // have waited on this phase
  cluster_arrive();
  // the decode grid may be scheduled now; it waits for this grid's completion
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // every input may still be being written by an earlier kernel of the stream
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const uint32_t keys_leader = map_shared(smem_u32(keys_s), 0);
  const uint32_t mm_leader = map_shared(smem_u32(misc), 0);
  const int64_t row0 = int64_t(b) * a.max_blocks;    // the sequence's first slot
  bool waited = false;                               // this thread has waited on phase 1

  if (warp == kIssueWarp) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();   // summaries are read once per step
      const uint32_t q_bytes = uint32_t(a.Hq) * a.d * 2;
      mbar_arrive_expect_tx(qbar, q_bytes);
      bulk_load(smem + L.q, a.q + int64_t(b) * a.Hq * a.d, q_bytes, qbar);
      // the first round before the sequence length is known: rows are
      // max_blocks long, so these reads stay inside the summary table
      for (int c = 0; c < min(S, nch); ++c) {
        const int cb = n_lo + c * CHB;
        const uint32_t bytes = uint32_t(min(CHB, n_hi - cb)) * block_bytes;
        mbar_arrive_expect_tx(&full[c], bytes);
        bulk_load_hint(stage + size_t(c) * SB, a.summaries + (row0 + cb) * NV * 8, bytes, &full[c], pol);
      }
    }
  } else if (warp >= kAppendWarp0 && warp < kAppendWarp0 + kAppendWarps) {
    if (a.append_pos) {
      const int N = seq_blocks(a, b);
      const int lo = min(a.n_sink, N), hi = max(lo, N - a.n_recent);
      cluster_wait();
      waited = true;
      append_open_blocks<VPL>(a, row0 + n_lo, row0 + n_hi, reinterpret_cast<uint4*>(smem + L.app_sum),
                              reinterpret_cast<float*>(smem + L.app_qf),
                              [&](int bb, int n, float score) {
                                const uint32_t key = order_key(score);
                                st_cluster(keys_leader + 4u * uint32_t(n), key);
                                if (a.scores) a.scores[int64_t(bb) * a.max_blocks + n] = score;
                                if (n >= lo && n < hi) {
                                  red_cluster_min(mm_leader, key);
                                  red_cluster_max(mm_leader + 4u, key);
                                }
                              });
    }
  } else if (warp == kInfoWarp) {
    if (rank == 0 && lane == 0) {
      misc[2] = uint32_t(a.seq_lens[b]);
      misc[3] = uint32_t(a.k_per_seq[b]);
    }
  } else if (warp < kCW) {
    // ---- consumer warps ----
    const int N = seq_blocks(a, b);
    const int lo = min(a.n_sink, N), hi = max(lo, N - a.n_recent);   // candidates [lo, hi)
    int n_open = -1;                    // the open block, scored by the append warps
    if (a.append_pos) {
      const int t = a.append_pos[b];
      n_open = t >= 0 && t < a.max_blocks * a.B ? t / a.B : -1;
    }
    const int HD = a.Hkv * a.d;
    const int G = a.Hq / a.Hkv;
    bool dead = false;
    int c_dead = nch;                   // first chunk not consumed after a failed wait
    if (!mbar_wait_bounded(qbar, 0u)) {
      dead = true;
      if (lane == 0) latch_error(a.err, KVSEL_ERR_TIMEOUT);
    }
    // fold q over each GQA group once for the CTA, 8 channels per thread
    for (int v = tid; v < HD / 8; v += kCW * 32) {
      const int j = (v * 8) / a.d, cc = (v * 8) % a.d;
      float f[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = 0.f;
      for (int r = 0; r < G; ++r) {
        const uint4 x = *reinterpret_cast<const uint4*>(q_s + (j * G + r) * a.d + cc);
        f[0] += bf16lo(x.x); f[1] += bf16hi(x.x);
        f[2] += bf16lo(x.y); f[3] += bf16hi(x.y);
        f[4] += bf16lo(x.z); f[5] += bf16hi(x.z);
        f[6] += bf16lo(x.w); f[7] += bf16hi(x.w);
      }
      float4* dq = reinterpret_cast<float4*>(qf_s + v * 8);
      dq[0] = make_float4(f[0], f[1], f[2], f[3]);
      dq[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
    consumers_sync();
    const int LPB = a.LPB, BPW = 32 / LPB;
    const int sub = lane / LPB, li = lane % LPB;
    const int h1 = LPB >> 1, h2 = LPB >> 2;
    const bool up1 = (li & h1) != 0, up2 = (li & h2) != 0;
    const int my_row = (up1 ? 2 : 0) + (up2 ? 1 : 0);   // the block row this lane's tree ends on
    const bool writer = (li & (h2 - 1)) == 0;
    uint64_t qreg[VPL <= 4 ? VPL : 1][4];     // folded q, channel pairs
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
    cluster_wait();                     // every CTA of the cluster is set up
    waited = true;
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
    const uint64_t pol = l2_evict_first_policy();
    for (int c = warp; c < nch; c += kCW) {
      const int s = c % S;
      const int cb = n_lo + c * CHB;
      const int nv = max(0, min(min(CHB, n_hi - cb), N - cb));   // blocks of the chunk with keys
      const bool copied = c < S || nv > 0;                         // a copy was issued for it
      if (!dead && copied && !mbar_wait_bounded(&full[s], uint32_t((c / S) & 1))) {
        dead = true;
        if (lane == 0) latch_error(a.err, KVSEL_ERR_TIMEOUT);
      }
      if (dead) {
        c_dead = min(c_dead, c);
        continue;
      }
      const unsigned char* st = stage + size_t(s) * SB;
      for (int p0 = 0; p0 < nv; p0 += 4 * BPW) {
        // rows past nv read stage bytes whose score is never stored
        const unsigned char* pr[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = p0 + j * BPW + sub;
          pr[j] = st + size_t(r < nv ? r : 0) * NV * 16;
        }
        uint64_t acc[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[j] = f32x2(0.f, 0.f);   // (even, odd) channel sums
        constexpr int kUnroll = VPL <= 4 ? VPL : 4;
#pragma unroll kUnroll
        for (int i = 0; i < VPL; ++i) {
          uint4 v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) v[j] = *reinterpret_cast<const uint4*>(pr[j] + (li + LPB * i) * 16);
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
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc[j] = ffma2(qv[0], bf16x2_f32x2(v[j].x), acc[j]);
            acc[j] = ffma2(qv[1], bf16x2_f32x2(v[j].y), acc[j]);
            acc[j] = ffma2(qv[2], bf16x2_f32x2(v[j].z), acc[j]);
            acc[j] = ffma2(qv[3], bf16x2_f32x2(v[j].w), acc[j]);
          }
        }
        // The xor trees of the four rows at once: at the first level the lanes
        // with the h1 bit keep rows 2 and 3 and hand rows 0 and 1 to their
        // partner (the others the reverse), at the second the lanes with the
        // h2 bit keep the second of their two rows; each later level works on
        // one value. Every sum is that of the row's own xor tree.
        const float s0 = f32x2_sum(acc[0]), s1 = f32x2_sum(acc[1]);
        const float s2 = f32x2_sum(acc[2]), s3 = f32x2_sum(acc[3]);
        const float x0 = (up1 ? s2 : s0) + __shfl_xor_sync(0xffffffffu, up1 ? s0 : s2, h1);
        const float x1 = (up1 ? s3 : s1) + __shfl_xor_sync(0xffffffffu, up1 ? s1 : s3, h1);
        float v = (up2 ? x1 : x0) + __shfl_xor_sync(0xffffffffu, up2 ? x0 : x1, h2);
        for (int off = h2 >> 1; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        const int r = p0 + my_row * BPW + sub;
        const int n = cb + r;
        if (writer && r < nv && n != n_open) {
          const uint32_t key = order_key(v);
          st_cluster(keys_leader + 4u * uint32_t(n), key);
          if (a.scores) a.scores[row0 + n] = v;
          if (n >= lo && n < hi) {
            kmin = min(kmin, key);
            kmax = max(kmax, key);
          }
        }
      }
      // Refill this stage with this warp's chunk S ahead (lane 0). Every value
      // the lanes read from the stage has been used by the scores above, so
      // those reads are complete before the warp barrier and the copy cannot
      // overwrite bytes still to be read.
      __syncwarp();
      const int c2 = c + S;
      if (c2 < nch && lane == 0) {
        const int cb2 = n_lo + c2 * CHB;
        const int n2 = min(min(CHB, n_hi - cb2), N - cb2);
        if (n2 > 0) {
          const uint32_t bytes = uint32_t(n2) * block_bytes;
          mbar_arrive_expect_tx(&full[s], bytes);
          bulk_load_hint(stage + size_t(s) * SB, a.summaries + (row0 + cb2) * NV * 8, bytes, &full[s], pol);
        }
      }
    }
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    if (lane == 0 && kmin <= kmax) {
      red_cluster_min(mm_leader, kmin);
      red_cluster_max(mm_leader + 4u, kmax);
    }
    // after a failed wait no copy may land once the CTA has exited: wait
    // (bounded) for every chunk of this warp still in flight
    if (dead && lane == 0) {
      (void)mbar_wait_bounded(qbar, 0u);
      for (int c = c_dead; c < min(nch, c_dead + S); c += kCW) {
        const int cb = n_lo + c * CHB;
        const int nv = min(min(CHB, n_hi - cb), N - cb);
        const bool issued = c < S || (c - S < c_dead && nv > 0);
        if (issued) (void)mbar_wait_bounded(&full[c % S], uint32_t((c / S) & 1));
      }
    }
  }

  __syncwarp();
  if (!waited) cluster_wait();
  cluster_arrive();                     // keys and key bounds are in the leader
  if (rank != 0) return;
  cluster_wait();

  // ---- leader: Top-k, spans and the gamma decision on the key row ----
  SelectSmem sel;
  sel.keys = keys_s;
  sel.flags = stage + kSelFlags;
  sel.hist = hist_s;
  sel.cand = reinterpret_cast<uint32_t*>(stage + kSelCand);
  sel.scratch = reinterpret_cast<int*>(stage + kSelScratch);
  sel.mm = nullptr;
  sel.bcast = reinterpret_cast<int*>(stage + kSelBcast);
  sel.binkey = reinterpret_cast<uint32_t*>(stage + kSelBinkey);
  if (tid < 8) sel.bcast[tid] = 0;
  const int N = blocks_of_len(a, int(misc[2]));
  const int kreq = int(misc[3]);
  const uint32_t kmin = misc[0], kmax = misc[1];
  __syncthreads();
  select_core(a, b, sel, N, kreq, kmin, kmax);
}

// ---- host side ----

int g_path = KVSEL_SCORE_PATH_AUTO;

struct ClusterKey {
  int dev;
  const void* fn;
  int C;
  size_t smem;
  int max_clusters;
};
std::mutex g_mu;
ClusterKey g_cache[128];
int g_cache_n = 0;

// Clusters of C CTAs of this kernel that fit on the device at once (cached).
int max_active_clusters(const void* fn, int C, size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  for (int i = 0; i < g_cache_n; ++i)
    if (g_cache[i].dev == dev && g_cache[i].fn == fn && g_cache[i].C == C && g_cache[i].smem == smem)
      return g_cache[i].max_clusters;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
      ensure_smem(fn, int(smem)) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  if (g_cache_n < 128) g_cache[g_cache_n++] = ClusterKey{dev, fn, C, smem, n};
  return n;
}

const void* kernel_for(int vpl) {
  switch (vpl) {
    case 1: return reinterpret_cast<const void*>(score_topk_cluster_kernel<1>);
    case 2: return reinterpret_cast<const void*>(score_topk_cluster_kernel<2>);
    case 4: return reinterpret_cast<const void*>(score_topk_cluster_kernel<4>);
    case 8: return reinterpret_cast<const void*>(score_topk_cluster_kernel<8>);
    case 16: return reinterpret_cast<const void*>(score_topk_cluster_kernel<16>);
    default: return nullptr;
  }
}

struct Plan {
  int C = 0, S = 0, CHB = 0, SB = 0;
  size_t smem = 0;
  const void* fn = nullptr;
};

// The cluster geometry for problem p, or C == 0 when the problem is outside
// the one-launch form (the two-grid form serves it).
Plan plan_cluster(const kvsel_problem& p, bool app) {
  Plan pl;
  if (p.batch <= 0 || p.max_blocks > kMaxClusterBlocks) return pl;
  const int NV = p.n_kvheads * p.head_dim / 8;
  int lpb = 32;
  while (NV % lpb) lpb >>= 1;
  const void* fn = kernel_for(NV / lpb);
  if (!fn || lpb < 4) return pl;
  const int block_bytes = NV * 16;   // a multiple of 128: NV is a multiple of 8
  const int pass_blocks = 4 * (32 / lpb);
  const int max_optin = max_smem_optin();
  const int sel_bytes = kSelFlags + p.max_blocks;
  // one or two stages per consumer warp, chunks a whole number of scoring
  // passes where they can be; the geometry with the most bytes in flight wins
  // (two stages per warp on a tie: smaller chunks, shorter tail)
  for (int spw = 2; spw >= 1; --spw) {
    const int S = kCW * spw;
    const Layout fixed(S, 0, p.n_qheads, p.n_kvheads, p.head_dim, p.max_blocks, NV, app);
    const int budget = max_optin - int(fixed.total) - 256;   // 256: static shared memory
    if (budget <= 0) continue;
    int chb = budget / S / block_bytes;
    if (chb >= pass_blocks) chb -= chb % pass_blocks;
    if (chb < 1 || chb * S <= pl.CHB * pl.S) continue;
    pl.S = S;
    pl.CHB = chb;
    pl.SB = chb * block_bytes;
  }
  if (pl.S == 0 || pl.S * pl.SB < sel_bytes) return Plan{};
  const Layout Lt(pl.S, pl.SB, p.n_qheads, p.n_kvheads, p.head_dim, p.max_blocks, NV, app);
  pl.smem = Lt.total;
  pl.fn = fn;
  // the largest cluster that keeps every sequence's cluster resident at once
  const int64_t row_bytes = int64_t(p.max_blocks) * block_bytes;
  for (int C = kMaxCluster; C >= 1; --C) {
    if (C > p.max_blocks || (C > 1 && row_bytes / C < kMinCtaBytes)) continue;
    if (max_active_clusters(fn, C, pl.smem) >= p.batch) {
      pl.C = C;
      break;
    }
  }
  return pl;
}

}  // namespace

void set_score_path(int path) { g_path = path; }
int score_path() { return g_path; }

int score_cluster_size(const kvsel_problem& p, bool app) { return plan_cluster(p, app).C; }

cudaError_t launch_score_topk_cluster(const kvsel_problem& p, const kvsel_bf16* q,
                                      const kvsel_bf16* summaries, const int32_t* seq_lens,
                                      const int32_t* k_per_seq, float gamma, float tau_rel,
                                      int32_t* sel_idx, int32_t* n_sel, int32_t* span_start,
                                      int32_t* span_len, int32_t* n_spans, uint8_t* dense_flag,
                                      float* scores_out, const kvsel_append_in* app, int n_sink,
                                      int n_recent, int* err, cudaStream_t s, bool* launched) {
  *launched = false;
  const Plan pl = plan_cluster(p, app != nullptr);
  if (pl.C == 0) return cudaSuccess;
  ScoreArgs a = make_score_args(p, q, summaries, seq_lens, k_per_seq, gamma, tau_rel, sel_idx, n_sel,
                                span_start, span_len, n_spans, dense_flag, scores_out, app, n_sink,
                                n_recent, err);
  a.stages = pl.S;
  a.chunk_blocks = pl.CHB;
  a.stage_bytes = pl.SB;
  a.csize = pl.C;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(p.batch) * unsigned(pl.C));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pl.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = ensure_smem(pl.fn, int(pl.smem));
  if (e != cudaSuccess) return e;
  switch (a.NV / a.LPB) {
    case 1: e = cudaLaunchKernelEx(&cfg, score_topk_cluster_kernel<1>, a); break;
    case 2: e = cudaLaunchKernelEx(&cfg, score_topk_cluster_kernel<2>, a); break;
    case 4: e = cudaLaunchKernelEx(&cfg, score_topk_cluster_kernel<4>, a); break;
    case 8: e = cudaLaunchKernelEx(&cfg, score_topk_cluster_kernel<8>, a); break;
    case 16: e = cudaLaunchKernelEx(&cfg, score_topk_cluster_kernel<16>, a); break;
    default: return cudaErrorInvalidValue;
  }
  count_launch();
  if (e == cudaSuccess) *launched = true;
  return e;
}

}  // namespace kvsel
