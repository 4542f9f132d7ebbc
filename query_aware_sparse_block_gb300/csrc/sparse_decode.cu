// Sparse decode attention over the selected KV blocks ("SparPR KV cache
// recovery on a consumer GPU", paragraph "On-demand local recomputation with
// cost-aware fallback": only the recovered blocks are attended, or all of
// them on the dense path), with split partial results merged by the
// flash-style log-sum-exp reduction of the DKV abstract.
//
// Design (GB300):
//  * Work unit: a tile is one attended block of one sequence for a group of
//    HPG consecutive KV heads. The selection is per sequence, so all heads of
//    a page are needed, and a page stores each head's K tile and V tile next
//    to each other, heads in order: a tile's K and V are one contiguous range
//    (32 KiB for d = 128 and HPG * B = 64 rows), moved into shared memory by a
//    single 1-D bulk (TMA) copy. Scattered 32 KiB copies stream markedly
//    faster than pairs of 16 KiB ones on GB300 HBM3e. The tiled layout already
//    carries the 16-byte chunk swizzle (chunk c of row t at c ^ (t % 8)), so
//    ldmatrix reads are conflict-free.
//  * Work list: the flattened (sequence, head group, block) tiles. When every
//    (sequence, head group) segment that has tiles has the same number nb of
//    them (every sequence of the batch at the same length and k), each
//    segment gets the same number m of CTAs, m = min(grid / segments,
//    nb / kMinTilesPerCta rounded up), and CTA c takes part c % m of segment
//    c / m: no CTA's range crosses a segment boundary, so a warp loads one
//    query and stores one state, and the SMs left over stay free for the
//    Top-k still running in the previous kernel (64 segments on 152 SMs: 128
//    CTAs; the call is about 4 % shorter than with 152 CTAs whose ranges cross
//    segments, measured on GB300). Other
//    batches are split into equal contiguous ranges, one per CTA, so that the
//    HBM stream is balanced whatever the per-sequence selection sizes are. At
//    the end of each (sequence, head group) segment every warp stores its online-
//    softmax state (max, sum, unnormalised output) to global memory and moves
//    on without any synchronisation; a second small kernel, launched as a
//    programmatic dependent of the first so that it is already resident,
//    merges the states of each output row by log-sum-exp.
//  * Pipeline: two rings of 4 warps; ring r takes every other tile of the
//    CTA's range and keeps S of them in flight. Each warp of a ring owns one
//    (head, 16-token slice) of its ring's tiles; the last warp to finish a
//    slot (a shared-memory counter) refills it, so no warp waits on another
//    and the two rings drift apart instead of hitting the tensor pipe in
//    lockstep.
//  * Math: tokens are the M dimension of mma.m16n8k16 bf16 tensor-core tiles:
//    S^T = K Q^T with K read by ldmatrix from the swizzled tile and the GQA
//    group's query heads (G <= 16, zero-padded to 8 or 16 columns) as N, online
//    softmax in fp32 per head column (exp2 of log2-scaled logits, accumulators
//    rescaled only when a running max moves), then O^T += V^T P^T with V read
//    by ldmatrix.trans and P transposed into B fragments by movmatrix; P is
//    split into bf16 high and low parts so the product keeps ~16 bits.
//  * Every wait on a copy is bounded; a wait that runs out latches
//    KVSEL_ERR_TIMEOUT and the warp stops issuing work.
#include <climits>
#include <type_traits>

#include "kvsel_common.cuh"
#include "kvsel_internal.h"

namespace kvsel {
namespace {

constexpr int kW = 8;                  // warps per CTA
constexpr int kRingWarps = 4;          // warps sharing one tile ring: one (head, 16-token slice) each
constexpr int kRings = kW / kRingWarps;
constexpr int kThreads = kW * 32;
constexpr int kMaxCtas = 512;          // partial-slot capacity of the workspace
constexpr int kMinTilesPerCta = 4;
constexpr int kMaxStages = 8;

// Heads per tile for block size B and H_kv heads: as many as keep the tile
// at 64 token rows (4 warps x 16 rows), and a divisor of H_kv.
inline int heads_per_group(int B, int Hkv) {
  int h = std::min(Hkv, kRingWarps * 16 / B);
  while (h > 1 && Hkv % h) --h;
  return std::max(1, h);
}

struct DecodeArgs {
  const kvsel_bf16* kv_base;  // PAGED: KV pages; STAGED: staging; HOST_DIRECT: the host tier
                              // (device-mapped); all in the same page layout
  const kvsel_bf16* q;
  const int32_t* seq_lens;
  const int32_t* sel_idx;
  const int32_t* n_sel;
  const uint8_t* dense_flag;
  const int32_t* block_table;
  int64_t n_pages;
  int kind;
  int slots;
  int host_blocks;     // HOST_DIRECT: block stride of the host tier per sequence
  float scale_log2;
  float* out;
  kvsel_bf16* out_bf16;
  float* lse;
  float* partials;     // warp states: [(cta + segment) * W + warp][G][D + 4] (m, l, -, -, O)
  int2* seg_info;      // [batch * n_groups] (first CTA, CTA count) of each segment; count 0: no tile
  int* err;
  int batch, Hq, Hkv, G, B, max_blocks, k_max;
  int hpg, n_groups;   // heads per tile, head groups per sequence
  int stages;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ int find_seq(const int* base_s, int batch, int64_t g) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (base_s[mid] <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Copy unit of tile g (the head group's K+V range, in units of 2*HPG*B*d
// elements) and its valid token count (0 when the tile is skipped).
__device__ void tile_info(const DecodeArgs& a, const int* base_s, const int* tlen_s, int64_t g,
                          bool report, int& unit, int& cnt) {
  const int b = find_seq(base_s, a.batch, g);
  const int64_t r = g - base_s[b];
  const int nb = (base_s[b + 1] - base_s[b]) / a.n_groups;
  const int hg = int(r / nb);
  const int o = int(r % nb);
  const int T = tlen_s[b];
  const int N = (T + a.B - 1) / a.B;
  const bool dense = a.dense_flag && a.dense_flag[b];
  const int n = dense ? o : a.sel_idx[int64_t(b) * a.k_max + o];
  bool ok = (n >= 0 && n < N);
  cnt = ok ? min(a.B, T - n * a.B) : 0;
  if (a.kind == KVSEL_KV_PAGED) {
    int64_t page = ok ? a.block_table[int64_t(b) * a.max_blocks + n] : 0;
    if (page < 0 || page >= a.n_pages) { ok = false; page = 0; }
    unit = int(page * a.n_groups + hg);
  } else if (a.kind == KVSEL_KV_HOST_DIRECT) {
    if (n >= a.host_blocks) ok = false;
    unit = ok ? int((int64_t(b) * a.host_blocks + n) * a.n_groups + hg) : 0;
  } else {
    int64_t slot = o;
    if (slot >= a.slots) { ok = false; slot = 0; }
    unit = int((int64_t(b) * a.slots + slot) * a.n_groups + hg);
  }
  if (!ok) {
    cnt = 0;
    if (report) latch_error(a.err, KVSEL_ERR_BOUNDS);
  }
}

// Shared address of (head h of the group, kv = 0 for K / 1 for V, token row,
// channel c with c % 8 == 0) in a slot holding the tile as the page stores it:
// [head][K, V][d/64][row][64], 16-byte chunk c of row t at c ^ (t % 8).
__device__ __forceinline__ uint32_t swz(uint32_t stage, int h, int kv, int halves, int B, int row,
                                        int c) {
  const int half = c >> 6;
  const int chunk = (c & 63) >> 3;
  return stage + uint32_t((((h * 2 + kv) * halves + half) * B + row) * 128 + ((chunk ^ (row & 7)) << 4));
}

template <int D, int B, int NTH>
__global__ void __launch_bounds__(kThreads, 1) sparse_decode_kernel(DecodeArgs a) {
  constexpr int kWPH = B / 16;               // warps (16-token slices) per head
  constexpr int kMT = D / 16;                // 16-channel m-tiles of O^T
  static_assert(kWPH <= kRingWarps, "block larger than a ring");
  constexpr int kKS = D / 16;                // k-steps of K Q^T
  constexpr int kHalves = D / 64;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.stages;
  const int G = a.G;
  const int HPG = a.hpg;
  const int plane_elems = HPG * B * D;      // one head-group tile of K (or V)
  const int plane_bytes = plane_elems * 2;
  const int tile_bytes = 2 * plane_bytes;    // K + V
  unsigned char* tiles = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(tiles + size_t(S) * kRings * tile_bytes);
  int* done_s = reinterpret_cast<int*>(bars + S * kRings);          // [S][rings] consumer counts
  int* base_s = done_s + 2 * kMaxStages * kRings;                  // [batch+1]
  int* tlen_s = base_s + a.batch + 1;                              // [batch]
  __shared__ int scan_s[kW];
  __shared__ int nbmin_s[kW], nbmax_s[kW];   // per warp: smallest / largest non-zero tile count per segment

  // the merge kernel may be scheduled now; it waits for this grid's completion
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // every input may still be being written by an earlier kernel of the stream
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int NA = HPG * kWPH;                 // active warps per ring
  const int ring = warp / kRingWarps, task = warp % kRingWarps;
  const bool active = task < NA;
  const int h_local = task / kWPH, slice = task % kWPH;

  // ---- per-sequence tile counts and prefix; the range of the non-zero counts ----
  int carry = 0;
  int nb_lo = INT_MAX, nb_hi = 0;
  for (int b0 = 0; b0 < a.batch; b0 += kThreads) {
    const int b = b0 + tid;
    int tiles_b = 0;
    if (b < a.batch) {
      int T = a.seq_lens[b];
      if (T < 0 || T > a.max_blocks * B) {
        latch_error(a.err, KVSEL_ERR_BOUNDS);
        T = T < 0 ? 0 : a.max_blocks * B;
      }
      tlen_s[b] = T;
      const int N = (T + B - 1) / B;
      int nb;
      if (a.dense_flag && a.dense_flag[b]) {
        nb = N;
      } else {
        nb = a.n_sel[b];
        if (nb < 0 || nb > a.k_max) latch_error(a.err, KVSEL_ERR_BOUNDS);
        nb = max(0, min(nb, min(N, a.k_max)));
      }
      tiles_b = nb * a.n_groups;
    }
    {
      const int nb = tiles_b / a.n_groups;
      const int wmin = __reduce_min_sync(0xffffffffu, nb > 0 ? nb : INT_MAX);
      const int wmax = __reduce_max_sync(0xffffffffu, nb);
      if (lane == 0) {
        nbmin_s[warp] = wmin;
        nbmax_s[warp] = wmax;
      }
    }
    int x = tiles_b;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) scan_s[warp] = x;
    __syncthreads();
    int before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      if (w < warp) before += scan_s[w];
      tot += scan_s[w];
      nb_lo = min(nb_lo, nbmin_s[w]);
      nb_hi = max(nb_hi, nbmax_s[w]);
    }
    if (b < a.batch) base_s[b] = carry + before + x - tiles_b;
    carry += tot;
    __syncthreads();
  }
  if (tid == 0) base_s[a.batch] = carry;
  __syncthreads();
  const int64_t total = carry;
  // equal segments: m CTAs each, ranges inside one segment
  const int nbu = nb_lo == nb_hi ? nb_hi : 0;
  const int n_seg = nbu > 0 ? int(total / nbu) : 0;
  const int m = n_seg > 0 && n_seg <= int(gridDim.x)
                    ? min(int(gridDim.x) / n_seg, (nbu + kMinTilesPerCta - 1) / kMinTilesPerCta)
                    : 0;
  const int A = m > 0 ? n_seg * m
                      : int(min(int64_t(gridDim.x), max(int64_t(1), (total + kMinTilesPerCta - 1) / kMinTilesPerCta)));
  if (blockIdx.x == 0) {
    // the CTAs holding each segment's states, for the merge kernel
    for (int64_t seg = tid; seg < int64_t(a.batch) * a.n_groups; seg += kThreads) {
      const int b = int(seg / a.n_groups), hg = int(seg % a.n_groups);
      const int seg_tiles = (base_s[b + 1] - base_s[b]) / a.n_groups;
      int2 info = make_int2(0, 0);
      if (seg_tiles > 0) {
        const int64_t s_start = base_s[b] + int64_t(hg) * seg_tiles, s_end = s_start + seg_tiles;
        if (m > 0) {
          info = make_int2(int(s_start / nbu) * m, m);
        } else {
          const int first_c = int(((s_start + 1) * A - 1) / total);
          const int last_c = int((s_end * A - 1) / total);
          info = make_int2(first_c, last_c - first_c + 1);
        }
      }
      a.seg_info[seg] = info;
    }
  }

  // sequences with nothing to attend: out = 0, lse = -inf
  for (int64_t e = int64_t(blockIdx.x) * kThreads + tid; e < int64_t(a.batch) * a.Hq;
       e += int64_t(gridDim.x) * kThreads) {
    const int b = int(e / a.Hq);
    if (base_s[b + 1] != base_s[b]) continue;
    a.lse[e] = -INFINITY;
    for (int c = 0; c < D; ++c) {
      a.out[e * D + c] = 0.f;
      if (a.out_bf16) a.out_bf16[e * D + c] = 0;
    }
  }
  if (total == 0) return;
  if (int(blockIdx.x) >= A) return;
  int64_t g0, g1;
  if (m > 0) {
    const int k = int(blockIdx.x) / m, part = int(blockIdx.x) % m;
    g0 = int64_t(k) * nbu + nbu * part / m;
    g1 = int64_t(k) * nbu + nbu * (part + 1) / m;
  } else {
    g0 = total * blockIdx.x / A;
    g1 = total * (blockIdx.x + 1) / A;
  }
  if (g0 >= g1) return;
  const int L = int(g1 - g0);

  if (tid == 0) {
    for (int i = 0; i < S * kRings; ++i) {
      mbar_init(&bars[i], 1);
      done_s[i] = 0;
    }
    fence_barrier_init();
  }
  __syncthreads();

  // ---- this ring's tile stream: tiles g0 + ring + m * kRings ----
  const int LR = L > ring ? (L - ring + kRings - 1) / kRings : 0;
  const uint32_t tiles_base = smem_u32(tiles);
  auto slot_idx = [&](int m) -> int { return (m % S) * kRings + ring; };
  auto slot_bar = [&](int m) -> uint64_t* { return &bars[slot_idx(m)]; };
  // Tile descriptors, 32 at a time: lane i holds the copy unit and valid token
  // count of tile (cbase + i) in `cur` and of tile (cbase + 32 + i) in `nxt`;
  // their selection and block-table loads run a whole batch ahead.
  int cbase = 0;
  int cur_rk = 0, cur_cnt = 0, nxt_rk = 0, nxt_cnt = 0;
  auto load_batch = [&](int base, int& rk, int& cnt) {
    const int m = base + lane;
    rk = cnt = 0;
    if (m < LR) tile_info(a, base_s, tlen_s, g0 + ring + int64_t(m) * kRings, task == 0, rk, cnt);
  };
  auto tile_desc = [&](int m, int& rk, int& cnt) {   // all lanes; cbase <= m < cbase + 64
    const int i = m - cbase;
    const int src = i & 31;
    const int rk0 = __shfl_sync(0xffffffffu, cur_rk, src), rk1 = __shfl_sync(0xffffffffu, nxt_rk, src);
    const int c0 = __shfl_sync(0xffffffffu, cur_cnt, src), c1 = __shfl_sync(0xffffffffu, nxt_cnt, src);
    rk = i < 32 ? rk0 : rk1;
    cnt = i < 32 ? c0 : c1;
  };
  const uint64_t pol = l2_evict_first_policy();   // K/V are read once per step
  auto issue = [&](int m, int unit) {   // one lane
    uint64_t* bar = slot_bar(m);
    mbar_arrive_expect_tx(bar, uint32_t(tile_bytes));
    unsigned char* dst = tiles + size_t(slot_idx(m)) * tile_bytes;
    bulk_load_hint(dst, a.kv_base + int64_t(unit) * 2 * plane_elems, uint32_t(tile_bytes), bar, pol);
  };
  // From host-mapped memory the tile arrives by 16-byte cp.async reads of the
  // whole warp instead of one bulk copy (the same bytes land in the same
  // place); each lane's copies arrive on the slot's barrier when they have
  // landed, and lane 0's ordinary arrival completes the count of one.
  const bool host_direct = a.kind == KVSEL_KV_HOST_DIRECT;
  auto issue_warp = [&](int m, int unit) {   // whole warp
    uint64_t* bar = slot_bar(m);
    const uint32_t dst = smem_u32(tiles + size_t(slot_idx(m)) * tile_bytes);
    const unsigned char* src =
        reinterpret_cast<const unsigned char*>(a.kv_base + int64_t(unit) * 2 * plane_elems);
    for (int off = lane * 16; off < tile_bytes; off += 32 * 16) cp_async_16(dst + off, src + off);
    cp_async_mbar_arrive(bar);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
  };
  if (active) {
    load_batch(0, cur_rk, cur_cnt);
    load_batch(32, nxt_rk, nxt_cnt);
  }
  if (task == 0) {
    for (int m = 0; m < min(S, LR); ++m) {
      int rk, cnt;
      tile_desc(m, rk, cnt);
      if (host_direct) issue_warp(m, rk);
      else if (lane == 0) issue(m, rk);
    }
  }
  bool dead = false;
  int m_cur = 0;

  const int gq = lane >> 2, tq = lane & 3;   // mma group / thread-in-group
  const int r0 = slice * 16;                 // this warp's 16 token rows of its head
  int64_t g = g0;
  while (g < g1) {
    // ---- segment (sequence b, head group hg) containing g ----
    const int b = find_seq(base_s, a.batch, g);
    const int seg_tiles = (base_s[b + 1] - base_s[b]) / a.n_groups;
    const int hg = int((g - base_s[b]) / seg_tiles);
    const int64_t s_start = base_s[b] + int64_t(hg) * seg_tiles;
    const int64_t s_end = s_start + seg_tiles;
    const int64_t sg1 = min(g1, s_end);
    const int head = hg * HPG + h_local;      // this warp's KV head

    // O^T accumulators: o[mt][n] holds channels mt*16 + {g, g+8} of query heads
    // n*8 + {2t, 2t+1}; mh / lh: running max and (per-thread) sum of those heads
    float o[kMT][NTH][4];
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
      for (int n = 0; n < NTH; ++n) o[mt][n][0] = o[mt][n][1] = o[mt][n][2] = o[mt][n][3] = 0.f;
    float mh[NTH][2], lh[NTH][2];
#pragma unroll
    for (int n = 0; n < NTH; ++n) mh[n][0] = mh[n][1] = -INFINITY, lh[n][0] = lh[n][1] = 0.f;

    if (active) {
      // Q^T as the B operand: qb[ks][n] = q[head n*8 + g][ks*16 + {2t, 2t+1, 2t+8, 2t+9}]
      // (query heads >= G are zero columns)
      uint32_t qb[kKS][NTH][2];
      {
        const kvsel_bf16* qp = a.q + (int64_t(b) * a.Hq + int64_t(head) * G) * D;
#pragma unroll
        for (int n = 0; n < NTH; ++n) {
          const int hq = n * 8 + gq;
#pragma unroll
          for (int ks = 0; ks < kKS; ++ks) {
            const int c = ks * 16 + 2 * tq;
            qb[ks][n][0] = hq < G ? *reinterpret_cast<const uint32_t*>(qp + hq * D + c) : 0u;
            qb[ks][n][1] = hq < G ? *reinterpret_cast<const uint32_t*>(qp + hq * D + c + 8) : 0u;
          }
        }
      }
      while (m_cur < LR && g0 + ring + int64_t(m_cur) * kRings < sg1) {
        if (m_cur == cbase + 32) {             // advance the descriptor window
          cbase += 32;
          cur_rk = nxt_rk; cur_cnt = nxt_cnt;
          load_batch(cbase + 32, nxt_rk, nxt_cnt);
        }
        int t_rk, t_cnt;
        tile_desc(m_cur, t_rk, t_cnt);
        if (!dead && !mbar_wait_bounded(slot_bar(m_cur), uint32_t((m_cur / S) & 1))) {
          dead = true;
          if (lane == 0) latch_error(a.err, KVSEL_ERR_TIMEOUT);
        }
        if (host_direct) dead = __any_sync(0xffffffffu, dead);   // the refill is warp-wide
        const int cnt = t_cnt - slice * 16;    // valid tokens in this warp's 16 rows
        const uint32_t st = tiles_base + uint32_t(slot_idx(m_cur)) * uint32_t(tile_bytes);
        if (!dead && cnt > 0) {
          if (cnt < 16) {
            // rows past the sequence end: zero V so that 0 * garbage cannot poison P V
            for (int idx = lane; idx < (16 - cnt) * (D / 8); idx += 32) {
              const int row = r0 + cnt + idx / (D / 8);
              const int c = (idx % (D / 8)) * 8;
              const uint32_t ad = swz(st, h_local, 1, kHalves, B, row, c);
              asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(ad), "r"(0u) : "memory");
            }
            __syncwarp();
          }
          // S^T = K Q^T over this warp's 16 tokens (tokens are the M rows): even and
          // odd k-steps in separate accumulators to shorten the mma chains
          float sa[NTH][4], sb[NTH][4];
#pragma unroll
          for (int n = 0; n < NTH; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) sa[n][e] = sb[n][e] = 0.f;
          {
            const int row = r0 + (lane & 7) + (((lane >> 3) & 1) << 3);
            const int cofs = (lane >> 4) * 8;
#pragma unroll
            for (int ks = 0; ks < kKS; ++ks) {
              uint32_t ka[4];
              ldsm_x4(swz(st, h_local, 0, kHalves, B, row, ks * 16 + cofs), ka[0], ka[1],
                      ka[2], ka[3]);
#pragma unroll
              for (int n = 0; n < NTH; ++n) {
                if (ks & 1) mma_bf16_16816(sb[n], ka, qb[ks][n][0], qb[ks][n][1]);
                else mma_bf16_16816(sa[n], ka, qb[ks][n][0], qb[ks][n][1]);
              }
            }
          }
          // scale, mask; e & 1 selects head 2t / 2t+1, e >> 1 token g / g + 8
          float x[NTH][4], mx[NTH][2];
#pragma unroll
          for (int n = 0; n < NTH; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int tok = gq + 8 * (e >> 1);
              x[n][e] = tok < cnt ? (sa[n][e] + sb[n][e]) * a.scale_log2 : -INFINITY;
            }
            mx[n][0] = fmaxf(x[n][0], x[n][2]);
            mx[n][1] = fmaxf(x[n][1], x[n][3]);
          }
          bool grow = false;
#pragma unroll
          for (int n = 0; n < NTH; ++n)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
#pragma unroll
              for (int off = 4; off < 32; off <<= 1)
                mx[n][c] = fmaxf(mx[n][c], __shfl_xor_sync(0xffffffffu, mx[n][c], off));
              grow |= mx[n][c] > mh[n][c];
            }
          if (__any_sync(0xffffffffu, grow)) {
            // a running max moved: rescale the accumulators of every head
#pragma unroll
            for (int n = 0; n < NTH; ++n) {
              float alpha[2];
#pragma unroll
              for (int c = 0; c < 2; ++c) {
                const float mn = fmaxf(mh[n][c], mx[n][c]);
                const float m_use = (mn == -INFINITY) ? 0.f : mn;
                alpha[c] = ex2(mh[n][c] - m_use);
                mh[n][c] = mn;
                lh[n][c] *= alpha[c];
              }
#pragma unroll
              for (int mt = 0; mt < kMT; ++mt) {
                o[mt][n][0] *= alpha[0]; o[mt][n][2] *= alpha[0];
                o[mt][n][1] *= alpha[1]; o[mt][n][3] *= alpha[1];
              }
            }
          }
          // P^T (tokens x heads) as the B operand: bf16 high and low parts, each
          // 8x8 block transposed from the accumulator layout with movmatrix
          uint32_t ph[NTH][2], pl[NTH][2];
#pragma unroll
          for (int n = 0; n < NTH; ++n) {
            const float mu0 = (mh[n][0] == -INFINITY) ? 0.f : mh[n][0];
            const float mu1 = (mh[n][1] == -INFINITY) ? 0.f : mh[n][1];
            float pv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              pv[e] = ex2(x[n][e] - ((e & 1) ? mu1 : mu0));
              lh[n][e & 1] += pv[e];
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const uint32_t hi = pack_bf16x2(pv[2 * k], pv[2 * k + 1]);
              const uint32_t lo = pack_bf16x2(pv[2 * k] - bf16lo(hi), pv[2 * k + 1] - bf16hi(hi));
              ph[n][k] = movmatrix_t(hi);
              pl[n][k] = movmatrix_t(lo);
            }
          }
          // O^T += V^T P^T: V^T m-tiles (16 channels x 16 tokens) by ldmatrix.trans,
          // two m-tiles at a time, high parts then low parts
          {
            const int row = r0 + (lane & 7) + ((lane >> 4) << 3);
            const int cofs = ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int mt = 0; mt < kMT; mt += 2) {
              uint32_t va[2][4];
#pragma unroll
              for (int u = 0; u < 2; ++u)
                ldsm_x4_t(swz(st, h_local, 1, kHalves, B, row, (mt + u) * 16 + cofs),
                          va[u][0], va[u][1], va[u][2], va[u][3]);
#pragma unroll
              for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int n = 0; n < NTH; ++n) mma_bf16_16816(o[mt + u][n], va[u], ph[n][0], ph[n][1]);
#pragma unroll
              for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int n = 0; n < NTH; ++n) mma_bf16_16816(o[mt + u][n], va[u], pl[n][0], pl[n][1]);
            }
          }
        }
        // release the slot; the last warp to release it refills it S tiles ahead
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          const int before = atomicAdd(&done_s[slot_idx(m_cur)], 1);
          last = (before % NA) == NA - 1;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last && !dead && m_cur + S < LR) {
          int rk, cnt2;
          tile_desc(m_cur + S, rk, cnt2);
          if (host_direct) {
            issue_warp(m_cur + S, rk);
          } else if (lane == 0) {
            fence_proxy_async();
            issue(m_cur + S, rk);
          }
        }
        ++m_cur;
      }
    }

    // ---- store this warp's state for the segment; the merge kernel combines ----
#pragma unroll
    for (int n = 0; n < NTH; ++n)
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) lh[n][c] += __shfl_xor_sync(0xffffffffu, lh[n][c], off);
    if (active) {
      const int64_t seg = int64_t(b) * a.n_groups + hg;
      float* mw = a.partials + ((int64_t(blockIdx.x) + seg) * kW + warp) * G * (D + 4);
#pragma unroll
      for (int n = 0; n < NTH; ++n)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int hq = n * 8 + 2 * tq + c;
          if (hq < G) {
            float* dst = mw + hq * (D + 4);
            if (gq == 0) {
              dst[0] = mh[n][c];
              dst[1] = lh[n][c];
            }
#pragma unroll
            for (int mt = 0; mt < kMT; ++mt) {
              dst[4 + mt * 16 + gq] = o[mt][n][c];
              dst[4 + mt * 16 + gq + 8] = o[mt][n][c + 2];
            }
          }
        }
    }
    g = sg1;
  }

  // drain copies still in flight (only after a timeout)
  if (dead && lane == 0 && task == 0)
    for (int m = m_cur; m < min(LR, m_cur + S); ++m)
      (void)mbar_wait_bounded(slot_bar(m), uint32_t((m / S) & 1));
  if (host_direct) asm volatile("cp.async.wait_all;" ::: "memory");   // this thread's copies
}

// Log-sum-exp merge, per output row (sequence b, query head h), of the states
// every decode warp stored for the row's segment: one warp per row (MW = 1,
// four rows per CTA), or, when rows have many states, one CTA of four warps
// per row (MW = 4). Warp w takes every MW-th chunk of 16 states; lane l owns channels
// [l * D/32, (l + 1) * D/32), and every lane loads each state's (max, sum) and
// its own channel slice, so a chunk costs one round trip to L2. With MW = 4 the
// four partial results are then merged through shared memory by warp 0. A long
// sequence attended by few blocks per CTA (one sequence of 131072 tokens, say)
// spreads its segment over many CTAs and so gives a row many states; four
// warps read them in a quarter of the round trips. Launched as a programmatic
// dependent of the decode kernel: it can be resident early and waits for the
// decode grid's completion before it reads anything that grid wrote.
template <int D, int WPH, int MW>
__global__ void __launch_bounds__(128) merge_rows_kernel(DecodeArgs a) {
  constexpr int kCPL = D / 32;            // channels per lane
  constexpr int kChunk = 16;              // states in flight per lane
  constexpr int kPerCta = kRings * WPH;   // warps of one CTA holding a head
  static_assert(MW == 1 || MW == 4, "one or four warps per row");
  constexpr int kMW = MW;                 // warps sharing one row's states
  constexpr int kRowsPerCta = 4 / MW;
  using vec_t = typename std::conditional<kCPL == 4, float4, float2>::type;
  __shared__ float ml_s[4][2];
  __shared__ vec_t o_s[3][32];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31, wq = (threadIdx.x >> 5) % kMW;
  const int64_t row = int64_t(blockIdx.x) * kRowsPerCta + (threadIdx.x >> 5) / kMW;
  if (row >= int64_t(a.batch) * a.Hq) return;   // uniform in a CTA when kMW == 4
  const int b = int(row / a.Hq), hq = int(row % a.Hq);
  const int G = a.G, j = hq / G, r = hq % G;
  const int hg = j / a.hpg, h_local = j % a.hpg;
  const int64_t seg = int64_t(b) * a.n_groups + hg;
  const int2 info = __ldcg(a.seg_info + seg);
  if (info.y == 0) return;                // no attended token: written by the decode kernel
  const int first_c = info.x;
  const int NP = info.y * kPerCta;
  auto state = [&](int i) -> const float* {
    const int c = first_c + i / kPerCta, k = i % kPerCta;
    const int w = (k / WPH) * kRingWarps + h_local * WPH + (k % WPH);
    return a.partials + (((int64_t(c) + seg) * kW + w) * G + r) * (D + 4);
  };
  float M = -INFINITY, L = 0.f;           // running max and sum (log2 domain)
  float acc[kCPL];
#pragma unroll
  for (int u = 0; u < kCPL; ++u) acc[u] = 0.f;
  for (int i0 = wq * kChunk; i0 < NP; i0 += kMW * kChunk) {   // every kMW-th chunk
    float mi[kChunk], li[kChunk];
    vec_t oi[kChunk];
#pragma unroll
    for (int k = 0; k < kChunk; ++k) {
      mi[k] = -INFINITY;
      li[k] = 0.f;
      if (i0 + k < NP) {
        const float* st = state(i0 + k);
        mi[k] = __ldcg(st);
        li[k] = __ldcg(st + 1);
        oi[k] = __ldcg(reinterpret_cast<const vec_t*>(st + 4) + lane);
      }
    }
    float mc = M;
#pragma unroll
    for (int k = 0; k < kChunk; ++k) mc = fmaxf(mc, mi[k]);
    if (mc == -INFINITY) continue;
    const float rs = M == -INFINITY ? 0.f : ex2(M - mc);
    L *= rs;
#pragma unroll
    for (int u = 0; u < kCPL; ++u) acc[u] *= rs;
#pragma unroll
    for (int k = 0; k < kChunk; ++k) {
      if (i0 + k < NP && mi[k] != -INFINITY) {
        const float wk = ex2(mi[k] - mc);
        L += wk * li[k];
        const float* ov = reinterpret_cast<const float*>(&oi[k]);
#pragma unroll
        for (int u = 0; u < kCPL; ++u) acc[u] += wk * ov[u];
      }
    }
    M = mc;
  }
  // the kMW partial states of the row, merged by warp 0
  if constexpr (kMW > 1) {
  if (lane == 0) {
    ml_s[wq][0] = M;
    ml_s[wq][1] = L;
  }
  if (wq > 0) {
    vec_t v;
    float* vp = reinterpret_cast<float*>(&v);
#pragma unroll
    for (int u = 0; u < kCPL; ++u) vp[u] = acc[u];
    o_s[wq - 1][lane] = v;
  }
  __syncthreads();
  if (wq > 0) return;
  {
    float mx = M;
#pragma unroll
    for (int w = 1; w < kMW; ++w) mx = fmaxf(mx, ml_s[w][0]);
    if (mx != -INFINITY) {
      const float r0 = M == -INFINITY ? 0.f : ex2(M - mx);
      L *= r0;
#pragma unroll
      for (int u = 0; u < kCPL; ++u) acc[u] *= r0;
#pragma unroll
      for (int w = 1; w < kMW; ++w) {
        const float mw = ml_s[w][0];
        if (mw == -INFINITY) continue;
        const float rw = ex2(mw - mx);
        L += rw * ml_s[w][1];
        const vec_t v = o_s[w - 1][lane];
        const float* ov = reinterpret_cast<const float*>(&v);
#pragma unroll
        for (int u = 0; u < kCPL; ++u) acc[u] += rw * ov[u];
      }
      M = mx;
    }
  }
  }
  vec_t res;
  float* rv = reinterpret_cast<float*>(&res);
#pragma unroll
  for (int u = 0; u < kCPL; ++u) rv[u] = L > 0.f ? acc[u] / L : 0.f;
  reinterpret_cast<vec_t*>(a.out + row * D)[lane] = res;
  if (a.out_bf16) {
    uint32_t pk[kCPL / 2];
#pragma unroll
    for (int u = 0; u < kCPL / 2; ++u)
      pk[u] = uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(rv[2 * u]))) |
              (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(rv[2 * u + 1]))) << 16);
    if constexpr (kCPL == 4)
      reinterpret_cast<uint2*>(a.out_bf16 + row * D)[lane] = make_uint2(pk[0], pk[1]);
    else
      reinterpret_cast<uint32_t*>(a.out_bf16 + row * D)[lane] = pk[0];
  }
  if (lane == 0) a.lse[row] = L > 0.f ? (M + lg2(L)) * 0.6931471805599453f : -INFINITY;
}

template <int D, int B, int NTH>
cudaError_t launch_t(const kvsel_problem& p, const DecodeArgs& a0, cudaStream_t s) {
  DecodeArgs a = a0;
  const size_t tile_bytes = size_t(a.hpg) * B * D * 4;
  // 1024: manual alignment of the tile area; 256: static shared variables
  const size_t rest = 1024 + 256 + 8 * 2 * kMaxStages * kRings + (size_t(p.batch) * 2 + 1) * 4;
  const int max_optin = max_smem_optin();
  int stages = int((size_t(max_optin) - rest - 8 * kMaxStages * kRings) / (tile_bytes * kRings));
  stages = std::min(kMaxStages, stages);
  if (stages < 1) return cudaErrorInvalidConfiguration;
  a.stages = stages;
  const size_t smem = rest + size_t(stages) * kRings * tile_bytes + 8 * stages * kRings;
  auto kfn = sparse_decode_kernel<D, B, NTH>;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kfn), int(smem));
  if (e != cudaSuccess) return e;
  const int grid = std::min(kMaxCtas, sm_count());
  e = launch_pdl(kfn, dim3(grid), dim3(kThreads), smem, s, a);
  count_launch();
  if (e != cudaSuccess) return e;
  // The row merge, as a programmatic dependent of the decode grid. A row has
  // (CTAs its segment spans) x kRings x B/16 states; bound the span with the
  // decode's own split applied to k_max blocks per sequence, and give rows
  // with more than four chunks of states four warps each.
  const int64_t rows = int64_t(p.batch) * p.n_qheads;
  const int64_t total_max = int64_t(p.batch) * a.n_groups * p.k_max;
  const int64_t ctas = std::min<int64_t>(sm_count(), std::max<int64_t>(1, (total_max + kMinTilesPerCta - 1) / kMinTilesPerCta));
  const int64_t per_cta = std::max<int64_t>(1, total_max / ctas);
  const int64_t span = (p.k_max + per_cta - 1) / per_cta + 1;
  if (span * kRings * (B / 16) > 64)
    e = launch_pdl(merge_rows_kernel<D, B / 16, 4>, dim3(unsigned(rows)), dim3(128), 0, s, a);
  else
    e = launch_pdl(merge_rows_kernel<D, B / 16, 1>, dim3(unsigned((rows + 3) / 4)), dim3(128), 0, s, a);
  count_launch();
  return e;
}

}  // namespace

size_t decode_meta_bytes(const kvsel_problem& p) {
  const int hpg = heads_per_group(p.block_size, p.n_kvheads);
  return (size_t(p.batch) * (p.n_kvheads / hpg) * 8 + 255) / 256 * 256;
}

size_t sparse_decode_ws_bytes(const kvsel_problem& p) {
  const int G = p.n_qheads / std::max(1, p.n_kvheads);
  const int hpg = heads_per_group(p.block_size, p.n_kvheads);
  const size_t segments = size_t(p.batch) * (p.n_kvheads / hpg);
  const size_t parts = (size_t(kMaxCtas) + segments) * kW * G * (p.head_dim + 4) * 4;
  return decode_meta_bytes(p) + parts;
}

cudaError_t launch_sparse_decode(const kvsel_problem& p, const kvsel_bf16* q,
                                 const kvsel_kv_src& kv, const int32_t* seq_lens,
                                 const int32_t* sel_idx, const int32_t* n_sel,
                                 const uint8_t* dense_flag, float softmax_scale, float* out,
                                 kvsel_bf16* out_bf16, float* lse, void* ws, int* err,
                                 cudaStream_t s) {
  if (p.batch == 0) return cudaSuccess;
  DecodeArgs a{};
  a.q = q; a.seq_lens = seq_lens; a.sel_idx = sel_idx; a.n_sel = n_sel; a.dense_flag = dense_flag;
  a.block_table = kv.block_table; a.n_pages = kv.n_pages;
  a.kind = (kv.kind == KVSEL_KV_PAGED || kv.kind == KVSEL_KV_HOST_DIRECT) ? kv.kind : KVSEL_KV_STAGED;
  a.slots = kv.staging_slots;
  a.host_blocks = kv.host_blocks;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.out = out; a.out_bf16 = out_bf16; a.lse = lse;
  char* w = static_cast<char*>(ws);
  a.seg_info = reinterpret_cast<int2*>(w);
  a.partials = reinterpret_cast<float*>(w + decode_meta_bytes(p));
  a.hpg = heads_per_group(p.block_size, p.n_kvheads);
  a.n_groups = p.n_kvheads / a.hpg;
  a.err = err;
  a.batch = p.batch; a.Hq = p.n_qheads; a.Hkv = p.n_kvheads; a.G = p.n_qheads / p.n_kvheads;
  a.B = p.block_size; a.max_blocks = p.max_blocks; a.k_max = p.k_max;
  const int D = p.head_dim;
  a.kv_base = a.kind == KVSEL_KV_PAGED ? kv.kv_pages
              : a.kind == KVSEL_KV_HOST_DIRECT ? kv.host_kv : kv.staging;
  const int Bs = p.block_size;
  if (D == 128 && Bs == 16) return a.G <= 8 ? launch_t<128, 16, 1>(p, a, s) : launch_t<128, 16, 2>(p, a, s);
  if (D == 128 && Bs == 32) return a.G <= 8 ? launch_t<128, 32, 1>(p, a, s) : launch_t<128, 32, 2>(p, a, s);
  if (D == 128 && Bs == 64) return a.G <= 8 ? launch_t<128, 64, 1>(p, a, s) : launch_t<128, 64, 2>(p, a, s);
  if (D == 64 && Bs == 16) return a.G <= 8 ? launch_t<64, 16, 1>(p, a, s) : launch_t<64, 16, 2>(p, a, s);
  if (D == 64 && Bs == 32) return a.G <= 8 ? launch_t<64, 32, 1>(p, a, s) : launch_t<64, 32, 2>(p, a, s);
  if (D == 64 && Bs == 64) return a.G <= 8 ? launch_t<64, 64, 1>(p, a, s) : launch_t<64, 64, 2>(p, a, s);
  return cudaErrorInvalidValue;
}

}  // namespace kvsel
