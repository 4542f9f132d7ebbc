// Sparse decode attention over the selected KV blocks ("SparPR KV cache
// recovery on a consumer GPU", paragraph "On-demand local recomputation with
// cost-aware fallback": only the recovered blocks are attended, or all of
// them on the dense path), with split partial results merged by the
// flash-style log-sum-exp reduction of the DKV abstract.
//
// Design (GB300):
//  * Work list: for every sequence b and KV head j, the attended blocks of b
//    are cut into sub-tiles of BT = min(B, 32) tokens; the flattened list of
//    (b, j, block, half) sub-tiles is split into equal contiguous ranges, one
//    per CTA (one CTA per SM), so the HBM stream is balanced whatever the
//    per-sequence selection sizes are (stream-K style). A (b, j) segment that
//    a CTA owns entirely is finished in place; a segment cut between CTAs is
//    finished by the last contributor (an atomic ticket, no waiting).
//  * Movement: each K or V sub-tile is one or two 2-D TMA boxes (64 channels x
//    BT rows, 128-byte swizzle) landing in shared memory; each of the four
//    warps owns a ring of stages and issues its own copies S tiles ahead, so
//    up to 4*S tiles per SM are in flight.
//  * Math: the GQA group's query heads (G <= 16, zero-padded to 16 rows) form
//    the A operand of mma.m16n8k16 bf16 tensor-core tiles: S = Q K^T with K
//    read by ldmatrix from the swizzled tile, online softmax in fp32 (exp2 of
//    log2-scaled logits), then O += P V with V read by ldmatrix.trans; P is
//    split into bf16 high and low parts so the product keeps ~16 bits.
//  * Every wait on a copy is bounded; a wait that runs out latches
//    KVSEL_ERR_TIMEOUT and the warp stops issuing work.
#include <cudaTypedefs.h>

#include <mutex>

#include "kvsel_common.cuh"
#include "kvsel_internal.h"

namespace kvsel {
namespace {

constexpr int kW = 8;                  // consumer warps per CTA (16 token rows each per tile)
constexpr int kThreads = kW * 32;
constexpr int kMaxCtas = 512;          // partial-slot capacity of the workspace
constexpr int kMinTilesPerCta = 8;
constexpr int kMaxStages = 8;

struct DecodeArgs {
  const kvsel_bf16* q;
  const int32_t* seq_lens;
  const int32_t* sel_idx;
  const int32_t* n_sel;
  const uint8_t* dense_flag;
  const int32_t* block_table;
  int64_t n_pages;
  int kind;
  int slots;
  float scale_log2;
  float* out;
  kvsel_bf16* out_bf16;
  float* lse;
  float* partials;
  uint32_t* tickets;
  int* err;
  int batch, Hq, Hkv, G, B, max_blocks, k_max;
  int stages;
  int kv_swap;   // 1: V precedes K in the tensor map (V tile lands first)
};

struct Tile {
  int b, j, h, cnt;
  int rk;
  bool ok;
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

template <int BT>
__device__ __forceinline__ int sub_per_block(int B) { return B / BT; }

template <int BT>
__device__ Tile tile_info(const DecodeArgs& a, const int* base_s, const int* tlen_s, int64_t g,
                          bool report) {
  Tile t;
  const int SUB = sub_per_block<BT>(a.B);
  const int b = find_seq(base_s, a.batch, g);
  const int64_t r = g - base_s[b];
  const int nb = (base_s[b + 1] - base_s[b]) / (a.Hkv * SUB);
  const int seg = nb * SUB;
  t.b = b;
  t.j = int(r / seg);
  const int rr = int(r % seg);
  const int o = rr / SUB;
  t.h = rr % SUB;
  const int T = tlen_s[b];
  const int N = (T + a.B - 1) / a.B;
  const bool dense = a.dense_flag && a.dense_flag[b];
  const int n = dense ? o : a.sel_idx[int64_t(b) * a.k_max + o];
  bool ok = (n >= 0 && n < N);
  t.cnt = ok ? min(BT, T - n * a.B - t.h * BT) : 0;
  if (a.kind == KVSEL_KV_PAGED) {
    int64_t page = ok ? a.block_table[int64_t(b) * a.max_blocks + n] : 0;
    if (page < 0 || page >= a.n_pages) { ok = false; page = 0; }
    t.rk = int((page * a.Hkv + t.j) * a.B + t.h * BT);
  } else {
    int64_t slot = o;
    if (slot >= a.slots) { ok = false; slot = 0; }
    t.rk = int((((int64_t(b) * a.slots + slot) * 2) * a.Hkv + t.j) * a.B + t.h * BT);
  }
  if (!ok && report) latch_error(a.err, KVSEL_ERR_BOUNDS);
  t.ok = ok;
  return t;
}

// Swizzled shared address of (row, channel c, c % 8 == 0) in a tile made of
// 64-channel TMA boxes with the 128-byte swizzle (16-byte chunk ^= row % 8).
template <int BT>
__device__ __forceinline__ uint32_t swz(uint32_t tile, int row, int c) {
  const int box = c >> 6;
  const int chunk = (c & 63) >> 3;
  return tile + box * (BT * 128) + row * 128 + ((chunk ^ (row & 7)) << 4);
}

template <int D, int BT>
__global__ void __launch_bounds__(kThreads, 1) sparse_decode_kernel(
    const __grid_constant__ CUtensorMap tmKV, DecodeArgs a) {
  constexpr int kTileBytes = BT * D * 2;     // one of K or V
  constexpr int kStageBytes = 2 * kTileBytes;
  constexpr int kKS = D / 16;                // k-steps of Q K^T
  constexpr int kNT = D / 8;                 // n-tiles of P V
  constexpr int kWPR = BT / 16;              // warps sharing one tile ring (16 tokens each)
  constexpr int kRings = kW / kWPR;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // carve: [stages][rings] tiles (1024-aligned) | barriers | merge area | base | tlen
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.stages;
  const int G = a.G;
  unsigned char* tiles = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(tiles + size_t(S) * kRings * kStageBytes);
  float* merge = reinterpret_cast<float*>(bars + S * kRings);      // [W][G][D+2]
  int* base_s = reinterpret_cast<int*>(merge + kW * G * (D + 2));  // [batch+1]
  int* tlen_s = base_s + a.batch + 1;                              // [batch]
  __shared__ int flag_s;
  __shared__ int scan_s[kW];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ring = warp / kWPR, half = warp % kWPR;
  const int SUB = a.B / BT;

  // ---- per-sequence tile counts and prefix ----
  int carry = 0;
  for (int b0 = 0; b0 < a.batch; b0 += kThreads) {
    const int b = b0 + tid;
    int tiles_b = 0;
    if (b < a.batch) {
      int T = a.seq_lens[b];
      if (T < 0 || T > a.max_blocks * a.B) {
        latch_error(a.err, KVSEL_ERR_BOUNDS);
        T = T < 0 ? 0 : a.max_blocks * a.B;
      }
      tlen_s[b] = T;
      const int N = (T + a.B - 1) / a.B;
      int nb;
      if (a.dense_flag && a.dense_flag[b]) {
        nb = N;
      } else {
        nb = a.n_sel[b];
        if (nb < 0 || nb > a.k_max) latch_error(a.err, KVSEL_ERR_BOUNDS);
        nb = max(0, min(nb, min(N, a.k_max)));
      }
      tiles_b = nb * SUB * a.Hkv;
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
    }
    if (b < a.batch) base_s[b] = carry + before + x - tiles_b;
    carry += tot;
    __syncthreads();
  }
  if (tid == 0) base_s[a.batch] = carry;
  __syncthreads();
  const int64_t total = carry;

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
  const int A = int(min(int64_t(gridDim.x), max(int64_t(1), (total + kMinTilesPerCta - 1) / kMinTilesPerCta)));
  if (int(blockIdx.x) >= A) return;
  const int64_t g0 = total * blockIdx.x / A;
  const int64_t g1 = total * (blockIdx.x + 1) / A;
  if (g0 >= g1) return;

  if (tid == 0) {
    for (int i = 0; i < S * kRings; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
    prefetch_tensormap(&tmKV);
  }
  __syncthreads();

  // ---- this ring's tile stream: tiles g0 + ring + m * kRings ----
  const int64_t L = g1 - g0;
  const int count_r = L > ring ? int((L - ring + kRings - 1) / kRings) : 0;
  const uint32_t tiles_base = smem_u32(tiles);
  auto slot_off = [&](int m) -> int { return ((m % S) * kRings + ring) * kStageBytes; };
  auto slot_bar = [&](int m) -> uint64_t* { return &bars[(m % S) * kRings + ring]; };
  const bool leader = (half == 0);
  auto ring_sync = [&]() {
    if constexpr (kWPR > 1) {
      asm volatile("bar.sync %0, %1;" ::"r"(1 + ring), "r"(kWPR * 32) : "memory");
    } else {
      __syncwarp();
    }
  };
  int issued = 0;
  bool dead = false;
  // Tile descriptors, 32 at a time: lane i holds the TMA rows and the valid
  // token count of the ring's tile (cbase + i) in `cur` and of tile
  // (cbase + 32 + i) in `nxt`. Their block-table and selection loads are
  // issued a whole batch ahead, so no global load sits between a tile's
  // consumption and the next copy.
  int cbase = 0;
  int cur_rk = 0, cur_cnt = 0, nxt_rk = 0, nxt_cnt = 0;
  auto load_batch = [&](int base, int& rk, int& cnt) {
    const int m = base + lane;
    rk = cnt = 0;
    if (m < count_r) {
      const Tile t = tile_info<BT>(a, base_s, tlen_s, g0 + ring + int64_t(m) * kRings, leader);
      rk = t.rk;
      cnt = t.ok ? max(t.cnt, 0) : 0;
    }
  };
  // all lanes: descriptor of ring tile m, with cbase <= m < cbase + 64
  auto tile_desc = [&](int m, int& rk, int& cnt) {
    const int i = m - cbase;
    const int src = i & 31;
    const int rk0 = __shfl_sync(0xffffffffu, cur_rk, src), rk1 = __shfl_sync(0xffffffffu, nxt_rk, src);
    const int c0 = __shfl_sync(0xffffffffu, cur_cnt, src), c1 = __shfl_sync(0xffffffffu, nxt_cnt, src);
    rk = i < 32 ? rk0 : rk1;
    cnt = i < 32 ? c0 : c1;
  };
  // one 4-D box brings the K and V halves of a tile: [kv][half][row][64 channels]
  auto issue = [&](int m, int rk) {   // ring leader, lane 0 only
    uint64_t* bar = slot_bar(m);
    mbar_arrive_expect_tx(bar, kStageBytes);
    tma_load_4d(tiles + slot_off(m), &tmKV, 0, rk, 0, 0, bar);
  };
  load_batch(0, cur_rk, cur_cnt);
  load_batch(32, nxt_rk, nxt_cnt);
  for (int m = 0; m < min(S, count_r); ++m) {
    int rk, cnt;
    tile_desc(m, rk, cnt);
    if (leader && lane == 0) issue(m, rk);
  }
  issued = min(S, count_r);
  int m_cur = 0;

  const int gq = lane >> 2, tq = lane & 3;   // mma group / thread-in-group
  const int r0 = half * 16;                  // this warp's 16 token rows of each tile
  int64_t g = g0;
  while (g < g1) {
    // ---- segment (b, j) containing g ----
    const int b = find_seq(base_s, a.batch, g);
    const int seg_tiles = (base_s[b + 1] - base_s[b]) / a.Hkv;
    const int j = int((g - base_s[b]) / seg_tiles);
    const int64_t s_start = base_s[b] + int64_t(j) * seg_tiles;
    const int64_t s_end = s_start + seg_tiles;
    const int64_t sg1 = min(g1, s_end);
    const bool owned = (s_start >= g0 && s_end <= g1);

    // Q fragments (rows >= G are zero)
    uint32_t qa[kKS][4];
    {
      const kvsel_bf16* qb = a.q + (int64_t(b) * a.Hq + int64_t(j) * G) * D;
#pragma unroll
      for (int ks = 0; ks < kKS; ++ks) {
        const int c = ks * 16 + 2 * tq;
        qa[ks][0] = gq < G ? *reinterpret_cast<const uint32_t*>(qb + gq * D + c) : 0u;
        qa[ks][1] = gq + 8 < G ? *reinterpret_cast<const uint32_t*>(qb + (gq + 8) * D + c) : 0u;
        qa[ks][2] = gq < G ? *reinterpret_cast<const uint32_t*>(qb + gq * D + c + 8) : 0u;
        qa[ks][3] = gq + 8 < G ? *reinterpret_cast<const uint32_t*>(qb + (gq + 8) * D + c + 8) : 0u;
      }
    }
    float o[kNT][4];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY};
    float lrow[2] = {0.f, 0.f};

    while (m_cur < count_r && g0 + ring + int64_t(m_cur) * kRings < sg1) {
      if (m_cur == cbase + 32) {           // advance the descriptor window
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
      const int cnt = t_cnt - r0;            // valid tokens in this warp's 16 rows
      if (!dead && cnt > 0) {
        const int k_off = a.kv_swap ? kTileBytes : 0, v_off = a.kv_swap ? 0 : kTileBytes;
        const uint32_t kt_base = tiles_base + slot_off(m_cur) + k_off;
        const uint32_t vt_base = tiles_base + slot_off(m_cur) + v_off;
        if (cnt < 16) {
          // rows past the sequence end: zero V so that 0 * garbage cannot poison P V
          unsigned char* vt = tiles + slot_off(m_cur) + v_off;
          for (int idx = lane; idx < (16 - cnt) * (D / 8); idx += 32) {
            const int row = r0 + cnt + idx / (D / 8);
            const int c = (idx % (D / 8)) * 8;
            *reinterpret_cast<uint4*>(vt + swz<BT>(0, row, c)) = make_uint4(0, 0, 0, 0);
          }
          __syncwarp();
        }
        // S = Q K^T over 16 tokens: two n-tiles, even / odd k-steps in separate
        // accumulators so that four independent mma chains are in flight
        float sa[2][4], sb[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sa[nt][e] = sb[nt][e] = 0.f;
        {
          const int row = r0 + (lane & 7) + ((lane >> 4) << 3);
          const int cofs = ((lane >> 3) & 1) * 8;
#pragma unroll
          for (int ks = 0; ks < kKS; ++ks) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(swz<BT>(kt_base, row, ks * 16 + cofs), b0, b1, b2, b3);
            if (ks & 1) {
              mma_bf16_16816(sb[0], qa[ks], b0, b1);
              mma_bf16_16816(sb[1], qa[ks], b2, b3);
            } else {
              mma_bf16_16816(sa[0], qa[ks], b0, b1);
              mma_bf16_16816(sa[1], qa[ks], b2, b3);
            }
          }
        }
        float s[2][4];
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int tok = nt * 8 + 2 * tq + (e & 1);
            const float x = tok < cnt ? (sa[nt][e] + sb[nt][e]) * a.scale_log2 : -INFINITY;
            s[nt][e] = x;
            mx[e >> 1] = fmaxf(mx[e >> 1], x);
          }
        float mu[2];
        bool grow = false;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
          mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
          grow |= mx[r] > mrow[r];
        }
        if (__any_sync(0xffffffffu, grow)) {
          // a running max moved: rescale the accumulators of every row
          float alpha[2];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const float mn = fmaxf(mrow[r], mx[r]);
            const float m_use = (mn == -INFINITY) ? 0.f : mn;
            alpha[r] = ex2(mrow[r] - m_use);
            mrow[r] = mn;
            lrow[r] *= alpha[r];
          }
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            o[nt][0] *= alpha[0]; o[nt][1] *= alpha[0];
            o[nt][2] *= alpha[1]; o[nt][3] *= alpha[1];
          }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) mu[r] = (mrow[r] == -INFINITY) ? 0.f : mrow[r];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float p = ex2(s[nt][e] - mu[e >> 1]);
            s[nt][e] = p;
            lrow[e >> 1] += p;
          }
        uint32_t ph[4], pl[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float x0 = s[i >> 1][(i & 1) * 2 + 0];
          const float x1 = s[i >> 1][(i & 1) * 2 + 1];
          ph[i] = pack_bf16x2(x0, x1);
          pl[i] = pack_bf16x2(x0 - bf16lo(ph[i]), x1 - bf16hi(ph[i]));
        }
        {
          const int row = r0 + (lane & 7) + (((lane >> 3) & 1) << 3);
          const int cofs = (lane >> 4) * 8;
#pragma unroll
          for (int dc = 0; dc < D / 16; ++dc) {
            uint32_t v0, v1, v2, v3;
            ldsm_x4_t(swz<BT>(vt_base, row, dc * 16 + cofs), v0, v1, v2, v3);
            mma_bf16_16816(o[2 * dc], ph, v0, v1);
            mma_bf16_16816(o[2 * dc + 1], ph, v2, v3);
            mma_bf16_16816(o[2 * dc], pl, v0, v1);
            mma_bf16_16816(o[2 * dc + 1], pl, v2, v3);
          }
        }
      }
      // release the slot (both warps of the ring are done) and refill it S tiles ahead
      ring_sync();
      if (!dead && m_cur + S < count_r) {
        int rk, cnt2;
        tile_desc(m_cur + S, rk, cnt2);
        if (leader && lane == 0) {
          fence_proxy_async();
          issue(m_cur + S, rk);
        }
        issued = m_cur + S + 1;
      }
      ++m_cur;
    }

    // ---- merge the warps' states for this segment ----
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 1);
      lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 2);
    }
    {
      float* mw = merge + warp * G * (D + 2);
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int row = gq + 8 * r;
        if (row < G) {
          float* dst = mw + row * (D + 2);
          if (tq == 0) {
            dst[0] = mrow[r];
            dst[1] = lrow[r];
          }
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            dst[2 + nt * 8 + 2 * tq] = o[nt][2 * r];
            dst[2 + nt * 8 + 2 * tq + 1] = o[nt][2 * r + 1];
          }
        }
      }
    }
    __syncthreads();
    const int slot = (g0 >= s_start) ? 0 : 1;
    float* part = a.partials + (int64_t(blockIdx.x) * 2 + slot) * G * (D + 2);
    for (int e = tid; e < G * D; e += kThreads) {
      const int r = e / D, c = e % D;
      float ms = -INFINITY;
#pragma unroll
      for (int w = 0; w < kW; ++w) ms = fmaxf(ms, merge[(w * G + r) * (D + 2)]);
      float l = 0.f, acc = 0.f;
      if (ms != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kW; ++w) {
          const float* src = merge + (w * G + r) * (D + 2);
          const float f = ex2(src[0] - ms);
          l += src[1] * f;
          acc += src[2 + c] * f;
        }
      }
      const int64_t orow = int64_t(b) * a.Hq + int64_t(j) * G + r;
      if (owned) {
        const float v = l > 0.f ? acc / l : 0.f;
        a.out[orow * D + c] = v;
        if (a.out_bf16) a.out_bf16[orow * D + c] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
        if (c == 0) a.lse[orow] = l > 0.f ? (ms + lg2(l)) * 0.6931471805599453f : -INFINITY;
      } else {
        float* pr = part + r * (D + 2);
        if (c == 0) {
          pr[0] = ms;
          pr[1] = l;
        }
        pr[2 + c] = acc;
      }
    }
    if (!owned) {
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const int64_t first_c = ((s_start + 1) * A - 1) / total;
        const int64_t last_c = ((s_end) * A - 1) / total;
        const uint32_t expect = uint32_t(last_c - first_c + 1);
        const uint32_t before = atomicAdd(&a.tickets[b * a.Hkv + j], 1u);
        if (before + 1 == expect) {
          a.tickets[b * a.Hkv + j] = 0;   // leave the workspace zero-filled
          __threadfence();
        }
        flag_s = (before + 1 == expect) ? int(first_c) : -1;
        scan_s[0] = int(last_c);
      }
      __syncthreads();
      if (flag_s >= 0) {
        const int c_first = flag_s, c_last = scan_s[0];
        for (int e = tid; e < G * D; e += kThreads) {
          const int r = e / D, c = e % D;
          float ms = -INFINITY;
          for (int cc = c_first; cc <= c_last; ++cc) {
            const int sl = (total * cc / A >= s_start) ? 0 : 1;
            const float* pr = a.partials + ((int64_t(cc) * 2 + sl) * G + r) * (D + 2);
            ms = fmaxf(ms, __ldcg(pr));
          }
          float l = 0.f, acc = 0.f;
          if (ms != -INFINITY) {
            for (int cc = c_first; cc <= c_last; ++cc) {
              const int sl = (total * cc / A >= s_start) ? 0 : 1;
              const float* pr = a.partials + ((int64_t(cc) * 2 + sl) * G + r) * (D + 2);
              const float f = ex2(__ldcg(pr) - ms);
              l += __ldcg(pr + 1) * f;
              acc += __ldcg(pr + 2 + c) * f;
            }
          }
          const int64_t orow = int64_t(b) * a.Hq + int64_t(j) * G + r;
          const float v = l > 0.f ? acc / l : 0.f;
          a.out[orow * D + c] = v;
          if (a.out_bf16) a.out_bf16[orow * D + c] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
          if (c == 0) a.lse[orow] = l > 0.f ? (ms + lg2(l)) * 0.6931471805599453f : -INFINITY;
        }
      }
    }
    __syncthreads();
    g = sg1;
  }

  // drain copies still in flight (only after a timeout)
  if (dead && leader && lane == 0)
    for (int m = m_cur; m < issued; ++m) (void)mbar_wait_bounded(slot_bar(m), uint32_t((m / S) & 1));
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tensor map over K and V together: dims (innermost first) are 64 channels,
// cache rows (stride D*2 bytes), the D/64 channel halves (stride 128 bytes)
// and K vs V (stride = distance between the two buffers). A box of
// {64, BT, D/64, 2} with the 128-byte swizzle lands as [kv][half][row][64] in
// shared memory, every 128-byte row swizzled by its row index.
bool encode_map(CUtensorMap* m, const void* base, int64_t rows, int64_t kv_stride, int D, int BT) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[4] = {64u, cuuint64_t(rows), cuuint64_t(D / 64), 2u};
  cuuint64_t strides[3] = {cuuint64_t(D) * 2, 128u, cuuint64_t(kv_stride)};
  cuuint32_t box[4] = {64u, cuuint32_t(BT), cuuint32_t(D / 64), 2u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A tensor map depends only on (address, rows, K/V distance, D, BT): cache the
// encodings so that a decode loop over the same buffers does no host-side
// encoding.
struct MapEntry {
  const void* base;
  int64_t rows, kv_stride;
  int D, BT;
  CUtensorMap map;
};
std::mutex g_map_mu;
MapEntry g_maps[64];
int g_map_next = 0, g_map_n = 0;

bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t kv_stride, int D, int BT) {
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    for (int i = 0; i < g_map_n; ++i) {
      const MapEntry& e = g_maps[i];
      if (e.base == base && e.rows == rows && e.kv_stride == kv_stride && e.D == D && e.BT == BT) {
        *m = e.map;
        return true;
      }
    }
  }
  if (!encode_map(m, base, rows, kv_stride, D, BT)) return false;
  std::lock_guard<std::mutex> lk(g_map_mu);
  MapEntry& e = g_maps[g_map_next];
  e.base = base; e.rows = rows; e.kv_stride = kv_stride; e.D = D; e.BT = BT; e.map = *m;
  g_map_next = (g_map_next + 1) % 64;
  if (g_map_n < 64) ++g_map_n;
  return true;
}

template <int D, int BT>
cudaError_t launch_t(const kvsel_problem& p, const DecodeArgs& a0, const CUtensorMap& mkv,
                     cudaStream_t s) {
  DecodeArgs a = a0;
  constexpr int kRings = kW / (BT / 16);
  constexpr int kGroupBytes = kRings * 2 * BT * D * 2;   // one stage of every ring
  // 1024: manual alignment of the tile area; 256: static shared variables
  const size_t rest = 1024 + 256 + size_t(kW) * a.G * (D + 2) * 4 + (size_t(p.batch) * 2 + 1) * 4;
  const int max_optin = max_smem_optin();
  int stages = int((size_t(max_optin) - rest - 8 * kRings * kMaxStages) / size_t(kGroupBytes));
  stages = std::min(kMaxStages, stages);
  if (stages < 1) return cudaErrorInvalidConfiguration;
  a.stages = stages;
  const size_t smem = rest + size_t(stages) * kGroupBytes + 8 * kRings * stages;
  auto kfn = sparse_decode_kernel<D, BT>;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kfn), int(smem));
  if (e != cudaSuccess) return e;
  const int grid = std::min(kMaxCtas, sm_count());
  kfn<<<grid, kThreads, smem, s>>>(mkv, a);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

size_t sparse_decode_ws_bytes(const kvsel_problem& p) {
  const int G = p.n_qheads / std::max(1, p.n_kvheads);
  const size_t tickets = (size_t(p.batch) * p.n_kvheads * 4 + 255) / 256 * 256;
  const size_t parts = size_t(kMaxCtas) * 2 * G * (p.head_dim + 2) * 4;
  return tickets + parts;
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
  a.kind = (kv.kind == KVSEL_KV_PAGED) ? KVSEL_KV_PAGED : KVSEL_KV_STAGED;
  a.slots = kv.staging_slots;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.out = out; a.out_bf16 = out_bf16; a.lse = lse;
  char* w = static_cast<char*>(ws);
  a.tickets = reinterpret_cast<uint32_t*>(w);
  a.partials = reinterpret_cast<float*>(w + (size_t(p.batch) * p.n_kvheads * 4 + 255) / 256 * 256);
  a.err = err;
  a.batch = p.batch; a.Hq = p.n_qheads; a.Hkv = p.n_kvheads; a.G = p.n_qheads / p.n_kvheads;
  a.B = p.block_size; a.max_blocks = p.max_blocks; a.k_max = p.k_max;
  const int D = p.head_dim;
  const int BT = std::min(p.block_size, 32);
  CUtensorMap mkv;
  if (a.kind == KVSEL_KV_PAGED) {
    const int64_t rows = kv.n_pages * p.n_kvheads * p.block_size;
    const char* kb = reinterpret_cast<const char*>(kv.k_pages);
    const char* vb = reinterpret_cast<const char*>(kv.v_pages);
    const int64_t dist = vb > kb ? int64_t(vb - kb) : int64_t(kb - vb);
    a.kv_swap = vb < kb ? 1 : 0;
    if (dist == 0 || (dist & 15) || dist >= (int64_t(1) << 40)) return cudaErrorInvalidValue;
    if (!make_map(&mkv, a.kv_swap ? kv.v_pages : kv.k_pages, rows, dist, D, BT))
      return cudaErrorInvalidValue;
  } else {
    const int64_t rows = int64_t(p.batch) * kv.staging_slots * 2 * p.n_kvheads * p.block_size;
    const int64_t dist = int64_t(p.n_kvheads) * p.block_size * D * 2;
    a.kv_swap = 0;
    if (!make_map(&mkv, kv.staging, rows, dist, D, BT)) return cudaErrorInvalidValue;
  }
  if (D == 128 && BT == 32) return launch_t<128, 32>(p, a, mkv, s);
  if (D == 128 && BT == 16) return launch_t<128, 16>(p, a, mkv, s);
  if (D == 64 && BT == 32) return launch_t<64, 32>(p, a, mkv, s);
  if (D == 64 && BT == 16) return launch_t<64, 16>(p, a, mkv, s);
  return cudaErrorInvalidValue;
}

}  // namespace kvsel
