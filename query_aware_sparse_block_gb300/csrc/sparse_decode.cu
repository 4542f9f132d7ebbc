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

constexpr int kW = 4;                  // warps per CTA, each with its own tile ring
constexpr int kThreads = kW * 32;
constexpr int kMaxCtas = 512;          // partial-slot capacity of the workspace
constexpr int kMinTilesPerCta = 2 * kW;
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
};

struct Tile {
  int b, j, h, cnt;
  int rk, rv;
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
    t.rv = t.rk;
  } else {
    int64_t slot = o;
    if (slot >= a.slots) { ok = false; slot = 0; }
    t.rk = int((((int64_t(b) * a.slots + slot) * 2) * a.Hkv + t.j) * a.B + t.h * BT);
    t.rv = t.rk + a.Hkv * a.B;
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
    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
    DecodeArgs a) {
  constexpr int kTileBytes = BT * D * 2;     // one of K or V
  constexpr int kStageBytes = 2 * kTileBytes;
  constexpr int kBoxes = D / 64;
  constexpr int kKS = D / 16;                // k-steps of Q K^T
  constexpr int kNT = D / 8;                 // n-tiles of P V
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // carve: [stages][W] tiles (1024-aligned) | barriers | merge area | base | tlen
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.stages;
  const int G = a.G;
  unsigned char* tiles = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(tiles + size_t(S) * kW * kStageBytes);
  float* merge = reinterpret_cast<float*>(bars + S * kW);          // [W][G][D+2]
  int* base_s = reinterpret_cast<int*>(merge + kW * G * (D + 2));  // [batch+1]
  int* tlen_s = base_s + a.batch + 1;                              // [batch]
  __shared__ int flag_s;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int SUB = a.B / BT;

  // ---- per-sequence tile counts and prefix ----
  __shared__ int scan_s[kW];
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
    for (int i = 0; i < S * kW; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  __syncthreads();

  // ---- this warp's tile stream ----
  const int64_t L = g1 - g0;
  const int count_w = L > warp ? int((L - warp + kW - 1) / kW) : 0;
  const uint32_t tiles_base = smem_u32(tiles);
  auto slot_addr = [&](int m) -> uint32_t {
    return tiles_base + uint32_t(((m % S) * kW + warp) * kStageBytes);
  };
  auto slot_bar = [&](int m) -> uint64_t* { return &bars[(m % S) * kW + warp]; };
  int issued = 0;
  bool dead = false;
  auto issue = [&](int m) {
    const Tile t = tile_info<BT>(a, base_s, tlen_s, g0 + warp + int64_t(m) * kW, true);
    uint64_t* bar = slot_bar(m);
    mbar_arrive_expect_tx(bar, kStageBytes);
    unsigned char* dst = tiles + ((m % S) * kW + warp) * kStageBytes;
#pragma unroll
    for (int x = 0; x < kBoxes; ++x) {
      tma_load_2d(dst + x * BT * 128, &tmK, x * 64, t.rk, bar);
      tma_load_2d(dst + kTileBytes + x * BT * 128, &tmV, x * 64, t.rv, bar);
    }
  };
  if (lane == 0)
    for (int m = 0; m < min(S, count_w); ++m) issue(m);
  issued = min(S, count_w);
  int m_cur = 0;

  const int gq = lane >> 2, tq = lane & 3;   // mma group / thread-in-group
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

    while (m_cur < count_w && g0 + warp + int64_t(m_cur) * kW < sg1) {
      const int64_t gt = g0 + warp + int64_t(m_cur) * kW;
      const Tile t = tile_info<BT>(a, base_s, tlen_s, gt, false);
      if (!dead && !mbar_wait_bounded(slot_bar(m_cur), uint32_t((m_cur / S) & 1))) {
        dead = true;
        if (lane == 0) latch_error(a.err, KVSEL_ERR_TIMEOUT);
      }
      if (!dead && t.ok && t.cnt > 0) {
        const uint32_t kt_base = slot_addr(m_cur);
        const uint32_t vt_base = kt_base + kTileBytes;
        if (t.cnt < BT) {
          // rows past the sequence end: zero V so that 0 * garbage cannot poison P V
          unsigned char* vt = tiles + ((m_cur % S) * kW + warp) * kStageBytes + kTileBytes;
          for (int idx = lane; idx < (BT - t.cnt) * (D / 8); idx += 32) {
            const int row = t.cnt + idx / (D / 8);
            const int c = (idx % (D / 8)) * 8;
            const uint32_t off = swz<BT>(0, row, c);
            *reinterpret_cast<uint4*>(vt + off) = make_uint4(0, 0, 0, 0);
          }
          __syncwarp();
        }
#pragma unroll
        for (int kt = 0; kt < BT / 16; ++kt) {
          float s[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
          {
            const int row = kt * 16 + (lane & 7) + ((lane >> 4) << 3);
            const int cofs = ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int ks = 0; ks < kKS; ++ks) {
              uint32_t b0, b1, b2, b3;
              ldsm_x4(swz<BT>(kt_base, row, ks * 16 + cofs), b0, b1, b2, b3);
              mma_bf16_16816(s[0], qa[ks], b0, b1);
              mma_bf16_16816(s[1], qa[ks], b2, b3);
            }
          }
          // scale, mask, online softmax (rows gq and gq + 8)
          float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int tok = kt * 16 + nt * 8 + 2 * tq + (e & 1);
              const float x = tok < t.cnt ? s[nt][e] * a.scale_log2 : -INFINITY;
              s[nt][e] = x;
              mx[e >> 1] = fmaxf(mx[e >> 1], x);
            }
          float alpha[2], mu[2];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
            const float mn = fmaxf(mrow[r], mx[r]);
            mu[r] = (mn == -INFINITY) ? 0.f : mn;
            alpha[r] = ex2(mrow[r] - mu[r]);
            mrow[r] = mn;
          }
          float psum[2] = {0.f, 0.f};
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float p = ex2(s[nt][e] - mu[e >> 1]);
              s[nt][e] = p;
              psum[e >> 1] += p;
            }
#pragma unroll
          for (int r = 0; r < 2; ++r) lrow[r] = lrow[r] * alpha[r] + psum[r];
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            o[nt][0] *= alpha[0]; o[nt][1] *= alpha[0];
            o[nt][2] *= alpha[1]; o[nt][3] *= alpha[1];
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
            const int row = kt * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
            const int cofs = (lane >> 4) * 8;
#pragma unroll
            for (int dc = 0; dc < D / 16; ++dc) {
              uint32_t v0, v1, v2, v3;
              ldsm_x4_t(swz<BT>(vt_base, row, dc * 16 + cofs), v0, v1, v2, v3);
              mma_bf16_16816(o[2 * dc], ph, v0, v1);
              mma_bf16_16816(o[2 * dc], pl, v0, v1);
              mma_bf16_16816(o[2 * dc + 1], ph, v2, v3);
              mma_bf16_16816(o[2 * dc + 1], pl, v2, v3);
            }
          }
        }
      }
      // release the slot and refill it S tiles ahead
      __syncwarp();
      if (!dead && m_cur + S < count_w) {
        if (lane == 0) {
          fence_proxy_async();
          issue(m_cur + S);
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
  if (dead && lane == 0)
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

bool make_map(CUtensorMap* m, const void* base, int64_t rows, int D, int BT) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {cuuint64_t(D), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(D) * 2};
  cuuint32_t box[2] = {64u, cuuint32_t(BT)};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, int BT>
cudaError_t launch_t(const kvsel_problem& p, const DecodeArgs& a0, const CUtensorMap& mk,
                     const CUtensorMap& mv, cudaStream_t s) {
  DecodeArgs a = a0;
  constexpr int kStageBytes = 2 * BT * D * 2;
  // 1024: manual alignment of the tile area; 256: static shared variables
  const size_t rest = 1024 + 256 + size_t(kW) * a.G * (D + 2) * 4 + (size_t(p.batch) * 2 + 1) * 4;
  int dev = 0;
  cudaGetDevice(&dev);
  int max_optin = 0;
  cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  int stages = int((size_t(max_optin) - rest - 8 * kW * kMaxStages) / (size_t(kW) * kStageBytes));
  stages = std::min(kMaxStages, stages);
  if (stages < 1) return cudaErrorInvalidConfiguration;
  a.stages = stages;
  const size_t smem = rest + size_t(stages) * kW * kStageBytes + 8 * kW * stages;
  auto kfn = sparse_decode_kernel<D, BT>;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  const int grid = std::min(kMaxCtas, sm_count());
  kfn<<<grid, kThreads, smem, s>>>(mk, mv, a);
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
  CUtensorMap mk, mv;
  if (a.kind == KVSEL_KV_PAGED) {
    const int64_t rows = kv.n_pages * p.n_kvheads * p.block_size;
    if (!make_map(&mk, kv.k_pages, rows, D, BT) || !make_map(&mv, kv.v_pages, rows, D, BT))
      return cudaErrorInvalidValue;
  } else {
    const int64_t rows = int64_t(p.batch) * kv.staging_slots * 2 * p.n_kvheads * p.block_size;
    if (!make_map(&mk, kv.staging, rows, D, BT)) return cudaErrorInvalidValue;
    mv = mk;
  }
  if (D == 128 && BT == 32) return launch_t<128, 32>(p, a, mk, mv, s);
  if (D == 128 && BT == 16) return launch_t<128, 16>(p, a, mk, mv, s);
  if (D == 64 && BT == 32) return launch_t<64, 32>(p, a, mk, mv, s);
  if (D == 64 && BT == 16) return launch_t<64, 16>(p, a, mk, mv, s);
  return cudaErrorInvalidValue;
}

}  // namespace kvsel
