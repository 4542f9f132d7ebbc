// Arithmetic of one block summary, shared by the summary kernels and the
// append step folded into the score grid: the tiled position of a cached K/V
// row, and the mean of a block's keys rounded once to bf16.
//
// A summary element is the fp64 sum of the block's keys taken in token order
// from +0.0, divided by the token count in fp64 and rounded once to bf16
// (nearest, ties to even). The rounding from fp64 goes through fp32 with
// round-to-odd, which gives the same result as one direct rounding whenever
// the intermediate format carries at least two more bits than the target
// (Boldo and Melquiond, "Emulation of FMA and correctly rounded sums: proved
// algorithms using rounding to odd", IEEE Trans. Computers, 2008); fp32
// carries 24 bits against bf16's 8.
#pragma once

#include "kvsel_common.cuh"

namespace kvsel {

// Element offset, inside one K (or V) tile of a (page, head) in the tiled
// layout, of the 8-channel vector starting at channel c0 (c0 % 8 == 0) of
// token row t. The page of head j holds the K tile at element (page * H + j)
// * 2 * B * d and the V tile right after it.
__device__ __forceinline__ int64_t tiled_off(int t, int c0, int B) {
  const int half = c0 >> 6, chunk = (c0 & 63) >> 3;
  return (int64_t(half) * B + t) * 64 + ((chunk ^ (t & 7)) << 3);
}

__device__ __forceinline__ uint16_t f64_to_bf16_rne(double x) {
  float f = __double2float_rz(x);
  if (static_cast<double>(f) != x) f = __uint_as_float(__float_as_uint(f) | 1u);  // round to odd
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// The fp64 value of a bf16 bit pattern h (low 16 bits), exactly. A normal
// number, an infinity or a NaN is re-encoded with integer operations (exponent
// rebiased from 127 to 1023, the 7 fraction bits moved to the top of the 52),
// so the conversion does not occupy the fp64 pipe, which this part runs at a
// small fraction of its fp32 rate; +-0 is built the same way and only a
// subnormal (exponent field 0, fraction non-zero) takes the fp32 -> fp64
// conversion instruction.
__device__ __forceinline__ double bf16_to_f64(uint32_t h) {
  const uint32_t e = (h >> 7) & 0xFFu;
  const uint64_t sign = uint64_t(h & 0x8000u) << 48;
  if (e == 0u) {
    if ((h & 0x7Fu) == 0u) return __longlong_as_double(static_cast<long long>(sign));
    return static_cast<double>(__uint_as_float(h << 16));
  }
  const uint64_t ex = e == 0xFFu ? 0x7FFull : uint64_t(e + (1023u - 127u));
  const uint64_t man = uint64_t(h & 0x7Fu) << 45;
  return __longlong_as_double(static_cast<long long>(sign | (ex << 52) | man));
}

// The sum of a block column (at most 64 bf16 values) on the integer pipe.
// A bf16 value is m * 2^(E - 134) with an integer m < 2^8 and E its biased
// exponent (E = 1 for subnormals). Let r and E_max be the lowest and highest
// E among the column's non-zero values. If E_max - r <= 39, every partial sum
// of the column is an integer multiple of 2^(r - 134) below 2^53 of those
// units, so each fp64 addition of the sequential sum the summary definition
// prescribes is exact, and that sum equals the exact sum: accumulated here as
// an int64 count of units and converted at the end without rounding. A column
// with a wider spread, an infinity or a NaN is marked `bad`; its caller takes
// the fp64 sum in token order instead.
struct ExactSum {
  long long acc;   // the sum in units of 2^(r - 134)
  int r, emax;     // lowest and highest biased exponent of the non-zero values
  bool bad;
};

__device__ __forceinline__ void exact_init(ExactSum& s) {
  s.acc = 0;
  s.r = 255;
  s.emax = 0;
  s.bad = false;
}

__device__ __forceinline__ void exact_add(ExactSum& s, uint32_t h) {
  if (s.bad) return;
  const uint32_t e = (h >> 7) & 0xFFu, f = h & 0x7Fu;
  if (e == 0xFFu) {
    s.bad = true;
    return;
  }
  if (e == 0u && f == 0u) return;                        // +-0 adds nothing
  const int ee = e ? int(e) : 1;
  const int nr = min(s.r, ee), nmax = max(s.emax, ee);
  if (nmax - nr > 39) {
    s.bad = true;
    return;
  }
  if (nr < s.r) {
    if (s.acc != 0) s.acc <<= (s.r - nr);                // at most 39, and |acc| stays < 2^53
    s.r = nr;
  }
  s.emax = nmax;
  const long long v = static_cast<long long>(e ? (0x80u | f) : f) << (ee - s.r);
  s.acc += (h & 0x8000u) ? -v : v;
}

// The exact sum as fp64 (|acc| < 2^53 converts exactly; the power of two
// 2^(r - 134) is a normal number, so the product is exact). An empty or
// cancelling column gives +0, as the sequential sum from +0.0 does.
__device__ __forceinline__ double exact_result(const ExactSum& s) {
  if (s.acc == 0) return 0.0;
  const double scale = __longlong_as_double(static_cast<long long>(s.r - 134 + 1023) << 52);
  return __ll2double_rn(s.acc) * scale;
}

__device__ __forceinline__ void unpack8(const uint4& v, double (&x)[8]) {
  x[0] = bf16_to_f64(v.x & 0xFFFFu); x[1] = bf16_to_f64(v.x >> 16);
  x[2] = bf16_to_f64(v.y & 0xFFFFu); x[3] = bf16_to_f64(v.y >> 16);
  x[4] = bf16_to_f64(v.z & 0xFFFFu); x[5] = bf16_to_f64(v.z >> 16);
  x[6] = bf16_to_f64(v.w & 0xFFFFu); x[7] = bf16_to_f64(v.w >> 16);
}

// x / c correctly rounded for a positive integer c, from r = RN(1/c): the
// product q = RN(x r), its exact residual e = x - q c (one FMA) and the
// corrected quotient RN(q + e r) (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Develop.
// 34(1), 1990). fp64 division is slow on this part; one reciprocal then
// serves the eight channels of a vector. A zero quotient keeps the sign of x;
// an infinite or NaN quotient is returned as it is (the residual of an
// infinity would be inf - inf = NaN, where IEEE division gives the infinity).
// Checked against IEEE division on 2^32 operands shaped like block sums.
__device__ __forceinline__ double div_by_count(double x, double c, double r) {
  const double q = x * r;
  if (q == 0.0 || !(fabs(q) <= 1.7976931348623157e308)) return q;
  const double e = fma(-q, c, x);
  return fma(e, r, q);
}

__device__ __forceinline__ uint4 mean_to_bf16x8(const double (&acc)[8], int cnt) {
  const double c = static_cast<double>(cnt);
  const double rc = 1.0 / c;
  uint16_t h[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) h[i] = f64_to_bf16_rne(div_by_count(acc[i], c, rc));
  uint4 r;
  r.x = h[0] | (uint32_t(h[1]) << 16);
  r.y = h[2] | (uint32_t(h[3]) << 16);
  r.z = h[4] | (uint32_t(h[5]) << 16);
  r.w = h[6] | (uint32_t(h[7]) << 16);
  return r;
}

}  // namespace kvsel
