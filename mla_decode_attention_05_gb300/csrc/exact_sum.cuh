// Exact sum of squares of a warp's bf16 values, rounded once to fp32.
//
// A bf16 value is m * 2^(ee - 134): m the 8-bit significand (hidden bit
// included), ee the biased exponent (1 for subnormals).  Its square m^2 *
// 2^(2 ee - 268) is an integer below 2^16 times a power of two, so the
// squares of a row can be added exactly as integers in a fixed-point frame
// aligned to the largest one; the sum then does not depend on the order of
// additions.  Each lane holds kWords 32-bit words (two bf16 values each, the
// first in the low half); the warp's sum is returned to every lane.
#pragma once

#include "common.cuh"

namespace mla {

template <int kWords>
struct LaneBf16 {
  uint32_t w[kWords];
};

// v << s with the PTX rule for large shifts: an amount of 32 or more (a
// negative s reads as a large unsigned amount) gives 0.
__device__ __forceinline__ uint32_t shl_or_zero(uint32_t v, int s) {
  uint32_t r;
  asm("shl.b32 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(s));
  return r;
}

__device__ __forceinline__ void split_bf16(uint32_t h, uint32_t &m, int &ee) {
  const int e = (h >> 7) & 0xFF;
  m = (h & 0x7Fu) | (e ? 0x80u : 0u);
  ee = e ? e : 1;
}

template <int kWords>
__device__ __forceinline__ uint32_t half_of(const LaneBf16<kWords> &x, int i) {
  return (x.w[i >> 1] >> ((i & 1) * 16)) & 0xFFFFu;
}

// acc * 2^e0 (acc < 2^127; sticky: the true value lies strictly above acc,
// by less than one unit of acc's lowest bit) rounded to fp32, ties to even.
__device__ __forceinline__ float round_to_f32(unsigned __int128 acc, int e0, bool sticky) {
  if (sticky) acc |= 1u;
  const uint64_t hi = (uint64_t)(acc >> 64);
  const int lead = hi ? 127 - __clzll((long long)hi) : 63 - __clzll((long long)(uint64_t)acc);
  const int q = max(lead - 23, -149 - e0);  // position of the fp32 quantum in acc
  if (q <= 0) return ldexpf((float)(uint32_t)acc, e0);  // exact: acc < 2^24
  if (q >= lead + 2) return 0.f;                         // below half the smallest subnormal
  unsigned __int128 keep = acc >> q;
  const unsigned __int128 rem = acc & (((unsigned __int128)1 << q) - 1);
  const unsigned __int128 half = (unsigned __int128)1 << (q - 1);
  if (rem > half || (rem == half && (keep & 1))) keep += 1;
  return ldexpf((float)(uint32_t)keep, q + e0);  // keep <= 2^24: exact; overflow -> inf
}

// Wide form, for rows whose values span more than 2^31 (or that hold
// subnormals): squares placed relative to the largest one at bit kTop
// (a warp's at most 1536 squares below 2^16 stay below 2^127); those that
// fall below bit 0 leave their remainder as a sticky bit.
template <int kWords>
__device__ __noinline__ float sum_sq_wide(const LaneBf16<kWords> x, int emax) {
  constexpr int kTop = 100;
  static_assert(32 * 2 * kWords <= 1536, "accumulator range");
  unsigned __int128 acc = 0;
  bool sticky = false;
#pragma unroll
  for (int i = 0; i < 2 * kWords; i++) {
    uint32_t m;
    int ee;
    split_bf16(half_of(x, i), m, ee);
    const uint32_t t = m * m;
    const int sh = kTop - 2 * (emax - ee);
    if (sh >= 0) {
      acc += (unsigned __int128)t << sh;
    } else if (sh > -32) {
      acc += t >> -sh;
      sticky |= (t & ((1u << -sh) - 1u)) != 0u;
    } else {
      sticky |= t != 0u;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t lo = __shfl_xor_sync(0xffffffffu, (unsigned long long)acc, o);
    const uint64_t hi = __shfl_xor_sync(0xffffffffu, (unsigned long long)(acc >> 64), o);
    acc += ((unsigned __int128)hi << 64) | lo;
  }
  return round_to_f32(acc, 2 * emax - 268 - kTop, __any_sync(0xffffffffu, sticky));
}

// Relative to the largest exponent emax a square sits at bit
// s = 2 (ee - emax) + 31.  Squares with s in [0, 31] go to `hi` at bit s,
// those with s in [-32, -1] to `lo` at bit s + 32, so hi * 2^32 + lo is the
// exact sum in units of 2^(2 emax - 331) (each part stays below 2^58 for
// 1536 squares).  When emax >= 32 every zero lands below bit -32 and adds
// nothing, so every value can take the normal significand 0x80 | mantissa.
// A row with a nonzero value below the window (its exponent under emax - 31:
// subnormals included) or with emax < 32 takes the wide form.  A row whose
// nonzero values all lie within 2^15 of the largest (exponents emax - 15 ..
// emax, the common case) puts every square into `hi` (s in [1, 31]) and
// needs only that window.  emax and the smallest nonzero magnitude come from
// the 15-bit magnitude patterns, which order like the values.
// n * 2^e (n >= 1) rounded to fp32, ties to even: the correctly rounded
// conversion of n, then e added to the exponent, which is exact while the
// result is normal; a result that would be subnormal or zero takes the
// general rounding (one rounding at the subnormal quantum).
__device__ __forceinline__ float scaled_u64_to_f32(uint64_t n, int e) {
  const uint32_t f = __float_as_uint(__ull2float_rn(n));
  const int re = (int)(f >> 23) + e;  // biased exponent of the result
  if (re >= 255) return __int_as_float(0x7F800000);
  if (re >= 1) return __uint_as_float(f + ((uint32_t)e << 23));
  return round_to_f32((unsigned __int128)n, e, false);
}

template <int kWords>
__device__ __forceinline__ float sum_sq_rn(const LaneBf16<kWords> &x) {
  // per 16-bit half: the largest magnitude, and the smallest of (magnitude -
  // 1) over nonzero magnitudes (0x7FFF for a zero): with bit 15 set in both
  // halves the subtraction of 1 never borrows across them
  uint32_t amax2 = 0, aminm2 = 0xFFFFFFFFu;
#pragma unroll
  for (int k = 0; k < kWords; k++) {
    amax2 = __vmaxu2(amax2, x.w[k] & 0x7FFF7FFFu);
    aminm2 = __vminu2(aminm2, ((x.w[k] | 0x80008000u) - 0x00010001u) & 0x7FFF7FFFu);
  }
  const uint32_t amax = __reduce_max_sync(0xffffffffu, max(amax2 & 0xFFFFu, amax2 >> 16));
  if (amax == 0) return 0.f;  // all zeros
  const uint32_t amin = __reduce_min_sync(0xffffffffu, min(aminm2 & 0xFFFFu, aminm2 >> 16)) + 1u;
  const int emax = (int)(amax >> 7);
  if (emax < 32 || (int)(amin >> 7) < emax - 31) return sum_sq_wide<kWords>(x, max(emax, 1));
  const int base = 31 - 2 * emax;
  if ((int)(amin >> 7) >= emax - 15) {
    uint64_t hi = 0;
#pragma unroll
    for (int i = 0; i < 2 * kWords; i++) {
      const uint32_t h = half_of(x, i);
      const uint32_t m = (h & 0x7Fu) | 0x80u;
      hi += (uint64_t)(m * m) * shl_or_zero(1u, 2 * (int)((h >> 7) & 0xFFu) + base);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) hi += __shfl_xor_sync(0xffffffffu, (unsigned long long)hi, o);
    return scaled_u64_to_f32(hi, 2 * emax - 299);  // hi > 0: the largest square is in it
  }
  uint64_t hi = 0, lo = 0;
#pragma unroll
  for (int i = 0; i < 2 * kWords; i++) {
    const uint32_t h = half_of(x, i);
    const uint32_t m = (h & 0x7Fu) | 0x80u;
    const uint32_t t = m * m;
    const int s = 2 * (int)((h >> 7) & 0xFFu) + base;
    hi += (uint64_t)t * shl_or_zero(1u, s);
    lo += (uint64_t)t * shl_or_zero(1u, s + 32);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    hi += __shfl_xor_sync(0xffffffffu, (unsigned long long)hi, o);
    lo += __shfl_xor_sync(0xffffffffu, (unsigned long long)lo, o);
  }
  return round_to_f32(((unsigned __int128)hi << 32) + lo, 2 * emax - 331, false);
}

}  // namespace mla
