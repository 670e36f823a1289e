// f64emu.h -- correctly rounded binary64 operations in 64-bit integer
// arithmetic, for the few fp64 step scalars every CTA forms.
//
// The Adam bias corrections are defined on fp64 state: beta^(t+1) is the
// rounded product of the stored power and beta, and the correction is
// 1 - beta^(t+1) rounded to fp64 and then to fp32. On GB300 the fp64 pipe
// is narrow, and when every CTA of a short step forms these scalars at once
// the fp64 instructions queue behind one another on the critical path. The
// same results come exactly from integer arithmetic on the bit patterns:
// IEEE 754 round-to-nearest-even of the exact product, difference and
// narrowing, written out from the definition of rounding (keep the leading
// p bits, look at the next bit and at whether anything below it is
// nonzero). Each function handles the normal positive range the step needs
// and returns false elsewhere (zero, subnormal, infinite or NaN operands or
// results); the caller then uses the hardware fp64 operations, so the
// results never depend on which way was taken.
//
// The functions compile for the device and the host, so a host test can
// compare them with the host's IEEE arithmetic bit for bit.
#ifndef ZERO_F64EMU_H
#define ZERO_F64EMU_H

#include <stdint.h>

#if defined(__CUDACC__)
#define F64EMU_FN __host__ __device__ __forceinline__
#else
#define F64EMU_FN static inline
#endif

namespace f64emu {

constexpr uint64_t kFrac = (uint64_t(1) << 52) - 1;
constexpr uint64_t kHidden = uint64_t(1) << 52;

F64EMU_FN uint64_t mul_hi(uint64_t a, uint64_t b) {
#if defined(__CUDA_ARCH__)
  return __umul64hi(a, b);
#else
  return static_cast<uint64_t>((static_cast<unsigned __int128>(a) * b) >> 64);
#endif
}

F64EMU_FN int clz64(uint64_t x) {  // x != 0
#if defined(__CUDA_ARCH__)
  return __clzll(static_cast<long long>(x));
#else
  return __builtin_clzll(x);
#endif
}

// biased exponent of a positive normal double, or 0 if x is not one
F64EMU_FN int normal_exp(uint64_t x) {
  const int e = static_cast<int>((x >> 52) & 0x7FF);
  return (x >> 63) == 0 && e != 0 && e != 0x7FF ? e : 0;
}

// RN(x * y) for positive normal x, y with a normal result.
F64EMU_FN bool mul(uint64_t x, uint64_t y, uint64_t* out) {
  const int ex = normal_exp(x), ey = normal_exp(y);
  if (ex == 0 || ey == 0) return false;
  // significands as 64-bit integers with the leading bit on top:
  // a * b lies in [2^126, 2^128)
  const uint64_t a = ((x & kFrac) | kHidden) << 11;
  const uint64_t b = ((y & kFrac) | kHidden) << 11;
  const uint64_t hi = mul_hi(a, b), lo = a * b;
  // x * y = (a b) 2^(ex + ey - 2172); keep 53 bits below the leading one
  const int top = static_cast<int>(hi >> 63);  // 1: leading bit at 2^127
  const int rb = 9 + top;                      // the round bit's place in hi
  uint64_t m = hi >> (rb + 1);
  const uint64_t round = (hi >> rb) & 1;
  const bool sticky = (hi & ((uint64_t(1) << rb) - 1)) != 0 || lo != 0;
  int e = ex + ey - 1023 + top;
  if (e < 1) return false;  // below the normal range: IEEE rounds to fewer bits there
  if (round && (sticky || (m & 1))) {
    m += 1;
    if (m == (uint64_t(1) << 53)) {
      m >>= 1;
      e += 1;
    }
  }
  if (e > 2046) return false;
  *out = (static_cast<uint64_t>(e) << 52) | (m & kFrac);
  return true;
}

// RN(1 - p) for a normal p in (0, 1).
F64EMU_FN bool one_minus(uint64_t p, uint64_t* out) {
  const int ep = normal_exp(p);
  if (ep == 0 || ep > 1022) return false;
  const uint64_t mp = (p & kFrac) | kHidden;
  if (ep == 1022) {
    // p in [1/2, 1): 1 - p = (2^53 - mp) 2^-53 exactly
    const uint64_t d = (uint64_t(1) << 53) - mp;  // in (0, 2^52]
    const int lead = 63 - clz64(d);
    *out = (static_cast<uint64_t>(lead + 970) << 52) | ((d << (52 - lead)) & kFrac);
    return true;
  }
  // p < 1/2: in units of 2^-54, 1 = 2^54 and p = mp 2^-r with r >= 0;
  // 1 - p lies in (1/2, 1), so its 53 bits are the units above 2^-54
  const int r = 1021 - ep;
  uint64_t q, frac;
  if (r >= 64) {
    q = 0;
    frac = mp;
  } else {
    q = r == 0 ? mp : mp >> r;
    frac = r == 0 ? 0 : mp & ((uint64_t(1) << r) - 1);
  }
  // integer part of 1 - p in units, and whether a fraction of a unit remains
  const uint64_t units = (uint64_t(1) << 54) - q - (frac != 0 ? 1 : 0);
  uint64_t m = units >> 1;
  const uint64_t round = units & 1;
  const bool sticky = frac != 0;
  if (round && (sticky || (m & 1))) m += 1;
  if (m == (uint64_t(1) << 53)) {
    *out = uint64_t(1023) << 52;  // 1.0
    return true;
  }
  *out = (uint64_t(1022) << 52) | (m & kFrac);
  return true;
}

// RN_fp32(x) for a positive normal double x with a normal fp32 result;
// returns the fp32 bit pattern.
F64EMU_FN bool to_f32(uint64_t x, uint32_t* out) {
  const int ex = normal_exp(x);
  if (ex == 0) return false;
  const uint64_t md = (x & kFrac) | kHidden;  // 53 bits
  uint32_t m = static_cast<uint32_t>(md >> 29);  // 24 bits
  const uint64_t round = (md >> 28) & 1;
  const bool sticky = (md & ((uint64_t(1) << 28) - 1)) != 0;
  int e = ex - 1023 + 127;
  if (e < 1) return false;  // an fp32 subnormal: fewer bits
  if (round && (sticky || (m & 1))) {
    m += 1;
    if (m == (1u << 24)) {
      m >>= 1;
      e += 1;
    }
  }
  if (e > 254) return false;
  *out = (static_cast<uint32_t>(e) << 23) | (m & 0x7FFFFFu);
  return true;
}

}  // namespace f64emu

#endif
