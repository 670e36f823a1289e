// Host test of csrc/f64emu.h: every emulated product, difference and
// narrowing that reports success must equal the host's IEEE double and
// float arithmetic bit for bit, and the emulation must cover the whole
// range the step meets (Adam's beta powers from beta^0 = 1 down to the
// normal limit). Built with -ffp-contract=off, so a * b and 1 - p are
// single IEEE operations.
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "f64emu.h"

static uint64_t bits(double x) {
  uint64_t u;
  memcpy(&u, &x, 8);
  return u;
}
static double dbl(uint64_t u) {
  double x;
  memcpy(&x, &u, 8);
  return x;
}
static uint32_t fbits(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  return u;
}

static uint64_t state = 0x9E3779B97F4A7C15ull;
static uint64_t next() {  // SplitMix64
  uint64_t z = (state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static long n_checked = 0, n_fail = 0, n_fallback = 0;

static bool is_normal_pos(double x) {
  const uint64_t u = bits(x);
  const int e = (int)((u >> 52) & 0x7FF);
  return (u >> 63) == 0 && e != 0 && e != 0x7FF;
}
static bool is_normal_f(float x) {
  const uint32_t u = fbits(x);
  const int e = (int)((u >> 23) & 0xFF);
  return e != 0 && e != 0xFF;
}

static void check_mul(double x, double y, bool must_cover) {
  uint64_t r;
  const double want = x * y;
  const bool ok = f64emu::mul(bits(x), bits(y), &r);
  ++n_checked;
  if (ok && r != bits(want)) {
    if (n_fail++ < 10) printf("mul %a * %a: %a want %a\n", x, y, dbl(r), want);
  }
  if (!ok) {
    ++n_fallback;
    if (must_cover && n_fail++ < 10) printf("mul %a * %a not covered\n", x, y);
  }
}

static void check_one_minus(double p, bool must_cover) {
  uint64_t r;
  const double want = 1.0 - p;
  const bool ok = f64emu::one_minus(bits(p), &r);
  ++n_checked;
  if (ok && r != bits(want)) {
    if (n_fail++ < 10) printf("1 - %a: %a want %a\n", p, dbl(r), want);
  }
  if (!ok) {
    ++n_fallback;
    if (must_cover && n_fail++ < 10) printf("1 - %a not covered\n", p);
  }
}

static void check_f32(double d, bool must_cover) {
  uint32_t r;
  const float want = (float)d;
  const bool ok = f64emu::to_f32(bits(d), &r);
  ++n_checked;
  if (ok && r != fbits(want)) {
    if (n_fail++ < 10) printf("f32(%a): %08x want %a\n", d, r, (double)want);
  }
  if (!ok) {
    ++n_fallback;
    if (must_cover && n_fail++ < 10) printf("f32(%a) not covered\n", d);
  }
}

// the step's chain for one beta: p = RN(pow * beta), bc = RN32(RN(1 - p))
static void beta_sequence(double beta, long max_t) {
  double pw = 1.0;
  for (long t = 0; t < max_t; ++t) {
    const double p = pw * beta;
    const bool normal = is_normal_pos(p);
    check_mul(pw, beta, normal);
    if (!normal) break;
    const double d = 1.0 - p;
    check_one_minus(p, true);
    check_f32(d, is_normal_f((float)d));
    pw = p;
  }
}

static double rand_normal_in(int emin, int emax) {  // biased exponents, inclusive
  const uint64_t e = (uint64_t)(emin + (int)(next() % (uint64_t)(emax - emin + 1)));
  return dbl((e << 52) | (next() & f64emu::kFrac));
}

int main(int argc, char** argv) {
  long scale = argc > 1 ? atol(argv[1]) : 1;
  // Adam's usual betas and others, each power chain to the normal limit
  const double betas[] = {0.9, 0.99, 0.999, 0.9999, 0.95, 0.98, 0.5, 0.1, 0.75, 0.3,
                          1.0 - 1.0 / 1048576.0, 1e-3};
  for (double b : betas) beta_sequence(b, 200000 * scale);
  for (int i = 0; i < 64; ++i) beta_sequence(rand_normal_in(1013, 1022), 20000 * scale);
  // random products over the whole exponent range (results of every kind)
  for (long i = 0; i < 2000000 * scale; ++i) {
    const double x = rand_normal_in(1, 2046), y = rand_normal_in(1, 2046);
    const double w = x * y;
    const int ew = (int)((bits(w) >> 52) & 0x7FF);
    check_mul(x, y, is_normal_pos(w) && ew > 1);
  }
  // products near 1 (the step's range), and exact ties: (1 + k 2^-52) * 1.5
  for (long i = 0; i < 2000000 * scale; ++i) check_mul(rand_normal_in(1015, 1023), rand_normal_in(1015, 1022), true);
  for (long k = 1; k < 4096; ++k) {
    const double x = 1.0 + (double)k * 0x1p-52;
    check_mul(x, 1.5, true);
    check_mul(x, 0.75, true);
    check_mul(1.5, x, true);
  }
  // 1 - p for p over (0, 1): every exponent, including p far below 2^-64
  for (long i = 0; i < 2000000 * scale; ++i) check_one_minus(rand_normal_in(1, 1022), true);
  for (long i = 0; i < 2000000 * scale; ++i) check_one_minus(rand_normal_in(1000, 1022), true);
  for (int e = 1; e <= 1022; ++e) {
    check_one_minus(dbl((uint64_t)e << 52), true);
    check_one_minus(dbl(((uint64_t)e << 52) | f64emu::kFrac), true);
    check_one_minus(dbl(((uint64_t)e << 52) | 1), true);
  }
  // narrowing: random doubles in and around the fp32 range, and exact ties
  for (long i = 0; i < 2000000 * scale; ++i) {
    const double d = rand_normal_in(1023 - 140, 1023 + 130);
    check_f32(d, is_normal_f((float)d) && ((bits(d) >> 52) & 0x7FF) >= 1023 - 126);
  }
  for (long i = 0; i < 100000 * scale; ++i) {
    // 24 kept bits, the round bit set, nothing below: a tie
    const uint64_t m = next() & 0x7FFFFFull;
    const double d = dbl((uint64_t(1000) << 52) | (m << 29) | (uint64_t(1) << 28));
    check_f32(d, true);
  }
  printf("checked %ld, fallbacks %ld, failures %ld\n", n_checked, n_fallback, n_fail);
  if (n_fail) return 1;
  printf("f64emu ok\n");
  return 0;
}
