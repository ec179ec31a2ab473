// Shared device/host helpers of the exact solver library: the prime set and
// modular reduction by small odd primes.
//
// Prime set (exact-solve card, §Method): the squarefree modulus is a product
// of primes q_j < 256; it must be odd (the residual update divides by P
// modulo 2^64), so the set is the 53 odd primes 3..251.
//
// Reduction (card §Method: Barrett's method instead of the hardware remainder):
// Barrett's method with a 32-bit reciprocal.  For an odd q < 256 let
// mu = floor(2^32 / q).  For any u < 2^32, t = floor(u * mu / 2^32)
// satisfies floor(u/q) - 1 <= t <= floor(u/q) because
// u*mu/2^32 = u/q - u*eps/2^32 with eps = 2^32/q - mu in [0, 1) and
// u < 2^32; hence r = u - t*q lies in [0, 2q) and one conditional
// subtraction finishes the reduction.  Signed inputs are shifted by a
// multiple of q first.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define ES_HD __host__ __device__ __forceinline__
#else
#define ES_HD inline
#endif

namespace es {

constexpr int kNumPrimes = 53;
constexpr int kDigitLimbs = 6;  // 6 x 64 bits hold a balanced base-P digit (P < 2^334)
constexpr int kCrtWords = 12;   // the same in 32-bit words

struct ModQ {
  uint32_t q;     // the prime
  uint32_t mu;    // floor(2^32 / q)
  uint32_t half;  // (q - 1) / 2
  uint32_t off;   // q * ceil(2^31 / q): makes any int32 x > -2^31 non-negative
  uint32_t r32;   // 2^32 mod q
  uint32_t r64;   // 2^64 mod q
};

// The odd primes below 256, ascending.
constexpr uint32_t kPrimes[kNumPrimes] = {
    3,   5,   7,   11,  13,  17,  19,  23,  29,  31,  37,  41,  43,  47,  53,  59,  61,  67,
    71,  73,  79,  83,  89,  97,  101, 103, 107, 109, 113, 127, 131, 137, 139, 149, 151, 157,
    163, 167, 173, 179, 181, 191, 193, 197, 199, 211, 223, 227, 229, 233, 239, 241, 251};

constexpr ModQ make_modq(uint32_t q) {
  return ModQ{q,
              (uint32_t)(0x100000000ull / q),
              (q - 1) / 2,
              (uint32_t)(q * ((0x80000000ull + q - 1) / q)),
              (uint32_t)(0x100000000ull % q),
              (uint32_t)(((0x100000000ull % q) * (0x100000000ull % q)) % q)};
}

ES_HD uint32_t umulhi32(uint32_t a, uint32_t b) {
#if defined(__CUDA_ARCH__)
  return __umulhi(a, b);
#else
  return (uint32_t)(((uint64_t)a * b) >> 32);
#endif
}

// u mod q for any u < 2^32.
ES_HD uint32_t barrett(uint32_t u, const ModQ& m) {
  uint32_t t = umulhi32(u, m.mu);
  uint32_t r = u - t * m.q;
  return r >= m.q ? r - m.q : r;
}

// Balanced residue of a signed accumulator x with -2^31 < x < 2^31 - 256.
// (x + off) is computed modulo 2^32 and is the exact value in [0, 2^32).
ES_HD int32_t reduce_bal(int32_t x, const ModQ& m) {
  uint32_t r = barrett((uint32_t)x + m.off, m);
  return r > m.half ? (int32_t)r - (int32_t)m.q : (int32_t)r;
}

// Residue in [0, q) of any int64 (two's complement split into 32-bit halves).
ES_HD uint32_t mod_i64(int64_t a, const ModQ& m) {
  uint64_t u = (uint64_t)a;
  uint32_t h = barrett((uint32_t)(u >> 32), m);
  uint32_t l = barrett((uint32_t)u, m);
  uint32_t s = barrett(h * m.r32 + l, m);  // < 256*256 + 256
  if (a < 0) {                              // value = u - 2^64
    s = s + m.q - m.r64;
    s = s >= m.q ? s - m.q : s;
  }
  return s;
}

ES_HD int32_t bal_from_unsigned(uint32_t r, const ModQ& m) {
  return r > m.half ? (int32_t)r - (int32_t)m.q : (int32_t)r;
}

ES_HD int32_t reduce_i64_bal(int64_t a, const ModQ& m) { return bal_from_unsigned(mod_i64(a, m), m); }

// v^{-1} mod q for v != 0 mod q, by Fermat's little theorem (q prime).
ES_HD uint32_t inv_mod(uint32_t v, const ModQ& m) {
  uint32_t base = barrett(v, m), e = m.q - 2, r = 1;
  while (e) {
    if (e & 1) r = barrett(r * base, m);
    base = barrett(base * base, m);
    e >>= 1;
  }
  return r;
}

}  // namespace es

namespace es {
struct ModQTable {
  ModQ v[kNumPrimes];
};
constexpr ModQTable make_modq_table() {
  ModQTable t{};
  for (int i = 0; i < kNumPrimes; ++i) t.v[i] = make_modq(kPrimes[i]);
  return t;
}
}  // namespace es

#if defined(__CUDACC__)
// Per-prime reduction constants in constant memory (one copy per translation unit).
static __constant__ es::ModQTable c_modq = es::make_modq_table();

namespace es {
// Four signed bytes -> f16x2 of bytes 0, 1 (lo) and of bytes 2, 3 (hi): with
// u = x + 128 (the top bit flipped), 0x64uu is the f16 1024 + u, and
// 1024 + u - 1152 = x exactly.
__device__ __forceinline__ void s8x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  lo = __byte_perm(u, 0x64646464u, 0x4140);
  hi = __byte_perm(u, 0x64646464u, 0x4342);
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(0x64806480u));
}
}  // namespace es
#endif
