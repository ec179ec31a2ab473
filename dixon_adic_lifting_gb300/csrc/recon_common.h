// Host helpers shared by the two reconstruction paths (recon.cpp: all on the
// host; k_recon.cu: numerators on the GPU).
#pragma once

#include <atomic>
#include <thread>
#include <vector>

#include "bigint.h"
#include "es_common.cuh"

namespace es {

// P' (product of the good primes) and its balanced-digit offset (P'-1)/2.
struct PrimeSet {
  big::Nat P, half;
  uint64_t P6[kDigitLimbs];
  uint64_t half6[kDigitLimbs];
  int plen = 0;
  int E = 0;
};
PrimeSet make_prime_set(const uint8_t* good);
big::Nat pow_nat(const big::Nat& b, int64_t e);

// sum_{i < m} x_i P'^i + (P'^m - 1)/2 for balanced digits x_i stored as 6
// little-endian two's complement limbs at base + i * stride (in limbs):
// Horner on the shifted digits x_i + (P'-1)/2 in [0, P'-1].
big::Nat assemble_shifted(const PrimeSet& ps, const uint64_t* base, size_t stride, int32_t m);
// u = X mod M in [0, M) from the shifted sum X' (M = P'^m, Mhalf = (M-1)/2).
big::Nat shifted_to_residue(big::Nat X, const big::Nat& Mhalf, const big::Nat& Mhalf1);

// d <- lcm(d, v)
void lcm_in(big::Nat& d, const big::Nat& v);

// Rational reconstruction of one component's denominator (Wang; bounds
// Nb = 2^num_bits, Db = 2^den_bits); false when it does not exist.
bool component_denominator(const big::Nat& M, const big::Nat& u, int64_t num_bits, int64_t den_bits,
                           big::Nat* den);

// Two's complement little-endian limbs of +-mag into out[0..W).
void to_limbs(const big::Nat& mag, bool neg, int64_t W, uint64_t* out);

template <typename F>
void parallel_for(int64_t count, int threads, F&& fn) {
  if (count <= 0) return;
  int T = threads > 0 ? threads : (int)std::thread::hardware_concurrency();
  if (T < 1) T = 1;
  if ((int64_t)T > count) T = (int)count;
  std::atomic<int64_t> next(0);
  auto worker = [&]() {
    for (;;) {
      int64_t k = next.fetch_add(1);
      if (k >= count) break;
      fn(k);
    }
  };
  if (T == 1) {
    worker();
    return;
  }
  std::vector<std::thread> pool;
  for (int t = 0; t < T; ++t) pool.emplace_back(worker);
  for (auto& th : pool) th.join();
}

}  // namespace es
