// Host helpers shared by the two reconstruction paths (recon.cpp: all on the
// host; k_recon.cu: numerators on the GPU).
#pragma once

#include <atomic>
#include <functional>
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
// The same sum split in halves down to short runs of digits (Horner on the
// runs), X = X_lo + P'^h X_hi.  The powers P'^h of every split length depend
// on m only and are built beforehand (from `table` when it reaches h).
struct AssemblePlan {
  int32_t m = 0;
  std::vector<std::pair<int32_t, big::Nat>> pw;  // (h, P'^h)
};
void assemble_plan_init(const PrimeSet& ps, int32_t m, AssemblePlan* ap,
                        const std::vector<big::Nat>* table = nullptr);
big::Nat assemble_shifted_dc(const PrimeSet& ps, const AssemblePlan& ap, const uint64_t* base, size_t stride);
// The shifted sum of one streamed component (entry s of every step's `rows`
// entries of `words` words in `host`: twelve words, each a 32-bit part of the
// digit's six limbs under the tag step + 1 in its high half), formed from the
// low digit up as the digits arrive: X' += (x_i + (P'-1)/2) P'^i, the same
// value as assemble_shifted.  False when lift_over() says the lift has ended
// and a digit is still missing (or after a minute without progress).
bool assemble_streamed(const PrimeSet& ps, const volatile uint64_t* host, int s, int rows, int words, int32_t m,
                       const std::function<bool()>& lift_over, big::Nat* out);
// P'^k for k = 0 .. kmax, one multiplication by P' each
void power_table(const PrimeSet& ps, int32_t kmax, std::vector<big::Nat>* pw);
// u = X mod M in [0, M) from the shifted sum X' (M = P'^m, Mhalf = (M-1)/2).
big::Nat shifted_to_residue(big::Nat X, const big::Nat& Mhalf, const big::Nat& Mhalf1);

// d <- lcm(d, v)
void lcm_in(big::Nat& d, const big::Nat& v);

// Rational reconstruction of one component's denominator (Wang; bounds
// Nb = 2^num_bits, Db = 2^den_bits); false when it does not exist.  With the
// pipes of `o`, pool tasks serving them (big::cofactor_pipe_serve,
// big::low_pipe_serve) can keep the cofactors and the remainders' low limbs.
bool component_denominator(const big::Nat& M, const big::Nat& u, int64_t num_bits, int64_t den_bits,
                           big::Nat* den, const big::ReconOpts& o = big::ReconOpts());
// Low-limb servers per reconstruction when the pool is wide enough.
constexpr int64_t kLowServers = 2;
// Denominators of `count` components at once on the host pool: run(t, opts)
// reconstructs component t (passing the options on).  When the pool is at
// least twice as wide as count, each run gets a cofactor pipe and a second
// pool task serves it; when it is wider still, a low-limb pipe as well with up
// to kLowServers more tasks (the tasks are taken in index order: the runs come
// first, then the cofactor servers, so a narrower pool than planned only makes
// the servers return at once).
void denominators_parallel(int64_t count, int width,
                           const std::function<void(int64_t, const big::ReconOpts&)>& run);

// Two's complement little-endian limbs of +-mag into out[0..W).
void to_limbs(const big::Nat& mag, bool neg, int64_t W, uint64_t* out);

// Components whose denominators seed the common denominator.  Components of
// one column usually share its least denominator while columns differ, so the
// sample takes one component per column (rows spread out): `count` of them,
// where count = max(4, min(c, width)) for `width` host threads.
int64_t sample_count(int64_t c, int width);
std::vector<int64_t> sample_components(int64_t n, int64_t c, int64_t count);
// From the failed components in ascending order, the first of each column, at
// most `count` of them.
std::vector<int64_t> first_failure_per_column(const std::vector<int64_t>& failed, int64_t c, int64_t count);

// fn(i) for i in [0, count) on up to `threads` host threads (<= 0: all
// cores) of the process-wide pool (host_pool.cpp); returns when all are done.
void host_parallel_for(int64_t count, int threads, const std::function<void(int64_t)>& fn);
template <typename F>
void parallel_for(int64_t count, int threads, F&& fn) {
  host_parallel_for(count, threads, std::function<void(int64_t)>(std::forward<F>(fn)));
}

}  // namespace es
