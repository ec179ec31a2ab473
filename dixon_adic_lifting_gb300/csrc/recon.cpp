// Final rational reconstruction on the host.
//
// exact-solve card, §Method: the last stage reconstructs the rationals on
// the CPU -- a common denominator taken from a few sampled components, then a
// single modular multiplication for each numerator (the card runs it with a
// multiprecision package and worker processes).  Here: the library's own
// limb arithmetic (bigint.h) and a pool of host threads.
//
// From the digits x_0 .. x_{m-1} (balanced, base P') of every component:
//   u_k = sum_i x_{i,k} P'^i mod M,  M = P'^m > 2 Nb Db  (Nb = 2^num_bits, Db = 2^den_bits)
//   d   = lcm of the denominators of a few sampled components, each found by
//         Wang's rational reconstruction (extended Euclid on (M, u_k) stopped
//         at the first remainder <= Nb);
//   N_k = bal(d u_k mod M), accepted when |N_k| <= Nb.
// Acceptance certifies d x_k integral: N_k v = d u (mod M) with both sides
// below M/2 in absolute value forces v | d u, i.e. v = 1.  A component that
// fails has a denominator not dividing d: it is reconstructed, d grows to the
// lcm, and the pass repeats.  The final d is the least common denominator
// (it divides the true one and makes every d x_k integral), so the result is
// the canonical (N, d) whatever the sample.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <climits>
#include <new>
#include <cstring>
#include <mutex>
#include <thread>
#include <vector>

#include "bigint.h"
#include "es_common.cuh"
#include "es_internal.h"
#include "recon_common.h"

namespace es {

using big::Nat;

PrimeSet make_prime_set(const uint8_t* good) {
  PrimeSet ps;
  ps.P = big::from_u64(1);
  for (int j = 0; j < kNumPrimes; ++j)
    if (good[j]) {
      ps.P = big::mul_small(ps.P, kPrimes[j]);
      ++ps.E;
    }
  ps.half = big::shr(big::sub(ps.P, big::from_u64(1)), 1);
  std::memset(ps.P6, 0, sizeof(ps.P6));
  std::memset(ps.half6, 0, sizeof(ps.half6));
  for (size_t l = 0; l < ps.P.size() && l < (size_t)kDigitLimbs; ++l) ps.P6[l] = ps.P[l];
  for (size_t l = 0; l < ps.half.size() && l < (size_t)kDigitLimbs; ++l) ps.half6[l] = ps.half[l];
  ps.plen = (int)ps.P.size();
  return ps;
}

Nat pow_nat(const Nat& b, int64_t e) {
  Nat r = big::from_u64(1), base = b;
  for (; e; e >>= 1) {
    if (e & 1) r = big::mul(r, base);
    if (e > 1) base = big::mul(base, base);
  }
  return r;
}

Nat assemble_shifted(const PrimeSet& ps, const uint64_t* base, size_t stride, int32_t m) {
  Nat X;
  for (int32_t i = m - 1; i >= 0; --i) {
    const uint64_t* dg = base + (size_t)i * stride;
    uint64_t xp[kDigitLimbs];
    unsigned __int128 carry = 0;
    for (int l = 0; l < kDigitLimbs; ++l) {
      unsigned __int128 s = (unsigned __int128)dg[l] + ps.half6[l] + carry;
      xp[l] = (uint64_t)s;
      carry = s >> 64;
    }
    int alen = kDigitLimbs;
    while (alen && xp[alen - 1] == 0) --alen;
    big::mul_small_add_in(X, ps.P6, ps.plen, xp, alen);
  }
  return X;
}

bool assemble_streamed(const PrimeSet& ps, const volatile uint64_t* host, int s, int rows, int words, int32_t m,
                       const std::function<bool()>& lift_over, Nat* out) {
  Nat X, pw = big::from_u64(1);
  auto last = std::chrono::steady_clock::now();
  for (int32_t i = 0; i < m; ++i) {
    const volatile uint64_t* e = host + ((size_t)i * rows + (size_t)s) * words;
    const uint64_t tag = (uint64_t)i + 1;
    uint64_t w[2 * kDigitLimbs];
    for (int j = 0; j < 2 * kDigitLimbs; ++j) {
      for (uint32_t spins = 1; ((w[j] = e[j]) >> 32) != tag; ++spins) {
        if ((spins & 1023) == 0) {
          if (lift_over() && (e[j] >> 32) != tag) return false;
          if (std::chrono::steady_clock::now() - last > std::chrono::seconds(60)) return false;
          std::this_thread::yield();
        }
      }
    }
    uint64_t dg[kDigitLimbs];
    for (int l = 0; l < kDigitLimbs; ++l) dg[l] = (w[2 * l] & 0xffffffffull) | (w[2 * l + 1] << 32);
    uint64_t xp[kDigitLimbs];
    unsigned __int128 carry = 0;
    for (int l = 0; l < kDigitLimbs; ++l) {
      const unsigned __int128 v = (unsigned __int128)dg[l] + ps.half6[l] + carry;
      xp[l] = (uint64_t)v;
      carry = v >> 64;
    }
    int alen = kDigitLimbs;
    while (alen && xp[alen - 1] == 0) --alen;
    if (alen) big::add_in(X, big::mul(Nat(xp, xp + alen), pw));
    if (i + 1 < m) pw = big::mul(pw, ps.P);
    last = std::chrono::steady_clock::now();
  }
  *out = std::move(X);
  return true;
}

namespace {
constexpr int32_t kAssembleLeaf = 24;
void split_lengths(int32_t len, std::vector<int32_t>& out) {
  if (len <= kAssembleLeaf) return;
  const int32_t h = len / 2;
  out.push_back(h);
  split_lengths(h, out);
  split_lengths(len - h, out);
}
Nat assemble_range(const PrimeSet& ps, const AssemblePlan& ap, const uint64_t* base, size_t stride, int32_t lo,
                   int32_t len) {
  if (len <= kAssembleLeaf) return assemble_shifted(ps, base + (size_t)lo * stride, stride, len);
  const int32_t h = len / 2;
  const Nat* ph = nullptr;
  for (const auto& e : ap.pw)
    if (e.first == h) ph = &e.second;
  if (!ph) return assemble_shifted(ps, base + (size_t)lo * stride, stride, len);
  Nat r = big::mul(assemble_range(ps, ap, base, stride, lo + h, len - h), *ph);
  big::add_in(r, assemble_range(ps, ap, base, stride, lo, h));
  return r;
}
}  // namespace

void power_table(const PrimeSet& ps, int32_t kmax, std::vector<Nat>* pw) {
  pw->assign((size_t)kmax + 1, Nat{});
  (*pw)[0] = big::from_u64(1);
  for (int32_t k = 1; k <= kmax; ++k) {
    Nat v = (*pw)[(size_t)k - 1];
    big::mul_small_add_in(v, ps.P6, ps.plen, nullptr, 0);
    (*pw)[(size_t)k] = std::move(v);
  }
}

void assemble_plan_init(const PrimeSet& ps, int32_t m, AssemblePlan* ap, const std::vector<Nat>* table) {
  ap->m = m;
  ap->pw.clear();
  std::vector<int32_t> hs;
  split_lengths(m, hs);
  std::sort(hs.begin(), hs.end());
  hs.erase(std::unique(hs.begin(), hs.end()), hs.end());
  for (int32_t h : hs)
    ap->pw.emplace_back(h, table && (size_t)h < table->size() ? (*table)[(size_t)h] : pow_nat(ps.P, h));
}

Nat assemble_shifted_dc(const PrimeSet& ps, const AssemblePlan& ap, const uint64_t* base, size_t stride) {
  return assemble_range(ps, ap, base, stride, 0, ap.m);
}

Nat shifted_to_residue(Nat X, const Nat& Mhalf, const Nat& Mhalf1) {
  if (big::cmp(X, Mhalf) >= 0)
    big::sub_in(X, Mhalf);
  else
    big::add_in(X, Mhalf1);
  return X;
}

void lcm_in(Nat& d, const Nat& v) {
  if (big::cmp(d, v) == 0 || v.empty()) return;
  if (d.size() == 1 && d[0] == 1) {  // lcm(1, v) = v
    d = v;
    return;
  }
  Nat g = big::gcd(d, v), q;
  big::divmod(v, g, &q, nullptr);
  d = big::mul(d, q);
}

bool component_denominator(const Nat& M, const Nat& u, int64_t num_bits, int64_t den_bits, Nat* den,
                           const big::ReconOpts& o) {
  Nat num;
  bool neg;
  return big::rational_reconstruct(M, u, (size_t)num_bits, &num, &neg, den, o) &&
         big::le_pow2(*den, (size_t)den_bits);
}

void denominators_parallel(int64_t count, int width, const std::function<void(int64_t, const big::ReconOpts&)>& run) {
  std::vector<big::ReconOpts> opts((size_t)std::max<int64_t>(count, 0));
  int64_t low = 0;  // low-limb servers per run
  if (count > 0 && 2 * count <= (int64_t)width) {
    low = std::min<int64_t>(kLowServers, ((int64_t)width - 2 * count) / count);
    for (auto& o : opts) {
      o.pipe = big::cofactor_pipe_new();
      if (low > 0) o.low = big::low_pipe_new();
    }
  }
  const int64_t tasks = opts.empty() || !opts[0].pipe ? count : (2 + low) * count;
  parallel_for(tasks, width, [&](int64_t t) {
    if (t < count) {
      run(t, opts[(size_t)t]);
      // the servers return even if the run never reached the reconstruction
      big::cofactor_pipe_close(opts[(size_t)t].pipe);
      big::low_pipe_close(opts[(size_t)t].low);
    } else if (t < 2 * count)
      big::cofactor_pipe_serve(opts[(size_t)(t - count)].pipe);
    else
      big::low_pipe_serve(opts[(size_t)((t - 2 * count) % count)].low);
  });
  for (auto& o : opts) {
    big::cofactor_pipe_free(o.pipe);
    big::low_pipe_free(o.low);
  }
}

void to_limbs(const Nat& mag, bool neg, int64_t W, uint64_t* out) {
  for (int64_t l = 0; l < W; ++l) out[l] = l < (int64_t)mag.size() ? mag[(size_t)l] : 0;
  if (neg) {
    unsigned __int128 carry = 1;
    for (int64_t l = 0; l < W; ++l) {
      unsigned __int128 s = (unsigned __int128)(~out[l]) + carry;
      out[l] = (uint64_t)s;
      carry = s >> 64;
    }
  }
}

int64_t sample_count(int64_t c, int width) { return std::max<int64_t>(4, std::min<int64_t>(c, width)); }

std::vector<int64_t> sample_components(int64_t n, int64_t c, int64_t count) {
  const int64_t ns = std::min(n * c, count);
  std::vector<int64_t> k((size_t)ns);
  for (int64_t t = 0; t < ns; ++t) k[(size_t)t] = ((t * n) / ns) * c + (t * c) / ns;
  return k;
}

std::vector<int64_t> first_failure_per_column(const std::vector<int64_t>& failed, int64_t c, int64_t count) {
  std::vector<int64_t> out;
  std::vector<uint8_t> taken((size_t)c, 0);
  for (int64_t k : failed) {
    if ((int64_t)out.size() >= count) break;
    if (taken[(size_t)(k % c)]) continue;
    taken[(size_t)(k % c)] = 1;
    out.push_back(k);
  }
  return out;
}

es_status reconstruct(const uint64_t* digits, int64_t n, int64_t c, int32_t m, const uint8_t* good,
                      int64_t num_bits, int64_t den_bits, int threads, bool inject_fault, Solution* out) {
  if (inject_fault) return ES_ERR_INTERNAL;
  if (!digits || n < 1 || c < 1 || m < 1 || !good || num_bits < 0 || den_bits < 0) return ES_ERR_ARG;
  const PrimeSet ps = make_prime_set(good);
  if (ps.E == 0) return ES_ERR_ARG;
  const int64_t nc = n * c;
  const Nat M = pow_nat(ps.P, m);
  // Wang's uniqueness condition M > 2 Nb Db = 2^(num_bits + den_bits + 1)
  if (big::le_pow2(M, (size_t)(num_bits + den_bits + 1))) return ES_ERR_INTERNAL;
  const Nat Mhalf = big::shr(big::sub(M, big::from_u64(1)), 1);
  const Nat Mhalf1 = big::add(Mhalf, big::from_u64(1));
  AssemblePlan ap;
  assemble_plan_init(ps, m, &ap);
  auto residue = [&](int64_t k) {
    return shifted_to_residue(assemble_shifted_dc(ps, ap, digits + (size_t)k * kDigitLimbs, (size_t)nc * kDigitLimbs),
                              Mhalf, Mhalf1);
  };

  // common denominator from a sample of components
  const int width = threads > 0 ? threads : std::max(1, (int)std::thread::hardware_concurrency());
  const int64_t per_round = sample_count(c, width);
  const std::vector<int64_t> sk = sample_components(n, c, per_round);
  const int64_t ns = (int64_t)sk.size();
  std::vector<Nat> sden((size_t)ns);
  std::atomic<int> fail(0);
  denominators_parallel(ns, width, [&](int64_t t, const big::ReconOpts& ro) {
    if (!component_denominator(M, residue(sk[(size_t)t]), num_bits, den_bits, &sden[(size_t)t], ro)) fail = 1;
  });
  if (fail) return ES_ERR_INTERNAL;
  Nat d = big::from_u64(1);
  for (auto& v : sden) lcm_in(d, v);

  const int64_t W0 = (num_bits + 2 + 63) / 64, W1 = (den_bits + 1 + 63) / 64;
  const int64_t W = W0 > W1 ? W0 : W1;
  out->n = n;
  out->c = c;
  out->limbs = W;
  out->num.resize((size_t)(nc * W));  // every component writes its W limbs before the round ends
  for (int round = 0;; ++round) {
    if (round > 64) return ES_ERR_INTERNAL;
    std::mutex mu;
    std::vector<int64_t> failed;
    parallel_for(nc, threads, [&](int64_t k) {
      Nat prod = big::mul(d, residue(k)), rem;
      big::divmod(prod, M, nullptr, &rem);
      bool neg = big::cmp(rem, Mhalf) > 0;
      Nat mag = neg ? big::sub(M, rem) : rem;
      if (!big::le_pow2(mag, (size_t)num_bits)) {
        std::lock_guard<std::mutex> lk(mu);
        failed.push_back(k);
        return;
      }
      to_limbs(mag, neg, W, out->num.data() + (size_t)k * (size_t)W);
    });
    if (failed.empty()) break;
    std::sort(failed.begin(), failed.end());
    failed = first_failure_per_column(failed, c, per_round);
    // Every failing component's denominator does not divide d, so the round's
    // lcm must grow d (a later one may already be covered by an earlier one).
    const Nat before = d;
    std::vector<Nat> fden(failed.size());
    denominators_parallel((int64_t)failed.size(), width, [&](int64_t t, const big::ReconOpts& ro) {
      if (!component_denominator(M, residue(failed[(size_t)t]), num_bits, den_bits, &fden[(size_t)t], ro))
        fail = 1;
    });
    if (fail) return ES_ERR_INTERNAL;
    for (auto& v : fden) lcm_in(d, v);
    if (big::cmp(before, d) == 0) return ES_ERR_INTERNAL;  // no progress: digits inconsistent
  }
  if (!big::le_pow2(d, (size_t)den_bits)) return ES_ERR_INTERNAL;
  out->den.assign((size_t)W, 0);
  to_limbs(d, false, W, out->den.data());
  out->primes_used = ps.E;
  out->m = m;
  return ES_OK;
}

}  // namespace es

extern "C" es_status es_reconstruct(const uint64_t* digits, int64_t n, int64_t c, int32_t m, const uint8_t* good,
                                    int64_t num_bits, int64_t den_bits, const es_options* opt, es_solution** out) {
  if (!out) return ES_ERR_ARG;
  *out = nullptr;
  es_solution* s = new (std::nothrow) es_solution;
  if (!s) return ES_ERR_NOMEM;
  auto t0 = std::chrono::steady_clock::now();
  es_status st = es::reconstruct(digits, n, c, m, good, num_bits, den_bits, opt ? opt->threads : 0,
                                 opt && opt->fault_stage == ES_FAULT_RECON, &s->s);
  if (st != ES_OK) {
    delete s;
    return st;
  }
  s->s.ms[4] = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
  s->s.ms[5] = s->s.ms[4];
  *out = s;
  return ES_OK;
}

extern "C" int64_t es_selftest_modular(int64_t lo, int64_t hi, int64_t samples) {
  if (lo > hi || lo < INT32_MIN || hi > (int64_t)INT32_MAX - 255 || samples < 0) return -1;
  int64_t bad = 0;
  for (int j = 0; j < es::kNumPrimes; ++j) {
    const es::ModQ mq = es::make_modq(es::kPrimes[j]);
    const int64_t q = es::kPrimes[j], h = (q - 1) / 2;
    for (int64_t x = lo; x < hi; ++x) {
      int64_t r = x % q;
      if (r > h) r -= q;
      if (r < -h) r += q;
      if (es::reduce_bal((int32_t)x, mq) != r) ++bad;
    }
    uint64_t s = 0x9E3779B97F4A7C15ull ^ (uint64_t)j;
    for (int64_t t = 0; t < samples; ++t) {
      s ^= s << 13;
      s ^= s >> 7;
      s ^= s << 17;
      int64_t a = (int64_t)s;
      if (t < 8) {  // edge values
        const int64_t edges[8] = {INT64_MIN, INT64_MIN + 1, -1, 0, 1, INT64_MAX, INT64_MAX - 1, -q};
        a = edges[t];
      }
      __int128 r = (__int128)a % q;
      if (r > h) r -= q;
      if (r < -h) r += q;
      if (es::reduce_i64_bal(a, mq) != (int32_t)r) ++bad;
      if (a % q != 0) {
        uint32_t au = es::mod_i64(a, mq);
        if (es::barrett(au * es::inv_mod(au, mq), mq) != 1) ++bad;
      }
    }
  }
  return bad;
}

// rational_reconstruct in one of the ways the library can run it: way & 1: a
// cofactor pipe served by a second thread that starts before the run (way & 4:
// after it, so the run keeps the work); with way & 1, a low-limb pipe as well,
// served by two more threads (way & 8), one (way & 16) or five, one more than
// a pipe takes (way & 32), started at the same point (way & 64: each after a
// short delay of its own, so that they join while the run is under way);
// way & 2: half-gcd stages from any length.
static const int kWays[] = {0, 1, 2, 3, 5, 9, 11, 13, 17, 33, 73, 81};
static bool reconstruct_way(const es::big::Nat& M, const es::big::Nat& u, size_t nbits, int way, es::big::Nat* num,
                            bool* neg, es::big::Nat* den) {
  namespace big = es::big;
  big::ReconOpts o;
  if (way & 2) o.hgcd_min_bits = 0;
  if (!(way & 1)) return big::rational_reconstruct(M, u, nbits, num, neg, den, o);
  const int servers = (way & 8) ? 2 : (way & 16) ? 1 : (way & 32) ? 5 : 0;
  big::CofactorPipe* pipe = big::cofactor_pipe_new();
  big::LowPipe* low = servers ? big::low_pipe_new() : nullptr;
  if (!pipe || (servers && !low)) {
    big::cofactor_pipe_free(pipe);
    big::low_pipe_free(low);
    return false;
  }
  o.pipe = pipe;
  o.low = low;
  auto serve = [&] {
    std::vector<std::thread> th;
    th.emplace_back([&] { big::cofactor_pipe_serve(pipe); });
    for (int i = 0; i < servers; ++i)
      th.emplace_back([&, i] {
        if (way & 64) std::this_thread::sleep_for(std::chrono::microseconds(20 + 40 * i));
        big::low_pipe_serve(low);
      });
    return th;
  };
  bool ok = false;
  if (way & 4) {
    ok = big::rational_reconstruct(M, u, nbits, num, neg, den, o);
    for (auto& t : serve()) t.join();
  } else {
    std::vector<std::thread> th = serve();
    ok = big::rational_reconstruct(M, u, nbits, num, neg, den, o);
    for (auto& t : th) t.join();
  }
  big::cofactor_pipe_free(pipe);
  big::low_pipe_free(low);
  return ok;
}

extern "C" int64_t es_selftest_bigint(uint64_t seed, int64_t rounds) {
  using es::big::Nat;
  namespace big = es::big;
  if (rounds < 0) return -1;
  uint64_t st = seed * 0x9E3779B97F4A7C15ull + 1;
  auto rnd = [&]() {
    st ^= st << 13;
    st ^= st >> 7;
    st ^= st << 17;
    return st;
  };
  auto number = [&](size_t limbs) {
    Nat x(limbs);
    const uint64_t kind = rnd() % 4;
    for (auto& v : x) v = kind == 1 ? ~0ull : kind == 2 ? (rnd() % 8 == 0 ? rnd() : 0) : rnd();
    if (!x.empty() && x.back() == 0) x.back() = 1;
    big::trim(x);
    return x;
  };
  // plain O(n m) product, independent of the library's multiplication
  auto school = [](const Nat& a, const Nat& b) {
    Nat r(a.size() + b.size(), 0);
    for (size_t i = 0; i < a.size(); ++i) {
      unsigned __int128 carry = 0;
      for (size_t j = 0; j < b.size(); ++j) {
        const unsigned __int128 t = (unsigned __int128)a[i] * b[j] + r[i + j] + carry;
        r[i + j] = (uint64_t)t;
        carry = t >> 64;
      }
      for (size_t k = i + b.size(); carry; ++k) {
        const unsigned __int128 t = (unsigned __int128)r[k] + carry;
        r[k] = (uint64_t)t;
        carry = t >> 64;
      }
    }
    big::trim(r);
    return r;
  };
  int64_t bad = 0;
  for (int64_t t = 0; t < rounds; ++t) {
    const size_t an = 1 + rnd() % 1200, bn = (t % 3 == 0) ? an : 1 + rnd() % 1200;
    const Nat a = number(an), b = number(bn);
    // products
    if (big::mul(a, b) != school(a, b)) ++bad;
    // division: a = q b + r, 0 <= r < b
    if (!b.empty()) {
      Nat q, r;
      big::divmod(a, b, &q, &r);
      Nat back = big::mul(q, b);
      big::add_in(back, r);
      if (back != a || big::cmp(r, b) >= 0) ++bad;
    }
    // shifts
    const size_t sh = rnd() % 200;
    if (big::shr(big::shl(a, sh), sh) != a) ++bad;
    // rational reconstruction: num = +-den u (mod M), |num| <= 2^nbits, den > 0
    if (t % 4 == 0) {
      const size_t ml = 2 + rnd() % 120;
      Nat M = number(ml);
      if (M.empty()) continue;
      M[0] |= 1;
      Nat u;
      big::divmod(number(ml), M, nullptr, &u);
      const size_t nbits = big::bitlen(M) / 2;
      Nat num, den;
      bool neg = false;
      if (big::rational_reconstruct(M, u, nbits, &num, &neg, &den)) {
        Nat du, rem, nm;
        big::divmod(big::mul(den, u), M, nullptr, &du);
        big::divmod(num, M, nullptr, &nm);
        // den u = num (mod M) for num >= 0, or = M - num for a negative one
        if (neg && !nm.empty()) nm = big::sub(M, nm);
        if (den.empty() || !big::le_pow2(num, nbits) || du != nm) ++bad;
      }
    }
    // planted fraction num / den: with M = den k + 1, den^{-1} = M - k (mod M),
    // so u = -num k (mod M) represents it; with 2^(nbits+1) den < M the stopped
    // Euclid must return exactly (num, den), sign included
    if (t % 4 == 1) {
      // every eighth planted case long enough for the half-gcd stages and the
      // cofactor thread
      const size_t lmax = t % 32 == 1 ? 400 : 40;
      Nat den = number(1 + rnd() % lmax), k = number(1 + rnd() % lmax);
      if (den.empty() || k.empty()) continue;
      Nat M = big::mul(den, k);
      big::add_in(M, big::from_u64(1));
      const size_t dbits = big::bitlen(den), mbits = big::bitlen(M);
      if (mbits < dbits + 4) continue;
      const size_t nbits = mbits - dbits - 2;
      Nat num = big::shr(number((nbits + 63) / 64 + 1), 64 * ((nbits + 63) / 64 + 1) - nbits);  // < 2^nbits
      if (num.empty()) num = big::from_u64(1);
      const bool neg = (rnd() & 1) != 0;
      Nat u;
      big::divmod(big::mul(num, k), M, nullptr, &u);  // num k mod M
      if (!neg && !u.empty()) u = big::sub(M, u);    // -num k mod M
      const Nat g = big::gcd(num, den);
      if (!(g.size() == 1 && g[0] == 1)) {  // the expected result is the reduced fraction
        big::divmod(Nat(num), g, &num, nullptr);
        big::divmod(Nat(den), g, &den, nullptr);
      }
      // the same result on every way the reconstruction can run
      for (int way : kWays) {
        Nat rn, rd;
        bool rneg = false;
        if (!reconstruct_way(M, u, nbits, way, &rn, &rneg, &rd) || rn != num || rd != den || rneg != neg) ++bad;
      }
    }
    // a residue with no small fraction behind it: the other ways agree with
    // the plain one, failure included
    if (t % 8 == 2) {
      const size_t ml = 64 + rnd() % 400;
      Nat M = number(ml);
      if (M.empty()) continue;
      Nat u;
      big::divmod(number(ml), M, nullptr, &u);
      const size_t nbits = big::bitlen(M) / 2 - rnd() % 64;
      Nat n0, d0;
      bool g0 = false;
      const bool ok0 = big::rational_reconstruct(M, u, nbits, &n0, &g0, &d0);
      for (int way : kWays) {
        if (way == 0) continue;
        Nat n1, d1;
        bool g1 = false;
        const bool ok1 = reconstruct_way(M, u, nbits, way, &n1, &g1, &d1);
        if (ok1 != ok0 || (ok0 && (n1 != n0 || d1 != d0 || g1 != g0))) ++bad;
      }
    }
  }
  return bad;
}
