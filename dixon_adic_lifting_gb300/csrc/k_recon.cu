// Rational reconstruction with the numerator pass on the GPU.
//
// exact-solve card, §Method: the final reconstruction takes a common
// denominator from a small sample of components, then one modular multiply
// per numerator.  The sample's rational reconstruction (extended Euclid,
// inherently sequential) stays on the host; the per-numerator pass, which is
// the bulk of the work and independent per component, runs here.
//
// Low-digit certificate.  With Q = P'^m' and X_lo = sum_{i<m'} x_i P'^i the
// lift guarantees A X_lo = b (mod Q) exactly (b = A sum_{i<m'} x_i P'^i +
// P'^m' r_m').  For a candidate d (lcm of sampled denominators, so d | the
// least common denominator and d <= Db) let N_k = bal_Q(d X_lo,k).  If every
// |N_k| <= Nb then A N = d b (mod Q) and |A N - d b| <= n max|A| Nb +
// Db max|b| < Q/2, hence A N = d b exactly: N / d is the solution and d is the
// least common denominator.  So only m' digits are read, with
// Q > 2 (n max|A| 2^num_bits + 2^den_bits max|b|) -- about half of m.
//
// Per component k (one CTA): with G_i = d P'^i mod Q (host-precomputed) and
// the shifted digits x'_i = x_i + (P'-1)/2 in [0, P'-1],
//   Z = sum_i x'_i G_i + (Q - H),  H = ((P'-1)/2) sum_i G_i mod Q,
// so Z = d X_lo (mod Q) with 0 <= Z < (m' P' + 1) Q.  Z is formed as 32-bit
// word column sums (64-bit accumulators plus carry counts), normalised, and
// reduced mod Q by Barrett's method with a 13-word reciprocal; then the sign
// is balanced and |N| <= 2^num_bits is tested.
#include <cuda_runtime.h>

#include <memory>
#include <new>

#include <algorithm>
#include <cstring>
#include <vector>

#include "bigint.h"
#include "es_common.cuh"
#include "es_internal.h"
#include "recon_common.h"

namespace es {

using big::Nat;

namespace {
constexpr int kMuWords = 13;  // Barrett reciprocal floor(b^(LG-1+13) / Q), b = 2^32
constexpr int kZExtra = 12;   // Z < b^(LG + 11)
constexpr int kDigitWords = 2 * kDigitLimbs;
// G rows: word w of G_i at [i * g_stride(LG) + kGPad + w], zeros around it,
// so a thread can load the 16 words ending at its 4 output columns aligned.
constexpr int kGPad = 16;
inline int64_t g_stride(int64_t LG) { return (LG + 3) / 4 * 4 + 2 * kGPad; }

struct RParams {
  const uint32_t* D;      // digits as 32-bit words: [m][nc][12]
  int64_t nc;
  int mp;                 // digits used (m')
  int LG;                 // 32-bit words of Q
  const uint32_t* G;      // [mp][GS]  G_i = d P'^i mod Q (see g_stride)
  int64_t GS;
  const uint32_t* OFF;    // [LG]      Q - H
  const uint32_t* Q;      // [LG]
  const uint32_t* Qhalf;  // [LG]      (Q - 1) / 2
  const uint32_t* MU;     // [13]
  const uint32_t* H12;    // [12]      (P' - 1) / 2
  int64_t nb;             // accept |N| <= 2^nb
  int W;                  // output 64-bit limbs per numerator
  uint64_t* N;            // [nc][W] two's complement
  uint8_t* ok;            // [nc]
};

__device__ __forceinline__ void mac(uint64_t& lo, uint32_t& hi, uint32_t a, uint32_t b) {
  uint64_t p = (uint64_t)a * b;
  lo += p;
  hi += (lo < p) ? 1u : 0u;
}

// acc (96 bits, little-endian words) += x y, one carry chain
__device__ __forceinline__ void mac96(uint32_t (&acc)[3], uint32_t x, uint32_t y) {
  asm("mad.lo.cc.u32 %0, %3, %4, %0;\n\tmadc.hi.cc.u32 %1, %3, %4, %1;\n\taddc.u32 %2, %2, 0;"
      : "+r"(acc[0]), "+r"(acc[1]), "+r"(acc[2])
      : "r"(x), "r"(y));
}

__global__ void __launch_bounds__(256) k_recon_numerators(RParams p) {
  const int64_t k = blockIdx.x;
  const int mp = p.mp, LG = p.LG, LZ = LG + kZExtra;
  const int tid = threadIdx.x, nt = blockDim.x;
  extern __shared__ __align__(16) unsigned char sm[];
  uint64_t* Zlo = reinterpret_cast<uint64_t*>(sm);          // LZ + 1
  uint32_t* Zhi = reinterpret_cast<uint32_t*>(Zlo + LZ + 1);  // LZ + 1
  uint32_t* Zn = Zhi + LZ + 1;                              // LZ + 1
  uint32_t* xs = Zn + LZ + 1;                               // mp * 12
  __shared__ uint32_t qh[kMuWords];
  __shared__ int s_ok, s_neg, s_z;

  // shifted digits x'_i = x_i + (P'-1)/2  (384-bit two's complement add)
  for (int i = tid; i < mp; i += nt) {
    const uint32_t* src = p.D + ((size_t)i * (size_t)p.nc + (size_t)k) * kDigitWords;
    uint64_t carry = 0;
#pragma unroll
    for (int l = 0; l < kDigitWords; ++l) {
      uint64_t s = (uint64_t)src[l] + p.H12[l] + carry;
      xs[i * kDigitWords + l] = (uint32_t)s;
      carry = s >> 32;
    }
  }
  __syncthreads();
  // Z word columns: Z[w] = OFF[w] + sum_i sum_l x'_i[l] G_i[w - l].  A thread
  // owns 4 consecutive columns: per digit it loads the 16 words of G_i they
  // need (4 aligned 16-byte loads) and the digit's 12 words, then 48 96-bit MACs.
  for (int w0 = 4 * tid; w0 < LZ; w0 += 4 * nt) {
    uint32_t acc[4][3];
#pragma unroll
    for (int o = 0; o < 4; ++o) {
      acc[o][0] = w0 + o < LG ? p.OFF[w0 + o] : 0u;
      acc[o][1] = 0u;
      acc[o][2] = 0u;
    }
    for (int i = 0; i < mp; ++i) {
      const uint4* gr = reinterpret_cast<const uint4*>(p.G + (size_t)i * p.GS + kGPad + w0 - 12);
      const uint4* xr = reinterpret_cast<const uint4*>(xs + i * kDigitWords);
      uint32_t g[16], x[kDigitWords];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const uint4 v = __ldg(gr + h);
        g[4 * h] = v.x, g[4 * h + 1] = v.y, g[4 * h + 2] = v.z, g[4 * h + 3] = v.w;
      }
#pragma unroll
      for (int h = 0; h < kDigitWords / 4; ++h) {
        const uint4 v = xr[h];
        x[4 * h] = v.x, x[4 * h + 1] = v.y, x[4 * h + 2] = v.z, x[4 * h + 3] = v.w;
      }
#pragma unroll
      for (int o = 0; o < 4; ++o)
#pragma unroll
        for (int l = 0; l < kDigitWords; ++l) mac96(acc[o], x[l], g[o + 12 - l]);
    }
#pragma unroll
    for (int o = 0; o < 4; ++o)
      if (w0 + o < LZ) {
        Zlo[w0 + o] = (uint64_t)acc[o][0] | ((uint64_t)acc[o][1] << 32);
        Zhi[w0 + o] = acc[o][2];
      }
  }
  __syncthreads();
  if (tid == 0) {
    // normalise the columns into 32-bit words
    uint64_t carry = 0;
    for (int w = 0; w < LZ; ++w) {
      unsigned __int128 s = (unsigned __int128)Zlo[w] + ((unsigned __int128)Zhi[w] << 64) + carry;
      Zn[w] = (uint32_t)s;
      carry = (uint64_t)(s >> 32);
    }
    // q^ = floor(Z1 MU / b^13) with Z1 = floor(Z / b^(LG-1)) (13 words)
    uint32_t prod[2 * kMuWords];
    for (int t = 0; t < 2 * kMuWords; ++t) prod[t] = 0;
    for (int a = 0; a < kMuWords; ++a) {
      uint64_t c = 0;
      const uint64_t za = Zn[LG - 1 + a];
      for (int b = 0; b < kMuWords; ++b) {
        uint64_t t = za * p.MU[b] + prod[a + b] + c;
        prod[a + b] = (uint32_t)t;
        c = t >> 32;
      }
      prod[a + kMuWords] = (uint32_t)c;
    }
    for (int t = 0; t < kMuWords; ++t) qh[t] = prod[kMuWords + t];
  }
  __syncthreads();
  // q^ Q, words 0 .. LG (enough: the remainder is below 3Q < b^(LG+1))
  for (int w = tid; w <= LG; w += nt) {
    uint64_t lo = 0;
    uint32_t hi = 0;
    for (int j = 0; j < kMuWords; ++j) {
      const int t = w - j;
      if (t >= 0 && t < LG) mac(lo, hi, qh[j], p.Q[t]);
    }
    Zlo[w] = lo;
    Zhi[w] = hi;
  }
  __syncthreads();
  if (tid == 0) {
    // r = Z - q^ Q  (mod b^(LG+1))
    uint64_t carry = 0;
    int64_t borrow = 0;
    for (int w = 0; w <= LG; ++w) {
      unsigned __int128 s = (unsigned __int128)Zlo[w] + ((unsigned __int128)Zhi[w] << 64) + carry;
      const uint32_t qq = (uint32_t)s;
      carry = (uint64_t)(s >> 32);
      const int64_t d = (int64_t)Zn[w] - (int64_t)qq + borrow;
      Zn[w] = (uint32_t)d;
      borrow = d >> 32;
    }
    // at most two subtractions of Q
    for (int rep = 0; rep < 3; ++rep) {
      bool ge = Zn[LG] != 0;
      if (!ge) {
        ge = true;
        for (int w = LG - 1; w >= 0; --w)
          if (Zn[w] != p.Q[w]) {
            ge = Zn[w] > p.Q[w];
            break;
          }
      }
      if (!ge) break;
      borrow = 0;
      for (int w = 0; w <= LG; ++w) {
        const int64_t d = (int64_t)Zn[w] - (int64_t)(w < LG ? p.Q[w] : 0u) + borrow;
        Zn[w] = (uint32_t)d;
        borrow = d >> 32;
      }
    }
    // balanced: r > (Q-1)/2 -> N = r - Q, magnitude Q - r
    bool neg = false;
    for (int w = LG - 1; w >= 0; --w)
      if (Zn[w] != p.Qhalf[w]) {
        neg = Zn[w] > p.Qhalf[w];
        break;
      }
    if (neg) {
      borrow = 0;
      for (int w = 0; w < LG; ++w) {
        const int64_t d = (int64_t)p.Q[w] - (int64_t)Zn[w] + borrow;
        Zn[w] = (uint32_t)d;
        borrow = d >> 32;
      }
    }
    Zn[LG] = 0;
    // |N| <= 2^nb ?
    int top = LG - 1;
    while (top >= 0 && Zn[top] == 0) --top;
    bool ok = true;
    if (top >= 0) {
      const int64_t bl = 32 * (int64_t)top + (32 - __clz(Zn[top]));
      if (bl > p.nb + 1) {
        ok = false;
      } else if (bl == p.nb + 1) {  // equal to 2^nb only
        ok = Zn[top] == (1u << (p.nb % 32));
        for (int w = 0; ok && w < top; ++w) ok = Zn[w] == 0;
      }
    }
    int z = 0;
    while (z < LG && Zn[z] == 0) ++z;
    s_ok = ok ? 1 : 0;
    s_neg = neg ? 1 : 0;
    s_z = z;
  }
  __syncthreads();
  // two's complement output: -mag = ~mag + 1 (words below the lowest nonzero stay 0)
  const int neg = s_neg, z = s_z;
  uint64_t* out = p.N + (size_t)k * p.W;
  for (int t = tid; t < p.W; t += nt) {
    uint32_t wv[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int w = 2 * t + h;
      const uint32_t m = w < LG ? Zn[w] : 0u;
      wv[h] = !neg ? m : (w < z ? 0u : (w == z ? (uint32_t)(0u - m) : ~m));
    }
    out[t] = (uint64_t)wv[0] | ((uint64_t)wv[1] << 32);
  }
  if (tid == 0) p.ok[k] = (uint8_t)s_ok;
}

// little-endian 32-bit words of a natural, zero-extended to `words`
void to_words(const Nat& a, int64_t words, uint32_t* out) {
  for (int64_t w = 0; w < words; ++w) {
    const size_t limb = (size_t)(w / 2);
    const uint64_t v = limb < a.size() ? a[limb] : 0;
    out[w] = (uint32_t)(w % 2 ? v >> 32 : v);
  }
}

int64_t u64_bitlen(uint64_t v) { return v ? 64 - __builtin_clzll(v) : 0; }

}  // namespace

bool recon_device_applicable(int64_t n, int32_t m, const uint8_t* good, int64_t num_bits, int64_t den_bits,
                             const Stats& stats, int32_t* mp_out) {
  // Q = P'^m' > 2 (n max|A| 2^num_bits + 2^den_bits max|b|): it suffices that
  // Q > 2^(max(num_bits + bitlen(n max|A|), den_bits + bitlen(max|b|)) + 2)
  const int64_t na = u64_bitlen((uint64_t)n * stats.max_abs_a);  // n max|A| < 2^63
  const int64_t need = std::max(num_bits + na, den_bits + u64_bitlen(stats.max_abs_b)) + 2;
  double log2P = 0.0;
  for (int j = 0; j < kNumPrimes; ++j)
    if (good[j]) log2P += std::log2((double)kPrimes[j]);
  int32_t mp = (int32_t)((double)need / log2P) + 2;  // checked exactly on the host later
  if (mp > m) return false;
  *mp_out = mp;
  return true;
}

size_t recon_device_bytes(int64_t nc, int32_t mp, const uint8_t* good, int64_t num_bits, int64_t den_bits) {
  double log2P = 0.0;
  for (int j = 0; j < kNumPrimes; ++j)
    if (good[j]) log2P += std::log2((double)kPrimes[j]);
  const int64_t LG = (int64_t)(mp * log2P / 32.0) + 2;
  const int64_t W0 = (num_bits + 2 + 63) / 64, W1 = (den_bits + 1 + 63) / 64;
  const int64_t W = W0 > W1 ? W0 : W1;
  Layout L;
  L.add((size_t)mp * g_stride(LG) * 4);
  L.add((size_t)LG * 4 * 3);
  L.add(kMuWords * 4 + kDigitWords * 4);
  L.add((size_t)nc * W * 8);
  L.add((size_t)nc);
  return L.total;
}

// G_{i+1} = G_i P' mod Q for i < mp, written as LG 32-bit words each (row i
// at out + i GS + kGPad), and
// their sum.  Knuth's division with the divisor normalised once: G is kept
// shifted left by the normalising shift s, so each step is one multiply by
// the 6-limb P' and a division whose quotient has at most 6 limbs, in place.
static void g_chain(const Nat& Q, const Nat& P, const Nat& g0, int32_t mp, int64_t LG, int64_t GS, uint32_t* out,
                    Nat* sum) {
  using limb = big::limb;
  using u128 = unsigned __int128;
  const size_t n = Q.size(), pn = P.size();
  const int s = __builtin_clzll(Q.back());
  std::vector<limb> qn(n), g(n + 1, 0), t(n + pn + 1, 0), plain(n);
  for (size_t i = n - 1; i > 0; --i) qn[i] = (Q[i] << s) | (s ? Q[i - 1] >> (64 - s) : 0);
  qn[0] = Q[0] << s;
  // g = g0 << s (g0 < Q, so it fits in n limbs)
  for (size_t i = 0; i < n; ++i) {
    const limb lo = i < g0.size() ? g0[i] : 0, below = (i > 0 && i - 1 < g0.size()) ? g0[i - 1] : 0;
    g[i] = (lo << s) | (s && i > 0 ? below >> (64 - s) : 0);
  }
  const limb vtop = qn[n - 1], vsec = n > 1 ? qn[n - 2] : 0;
  sum->clear();
  for (int32_t i = 0; i < mp; ++i) {
    // output G_i = g >> s
    for (size_t l = 0; l < n; ++l) plain[l] = (g[l] >> s) | (s && l + 1 < n ? g[l + 1] << (64 - s) : 0);
    Nat gi(plain.begin(), plain.end());
    big::trim(gi);
    for (int64_t w = 0; w < LG; ++w) {
      const size_t l = (size_t)w / 2;
      out[(size_t)i * GS + kGPad + w] = l < n ? (uint32_t)(plain[l] >> (32 * (w & 1))) : 0u;
    }
    big::add_in(*sum, gi);
    if (i + 1 == mp) break;
    // t = g P (n + pn limbs), then t mod qn -> g
    std::fill(t.begin(), t.end(), 0);
    for (size_t a = 0; a < pn; ++a) {
      limb carry = 0;
      for (size_t b = 0; b < n; ++b) {
        const u128 pr = (u128)P[a] * g[b] + t[a + b] + carry;
        t[a + b] = (limb)pr;
        carry = (limb)(pr >> 64);
      }
      t[a + n] = carry;
    }
    for (ptrdiff_t j = (ptrdiff_t)pn; j >= 0; --j) {
      if (j + n >= t.size()) continue;
      const u128 num = ((u128)t[j + n] << 64) | t[j + n - 1];
      u128 qhat = num / vtop, rhat = num % vtop;
      while ((qhat >> 64) != 0 || (n > 1 && qhat * vsec > ((rhat << 64) | t[j + n - 2]))) {
        qhat -= 1;
        rhat += vtop;
        if ((rhat >> 64) != 0) break;
      }
      if (qhat == 0) continue;
      limb borrow = 0, carry = 0;
      const limb qh = (limb)qhat;
      for (size_t b = 0; b < n; ++b) {
        const u128 pr = (u128)qh * qn[b] + carry;
        carry = (limb)(pr >> 64);
        const limb pl = (limb)pr, x = t[b + j];
        const limb t1 = x - pl, b1 = x < pl;
        const limb t2 = t1 - borrow, b2 = t1 < borrow;
        t[b + j] = t2;
        borrow = b1 | b2;
      }
      const limb x = t[j + n];
      const limb t1 = x - carry, b1 = x < carry;
      const limb t2 = t1 - borrow, b2 = t1 < borrow;
      t[j + n] = t2;
      if (b1 | b2) {  // went negative: add back once
        limb c = 0;
        for (size_t b = 0; b < n; ++b) {
          const u128 sm = (u128)t[b + j] + qn[b] + c;
          t[b + j] = (limb)sm;
          c = (limb)(sm >> 64);
        }
        t[j + n] += c;
      }
    }
    for (size_t l = 0; l < n; ++l) g[l] = t[l];
    g[n] = 0;
  }
}

// The digit-independent part of the device reconstruction: P'^m, Q = P'^m',
// the reciprocal and word images of Q, sizes and offsets.  Built on the host
// while the lift runs.
struct ReconPlan {
  int64_t n = 0, c = 0, nc = 0, num_bits = 0, den_bits = 0;
  int32_t m = 0, mp = 0;
  PrimeSet ps;
  Nat M, Mhalf, Mhalf1, Q;
  std::vector<Nat> ppow;  // P'^k, k = 0 .. max(mp, m / 2)
  AssemblePlan ap;
  int64_t LG = 0, W = 0;
  size_t oG = 0, oC = 0, oM = 0, oN = 0, oK = 0, total = 0;
  std::vector<uint32_t> hC, hM;
  int dyn = 0;
};

void recon_plan_free(ReconPlan* p) { delete p; }

es_status recon_device_prepare(int64_t n, int64_t c, int32_t m, int32_t mp, const uint8_t* good, int64_t num_bits,
                               int64_t den_bits, const Stats& stats, ReconPlan** out) {
  *out = nullptr;
  std::unique_ptr<ReconPlan> rp(new (std::nothrow) ReconPlan);
  if (!rp) return ES_ERR_NOMEM;
  ReconPlan& R = *rp;
  R.n = n;
  R.c = c;
  R.nc = n * c;
  R.m = m;
  R.mp = mp;
  R.num_bits = num_bits;
  R.den_bits = den_bits;
  R.ps = make_prime_set(good);
  if (R.ps.E == 0) return ES_ERR_ARG;
  R.M = pow_nat(R.ps.P, m);
  power_table(R.ps, std::max(mp, m / 2 + 1), &R.ppow);
  assemble_plan_init(R.ps, m, &R.ap, &R.ppow);
  if (big::le_pow2(R.M, (size_t)(num_bits + den_bits + 1))) return ES_ERR_INTERNAL;
  R.Mhalf = big::shr(big::sub(R.M, big::from_u64(1)), 1);
  R.Mhalf1 = big::add(R.Mhalf, big::from_u64(1));
  // exact check of the low-digit certificate's modulus
  R.Q = pow_nat(R.ps.P, mp);
  {
    const int64_t na = u64_bitlen((uint64_t)n * stats.max_abs_a);
    const int64_t need = std::max(num_bits + na, den_bits + u64_bitlen(stats.max_abs_b)) + 2;
    if (big::le_pow2(R.Q, (size_t)need)) return ES_ERR_INTERNAL;
  }
  const Nat& Q = R.Q;
  const int64_t LG = (int64_t)((big::bitlen(Q) + 31) / 32);
  const int64_t W0 = (num_bits + 2 + 63) / 64, W1 = (den_bits + 1 + 63) / 64;
  R.LG = LG;
  R.W = W0 > W1 ? W0 : W1;
  Layout L;
  R.oG = L.add((size_t)mp * g_stride(LG) * 4);
  R.oC = L.add((size_t)LG * 4 * 3);
  R.oM = L.add(kMuWords * 4 + kDigitWords * 4);
  R.oN = L.add((size_t)R.nc * R.W * 8);
  R.oK = L.add((size_t)R.nc);
  R.total = L.total;
  R.hC.assign((size_t)LG * 3, 0);
  R.hM.assign(kMuWords + kDigitWords, 0);
  const Nat Qhalf = big::shr(big::sub(Q, big::from_u64(1)), 1);
  to_words(Q, LG, R.hC.data() + LG);
  to_words(Qhalf, LG, R.hC.data() + 2 * LG);
  Nat mu;
  big::divmod(big::shl(big::from_u64(1), (size_t)(32 * (LG - 1 + kMuWords))), Q, &mu, nullptr);
  if ((int64_t)((big::bitlen(mu) + 31) / 32) > kMuWords) return ES_ERR_INTERNAL;
  to_words(mu, kMuWords, R.hM.data());
  to_words(R.ps.half, kDigitWords, R.hM.data() + kMuWords);
  R.dyn = (int)((3 * (LG + kZExtra + 1)) * 4 + (LG + kZExtra + 1) * 4 + (size_t)mp * kDigitWords * 4);
  *out = rp.release();
  return ES_OK;
}

es_status reconstruct_device(ReconPlan* plan, const uint64_t* D_dev, int threads, char* scratch,
                             size_t scratch_bytes, void* stream, Solution* out) {
  cudaStream_t st = (cudaStream_t)stream;
  const ReconPlan& R = *plan;
  const int64_t n = R.n, c = R.c, nc = R.nc, num_bits = R.num_bits, den_bits = R.den_bits;
  const int32_t m = R.m, mp = R.mp;
  const PrimeSet& ps = R.ps;
  const Nat &M = R.M, &Mhalf = R.Mhalf, &Mhalf1 = R.Mhalf1, &Q = R.Q;
  const int hw_threads = threads > 0 ? threads : std::max(1, (int)std::thread::hardware_concurrency());
  // components' full digits -> residues mod M -> denominators (host threads)
  auto denominators = [&](const std::vector<int64_t>& ks, std::vector<Nat>* dens) -> es_status {
    std::vector<uint64_t> hd(ks.size() * (size_t)m * kDigitLimbs);
    for (size_t t = 0; t < ks.size(); ++t)
      ES_CHECK(cuda_status(cudaMemcpy2DAsync(hd.data() + t * (size_t)m * kDigitLimbs, kDigitLimbs * 8,
                                             D_dev + (size_t)ks[t] * kDigitLimbs, (size_t)nc * kDigitLimbs * 8,
                                             kDigitLimbs * 8, (size_t)m, cudaMemcpyDeviceToHost, st),
                           "sample digits D2H"));
    ES_CHECK(cuda_status(cudaStreamSynchronize(st), "sample digits sync"));
    dens->assign(ks.size(), Nat{});
    std::atomic<int> fail(0);
    parallel_for((int64_t)ks.size(), hw_threads, [&](int64_t t) {
      const Nat u = shifted_to_residue(
          assemble_shifted_dc(ps, R.ap, hd.data() + (size_t)t * m * kDigitLimbs, kDigitLimbs), Mhalf, Mhalf1);
      if (!component_denominator(M, u, num_bits, den_bits, &(*dens)[(size_t)t])) fail = 1;
    });
    return fail ? ES_ERR_INTERNAL : ES_OK;
  };
  const int64_t per_round = sample_count(c, hw_threads);
  const std::vector<int64_t> sk = sample_components(n, c, per_round);
  std::vector<Nat> sden;
  ES_CHECK(denominators(sk, &sden));
  Nat d = big::from_u64(1);
  for (auto& v : sden) lcm_in(d, v);

  // device constants that do not depend on d
  const int64_t LG = R.LG, W = R.W;
  const size_t oG = R.oG, oC = R.oC, oM = R.oM, oN = R.oN, oK = R.oK;
  if (R.total > scratch_bytes) return ES_ERR_INTERNAL;
  std::vector<uint32_t> hC = R.hC;
  ES_CHECK(cuda_status(cudaMemcpyAsync(scratch + oM, R.hM.data(), R.hM.size() * 4, cudaMemcpyHostToDevice, st),
                       "recon constants H2D"));
  const int dyn = R.dyn;
  if (dyn > 48 * 1024)
    ES_CHECK(cuda_status(cudaFuncSetAttribute(k_recon_numerators, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn),
                         "recon smem attribute"));
  out->n = n;
  out->c = c;
  out->limbs = W;
  out->num.resize((size_t)(nc * W));
  // A page-locked result buffer is written by the kernel directly.  A
  // pageable one is filled before the device copy: the fill touches its fresh
  // pages far faster than a copy into untouched pageable memory would.
  uint64_t* Nout = reinterpret_cast<uint64_t*>(scratch + oN);
  bool direct = false;
  if (out->num.pinned()) {
    void* dp = nullptr;
    if (cudaHostGetDevicePointer(&dp, out->num.data(), 0) == cudaSuccess) {
      Nout = static_cast<uint64_t*>(dp);
      direct = true;
    } else {
      cudaGetLastError();
    }
  }
  if (!direct) std::memset(out->num.data(), 0, out->num.size() * 8);
  std::vector<uint8_t> okh((size_t)nc);
  const int64_t GS = g_stride(LG);
  std::vector<uint32_t> hG((size_t)mp * GS, 0u);
  for (int round = 0;; ++round) {
    if (round > 64) return ES_ERR_INTERNAL;
    // G_i = d P'^i mod Q, OFF = Q - ((P'-1)/2 sum_i G_i mod Q).  The chain is
    // cut into segments run on host threads: since Q = P'^mp, a segment's
    // first term is G_i0 = (d mod P'^(mp - i0)) P'^i0, below Q already.
    Nat sum, rem;
    const int nseg = std::max(1, std::min(mp / 4, hw_threads));
    std::vector<Nat> ssum((size_t)nseg);
    parallel_for(nseg, nseg, [&](int64_t t) {
      const int32_t i0 = (int32_t)(t * mp / nseg), i1 = (int32_t)((t + 1) * mp / nseg);
      Nat g;
      if (i0 == 0) {
        big::divmod(d, Q, nullptr, &g);
      } else {
        Nat low;
        big::divmod(d, R.ppow[(size_t)(mp - i0)], nullptr, &low);
        g = big::mul(low, R.ppow[(size_t)i0]);
      }
      g_chain(Q, ps.P, g, i1 - i0, LG, GS, hG.data() + (size_t)i0 * GS, &ssum[(size_t)t]);
    });
    for (auto& v : ssum) big::add_in(sum, v);
    big::divmod(big::mul(sum, ps.half), Q, nullptr, &rem);
    const Nat off = rem.empty() ? Nat{} : big::sub(Q, rem);
    to_words(off, LG, hC.data());
    ES_CHECK(cuda_status(cudaMemcpyAsync(scratch + oG, hG.data(), hG.size() * 4, cudaMemcpyHostToDevice, st),
                         "recon G H2D"));
    ES_CHECK(cuda_status(cudaMemcpyAsync(scratch + oC, hC.data(), hC.size() * 4, cudaMemcpyHostToDevice, st),
                         "recon Q H2D"));
    RParams rp;
    rp.D = reinterpret_cast<const uint32_t*>(D_dev);
    rp.nc = nc;
    rp.mp = mp;
    rp.LG = (int)LG;
    rp.G = reinterpret_cast<const uint32_t*>(scratch + oG);
    rp.GS = GS;
    rp.OFF = reinterpret_cast<const uint32_t*>(scratch + oC);
    rp.Q = rp.OFF + LG;
    rp.Qhalf = rp.OFF + 2 * LG;
    rp.MU = reinterpret_cast<const uint32_t*>(scratch + oM);
    rp.H12 = rp.MU + kMuWords;
    rp.nb = num_bits;
    rp.W = (int)W;
    rp.N = Nout;
    rp.ok = reinterpret_cast<uint8_t*>(scratch + oK);
    k_recon_numerators<<<(unsigned)nc, 256, dyn, st>>>(rp);
    count_launch();
    ES_CHECK(cuda_status(cudaGetLastError(), "k_recon_numerators"));
    ES_CHECK(cuda_status(cudaMemcpyAsync(okh.data(), rp.ok, (size_t)nc, cudaMemcpyDeviceToHost, st), "ok D2H"));
    if (!direct)
      ES_CHECK(cuda_status(cudaMemcpyAsync(out->num.data(), rp.N, (size_t)nc * W * 8, cudaMemcpyDeviceToHost, st),
                           "numerators D2H"));
    ES_CHECK(cuda_status(cudaStreamSynchronize(st), "recon sync"));
    std::vector<int64_t> failed;
    for (int64_t k = 0; k < nc; ++k)
      if (!okh[(size_t)k]) failed.push_back(k);
    failed = first_failure_per_column(failed, c, per_round);
    if (failed.empty()) break;
    const Nat before = d;
    std::vector<Nat> fden;
    ES_CHECK(denominators(failed, &fden));
    for (auto& v : fden) lcm_in(d, v);
    if (big::cmp(before, d) == 0) return ES_ERR_INTERNAL;
  }
  if (!big::le_pow2(d, (size_t)den_bits)) return ES_ERR_INTERNAL;
  out->den.assign((size_t)W, 0);
  to_limbs(d, false, W, out->den.data());
  out->primes_used = ps.E;
  out->m = m;
  return ES_OK;
}

}  // namespace es
