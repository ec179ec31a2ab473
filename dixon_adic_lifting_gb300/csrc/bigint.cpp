// Host arbitrary-precision naturals for the reconstruction stage.
#include "bigint.h"

#include <algorithm>
#include <cstring>

namespace es {
namespace big {

using u128 = unsigned __int128;

void trim(Nat& a) {
  while (!a.empty() && a.back() == 0) a.pop_back();
}
bool is_zero(const Nat& a) { return a.empty(); }
int cmp(const Nat& a, const Nat& b) {
  if (a.size() != b.size()) return a.size() < b.size() ? -1 : 1;
  for (size_t i = a.size(); i-- > 0;)
    if (a[i] != b[i]) return a[i] < b[i] ? -1 : 1;
  return 0;
}
size_t bitlen(const Nat& a) {
  return a.empty() ? 0 : 64 * (a.size() - 1) + (64 - (size_t)__builtin_clzll(a.back()));
}
Nat from_u64(uint64_t v) { return v ? Nat{v} : Nat{}; }

bool le_pow2(const Nat& a, size_t k) {
  size_t bl = bitlen(a);
  if (bl <= k) return true;
  if (bl > k + 1) return false;
  // bl == k + 1: a <= 2^k iff a == 2^k
  size_t w = k / 64;
  if (a[w] != (limb(1) << (k % 64))) return false;
  for (size_t i = 0; i < w; ++i)
    if (a[i]) return false;
  return true;
}

void add_in(Nat& a, const Nat& b) {
  if (a.size() < b.size()) a.resize(b.size(), 0);
  limb carry = 0;
  for (size_t i = 0; i < b.size(); ++i) {
    u128 s = (u128)a[i] + b[i] + carry;
    a[i] = (limb)s;
    carry = (limb)(s >> 64);
  }
  for (size_t i = b.size(); carry && i < a.size(); ++i) {
    a[i] += 1;
    carry = (a[i] == 0);
  }
  if (carry) a.push_back(1);
}
Nat add(const Nat& a, const Nat& b) {
  Nat r = a;
  add_in(r, b);
  return r;
}

void sub_in(Nat& a, const Nat& b) {
  limb borrow = 0;
  for (size_t i = 0; i < b.size(); ++i) {
    limb x = a[i], y = b[i];
    limb t1 = x - y, b1 = x < y;
    limb t2 = t1 - borrow, b2 = t1 < borrow;
    a[i] = t2;
    borrow = b1 | b2;
  }
  for (size_t i = b.size(); borrow && i < a.size(); ++i) {
    borrow = (a[i] == 0);
    a[i] -= 1;
  }
  trim(a);
}
Nat sub(const Nat& a, const Nat& b) {
  Nat r = a;
  sub_in(r, b);
  return r;
}

// r[0 .. an+bn) = a * b (r zeroed by the caller)
static void mul_school(limb* r, const limb* a, size_t an, const limb* b, size_t bn) {
  for (size_t i = 0; i < an; ++i) {
    limb ai = a[i], carry = 0;
    for (size_t j = 0; j < bn; ++j) {
      u128 t = (u128)ai * b[j] + r[i + j] + carry;
      r[i + j] = (limb)t;
      carry = (limb)(t >> 64);
    }
    r[i + bn] = carry;
  }
}

static limb add_into(limb* r, size_t rn, const limb* a, size_t an) {  // r += a, returns carry out of rn
  limb carry = 0;
  size_t i = 0;
  for (; i < an; ++i) {
    u128 s = (u128)r[i] + a[i] + carry;
    r[i] = (limb)s;
    carry = (limb)(s >> 64);
  }
  for (; carry && i < rn; ++i) {
    r[i] += 1;
    carry = (r[i] == 0);
  }
  return carry;
}
static void sub_into(limb* r, size_t rn, const limb* a, size_t an) {  // r -= a (r >= a)
  limb borrow = 0;
  size_t i = 0;
  for (; i < an; ++i) {
    limb x = r[i], y = a[i];
    limb t1 = x - y, b1 = x < y;
    limb t2 = t1 - borrow, b2 = t1 < borrow;
    r[i] = t2;
    borrow = b1 | b2;
  }
  for (; borrow && i < rn; ++i) {
    borrow = (r[i] == 0);
    r[i] -= 1;
  }
}

constexpr size_t kKaraThreshold = 40;

// scratch limbs kara() needs for size n
static size_t kara_scratch(size_t n) {
  size_t total = 0;
  while (n >= kKaraThreshold) {
    const size_t hh = n - n / 2;
    total += 4 * (hh + 1);
    n = hh + 1;
  }
  return total;
}

// r[0 .. 2n) = a[0..n) * b[0..n); ws holds kara_scratch(n) limbs.  The two
// half products go straight into r; the middle one and the half sums use ws.
static void kara(limb* r, const limb* a, const limb* b, size_t n, limb* ws) {
  if (n < kKaraThreshold) {
    std::fill(r, r + 2 * n, 0);
    mul_school(r, a, n, b, n);
    return;
  }
  const size_t h = n / 2, hh = n - h;
  kara(r, a, b, h, ws);
  kara(r + 2 * h, a + h, b + h, hh, ws);
  limb* sa = ws;
  limb* sb = sa + (hh + 1);
  limb* z1 = sb + (hh + 1);
  limb* next = z1 + 2 * (hh + 1);
  std::copy(a + h, a + n, sa);
  std::copy(b + h, b + n, sb);
  sa[hh] = add_into(sa, hh, a, h);
  sb[hh] = add_into(sb, hh, b, h);
  kara(z1, sa, sb, hh + 1, next);
  sub_into(z1, 2 * (hh + 1), r, 2 * h);
  sub_into(z1, 2 * (hh + 1), r + 2 * h, 2 * hh);
  size_t z1n = 2 * (hh + 1);
  while (z1n && z1[z1n - 1] == 0) --z1n;
  add_into(r + h, 2 * n - h, z1, z1n);
}

Nat mul(const Nat& a, const Nat& b) {
  if (a.empty() || b.empty()) return {};
  const Nat& x = a.size() <= b.size() ? a : b;
  const Nat& y = a.size() <= b.size() ? b : a;
  size_t n = x.size(), m = y.size();
  Nat r(n + m, 0);
  if (n < kKaraThreshold) {
    mul_school(r.data(), x.data(), n, y.data(), m);
  } else {
    std::vector<limb> t(2 * n), ws(kara_scratch(n));
    for (size_t off = 0; off < m; off += n) {
      size_t len = std::min(n, m - off);
      if (len == n) {
        kara(t.data(), x.data(), y.data() + off, n, ws.data());
        add_into(r.data() + off, n + m - off, t.data(), 2 * n);
      } else {
        Nat part(y.begin() + off, y.begin() + off + len), xx = x;
        trim(part);
        Nat p = mul(xx, part);
        add_into(r.data() + off, n + m - off, p.data(), p.size());
      }
    }
  }
  trim(r);
  return r;
}

Nat mul_small(const Nat& a, limb s) {
  if (a.empty() || s == 0) return {};
  Nat r(a.size() + 1);
  limb carry = 0;
  for (size_t i = 0; i < a.size(); ++i) {
    u128 t = (u128)a[i] * s + carry;
    r[i] = (limb)t;
    carry = (limb)(t >> 64);
  }
  r[a.size()] = carry;
  trim(r);
  return r;
}

void mul_small_add_in(Nat& a, const limb* s, int slen, const limb* addv, int alen) {
  size_t an = a.size();
  Nat r(an + slen + 1, 0);
  if (an) mul_school(r.data(), a.data(), an, s, (size_t)slen);
  add_into(r.data(), r.size(), addv, (size_t)alen);
  trim(r);
  a.swap(r);
}

Nat shl(const Nat& a, size_t bits) {
  if (a.empty()) return {};
  size_t w = bits / 64, b = bits % 64;
  Nat r(a.size() + w + 1, 0);
  for (size_t i = 0; i < a.size(); ++i) {
    r[i + w] |= a[i] << b;
    if (b) r[i + w + 1] |= a[i] >> (64 - b);
  }
  trim(r);
  return r;
}

Nat shr(const Nat& a, size_t bits) {
  size_t w = bits / 64, b = bits % 64;
  if (w >= a.size()) return {};
  Nat r(a.size() - w, 0);
  for (size_t i = 0; i < r.size(); ++i) {
    r[i] = a[i + w] >> b;
    if (b && i + w + 1 < a.size()) r[i] |= a[i + w + 1] << (64 - b);
  }
  trim(r);
  return r;
}

// Knuth, TAOCP vol. 2, 4.3.1, Algorithm D, with 64-bit limbs.
void divmod(const Nat& u, const Nat& v, Nat* q, Nat* r) {
  const size_t n = v.size(), mlen = u.size();
  if (cmp(u, v) < 0) {
    if (q) q->clear();
    if (r) *r = u;
    return;
  }
  if (n == 1) {
    const limb d = v[0];
    Nat qq(mlen);
    u128 rem = 0;
    for (size_t i = mlen; i-- > 0;) {
      u128 cur = (rem << 64) | u[i];
      qq[i] = (limb)(cur / d);
      rem = cur % d;
    }
    trim(qq);
    if (q) q->swap(qq);
    if (r) *r = from_u64((limb)rem);
    return;
  }
  const int s = __builtin_clzll(v.back());
  Nat vn(n), un(mlen + 1);
  for (size_t i = n - 1; i > 0; --i) vn[i] = (v[i] << s) | (s ? v[i - 1] >> (64 - s) : 0);
  vn[0] = v[0] << s;
  un[mlen] = s ? u[mlen - 1] >> (64 - s) : 0;
  for (size_t i = mlen - 1; i > 0; --i) un[i] = (u[i] << s) | (s ? u[i - 1] >> (64 - s) : 0);
  un[0] = u[0] << s;
  Nat qq(mlen - n + 1, 0);
  const limb vtop = vn[n - 1], vsec = vn[n - 2];
  for (ptrdiff_t j = (ptrdiff_t)(mlen - n); j >= 0; --j) {
    u128 num = ((u128)un[j + n] << 64) | un[j + n - 1];
    u128 qhat = num / vtop, rhat = num % vtop;
    while ((qhat >> 64) != 0 || qhat * vsec > ((rhat << 64) | un[j + n - 2])) {
      qhat -= 1;
      rhat += vtop;
      if ((rhat >> 64) != 0) break;
    }
    limb borrow = 0, carry = 0;
    const limb qh = (limb)qhat;
    for (size_t i = 0; i < n; ++i) {
      u128 p = (u128)qh * vn[i] + carry;
      carry = (limb)(p >> 64);
      limb pl = (limb)p, x = un[i + j];
      limb t1 = x - pl, b1 = x < pl;
      limb t2 = t1 - borrow, b2 = t1 < borrow;
      un[i + j] = t2;
      borrow = b1 | b2;
    }
    limb x = un[j + n];
    limb t1 = x - carry, b1 = x < carry;
    limb t2 = t1 - borrow, b2 = t1 < borrow;
    un[j + n] = t2;
    limb qfinal = qh;
    if (b1 | b2) {  // went negative: add back once
      qfinal -= 1;
      limb c = 0;
      for (size_t i = 0; i < n; ++i) {
        u128 sum = (u128)un[i + j] + vn[i] + c;
        un[i + j] = (limb)sum;
        c = (limb)(sum >> 64);
      }
      un[j + n] += c;
    }
    qq[(size_t)j] = qfinal;
  }
  if (q) {
    trim(qq);
    q->swap(qq);
  }
  if (r) {
    Nat rr(n);
    for (size_t i = 0; i < n; ++i) rr[i] = (un[i] >> s) | (s ? un[i + 1] << (64 - s) : 0);
    trim(rr);
    r->swap(rr);
  }
}

// ------------------------------------------------------------ Lehmer
static uint64_t bits_at(const Nat& x, size_t sh) {  // floor(x / 2^sh) mod 2^64
  size_t w = sh / 64, b = sh % 64;
  uint64_t lo = w < x.size() ? x[w] : 0, hi = w + 1 < x.size() ? x[w + 1] : 0;
  return b ? (lo >> b) | (hi << (64 - b)) : lo;
}
static u128 bits128_at(const Nat& x, size_t sh) {  // floor(x / 2^sh) mod 2^128
  return (u128)bits_at(x, sh) | ((u128)bits_at(x, sh + 64) << 64);
}

static inline limb uabs(int64_t v) { return v < 0 ? (limb)(-v) : (limb)v; }

// Both rows of a Lehmer cofactor matrix in one pass:
//   o0 = A x + B y,  o1 = C x + D y   (|A|, |B|, |C|, |D| < 2^62, results >= 0)
// Each product |coef| * limb is below 2^126, so one signed 128-bit accumulator
// per output holds the limb sum and a signed carry; the signs are template
// parameters so the loop has no branches.
template <bool NA, bool NB, bool NC, bool ND>
static void lin2x2_pass(limb* o0, limb* o1, const limb* x, size_t xn, const limb* y, size_t yn, size_t len, limb a,
                        limb b, limb c, limb d) {
  __int128 c0 = 0, c1 = 0;
  for (size_t i = 0; i < len; ++i) {
    const limb xi = i < xn ? x[i] : 0, yi = i < yn ? y[i] : 0;
    const __int128 pa = (__int128)((u128)a * xi), pb = (__int128)((u128)b * yi);
    const __int128 pc = (__int128)((u128)c * xi), pd = (__int128)((u128)d * yi);
    const __int128 t0 = c0 + (NA ? -pa : pa) + (NB ? -pb : pb);
    const __int128 t1 = c1 + (NC ? -pc : pc) + (ND ? -pd : pd);
    o0[i] = (limb)t0;
    o1[i] = (limb)t1;
    c0 = t0 >> 64;
    c1 = t1 >> 64;
  }
  o0[len] = (limb)c0;
  o1[len] = (limb)c1;
}

static void comb2(Nat& o0, Nat& o1, int64_t A, int64_t B, int64_t C, int64_t D, const Nat& x, const Nat& y) {
  const size_t len = std::max(x.size(), y.size());
  o0.resize(len + 1);
  o1.resize(len + 1);
  const int code = (A < 0) << 3 | (B < 0) << 2 | (C < 0) << 1 | (D < 0);
  const limb a = uabs(A), b = uabs(B), c = uabs(C), d = uabs(D);
#define ES_LIN2X2(k)                                                                                              \
  case k:                                                                                                         \
    lin2x2_pass<(k >> 3) & 1, (k >> 2) & 1, (k >> 1) & 1, k & 1>(o0.data(), o1.data(), x.data(), x.size(),       \
                                                                  y.data(), y.size(), len, a, b, c, d);           \
    break;
  switch (code) {
    ES_LIN2X2(0) ES_LIN2X2(1) ES_LIN2X2(2) ES_LIN2X2(3) ES_LIN2X2(4) ES_LIN2X2(5) ES_LIN2X2(6) ES_LIN2X2(7)
    ES_LIN2X2(8) ES_LIN2X2(9) ES_LIN2X2(10) ES_LIN2X2(11) ES_LIN2X2(12) ES_LIN2X2(13) ES_LIN2X2(14) ES_LIN2X2(15)
  }
#undef ES_LIN2X2
  trim(o0);
  trim(o1);
}

// One Lehmer batch: the quotient steps simulated on the leading bits a >= b
// of (r0, r1) (at most 126 bits, same shift), Knuth's Algorithm L with two
// quotient checks, cofactors kept below 2^62 in magnitude, and no step whose
// simulated remainder falls below `stop`.  The batch maps (r0, r1) to
// (A r0 + B r1, C r0 + D r1); B == 0 means no step was certain.
struct LMat {
  int64_t A = 1, B = 0, C = 0, D = 1;
  size_t k = 0;  // quotient steps
};
static LMat lehmer_sim(__int128 a, __int128 b, __int128 stop) {
  const __int128 kCap = (__int128)1 << 62;
  LMat M;
  int64_t A = 1, B = 0, C = 0, D = 1;
  size_t k = 0;
  for (;;) {
    const __int128 bc = b + C, bd = b + D;
    if (bc <= 0 || bd <= 0) break;
    const __int128 ac = a + A, ad = a + B;
    if (ac < bc) break;
    // q = floor(ac / bc), small quotients by subtraction
    __int128 q = 1, rem = ac - bc;
    while (rem >= bc && q < 4) {
      rem -= bc;
      ++q;
    }
    if (rem >= bc) q = (__int128)((unsigned __int128)ac / (unsigned __int128)bc);
    // second check: floor(ad / bd) == q
    if (q >= kCap) break;
    const __int128 lo = q * bd;
    if (ad < lo || ad - lo >= bd) break;
    const __int128 nC = (__int128)A - q * C, nD = (__int128)B - q * D;
    if (nC >= kCap || -nC >= kCap || nD >= kCap || -nD >= kCap) break;
    const __int128 t = a - q * b;
    if (t < stop) break;
    A = C;
    C = (int64_t)nC;
    B = D;
    D = (int64_t)nD;
    a = b;
    b = t;
    ++k;
  }
  M.A = A, M.B = B, M.C = C, M.D = D, M.k = k;
  return M;
}

// Shared loop: r0 >= r1; stops when r1 <= 2^nbits (or r1 == 0 when nbits < 0).
// Lehmer batches (lehmer_sim), applied to the full numbers in fused passes.
// A batch never crosses the stopping point: with r = 2^sh a0 + alpha,
// 2^sh b0 + beta (0 <= alpha, beta < 2^sh) and cofactors |A|, |B| < 2^62 of
// opposite signs, the true remainder A r0 + B r1 differs from 2^sh times the
// simulated one, A a0 + B b0, by less than 2^(sh + 62); so a simulated
// remainder of at least 2^(nbits - sh) + 2^63 keeps the true one above
// 2^nbits.  Batches run until no certain step is left, then single
// division steps finish (a few near the stopping point).
static void euclid(Nat& r0, Nat& r1, Nat* T0, Nat* T1, size_t* steps, long nbits) {
  auto done = [&](const Nat& x) { return nbits < 0 ? x.empty() : le_pow2(x, (size_t)nbits); };
  Nat n0, n1, m0, m1;
  while (!done(r1)) {
    if (r1.size() >= 3) {
      const size_t bl0 = bitlen(r0);
      const size_t sh = bl0 > 126 ? bl0 - 126 : 0;
      __int128 stop = (__int128)1 << 63;
      if (nbits >= 0 && (size_t)nbits >= sh) {
        const size_t e = (size_t)nbits - sh;
        stop = e >= 126 ? ((__int128)1 << 126) : stop + ((__int128)1 << e);
      }
      const LMat L = lehmer_sim((__int128)bits128_at(r0, sh), (__int128)bits128_at(r1, sh), stop);
      const int64_t A = L.A, B = L.B, C = L.C, D = L.D;
      if (B != 0) {
        comb2(n0, n1, A, B, C, D, r0, r1);
        r0.swap(n0);
        r1.swap(n1);
        if (T0) {  // consecutive cofactors alternate in sign: the magnitudes add
          comb2(m0, m1, (int64_t)uabs(A), (int64_t)uabs(B), (int64_t)uabs(C), (int64_t)uabs(D), *T0, *T1);
          T0->swap(m0);
          T1->swap(m1);
        }
        *steps += L.k;
        continue;
      }
    }
    // one division step
    Nat q, rem;
    divmod(r0, r1, &q, &rem);
    r0.swap(r1);
    r1.swap(rem);
    if (T0) {
      Nat t = mul(q, *T1);
      add_in(t, *T0);
      T0->swap(*T1);
      T1->swap(t);
    }
    ++*steps;
  }
}

bool rational_reconstruct(const Nat& M, const Nat& u, size_t nbits, Nat* num, bool* num_neg, Nat* den) {
  Nat r0 = M, r1 = u, T0, T1 = from_u64(1);
  size_t steps = 0;
  euclid(r0, r1, &T0, &T1, &steps, (long)nbits);
  if (T1.empty()) return false;
  *num = r1;
  *num_neg = (steps & 1) && !r1.empty();
  *den = T1;
  return true;
}

Nat gcd(const Nat& a, const Nat& b) {
  Nat r0 = a, r1 = b;
  if (cmp(r0, r1) < 0) r0.swap(r1);
  size_t steps = 0;
  euclid(r0, r1, nullptr, nullptr, &steps, -1);
  return r0;
}

}  // namespace big
}  // namespace es
