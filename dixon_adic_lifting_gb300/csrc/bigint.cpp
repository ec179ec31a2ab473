// Host arbitrary-precision naturals for the reconstruction stage.
#include "bigint.h"

#include <algorithm>
#include <atomic>
#include <cstring>
#include <memory>
#include <thread>

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

// Both rows of a Lehmer cofactor matrix over limbs [lo, hi):
//   o0 = A x + B y,  o1 = C x + D y   (|A|, |B|, |C|, |D| < 2^62)
// with no carry coming in at lo; the carries out of limb hi - 1 are returned.
// Each product |coef| * limb is below 2^126, so one signed 128-bit accumulator
// per output holds the limb sum and a signed carry; the signs are template
// parameters so the loop has no branches.  Where both inputs have limbs, the
// range is cut in two halves that run as two independent carry chains side
// by side (the chain through the carries, not the multiplies, bounds one
// chain's speed); the lower half's carries are then added into the upper
// half, which rarely takes them past a limb or two.  In place (o0 == x,
// o1 == y) is allowed: every limb is read before it is written.
template <bool NA, bool NB, bool NC, bool ND>
static inline void lin2x2_limb(limb xi, limb yi, limb a, limb b, limb c, limb d, __int128& c0, __int128& c1,
                               limb* o0, limb* o1) {
  const __int128 pa = (__int128)((u128)a * xi), pb = (__int128)((u128)b * yi);
  const __int128 pc = (__int128)((u128)c * xi), pd = (__int128)((u128)d * yi);
  const __int128 t0 = c0 + (NA ? -pa : pa) + (NB ? -pb : pb);
  const __int128 t1 = c1 + (NC ? -pc : pc) + (ND ? -pd : pd);
  *o0 = (limb)t0;
  *o1 = (limb)t1;
  c0 = t0 >> 64;
  c1 = t1 >> 64;
}
static __int128 carry_into(limb* o, size_t from, size_t to, __int128 c) {  // o[from, to) += c; the carry out
  for (size_t k = from; k < to && c != 0; ++k) {
    const __int128 s = c + (__int128)o[k];
    o[k] = (limb)s;
    c = s >> 64;
  }
  return c;
}
template <bool NA, bool NB, bool NC, bool ND>
static void lin2x2_range(limb* o0, limb* o1, const limb* x, size_t xn, const limb* y, size_t yn, size_t lo,
                         size_t hi, limb a, limb b, limb c, limb d, __int128* cr0, __int128* cr1) {
  __int128 c0 = 0, c1 = 0;
  size_t i = lo;
  const size_t full = std::min(hi, std::min(xn, yn));
  if (full >= lo + 32) {
    const size_t half = (full - lo) / 2, mid = lo + half;
    __int128 e0 = 0, e1 = 0;
    for (size_t k = 0; k < half; ++k) {
      const limb xl = x[lo + k], yl = y[lo + k], xh = x[mid + k], yh = y[mid + k];
      lin2x2_limb<NA, NB, NC, ND>(xl, yl, a, b, c, d, c0, c1, o0 + lo + k, o1 + lo + k);
      lin2x2_limb<NA, NB, NC, ND>(xh, yh, a, b, c, d, e0, e1, o0 + mid + k, o1 + mid + k);
    }
    for (size_t k = mid + half; k < full; ++k) lin2x2_limb<NA, NB, NC, ND>(x[k], y[k], a, b, c, d, e0, e1, o0 + k, o1 + k);
    c0 = e0 + carry_into(o0, mid, full, c0);
    c1 = e1 + carry_into(o1, mid, full, c1);
    i = full;
  }
  for (; i < hi; ++i) {
    const limb xi = i < xn ? x[i] : 0, yi = i < yn ? y[i] : 0;
    lin2x2_limb<NA, NB, NC, ND>(xi, yi, a, b, c, d, c0, c1, o0 + i, o1 + i);
  }
  *cr0 = c0;
  *cr1 = c1;
}

static inline limb uabs(int64_t v) { return v < 0 ? (limb)(-v) : (limb)v; }
static int sign_code(int64_t A, int64_t B, int64_t C, int64_t D) {
  return (A < 0) << 3 | (B < 0) << 2 | (C < 0) << 1 | (D < 0);
}
static void comb2_range(int code, limb* o0, limb* o1, const limb* x, size_t xn, const limb* y, size_t yn, size_t lo,
                        size_t hi, limb a, limb b, limb c, limb d, __int128* cr0, __int128* cr1) {
#define ES_LIN2X2(k)                                                                                      \
  case k:                                                                                                 \
    lin2x2_range<(k >> 3) & 1, (k >> 2) & 1, (k >> 1) & 1, k & 1>(o0, o1, x, xn, y, yn, lo, hi, a, b, c, d, \
                                                                  cr0, cr1);                              \
    break;
  switch (code) {
    ES_LIN2X2(0) ES_LIN2X2(1) ES_LIN2X2(2) ES_LIN2X2(3) ES_LIN2X2(4) ES_LIN2X2(5) ES_LIN2X2(6) ES_LIN2X2(7)
    ES_LIN2X2(8) ES_LIN2X2(9) ES_LIN2X2(10) ES_LIN2X2(11) ES_LIN2X2(12) ES_LIN2X2(13) ES_LIN2X2(14) ES_LIN2X2(15)
  }
#undef ES_LIN2X2
}

// (o0, o1) = (A x + B y, C x + D y) for results known to be >= 0.
static void comb2(Nat& o0, Nat& o1, int64_t A, int64_t B, int64_t C, int64_t D, const Nat& x, const Nat& y) {
  const size_t len = std::max(x.size(), y.size());
  o0.resize(len + 1);
  o1.resize(len + 1);
  __int128 c0, c1;
  comb2_range(sign_code(A, B, C, D), o0.data(), o1.data(), x.data(), x.size(), y.data(), y.size(), 0, len, uabs(A),
              uabs(B), uabs(C), uabs(D), &c0, &c1);
  o0[len] = (limb)c0;
  o1[len] = (limb)c1;
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
// T0, T1 (optional) follow the magnitudes of the cofactors of the second
// number (r = s r0_in + t r1_in), S0, S1 (optional) those of the first; both
// alternate in sign from step to step.
static void euclid(Nat& r0, Nat& r1, Nat* T0, Nat* T1, size_t* steps, long nbits, Nat* S0 = nullptr,
                   Nat* S1 = nullptr) {
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
        if (S0) {
          comb2(m0, m1, (int64_t)uabs(A), (int64_t)uabs(B), (int64_t)uabs(C), (int64_t)uabs(D), *S0, *S1);
          S0->swap(m0);
          S1->swap(m1);
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
    if (S0) {
      Nat t = mul(q, *S1);
      add_in(t, *S0);
      S0->swap(*S1);
      S1->swap(t);
    }
    ++*steps;
  }
}

// ------------------------------------------------------------ cofactor pipe
// The Lehmer loop of rational_reconstruct can hand the cofactor updates to a
// second thread: every batch's matrix goes, in order, into a single-producer
// ring, and whoever claims the pipe first applies them to (T0, T1):
//   - a thread that calls cofactor_pipe_serve() (a pool task beside the run)
//     claims it and follows the ring until the run closes it;
//   - the run itself claims it whenever it needs the cofactors and nobody has
//     (a plain division step, a full ring, the end), and from then on applies
//     its batches directly; a late serve() then returns at once.
// So the run never waits for a thread that has not started, and a pool as
// narrow as one thread still finishes.  A division step with the pipe served
// waits for the ring to drain, then updates the cofactors itself.  (The
// remainder updates are split too, by the low-limb pipe below; a split that
// waits for the other thread at every batch did not pay: that handoff costs
// what the split saves.)
namespace {
inline void spin_wait(int& spins) {
  if (++spins > 512) std::this_thread::yield();
}
}  // namespace

struct CofactorPipe {
  struct Item {
    limb a, b, c, d;
  };
  static constexpr uint32_t kRing = 1024;
  static constexpr uint32_t kPublish = 4;
  enum : int { kFree = 0, kServed = 1, kOwned = 2 };
  Item ring[kRing];
  std::atomic<uint32_t> head{0}, tail{0};
  std::atomic<int> claim{kFree};
  std::atomic<bool> closed{false};
  uint32_t tail_seen = 0;  // the run's last look at tail
  uint32_t next = 0;       // the run's next ring slot (head trails it by under kPublish)
  Nat T0, T1{1};  // magnitudes of the cofactors of u in r0 and r1
  Nat m0, m1;

  void apply(const Item& it) {
    // consecutive cofactors alternate in sign: the magnitudes add
    comb2(m0, m1, (int64_t)it.a, (int64_t)it.b, (int64_t)it.c, (int64_t)it.d, T0, T1);
    T0.swap(m0);
    T1.swap(m1);
  }
  // the run's side: the cofactors are its own from here on
  void own() {
    int expect = kFree;
    if (claim.compare_exchange_strong(expect, kOwned, std::memory_order_acq_rel)) {
      for (uint32_t t = tail.load(std::memory_order_relaxed); t != next; ++t) apply(ring[t % kRing]);
      tail.store(next, std::memory_order_relaxed);
      head.store(next, std::memory_order_relaxed);
    }
  }
  void publish() {
    if (head.load(std::memory_order_relaxed) != next) head.store(next, std::memory_order_release);
  }
  // the run's side: every batch handed over so far is applied
  void sync() {
    if (claim.load(std::memory_order_acquire) == kFree) own();
    if (claim.load(std::memory_order_acquire) == kServed) {
      publish();
      int spins = 0;
      while (tail.load(std::memory_order_acquire) != next) spin_wait(spins);
    }
  }
  void push(limb a, limb b, limb c, limb d) {
    if (claim.load(std::memory_order_acquire) == kOwned) {
      apply(Item{a, b, c, d});
      return;
    }
    const uint32_t h = next;
    // the consumer's position is read only when the last one seen leaves no room
    if (h - tail_seen >= kRing) tail_seen = tail.load(std::memory_order_acquire);
    if (h - tail_seen >= kRing) {
      own();  // a full ring nobody serves: the run takes the work over
      if (claim.load(std::memory_order_acquire) == kOwned) {
        apply(Item{a, b, c, d});
        return;
      }
      publish();
      int spins = 0;
      while (h - tail.load(std::memory_order_acquire) >= kRing) spin_wait(spins);
    }
    ring[h % kRing] = Item{a, b, c, d};
    next = h + 1;
    // batches go out a few at a time: every store of head takes its cache
    // line away from the spinning server
    if (next - head.load(std::memory_order_relaxed) >= kPublish) head.store(next, std::memory_order_release);
  }
  void serve() {
    int expect = kFree;
    if (!claim.compare_exchange_strong(expect, kServed, std::memory_order_acq_rel)) return;
    uint32_t t = tail.load(std::memory_order_relaxed);
    for (;;) {
      int spins = 0;
      uint32_t h;
      while ((h = head.load(std::memory_order_acquire)) == t) {
        if (closed.load(std::memory_order_acquire) && head.load(std::memory_order_acquire) == t) return;
        spin_wait(spins);
      }
      for (; t != h; ++t) {
        apply(ring[t % kRing]);
        tail.store(t + 1, std::memory_order_release);
      }
    }
  }
};

CofactorPipe* cofactor_pipe_new() { return new (std::nothrow) CofactorPipe; }
void cofactor_pipe_free(CofactorPipe* p) { delete p; }
void cofactor_pipe_serve(CofactorPipe* p) {
  if (p) p->serve();
}
void cofactor_pipe_close(CofactorPipe* p) {
  if (p) p->closed.store(true, std::memory_order_release);
}

// ------------------------------------------------------------ low-limb pipe
// The remainder updates of the Lehmer loop split by limbs between the run and
// up to kLowSlots more threads.  At a round's start the run cuts both
// remainders at limb h and the part below into one range [lo_j, hi_j) per
// server: r = t 2^(64h) + sum_j l_j 2^(64 lo_j), 0 <= l_j < 2^(64(hi_j - lo_j)).
// The run keeps the high parts t (a copy) and updates them with each batch's
// matrix M as if nothing carried in from below; server j follows the same
// matrices over l_j in place, up to a ring's length behind, and keeps what
// carries out of its range as a small signed correction e_j (two's complement,
// at most kLowCorr limbs): a batch maps (l_j, e_j) to
// (M l_j mod 2^(64(hi_j - lo_j)), M e_j + floor(M l_j / 2^(64(hi_j - lo_j)))),
// so that throughout
//     r = t 2^(64h) + sum_j (l_j 2^(64 lo_j) + e_j 2^(64 hi_j)).
// Every |e_j| < 2^ebits, which grows by at most the bits of the batch's largest
// row sum plus one per batch, and the part below t is then below
// 2^(64h + ebits + 1) in magnitude; so as long as ebits + 3 <= sh' (the shift
// at which the run reads the leading 126 bits of t) the true leading parts
// differ from the simulated ones by less than 1/2, and a batch certified over
// the box [a0 - 1, a0 + 2] x [b0 - 1, b0 + 2] (lehmer_sim_wide) holds for the
// true remainders.  When that margin runs out (or no step is certain) the run
// waits for the servers, folds the corrections in from the bottom up, and
// starts the next round.  The run splits only while a server serves the pipe,
// and takes in servers that arrive late at the next round's start, so a pool
// narrower than planned changes nothing but the speed.
constexpr size_t kLowCorr = 64;        // limbs of a correction e_j
constexpr int kLowSlots = 4;            // servers one pipe takes
constexpr size_t kSplitMinLimbs = 160;  // shorter remainders stay on the run's thread

// As lehmer_sim, for leading parts known only to lie in (a - 1, a + 2) and
// (b - 1, b + 2).  Candidates come from plain quotient steps on the leading
// 64 bits of the current remainders (cofactors below 2^32 per level, at most
// three levels); a candidate is taken only when the composite matrix has
// alpha > beta > 0 at all four corners of the box [a - 1, a + 2] x
// [b - 1, b + 2], with alpha, beta its remainders: that makes its quotients
// the first ones of Euclid's algorithm at every point of the box (the
// continued fraction argument of the half-gcd below; alpha and beta are
// linear, so the corners decide), hence on the true remainders.  The longest
// such prefix of each level is kept; the stop condition is checked the same
// way.  Composite cofactors stay below 2^61 (row sums below 2^62), and every
// remainder at the base point fits in 127 bits (the steps only reduce them).
static LMat lehmer_sim_wide(__int128 a, __int128 b, __int128 stop) {
  const __int128 kMin = (__int128)1 << 66;
  const __int128 kCap = (__int128)1 << 61;
  const int64_t kLevelCap = (int64_t)1 << 32;
  constexpr int kSteps = 64;
  int64_t A = 1, B = 0, C = 0, D = 1;
  __int128 al = a, be = b;  // the composite's remainders at the base point
  size_t k = 0;
  for (int level = 0; level < 3; ++level) {
    if (be < kMin || al < be) break;
    const int sh = 64 - __builtin_clzll((uint64_t)(al >> 64));  // al >= 2^66: bitlen(al) - 64
    int64_t h[kSteps][4];
    int n = 0;
    {
      uint64_t x = (uint64_t)(al >> sh), y = (uint64_t)(be >> sh);
      int64_t a2 = 1, b2 = 0, c2 = 0, d2 = 1;
      while (n < kSteps && y >= ((uint64_t)1 << 34)) {
        uint64_t q = 1, r = x - y;
        if (r >= y) {
          r -= y;
          q = 2;
          if (r >= y) {
            r -= y;
            q = 3;
            if (r >= y) {
              q = x / y;
              r = x - q * y;
            }
          }
        }
        if (q >= (uint64_t)kLevelCap) break;
        const int64_t nc = a2 - (int64_t)q * c2, nd = b2 - (int64_t)q * d2;
        if (nc >= kLevelCap || -nc >= kLevelCap || nd >= kLevelCap || -nd >= kLevelCap) break;
        a2 = c2;
        b2 = d2;
        c2 = nc;
        d2 = nd;
        x = y;
        y = r;
        h[n][0] = a2, h[n][1] = b2, h[n][2] = c2, h[n][3] = d2;
        ++n;
      }
    }
    const int64_t alh = (int64_t)(al >> 64), beh = (int64_t)(be >> 64);
    const uint64_t all = (uint64_t)al, bel = (uint64_t)be;
    int got = -1;
    for (int j = n - 1; j >= 0 && got < 0; --j) {
      const int64_t a2 = h[j][0], b2 = h[j][1], c2 = h[j][2], d2 = h[j][3];
      const __int128 cA = (__int128)a2 * A + (__int128)b2 * C, cB = (__int128)a2 * B + (__int128)b2 * D;
      const __int128 cC = (__int128)c2 * A + (__int128)d2 * C, cD = (__int128)c2 * B + (__int128)d2 * D;
      if (cA >= kCap || -cA >= kCap || cB >= kCap || -cB >= kCap || cC >= kCap || -cC >= kCap || cD >= kCap ||
          -cD >= kCap)
        continue;
      // (a2 al + b2 be, c2 al + d2 be) with al, be split at 2^64: the high
      // parts nearly cancel, so no partial sum overflows
      const __int128 ra = ((__int128)a2 * alh + (__int128)b2 * beh) * ((__int128)1 << 64) +
                          ((__int128)a2 * (__int128)all + (__int128)b2 * (__int128)bel);
      const __int128 rb = ((__int128)c2 * alh + (__int128)d2 * beh) * ((__int128)1 << 64) +
                          ((__int128)c2 * (__int128)all + (__int128)d2 * (__int128)bel);
      bool ok = true;
      for (int c = 0; c < 4 && ok; ++c) {
        const int da = (c & 1) ? 2 : -1, db = (c & 2) ? 2 : -1;
        const __int128 x = ra + cA * da + cB * db, y = rb + cC * da + cD * db;
        ok = y > 0 && x > y && y >= stop;
      }
      if (!ok) continue;
      got = j;
      A = (int64_t)cA, B = (int64_t)cB, C = (int64_t)cC, D = (int64_t)cD;
      al = ra;
      be = rb;
      k += (size_t)j + 1;
    }
    if (got < 0) break;
  }
  LMat M;
  M.A = A, M.B = B, M.C = C, M.D = D, M.k = k;
  return M;
}

// x += c on a w-limb two's complement number (the result must fit).
static void add_carry_signed(limb* x, size_t w, __int128 c) {
  for (size_t i = 0; i < w && c != 0; ++i) {
    const __int128 s = c + (__int128)x[i];
    x[i] = (limb)s;
    c = s >> 64;
  }
}
// (x, y) <- (A x + B y + c0, C x + D y + c1) on w-limb two's complement numbers
// (in place; the results must fit): the unsigned limbs by comb2_range, the
// signed top limb apart, then the carries.
static void lin2x2_signed(limb* x, limb* y, size_t w, int64_t A, int64_t B, int64_t C, int64_t D, __int128 c0,
                          __int128 c1) {
  if (w == 0) return;
  __int128 h0 = 0, h1 = 0;
  if (w > 1)
    comb2_range(sign_code(A, B, C, D), x, y, x, w - 1, y, w - 1, 0, w - 1, uabs(A), uabs(B), uabs(C), uabs(D), &h0,
                &h1);
  const __int128 xt = (int64_t)x[w - 1], yt = (int64_t)y[w - 1];
  x[w - 1] = (limb)(h0 + (__int128)A * xt + (__int128)B * yt);
  y[w - 1] = (limb)(h1 + (__int128)C * xt + (__int128)D * yt);
  add_carry_signed(x, w, c0);
  add_carry_signed(y, w, c1);
}

struct LowPipe {
  struct Item {
    int64_t A, B, C, D;
    size_t w;  // limbs of the corrections that can be nonzero after this batch
  };
  static constexpr uint32_t kRing = 256;
  struct alignas(64) Slot {
    std::atomic<uint32_t> tail{0};
    std::atomic<bool> joined{false};
    // the round: set by the run while the slot is idle, published by the
    // release of the round's first item
    limb* x = nullptr;
    limb* y = nullptr;
    size_t lo = 0, hi = 0;
    size_t ew = 0;  // limbs of e in use (the ones above are its sign)
    limb e0[kLowCorr], e1[kLowCorr];

    void apply(const Item& it) {
      __int128 c0 = 0, c1 = 0;
      if (hi > lo)
        comb2_range(sign_code(it.A, it.B, it.C, it.D), x, y, x, hi, y, hi, lo, hi, uabs(it.A), uabs(it.B),
                    uabs(it.C), uabs(it.D), &c0, &c1);
      for (; ew < it.w; ++ew) {
        e0[ew] = ew && (e0[ew - 1] >> 63) ? ~(limb)0 : 0;
        e1[ew] = ew && (e1[ew - 1] >> 63) ? ~(limb)0 : 0;
      }
      lin2x2_signed(e0, e1, ew, it.A, it.B, it.C, it.D, c0, c1);
    }
  };
  Item ring[kRing];
  std::atomic<uint32_t> head{0};
  std::atomic<int> claimed{0};
  std::atomic<bool> closed{false};
  int joined = 0;           // the run's count of slots taken into rounds
  uint32_t tail_seen = 0;   // the run's last look at the slowest server
  uint32_t next = 0;        // the run's next ring slot (head trails it by under kPublish)
  static constexpr uint32_t kPublish = 4;
  Slot slot[kLowSlots];

  bool served() const { return claimed.load(std::memory_order_acquire) > 0; }
  // the run, between rounds: takes in the servers that have arrived
  int begin_round() {
    const int n = std::min(claimed.load(std::memory_order_acquire), kLowSlots);
    const uint32_t hd = next;  // every item so far is published and done
    for (; joined < n; ++joined) {
      slot[joined].tail.store(hd, std::memory_order_relaxed);
      slot[joined].joined.store(true, std::memory_order_release);
    }
    tail_seen = hd;  // every joined server has drained
    return joined;
  }
  uint32_t min_tail() const {
    uint32_t lag = 0;
    for (int j = 0; j < joined; ++j) lag = std::max(lag, next - slot[j].tail.load(std::memory_order_acquire));
    return next - lag;
  }
  void publish() {
    if (head.load(std::memory_order_relaxed) != next) head.store(next, std::memory_order_release);
  }
  void push(const LMat& L, size_t w) {
    int spins = 0;
    // the servers' positions are read only when the last ones seen leave no room
    while (next - tail_seen >= kRing) {
      publish();
      tail_seen = min_tail();
      if (next - tail_seen >= kRing) spin_wait(spins);
    }
    ring[next % kRing] = Item{L.A, L.B, L.C, L.D, w};
    ++next;
    // a few batches at a time: every store of head takes its cache line away
    // from the spinning servers
    if (next - head.load(std::memory_order_relaxed) >= kPublish) head.store(next, std::memory_order_release);
  }
  void drain() {
    publish();
    int spins = 0;
    while (min_tail() != next) spin_wait(spins);
  }
  void serve() {
    const int j = claimed.fetch_add(1, std::memory_order_acq_rel);
    if (j >= kLowSlots) return;
    Slot& s = slot[j];
    int spins = 0;
    while (!s.joined.load(std::memory_order_acquire)) {
      if (closed.load(std::memory_order_acquire)) return;
      spin_wait(spins);
    }
    uint32_t t = s.tail.load(std::memory_order_relaxed);
    for (;;) {
      spins = 0;
      uint32_t hd;
      while ((hd = head.load(std::memory_order_acquire)) == t) {
        if (closed.load(std::memory_order_acquire) && head.load(std::memory_order_acquire) == t) return;
        spin_wait(spins);
      }
      for (; t != hd; ++t) {
        s.apply(ring[t % kRing]);
        s.tail.store(t + 1, std::memory_order_release);
      }
    }
  }
};

LowPipe* low_pipe_new() { return new (std::nothrow) LowPipe; }
void low_pipe_free(LowPipe* p) { delete p; }
void low_pipe_serve(LowPipe* p) {
  if (p) p->serve();
}
void low_pipe_close(LowPipe* p) {
  if (p) p->closed.store(true, std::memory_order_release);
}

namespace {
size_t bitlen_n(const limb* x, size_t n) {
  while (n && !x[n - 1]) --n;
  return n ? 64 * (n - 1) + (64 - (size_t)__builtin_clzll(x[n - 1])) : 0;
}
size_t bits_u64(uint64_t v) { return v ? 64 - (size_t)__builtin_clzll(v) : 0; }

// One round of split batches (see LowPipe); false when none was taken.
bool split_round(Nat& r0, Nat& r1, CofactorPipe* P, LowPipe* S, size_t* steps, long nbits) {
  const int ns = S->begin_round();
  const size_t len = r0.size();
  // the run also simulates each batch: it keeps the top 3/16
  const size_t h = len * 13 / 16;
  const size_t lt = len - h + 1;
  if (ns < 1 || r1.size() < h + 8 || lt < 16 || h < (size_t)ns * (kLowCorr + 2)) return false;
  Nat t0(lt, 0), t1(lt, 0);
  std::copy(r0.begin() + (ptrdiff_t)h, r0.end(), t0.begin());
  std::copy(r1.begin() + (ptrdiff_t)h, r1.end(), t1.begin());
  for (int j = 0; j < ns; ++j) {
    LowPipe::Slot& sl = S->slot[j];
    sl.x = r0.data();
    sl.y = r1.data();
    sl.lo = h * (size_t)j / (size_t)ns;
    sl.hi = h * (size_t)(j + 1) / (size_t)ns;
    sl.ew = 0;
  }
  size_t ebits = 0, taken = 0;
  for (;;) {
    const size_t tb = bitlen_n(t0.data(), lt);
    if (tb < 126 + 64) break;
    const size_t shp = tb - 126;
    if (ebits + 3 > shp || ebits + 70 > 64 * kLowCorr) break;
    const size_t sh = shp + 64 * h;
    __int128 stop = (__int128)1 << 63;
    if ((size_t)nbits >= sh) {
      const size_t e = (size_t)nbits - sh;
      stop = e >= 126 ? ((__int128)1 << 126) : stop + ((__int128)1 << e);
    }
    const LMat L = lehmer_sim_wide((__int128)bits128_at(t0, shp), (__int128)bits128_at(t1, shp), stop);
    if (L.B == 0) break;
    const limb a = uabs(L.A), b = uabs(L.B), c = uabs(L.C), d = uabs(L.D);
    __int128 h0, h1;
    comb2_range(sign_code(L.A, L.B, L.C, L.D), t0.data(), t1.data(), t0.data(), lt, t1.data(), lt, 0, lt, a, b, c,
                d, &h0, &h1);
    ebits = std::max(ebits + bits_u64(std::max(a + b, c + d)), (size_t)64) + 1;
    S->push(L, ebits / 64 + 1);
    P->push(a, b, c, d);
    *steps += L.k;
    ++taken;
  }
  S->drain();
  // r = t 2^(64h) + sum_j (l_j 2^(64 lo_j) + e_j 2^(64 hi_j)), folded from the
  // bottom up with one signed carry; the total is below 2^(64(h + lt)) and at
  // least 0, so the top part's two's complement sum mod 2^(64 lt) is exact
  r0.resize(h + lt, 0);
  r1.resize(h + lt, 0);
  for (int q = 0; q < 2; ++q) {
    limb* r = q ? r1.data() : r0.data();
    const limb* t = q ? t1.data() : t0.data();
    __int128 carry = 0;
    const limb* e = nullptr;  // the correction entering the current range at its bottom
    size_t ew = 0;
    for (int j = 0; j <= ns; ++j) {
      const size_t lo = j < ns ? S->slot[j].lo : h, hi = j < ns ? S->slot[j].hi : h + lt;
      for (size_t i = lo; i < hi; ++i) {
        const size_t k = i - lo;
        __int128 s = carry + (__int128)(j < ns ? r[i] : t[i - h]);
        if (k + 1 < ew)
          s += (__int128)e[k];
        else if (k + 1 == ew)
          s += (__int128)(int64_t)e[k];
        r[i] = (limb)s;
        carry = s >> 64;
      }
      if (j < ns) {
        e = q ? S->slot[j].e1 : S->slot[j].e0;
        ew = S->slot[j].ew;
      }
    }
  }
  trim(r0);
  trim(r1);
  return taken > 0;
}
}  // namespace

namespace {
constexpr size_t kPipeMinLimbs = 48;  // shorter inputs keep their cofactors on the run's thread

// euclid() for rational_reconstruct (nbits >= 0) with the cofactors kept by
// the pipe (its T0, T1 are the starting cofactors; on return they are final
// and the run owns them or has seen every batch applied).
void euclid_piped(Nat& r0, Nat& r1, CofactorPipe* P, LowPipe* S, size_t* steps, long nbits) {
  auto done = [&](const Nat& x) { return le_pow2(x, (size_t)nbits); };
  Nat n0, n1;
  while (!done(r1)) {
    if (S && r1.size() >= kSplitMinLimbs && S->served() && split_round(r0, r1, P, S, steps, nbits)) continue;
    if (r1.size() >= 3) {
      const size_t bl0 = bitlen(r0);
      const size_t sh = bl0 > 126 ? bl0 - 126 : 0;
      __int128 stop = (__int128)1 << 63;
      if ((size_t)nbits >= sh) {
        const size_t e = (size_t)nbits - sh;
        stop = e >= 126 ? ((__int128)1 << 126) : stop + ((__int128)1 << e);
      }
      const LMat Lm = lehmer_sim((__int128)bits128_at(r0, sh), (__int128)bits128_at(r1, sh), stop);
      if (Lm.B != 0) {
        const size_t len = std::max(r0.size(), r1.size());
        n0.resize(len + 1);
        n1.resize(len + 1);
        const limb a = uabs(Lm.A), b = uabs(Lm.B), c = uabs(Lm.C), d = uabs(Lm.D);
        __int128 h0, h1;
        comb2_range(sign_code(Lm.A, Lm.B, Lm.C, Lm.D), n0.data(), n1.data(), r0.data(), r0.size(), r1.data(),
                    r1.size(), 0, len, a, b, c, d, &h0, &h1);
        n0[len] = (limb)h0;
        n1[len] = (limb)h1;
        trim(n0);
        trim(n1);
        r0.swap(n0);
        r1.swap(n1);
        P->push(a, b, c, d);
        *steps += Lm.k;
        continue;
      }
    }
    // one division step, with every earlier batch applied to the cofactors
    P->sync();
    Nat q, rem;
    divmod(r0, r1, &q, &rem);
    r0.swap(r1);
    r1.swap(rem);
    Nat t = mul(q, P->T1);
    add_in(t, P->T0);
    P->T0.swap(P->T1);
    P->T1.swap(t);
    ++*steps;
  }
  P->sync();
}
}  // namespace

// ------------------------------------------------------------ half-gcd
// A run of k Euclid quotient steps on (a, b) as the matrix
//   Q = Q(q_1) ... Q(q_k),  Q(q) = [[q, 1], [1, 0]],  (a; b) = Q (alpha; beta),
// entries >= 0, det Q = (-1)^k (odd = k odd).  Then
//   alpha = (-1)^k (m11 a - m01 b),  beta = (-1)^k (m00 b - m10 a),
// and m01, m00 are the magnitudes of the cofactors of b in alpha and beta.
// If alpha > beta > 0, a / b = [q_1; ..., q_{k-1}, q_k + beta / alpha] with
// every partial term strictly between q_i and q_i + 1, so the q_i are
// exactly the first k quotients of Euclid on (a, b) and (alpha, beta) its
// k-th remainder pair.  That check (qmat_apply_split) is the only thing trusted:
// quotients are computed from leading parts of the numbers, and a matrix
// that fails it is recomputed more conservatively or dropped.
struct QMat {
  Nat m00{1}, m01, m10, m11{1};
  bool odd = false;
  bool identity() const { return m01.empty() && m10.empty(); }
};

static Nat add_prod(const Nat& a, const Nat& b, const Nat& c, const Nat& d) {  // a b + c d
  Nat r = mul(a, b);
  add_in(r, mul(c, d));
  return r;
}
static QMat qmat_mul(const QMat& x, const QMat& y) {
  QMat r;
  r.m00 = add_prod(x.m00, y.m00, x.m01, y.m10);
  r.m01 = add_prod(x.m00, y.m01, x.m01, y.m11);
  r.m10 = add_prod(x.m10, y.m00, x.m11, y.m10);
  r.m11 = add_prod(x.m10, y.m01, x.m11, y.m11);
  r.odd = x.odd != y.odd;
  return r;
}
// (alpha, beta) = Q^{-1} (a, b), true when alpha > beta > 0, for
// a = a1 2^h + a0, b = b1 2^h + b0 (0 <= a0, b0 < 2^h) when
// (x, y) = Q^{-1} (a1, b1) is known already: alpha = x 2^h + (-1)^k (m11 a0 - m01 b0),
// beta = y 2^h + (-1)^k (m00 b0 - m10 a0), so only the short low parts are
// multiplied.
static bool qmat_apply_split(const QMat& Q, const Nat& x, const Nat& y, const Nat& a0, const Nat& b0, size_t h,
                             Nat* al, Nat* be) {
  const Nat p = mul(Q.m11, a0), q = mul(Q.m01, b0), r = mul(Q.m00, b0), t = mul(Q.m10, a0);
  Nat ap = shl(x, h), bp = shl(y, h);
  add_in(ap, Q.odd ? q : p);
  add_in(bp, Q.odd ? t : r);
  const Nat& am = Q.odd ? p : q;
  const Nat& bm = Q.odd ? r : t;
  if (cmp(ap, am) <= 0 || cmp(bp, bm) <= 0) return false;
  sub_in(ap, am);
  sub_in(bp, bm);
  al->swap(ap);
  be->swap(bp);
  return cmp(*al, *be) > 0;
}
static Nat low_bits(const Nat& a, size_t h) {  // a mod 2^h
  const size_t w = (h + 63) / 64;
  Nat r(a.begin(), a.begin() + (ptrdiff_t)std::min(w, a.size()));
  if (h % 64 && r.size() == w) r[w - 1] &= (~0ull >> (64 - h % 64));
  trim(r);
  return r;
}
// One plain division step appended to Q: (x, y) -> (y, x mod y).
static void qmat_step(QMat* Q, Nat* x, Nat* y) {
  Nat q, rem;
  divmod(*x, *y, &q, &rem);
  Nat n00 = mul(Q->m00, q), n10 = mul(Q->m10, q);
  add_in(n00, Q->m01);
  add_in(n10, Q->m11);
  Q->m01.swap(Q->m00);
  Q->m00.swap(n00);
  Q->m11.swap(Q->m10);
  Q->m10.swap(n10);
  Q->odd = !Q->odd;
  x->swap(*y);
  y->swap(rem);
}

constexpr size_t kHgcdBaseBits = 64 * 64;  // at most this: Lehmer batches on the numbers themselves
constexpr size_t kHgcdShiftMin = 512;      // a leading part is at least this much shorter than the number
constexpr size_t kHgcdMargin = 64;         // the leading part stops this far above its share of the target
constexpr size_t kHgcdTol = 192;           // a stage is done within this many bits of its target

// Euclid steps on (a, b), a > b > 0, while the remainders stay above about
// 2^s: returns their matrix Q and the remainder pair (alpha, beta) reached
// (alpha > beta > 0; Q may be the identity when no step is certain).
//   - small numbers: Lehmer batches (euclid) on the numbers themselves;
//   - target at most half of a's length away (2 s >= n + kHgcdShiftMin):
//     the quotients of the leading 2 (n - s) bits, reduced to their own
//     half (plus a margin), agree with those of (a, b) for all but possibly
//     the last few; the matrix is checked against (a, b) and recomputed
//     with a wider margin if the check fails;
//   - farther: stages, each one reduction of the previous kind over the
//     leading (n - s) bits, i.e. half of the remaining distance and then the
//     rest, with one division step wherever a stage makes no progress.
static void hgcd(const Nat& a, const Nat& b, size_t s, QMat* Q, Nat* al, Nat* be) {
  const size_t n = bitlen(a);
  *Q = QMat{};
  if (bitlen(b) <= s) {
    *al = a;
    *be = b;
    return;
  }
  if (n <= kHgcdBaseBits || s < kHgcdShiftMin) {
    Nat r0 = a, r1 = b, T0, T1 = from_u64(1), S0 = from_u64(1), S1;
    size_t steps = 0;
    euclid(r0, r1, &T0, &T1, &steps, (long)s, &S0, &S1);
    if (r1.empty()) {  // ran into the gcd: keep the pair before the last step (beta > 0)
      *Q = QMat{};
      *al = a;
      *be = b;
      return;
    }
    Q->m00.swap(T1);
    Q->m01.swap(T0);
    Q->m10.swap(S1);
    Q->m11.swap(S0);
    Q->odd = steps & 1;
    al->swap(r0);
    be->swap(r1);
    return;
  }
  if (2 * s >= n + kHgcdShiftMin) {
    const size_t h = 2 * s - n;
    const Nat a1 = shr(a, h), b1 = shr(b, h);
    if (b1.empty() || cmp(a1, b1) <= 0) {
      *al = a;
      *be = b;
      return;
    }
    const Nat a0 = low_bits(a, h), b0 = low_bits(b, h);
    for (size_t margin = kHgcdMargin; margin <= 3 * kHgcdMargin; margin += kHgcdMargin) {
      QMat Q1;
      Nat x, y;
      hgcd(a1, b1, s - h + margin, &Q1, &x, &y);
      if (Q1.identity()) break;
      if (qmat_apply_split(Q1, x, y, a0, b0, h, al, be)) {
        *Q = std::move(Q1);
        return;
      }
    }
    *Q = QMat{};
    *al = a;
    *be = b;
    return;
  }
  Nat x = a, y = b;
  while (bitlen(y) > s + kHgcdTol) {
    const size_t nx = bitlen(x);
    const size_t t = 2 * s >= nx + kHgcdShiftMin ? s : nx - (nx - s) / 2;
    QMat Qs;
    Nat x2, y2;
    hgcd(x, y, t, &Qs, &x2, &y2);
    if (Qs.identity()) {
      qmat_step(Q, &x, &y);
      if (y.empty()) break;  // the gcd: the caller's check rejects beta = 0
      continue;
    }
    if (Q->identity())
      *Q = std::move(Qs);
    else
      *Q = qmat_mul(*Q, Qs);
    x.swap(x2);
    y.swap(y2);
  }
  al->swap(x);
  be->swap(y);
}

bool rational_reconstruct(const Nat& M, const Nat& u, size_t nbits, Nat* num, bool* num_neg, Nat* den,
                          const ReconOpts& opts) {
  // a pipe is closed on every way out, so that a serve() waiting on it returns
  struct Closer {
    CofactorPipe* p;
    LowPipe* l;
    ~Closer() {
      if (p) p->closed.store(true, std::memory_order_release);
      if (l) l->closed.store(true, std::memory_order_release);
    }
  } closer{opts.pipe, opts.low};
  Nat r0 = M, r1 = u, T0, T1 = from_u64(1);
  size_t steps = 0;
  // Long inputs: most of the way by half-gcd stages, kept above 2^nbits; the
  // exact stopping point is then found by the Lehmer loop below.
  if (bitlen(M) >= std::max(opts.hgcd_min_bits, kHgcdBaseBits + 1) && !u.empty() && cmp(M, u) > 0 &&
      bitlen(u) > nbits + 4 * kHgcdTol) {
    QMat Q;
    Nat x, y;
    hgcd(M, u, nbits + kHgcdTol, &Q, &x, &y);
    if (!y.empty() && cmp(x, y) > 0 && !le_pow2(x, nbits)) {
      r0.swap(x);
      r1.swap(y);
      T0.swap(Q.m01);
      T1.swap(Q.m00);
      steps = Q.odd ? 1 : 0;
    }
  }
  CofactorPipe* P = opts.pipe;
  if (P && r1.size() >= kPipeMinLimbs && !le_pow2(r1, nbits) && P->head.load() == 0 &&
      P->claim.load() != CofactorPipe::kOwned) {
    // the pipe starts from these cofactors; a server reads them only after
    // the first batch is handed over
    P->T0 = T0;
    P->T1 = T1;
    euclid_piped(r0, r1, P, opts.low, &steps, (long)nbits);
    T0 = P->T0;
    T1 = P->T1;
  } else {
    euclid(r0, r1, &T0, &T1, &steps, (long)nbits);
  }
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
