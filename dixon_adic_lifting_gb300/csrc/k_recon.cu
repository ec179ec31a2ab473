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
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <memory>
#include <new>

#include <algorithm>
#include <cstring>
#include <string>
#include <vector>

#include "bigint.h"
#include "es_common.cuh"
#include "es_internal.h"
#include "recon_common.h"
#include "tc_common.cuh"

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

// acc (96 bits, little-endian words) += x y, one carry chain
__device__ __forceinline__ void mac96(uint32_t (&acc)[3], uint32_t x, uint32_t y) {
  asm("mad.lo.cc.u32 %0, %3, %4, %0;\n\tmadc.hi.cc.u32 %1, %3, %4, %1;\n\taddc.u32 %2, %2, 0;"
      : "+r"(acc[0]), "+r"(acc[1]), "+r"(acc[2])
      : "r"(x), "r"(y));
}

// ---- block-parallel multi-word arithmetic
// The numerator's big integers live in shared memory as 32-bit words, cut into
// groups of four (16 bytes) that one thread owns in each round of blockDim
// groups.  A carry (or borrow) between groups is resolved by a block-wide
// carry lookahead: a group generates a carry when its own sum overflows and
// propagates one when its sum is all ones (a borrow: when its difference is
// zero); with G and P the warp's ballots of the two, the carry into lane l is
// bit l of 2G + P + c_in, xor P's bit l, and bit 32 of that sum is the carry
// out of the warp.
constexpr int kGroup = 4;

struct Scratch {
  uint32_t g[32], pr[32];
  int hi[32], lo[32];
};

// Carry into this thread's group of the current round; *cin is the carry into
// the round's first group on entry and into the next round's on return.  gen
// and prop must not both hold.  Called by every thread of the block.
__device__ __forceinline__ uint32_t carry_in(bool gen, bool prop, uint32_t* cin, Scratch& sc) {
  const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const uint32_t G = __ballot_sync(~0u, gen), P = __ballot_sync(~0u, prop);
  if (lane == 0) {
    sc.g[wp] = G;
    sc.pr[wp] = P;
  }
  __syncthreads();
  uint64_t c = *cin;
  uint32_t mine = 0;
  for (int w = 0; w < nw; ++w) {
    const uint64_t gw = sc.g[w], pw = sc.pr[w];
    const uint64_t s = 2 * gw + pw + c;
    if (w == wp) mine = (uint32_t)(((s ^ pw) >> lane) & 1u);
    c = (s >> 32) & 1u;
  }
  __syncthreads();
  *cin = (uint32_t)c;
  return mine;
}

__device__ __forceinline__ unsigned __int128 ld_group(const uint32_t* Y, int g) {
  const uint4 v = reinterpret_cast<const uint4*>(Y)[g];
  return (unsigned __int128)v.x | ((unsigned __int128)v.y << 32) | ((unsigned __int128)v.z << 64) |
         ((unsigned __int128)v.w << 96);
}

__device__ __forceinline__ void st_group(uint32_t* Y, int g, unsigned __int128 v) {
  reinterpret_cast<uint4*>(Y)[g] = make_uint4((uint32_t)v, (uint32_t)(v >> 32), (uint32_t)(v >> 64), (uint32_t)(v >> 96));
}

// Y holds ng groups, each normalised on its own, and Cg[g] the carry out of
// group g (below 2^64); adds Cg[g - 1] into group g and resolves the ripple,
// so that Y becomes the normalised sum mod b^(4 ng).  Every thread calls it.
__device__ void settle(uint32_t* Y, int ng, const uint64_t* Cg, Scratch& sc) {
  uint32_t cin = 0;
  for (int r0 = 0; r0 < ng; r0 += blockDim.x) {
    const int g = r0 + threadIdx.x;
    unsigned __int128 v = 0;
    bool gen = false, prop = false;
    if (g < ng) {
      const unsigned __int128 y = ld_group(Y, g);
      v = y + (g ? Cg[g - 1] : 0ull);
      gen = v < y;
      prop = v == ~(unsigned __int128)0;
    }
    const uint32_t c = carry_in(gen, prop, &cin, sc);
    if (g < ng) st_group(Y, g, v + c);
  }
}

// Y = X - S mod b^L over words w < L (X, S word sources; Y may be either's
// storage: each thread reads and writes only its own groups).  Y has whole
// groups of storage; its words from L up to the group end are left as they are.
template <class FX, class FS>
__device__ void sub_words(uint32_t* Y, int L, FX x, FS s, Scratch& sc) {
  const int ng = (L + kGroup - 1) / kGroup;
  uint32_t bin = 0;
  for (int r0 = 0; r0 < ng; r0 += blockDim.x) {
    const int g = r0 + threadIdx.x;
    uint32_t d[kGroup] = {0u, 0u, 0u, 0u};
    bool gen = false, prop = false;
    if (g < ng) {
      int64_t br = 0;
#pragma unroll
      for (int j = 0; j < kGroup; ++j) {
        const int w = kGroup * g + j;
        const int64_t t = (w < L ? (int64_t)x(w) - (int64_t)s(w) : 0) + br;
        d[j] = (uint32_t)t;
        br = t >> 32;
      }
      gen = br != 0;
      prop = (d[0] | d[1] | d[2] | d[3]) == 0u;
    }
    uint32_t b = carry_in(gen, prop, &bin, sc);
    if (g < ng) {
#pragma unroll
      for (int j = 0; j < kGroup; ++j) {
        const int w = kGroup * g + j;
        const uint32_t v = d[j] - b;
        b = d[j] < b ? 1u : 0u;
        if (w < L) Y[w] = v;
      }
    }
  }
}

// Highest w < L with a(w) != b(w), or -1; the same value in every thread.
template <class FA, class FB>
__device__ int top_diff(int L, FA a, FB b, Scratch& sc) {
  int best = -1;
  for (int w = threadIdx.x; w < L; w += blockDim.x)
    if (a(w) != b(w)) best = w;
  best = __reduce_max_sync(~0u, best);
  if ((threadIdx.x & 31) == 0) sc.hi[threadIdx.x >> 5] = best;
  __syncthreads();
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) best = max(best, sc.hi[w]);
  __syncthreads();
  return best;
}

// From Z's words Zn[0 .. LG + kZExtra), normalised (Z < b^(LG + 11)): N =
// bal_Q(Z mod Q) by Barrett's method with the 13-word reciprocal, the
// acceptance test |N| <= 2^nb, and the two's complement output of component k.
// QQ is shared scratch of whole groups covering LG + 1 words, Cg one 64-bit
// carry per group.  Every thread calls it.
__device__ __forceinline__ void numerator_tail(const RParams& p, int64_t k, uint32_t* Zn, uint32_t* QQ, uint64_t* Cg,
                                               Scratch& sc) {
  const int LG = p.LG;
  const int tid = threadIdx.x, nt = blockDim.x;
  __shared__ uint32_t qc[2 * kMuWords][3];
  __shared__ uint32_t qh[kMuWords];
  // q^ = floor(Z1 MU / b^13) with Z1 = floor(Z / b^(LG-1)): 26 column sums,
  // then one short carry chain
  if (tid < 2 * kMuWords) {
    uint32_t acc[3] = {0u, 0u, 0u};
    for (int a = max(0, tid - (kMuWords - 1)); a <= min(kMuWords - 1, tid); ++a)
      mac96(acc, Zn[LG - 1 + a], p.MU[tid - a]);
    qc[tid][0] = acc[0];
    qc[tid][1] = acc[1];
    qc[tid][2] = acc[2];
  }
  __syncthreads();
  if (tid == 0) {
    unsigned __int128 s = 0;
    for (int t = 0; t < 2 * kMuWords; ++t) {
      s += (unsigned __int128)qc[t][0] | ((unsigned __int128)qc[t][1] << 32) | ((unsigned __int128)qc[t][2] << 64);
      if (t >= kMuWords) qh[t - kMuWords] = (uint32_t)s;
      s >>= 32;
    }
  }
  __syncthreads();
  // q^ Q mod b^(LG+1) (the remainder is below 3Q < b^(LG+1)): each group's four
  // column sums, normalised within the group, then settled
  const int nq = (LG + 1 + kGroup - 1) / kGroup;
  for (int g = tid; g < nq; g += nt) {
    unsigned __int128 s = 0;
    uint32_t v[kGroup];
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      const int w = kGroup * g + j;
      uint32_t acc[3] = {0u, 0u, 0u};
      if (w <= LG)
        for (int i = max(0, w - LG + 1); i <= min(kMuWords - 1, w); ++i) mac96(acc, qh[i], p.Q[w - i]);
      s += (unsigned __int128)acc[0] | ((unsigned __int128)acc[1] << 32) | ((unsigned __int128)acc[2] << 64);
      v[j] = (uint32_t)s;
      s >>= 32;
    }
    reinterpret_cast<uint4*>(QQ)[g] = make_uint4(v[0], v[1], v[2], v[3]);
    Cg[g] = (uint64_t)s;
  }
  __syncthreads();
  settle(QQ, nq, Cg, sc);
  __syncthreads();
  // r = Z - q^ Q  (mod b^(LG+1))
  auto zw = [&](int w) { return Zn[w]; };
  auto qw = [&](int w) { return w < LG ? p.Q[w] : 0u; };
  sub_words(Zn, LG + 1, zw, [&](int w) { return QQ[w]; }, sc);
  __syncthreads();
  // at most two subtractions of Q
  for (int rep = 0; rep < 3; ++rep) {
    const int t = top_diff(LG + 1, zw, qw, sc);
    if (t >= 0 && Zn[t] < qw(t)) break;  // r < Q
    if (t < 0) {                         // r == Q
      for (int w = tid; w <= LG; w += nt) Zn[w] = 0u;
      __syncthreads();
      break;
    }
    sub_words(Zn, LG + 1, zw, qw, sc);
    __syncthreads();
  }
  // balanced: r > (Q-1)/2 -> N = r - Q, magnitude Q - r
  const int th = top_diff(LG, zw, [&](int w) { return p.Qhalf[w]; }, sc);
  const bool neg = th >= 0 && Zn[th] > p.Qhalf[th];
  if (neg) {
    sub_words(Zn, LG, qw, zw, sc);
    __syncthreads();
  }
  // highest and lowest nonzero words
  int hi = -1, lo = LG;
  for (int w = tid; w < LG; w += nt)
    if (Zn[w] != 0u) {
      hi = w;
      lo = min(lo, w);
    }
  hi = __reduce_max_sync(~0u, hi);
  lo = __reduce_min_sync(~0u, lo);
  if ((tid & 31) == 0) {
    sc.hi[tid >> 5] = hi;
    sc.lo[tid >> 5] = lo;
  }
  __syncthreads();
  for (int w = 0; w < (nt >> 5); ++w) {
    hi = max(hi, sc.hi[w]);
    lo = min(lo, sc.lo[w]);
  }
  // |N| <= 2^nb ?
  bool ok = true;
  if (hi >= 0) {
    const int64_t bl = 32 * (int64_t)hi + (32 - __clz(Zn[hi]));
    if (bl > p.nb + 1)
      ok = false;
    else if (bl == p.nb + 1)  // equal to 2^nb only
      ok = Zn[hi] == (1u << (p.nb % 32)) && lo == hi;
  }
  // two's complement output: -mag = ~mag + 1 (words below the lowest nonzero stay 0)
  const int z = lo;
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
  if (tid == 0) p.ok[k] = ok ? 1 : 0;
}

// Shared memory of k_recon_numerators, in 32-bit words unless stated: Zn
// (whole groups over LG + kZExtra words), QQ (whole groups over LG + 1), the
// shifted digits (mp * 12), then one 64-bit carry per group of Zn.
__host__ __device__ inline int64_t zn_groups(int64_t LG) { return (LG + kZExtra + kGroup - 1) / kGroup; }
__host__ __device__ inline int64_t qq_groups(int64_t LG) { return (LG + 1 + kGroup - 1) / kGroup; }
inline int64_t numerator_smem(int64_t LG, int64_t mp) {
  return 4 * kGroup * (zn_groups(LG) + qq_groups(LG)) + 4 * mp * kDigitWords + 8 * zn_groups(LG);
}

// Five CTAs per SM (48 registers): 1024 components take 1.35 waves of 760 CTAs
// rather than 1.7 waves of 608.
__global__ void __launch_bounds__(256, 5) k_recon_numerators(RParams p) {
  const int64_t k = blockIdx.x;
  const int mp = p.mp, LG = p.LG;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int nz = (int)zn_groups(LG);
  extern __shared__ __align__(16) unsigned char sm[];
  __shared__ Scratch sc;
  uint32_t* Zn = reinterpret_cast<uint32_t*>(sm);             // kGroup nz
  uint32_t* QQ = Zn + kGroup * nz;                            // kGroup qq_groups(LG)
  uint32_t* xs = QQ + kGroup * qq_groups(LG);                 // mp * 12
  uint64_t* Cg = reinterpret_cast<uint64_t*>(xs + mp * kDigitWords);  // nz

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
  // owns a group of 4 consecutive columns: per digit it loads the 16 words of
  // G_i they need (4 aligned 16-byte loads) and the digit's 12 words, then 48
  // 96-bit MACs; the four sums are normalised into words in registers and the
  // group's carry out (below 2^64: every column is below 2^95) is kept apart.
  for (int g = tid; g < nz; g += nt) {
    const int w0 = kGroup * g;
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
      uint32_t g16[16], x[kDigitWords];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const uint4 v = __ldg(gr + h);
        g16[4 * h] = v.x, g16[4 * h + 1] = v.y, g16[4 * h + 2] = v.z, g16[4 * h + 3] = v.w;
      }
#pragma unroll
      for (int h = 0; h < kDigitWords / 4; ++h) {
        const uint4 v = xr[h];
        x[4 * h] = v.x, x[4 * h + 1] = v.y, x[4 * h + 2] = v.z, x[4 * h + 3] = v.w;
      }
#pragma unroll
      for (int o = 0; o < 4; ++o)
#pragma unroll
        for (int l = 0; l < kDigitWords; ++l) mac96(acc[o], x[l], g16[o + 12 - l]);
    }
    unsigned __int128 s = 0;
    uint32_t v[4];
#pragma unroll
    for (int o = 0; o < 4; ++o) {
      s += (unsigned __int128)acc[o][0] | ((unsigned __int128)acc[o][1] << 32) | ((unsigned __int128)acc[o][2] << 64);
      v[o] = (uint32_t)s;
      s >>= 32;
    }
    reinterpret_cast<uint4*>(Zn)[g] = make_uint4(v[0], v[1], v[2], v[3]);
    Cg[g] = (uint64_t)s;
  }
  __syncthreads();
  settle(Zn, nz, Cg, sc);  // Z < b^(LG + 11): nothing carries out of the top group
  __syncthreads();
  numerator_tail(p, k, Zn, QQ, Cg, sc);
}

// ------------------------------------------------------------------ tensor cores
// The numerators' products on the 5th-generation tensor cores.  With x_i the
// balanced digits of component k and G_i = d P'^i mod Q,
//     Z_k = sum_{i < m'} x_i G_i = sum_p 256^p S_p,
//     S_p = sum_i sum_{b < 48} X_i[b] G_i[p - b],
// where X_i[b] are the balanced bytes (in [-128, 127]) of x_i and G_i[u] those
// of G_i.  Over all components this is one GEMM: M = components, N = byte
// columns p, K = (digit, byte) = 48 m'; each product is at most 2^14, so the
// FP32 accumulator is exact over 1008 terms (21 digits) and is folded into
// int32 (|S_p| <= 48 m' 2^14 < 2^31 for m' < 2730).
//
// The B operand is Toeplitz: with b' = 47 - b (A's bytes reversed), row p of
// B holds G_i[p - 47 + b'].  In the canonical K-major layout without swizzle
// (core matrices of 8 rows x 16 bytes), the core matrix of rows 8q .. 8q + 7
// and K elements 8s .. 8s + 7 is, with T[j][r][e] = G_i[8 j + r + 1 + e] as
// f16, exactly T[j] for j = q + s - 6 (plus the tile's offset): a matrix
// descriptor whose two core-matrix strides are both 128 bytes reads B
// straight from one contiguous 128-byte-per-unit copy of T.  T is built once
// per digit (8 f16 per byte of G_i, all of it resident in L2) and each stage
// loads the 21 units a 128-column tile needs.
//
// CTA tile = 128 components (MMA M, A operand in tensor memory: eight
// converter warps, one per lane quarter and digit, widen each component's 48
// digit bytes, balanced and reversed, with tcgen05.st) x 128 byte columns
// (MMA N); a pipeline stage is two digits (six K = 16 MMAs), five stages in
// flight.  Persistent CTAs walk the tiles with the byte-column tile fastest,
// so the CTAs running together share a component tile and its digits stay in
// L2.  The epilogue (eight warps) folds each 20-digit chunk into int32 column
// sums, and at the tile's end normalises each component's 128 columns into 32
// words plus a signed carry, stored word-major (component fastest).
// k_recon_finish (one thread per component) adds the tiles, reduces mod Q and
// writes the numerator limbs, which k_recon_transpose puts in component order.
namespace rg {
constexpr int kM = 128;                     // components per tile
constexpr int kN = 128;                     // byte columns per tile
constexpr int kDig = 48;                    // bytes per digit (K per stage)
constexpr int kDPS = 2;                     // digits per pipeline stage
constexpr int kStages = 5;                  // pipeline stages (shared memory and A slots)
constexpr int kXBytes = kM * kDig;          // 6144 per digit
constexpr int kUnits = kN / 8 + kDig / 8 - 1;  // 21 core-matrix units per window
constexpr int kTBytes = kUnits * 128;       // 2688 per digit
constexpr int kFold = 10;                   // stages per exact FP32 chunk (20 digits: 960 K)
constexpr uint32_t kColA = 2 * kN;          // A slots after the two accumulators
constexpr uint32_t kSlotCols = 48;          // per stage: 24 columns per digit
constexpr uint32_t kTmemCols = 512;
constexpr int kZStride = kN + 1;            // words per row of the epilogue's staging (odd)
constexpr int kConvWarps = 4 * kDPS;        // one warp per lane quarter and digit of a stage
constexpr int kEpiWarp0 = 2 + kConvWarps;   // first epilogue warp
constexpr int kThreads = 32 * (kEpiWarp0 + 8);  // producer, MMA, converter and 8 epilogue warps
constexpr size_t kSmem =
    1024 + (size_t)kStages * kDPS * (kXBytes + kTBytes) + (size_t)kM * kZStride * 4 + 512;
static_assert(kColA + kSlotCols * kStages <= kTmemCols, "tensor memory");
static_assert(24 * kDPS <= (int)kSlotCols, "A slot");
}  // namespace rg

struct GParams {
  const uint8_t* X;    // digits as bytes: [m][nc][48]
  const uint8_t* T;    // [mp][NU][128]: f16 T units of every digit
  int64_t nc;
  int mp, NP, NU;
  int tiles;           // comp tiles x NP
  uint32_t* Zw;        // [NP * 32 + 1][nc] normalised words of the tiles, component fastest
  int32_t* Zc;         // [NP][nc]       carry out of each tile
  int* err;
};

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   tc::smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
               : "memory");
}
// K-major, no swizzle: core matrices of 8 rows x 16 bytes, `lbo` bytes apart
// along K and `sbo` bytes apart along M/N.
__device__ __forceinline__ uint64_t desc_interleave(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (saddr >> 4) & 0x3FFFull;
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version; base offset 0, no swizzle
  return d;
}
// f16 pairs of byte - 128 for the four unsigned bytes of w: 0x64uu is the f16
// 1024 + uu, and 1024 + uu - 1152 = uu - 128 exactly.
__device__ __forceinline__ void u8x4_m128_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = __byte_perm(w, 0x64646464u, 0x4140);
  hi = __byte_perm(w, 0x64646464u, 0x4342);
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(0x64806480u));
}

// T[i][u][r][e] = G_i[8 (u - 6) + r + 1 + e] as f16 (zero outside the bytes of
// G_i), from the balanced bytes Gb [mp][LGB1]; one thread per 16-byte row.
__global__ void k_recon_tbuild(const int8_t* __restrict__ Gb, int64_t LGB1, int NU, int mp,
                               uint8_t* __restrict__ T) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)mp * NU * 8) return;
  const int r = (int)(t & 7);
  const int64_t ui = t >> 3, i = ui / NU, u = ui - i * NU;
  const int64_t base = 8 * (u - 6) + r + 1;
  uint32_t w[4];
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    uint32_t pr = 0;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int64_t idx = base + 2 * h + q;
      const int v = (idx >= 0 && idx < LGB1) ? (int)Gb[i * LGB1 + idx] : 0;
      pr |= (uint32_t)__half_as_ushort(__int2half_rn(v)) << (16 * q);
    }
    w[h] = pr;
  }
  reinterpret_cast<uint4*>(T)[t] = make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void __launch_bounds__(rg::kThreads, 1) k_recon_gemm(GParams p) {
  using namespace rg;
  using namespace tc;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sX = smem;                                   // [S][DPS][128][48] digit bytes
  uint8_t* sT = sX + kStages * kDPS * kXBytes;          // [S][DPS][21][128] T windows
  int32_t* sZ = reinterpret_cast<int32_t*>(sT + kStages * kDPS * kTBytes);  // [128][129]
  uint64_t* full = reinterpret_cast<uint64_t*>(sZ + kM * kZStride);
  uint64_t* empty = full + kStages;
  uint64_t* conv = empty + kStages;
  uint64_t* accfull = conv + kStages;
  uint64_t* accempty = accfull + 2;
  uint64_t* drained = accempty + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drained + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mp = p.mp, nst = (mp + kDPS - 1) / kDPS, nch = (nst + kFold - 1) / kFold;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
      mbar_init(conv + s, 32 * kConvWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accfull + b, 1);
      mbar_init(accempty + b, 256);
    }
    mbar_init(drained, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(s_tmem)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = __shfl_sync(0xffffffffu, *s_tmem, 0);
  int* err = p.err;

  if (warp == 0) {  // producer: the digit bytes of the tile's components and the T window, per digit
    int g = 0;
    bool stop = false;
    for (int t = blockIdx.x; t < p.tiles && !stop; t += gridDim.x) {
      const int ct = t / p.NP, pt = t - ct * p.NP;
      const int64_t c0 = (int64_t)ct * kM;
      const uint32_t cnt = (uint32_t)(p.nc - c0 < kM ? p.nc - c0 : kM);
      for (int j = 0; j < nst; ++j, ++g) {
        const int s = g % kStages, nd = mp - kDPS * j < kDPS ? mp - kDPS * j : kDPS;
        if (g >= kStages && !mbar_wait_warp(empty + s, ((g / kStages) & 1) ^ 1, err, 21)) {
          stop = true;
          break;
        }
        if (elect_one()) {
          mbar_expect_tx(full + s, nd * (cnt * kDig + kTBytes));
          for (int d = 0; d < nd; ++d) {
            const int i = kDPS * j + d;
            bulk_g2s(sX + (s * kDPS + d) * kXBytes, p.X + ((int64_t)i * p.nc + c0) * kDig, cnt * kDig, full + s);
            bulk_g2s(sT + (s * kDPS + d) * kTBytes, p.T + ((int64_t)i * p.NU + 16 * pt) * 128, kTBytes, full + s);
          }
        }
        __syncwarp();
      }
    }
    for (int k = g > kStages ? g - kStages : 0; k < g; ++k) mbar_wait_drain(full + k % kStages, (k / kStages) & 1);
  } else if (warp == 1) {  // MMA issuer
    const uint32_t idesc = (1u << 4) | ((uint32_t)(kN >> 3) << 17) | ((uint32_t)(kM >> 4) << 24);
    int g = 0, gc = 0;
    bool stop = false;
    for (int t = blockIdx.x; t < p.tiles && !stop; t += gridDim.x) {
      for (int j = 0; j < nst; ++j, ++g) {
        const int s = g % kStages, buf = gc & 1, nd = mp - kDPS * j < kDPS ? mp - kDPS * j : kDPS;
        const bool first = (j % kFold) == 0;
        if (first && gc >= 2 && !mbar_wait_warp(accempty + buf, ((gc - 2) >> 1) & 1, err, 22)) {
          stop = true;
          break;
        }
        if (!mbar_wait_warp(full + s, (g / kStages) & 1, err, 23) ||
            !mbar_wait_warp(conv + s, (g / kStages) & 1, err, 24)) {
          stop = true;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          for (int d = 0; d < nd; ++d) {
            // K = 16 steps advance the window by two 128-byte units (16 in the address field)
            const uint64_t bd = desc_interleave(smem_u32(sT + (s * kDPS + d) * kTBytes), 128, 128);
#pragma unroll
            for (int k = 0; k < kDig / 16; ++k)
              mma_f16_ta(tmem + buf * kN, tmem + kColA + kSlotCols * s + 24 * d + 8 * k, bd + 16 * k, idesc,
                         (first && d == 0 && k == 0) ? 0u : 1u);
          }
          mma_commit(empty + s);
          if (j % kFold == kFold - 1 || j == nst - 1) mma_commit(accfull + buf);
        }
        __syncwarp();
        if (j % kFold == kFold - 1 || j == nst - 1) ++gc;
      }
    }
    if (elect_one()) mma_commit(drained);
    __syncwarp();
    mbar_wait_drain(drained, 0);
  } else if (warp < kEpiWarp0) {
    // converters: warp w touches tensor-memory lanes 32 (w % 4) .. + 31 and
    // takes digit d = (w - 2) / 4 of each stage; thread = one component (row):
    // its 48 digit bytes, balanced (bytes of x + 0x80..80, less 128) and
    // reversed (A's element b' = byte 47 - b'), as 24 columns
    const int quarter = warp & 3, d = (warp - 2) >> 2, r = 32 * quarter + lane;
    const uint32_t trow = tmem + ((uint32_t)(32 * quarter) << 16);
    int g = 0;
    bool stop = false;
    for (int t = blockIdx.x; t < p.tiles && !stop; t += gridDim.x) {
      const int ct = t / p.NP;
      const bool live = (int64_t)ct * kM + r < p.nc;
      for (int j = 0; j < nst; ++j, ++g) {
        const int s = g % kStages, nd = mp - kDPS * j < kDPS ? mp - kDPS * j : kDPS;
        // the slot's previous MMAs completed before its copy was issued (empty -> full)
        if (!mbar_wait_warp(full + s, (g / kStages) & 1, err, 25)) {
          stop = true;
          break;
        }
        tc_fence_after();
        if (d < nd) {
          uint32_t wv[24];
          if (live) {
            const uint4* src = reinterpret_cast<const uint4*>(sX + (s * kDPS + d) * kXBytes + r * kDig);
            const uint4 v0 = src[0], v1 = src[1], v2 = src[2];
            // x + 0x8080...80 over 384 bits
            uint64_t w64[6] = {(uint64_t)v0.x | ((uint64_t)v0.y << 32), (uint64_t)v0.z | ((uint64_t)v0.w << 32),
                               (uint64_t)v1.x | ((uint64_t)v1.y << 32), (uint64_t)v1.z | ((uint64_t)v1.w << 32),
                               (uint64_t)v2.x | ((uint64_t)v2.y << 32), (uint64_t)v2.z | ((uint64_t)v2.w << 32)};
            uint32_t cy = 0;
#pragma unroll
            for (int l = 0; l < 6; ++l) {
              const uint64_t a = w64[l] + 0x8080808080808080ull, b = a + cy;
              cy = (a < w64[l] || b < a) ? 1u : 0u;
              w64[l] = b;
            }
            // reversed bytes: word k' of the reversal = bytes 47 - 4k' .. 44 - 4k'
#pragma unroll
            for (int kk = 0; kk < 12; ++kk) {
              const int src_w = 11 - kk;
              const uint32_t word = (uint32_t)(w64[src_w >> 1] >> (32 * (src_w & 1)));
              u8x4_m128_to_f16(__byte_perm(word, 0, 0x0123), wv[2 * kk], wv[2 * kk + 1]);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < 24; ++kk) wv[kk] = 0;
          }
          uint32_t lo[16], hi[8];
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) lo[kk] = wv[kk];
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) hi[kk] = wv[16 + kk];
          tmem_st16(trow + kColA + kSlotCols * s + 24 * d, lo);
          tmem_st8(trow + kColA + kSlotCols * s + 24 * d + 16, hi);
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(conv + s);
      }
    }
  } else {
    // epilogue: warp w folds columns 64 h .. 64 h + 63 (h = (w - kEpiWarp0) / 4) of the
    // rows of lane quarter w % 4; at a tile's end the rows are normalised into
    // bytes and a carry through the staging area
    const int quarter = warp & 3, h = (warp - kEpiWarp0) >> 2, r = 32 * quarter + lane;
    int gc = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.tiles && ok; t += gridDim.x) {
      const int ct = t / p.NP, pt = t - ct * p.NP;
      int32_t acc[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] = 0;
      for (int ch = 0; ch < nch; ++ch, ++gc) {
        const int buf = gc & 1;
        if (!mbar_wait(accfull + buf, (gc >> 1) & 1, err, 26)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c16 = 0; c16 < 4; ++c16) {
          float f[16];
          tmem_ld<16>(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(buf * kN + 64 * h + 16 * c16), f);
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[16 * c16 + j] += __float2int_rn(f[j]);
        }
        tc_fence_before();
        mbar_arrive(accempty + buf);
      }
      if (!ok) break;
#pragma unroll
      for (int j = 0; j < 64; ++j) sZ[r * kZStride + 64 * h + j] = acc[j];
      asm volatile("bar.sync 1, 256;" ::: "memory");
      const int64_t comp = (int64_t)ct * kM + r;
      if (h == 0 && comp < p.nc) {
        // words of the tile, component fastest: a warp's stores are 128 contiguous bytes
        int64_t carry = 0;
        uint32_t* zw = p.Zw + (int64_t)(kN / 4) * pt * p.nc + comp;
#pragma unroll 1
        for (int q = 0; q < kN / 4; ++q) {
          uint32_t word = 0;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int64_t v = (int64_t)sZ[r * kZStride + 4 * q + e] + carry;
            word |= (uint32_t)(v & 255) << (8 * e);
            carry = v >> 8;
          }
          zw[(int64_t)q * p.nc] = word;
        }
        p.Zc[(int64_t)pt * p.nc + comp] = (int32_t)carry;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(rg::kTmemCols));
  }
}

struct FParams {
  uint32_t* Zw;          // [LZ2][nc] words, component fastest (in: the tiles' words)
  const int32_t* Zc;     // [NP][nc]
  const uint32_t* OFF2;  // [LZ2] words of m' ((P'+1)/2) Q, so that Z + OFF2 >= 0
  const uint32_t* Q;     // [LG]
  const uint32_t* Qhalf; // [LG]  (Q - 1) / 2
  const uint32_t* MU;    // [13]  floor(b^(LG-1+13) / Q)
  int64_t nc, nb;
  int LG, NP, LZ2, W;
  uint64_t* Nw;          // [W][nc] numerator limbs, component fastest
  uint8_t* ok;           // [nc]
};

// One thread per component (every step of the finish is a carry chain, so
// the components, not the words, are spread over the threads; the word-major
// layout keeps each warp's accesses contiguous):
//   Z' = OFF2 + sum_t (words of tile t + carry_t b^32) b^(32 t) = d X_lo (mod Q),
//   r = Z' - q^ Q with q^ = floor(floor(Z' / b^(LG-1)) MU / b^13) (Barrett),
//   at most two subtractions of Q, the balanced N = r or r - Q, |N| <= 2^nb,
//   and N's two's complement limbs.
__global__ void __launch_bounds__(128) k_recon_finish(FParams f) {
  const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= f.nc) return;
  const int64_t nc = f.nc;
  const int LG = f.LG, LZ2 = f.LZ2, LW = 32 * f.NP;
  uint32_t* Z = f.Zw + k;  // word w at Z[w * nc]
  // Z' normalised into words
  {
    int64_t carry = 0;
    for (int w = 0; w < LZ2; ++w) {
      int64_t v = (int64_t)f.OFF2[w] + carry;
      if (w < LW) v += Z[(int64_t)w * nc];
      if (w >= 32 && (w & 31) == 0 && (w >> 5) - 1 < f.NP) v += f.Zc[(int64_t)((w >> 5) - 1) * nc + k];
      Z[(int64_t)w * nc] = (uint32_t)v;
      carry = v >> 32;  // arithmetic: the columns may be negative
    }
  }
  // q^ from the top 13 words
  uint32_t qh[kMuWords];
  {
    uint32_t prod[2 * kMuWords];
#pragma unroll
    for (int t = 0; t < 2 * kMuWords; ++t) prod[t] = 0;
#pragma unroll 1
    for (int a = 0; a < kMuWords; ++a) {
      uint64_t c = 0;
      const uint64_t za = Z[(int64_t)(LG - 1 + a) * nc];
#pragma unroll
      for (int b = 0; b < kMuWords; ++b) {
        const uint64_t t = za * f.MU[b] + prod[a + b] + c;
        prod[a + b] = (uint32_t)t;
        c = t >> 32;
      }
      prod[a + kMuWords] = (uint32_t)c;
    }
#pragma unroll
    for (int t = 0; t < kMuWords; ++t) qh[t] = prod[kMuWords + t];
  }
  // r = Z' - q^ Q over words 0 .. LG (the remainder is below 3Q < b^(LG+1))
  {
    uint64_t plo = 0;  // running column sum of q^ Q (96 bits: plo + 2^64 phi)
    uint32_t phi = 0;
    int64_t borrow = 0;
    for (int w = 0; w <= LG; ++w) {
#pragma unroll
      for (int j = 0; j < kMuWords; ++j) {
        const int t = w - j;
        if (t >= 0 && t < LG) {
          const uint64_t pr = (uint64_t)qh[j] * f.Q[t];
          plo += pr;
          phi += plo < pr ? 1u : 0u;
        }
      }
      const uint32_t qq = (uint32_t)plo;
      plo = (plo >> 32) | ((uint64_t)phi << 32);
      phi = 0;
      const int64_t d = (int64_t)Z[(int64_t)w * nc] - (int64_t)qq + borrow;
      Z[(int64_t)w * nc] = (uint32_t)d;
      borrow = d >> 32;
    }
  }
  // at most two subtractions of Q
  for (int rep = 0; rep < 3; ++rep) {
    bool ge = Z[(int64_t)LG * nc] != 0;
    if (!ge) {
      ge = true;
      for (int w = LG - 1; w >= 0; --w) {
        const uint32_t zw = Z[(int64_t)w * nc], qw = f.Q[w];
        if (zw != qw) {
          ge = zw > qw;
          break;
        }
      }
    }
    if (!ge) break;
    int64_t borrow = 0;
    for (int w = 0; w <= LG; ++w) {
      const int64_t d = (int64_t)Z[(int64_t)w * nc] - (int64_t)(w < LG ? f.Q[w] : 0u) + borrow;
      Z[(int64_t)w * nc] = (uint32_t)d;
      borrow = d >> 32;
    }
  }
  // balanced: r > (Q-1)/2 -> N = r - Q, magnitude Q - r
  bool neg = false;
  for (int w = LG - 1; w >= 0; --w) {
    const uint32_t zw = Z[(int64_t)w * nc], hw = f.Qhalf[w];
    if (zw != hw) {
      neg = zw > hw;
      break;
    }
  }
  if (neg) {
    int64_t borrow = 0;
    for (int w = 0; w < LG; ++w) {
      const int64_t d = (int64_t)f.Q[w] - (int64_t)Z[(int64_t)w * nc] + borrow;
      Z[(int64_t)w * nc] = (uint32_t)d;
      borrow = d >> 32;
    }
  }
  // |N| <= 2^nb ?
  int top = LG - 1;
  while (top >= 0 && Z[(int64_t)top * nc] == 0) --top;
  bool ok = true;
  if (top >= 0) {
    const uint32_t zt = Z[(int64_t)top * nc];
    const int64_t bl = 32 * (int64_t)top + (32 - __clz(zt));
    if (bl > f.nb + 1) {
      ok = false;
    } else if (bl == f.nb + 1) {  // equal to 2^nb only
      ok = zt == (1u << (f.nb % 32));
      for (int w = 0; ok && w < top; ++w) ok = Z[(int64_t)w * nc] == 0;
    }
  }
  f.ok[k] = ok ? 1 : 0;
  // two's complement limbs: -mag = ~mag + 1
  uint32_t cy = neg ? 1u : 0u;
  for (int t = 0; t < f.W; ++t) {
    uint32_t wv[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int w = 2 * t + hh;
      const uint32_t m = w < LG ? Z[(int64_t)w * nc] : 0u;
      if (neg) {
        const uint64_t v = (uint64_t)(~m) + cy;
        wv[hh] = (uint32_t)v;
        cy = (uint32_t)(v >> 32);
      } else {
        wv[hh] = m;
      }
    }
    f.Nw[(int64_t)t * nc + k] = (uint64_t)wv[0] | ((uint64_t)wv[1] << 32);
  }
}

// out[k][t] = Nw[t][k]: 32 x 32 tiles through shared memory, both sides
// contiguous (the destination may be page-locked host memory).
__global__ void k_recon_transpose(const uint64_t* __restrict__ Nw, int64_t nc, int W, uint64_t* __restrict__ out) {
  __shared__ uint64_t tile[32][33];
  const int64_t k0 = (int64_t)blockIdx.x * 32, t0 = (int64_t)blockIdx.y * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
  for (int yy = ty; yy < 32; yy += 8) {
    const int64_t t = t0 + yy, k = k0 + tx;
    if (t < W && k < nc) tile[yy][tx] = Nw[t * nc + k];
  }
  __syncthreads();
  for (int yy = ty; yy < 32; yy += 8) {
    const int64_t k = k0 + yy, t = t0 + tx;
    if (t < W && k < nc) out[k * W + t] = tile[tx][yy];
  }
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

// The tensor-core numerator product pays off once there are enough
// components to fill the GPU with 128-component tiles (measured: at 4096 and
// 8192 components the per-component kernel is still faster); its int32 column sums
// stay exact for m' < 2730 (48 m' 2^14 < 2^31).
constexpr int64_t kReconTcMinComponents = 16384;
bool tc_numerators(int64_t nc, int32_t mp) { return nc >= kReconTcMinComponents && mp >= 1 && mp < 2730; }
struct TcSizes {
  int64_t LGB1 = 0;
  int NP = 0, NU = 0, LZ2 = 0;
};
TcSizes tc_sizes(int64_t LG) {
  TcSizes z;
  z.LGB1 = 4 * LG + 1;  // balanced bytes of G_i < Q < b^LG (one more for the top carry)
  z.NP = (int)((z.LGB1 + rg::kDig - 1 + rg::kN - 1) / rg::kN);  // byte columns p < LGB1 + 47
  z.NU = 16 * z.NP + 6;
  z.LZ2 = (int)std::max<int64_t>(LG + kZExtra, 32 * (int64_t)z.NP + 1);
  return z;
}
void tc_layout_add(Layout& L, int64_t nc, int32_t mp, int64_t W, const TcSizes& z, size_t* o) {
  o[0] = L.add((size_t)mp * z.NU * 128);             // T
  o[1] = L.add((size_t)mp * z.LGB1);                 // balanced bytes of G_i
  o[2] = L.add((size_t)nc * z.LZ2 * 4);              // Z' words, component fastest
  o[3] = L.add((size_t)nc * z.NP * 4);               // tile carries
  o[4] = L.add((size_t)z.LZ2 * 4);                   // OFF2
  o[5] = L.add(sizeof(int));                         // error flag
  o[6] = L.add((size_t)nc * W * 8);                  // numerator limbs, component fastest
}

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
  if (tc_numerators(nc, mp)) {
    size_t o[7];
    tc_layout_add(L, nc, mp, W, tc_sizes(LG), o);
  }
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
  // tensor-core numerator product
  bool tc = false;
  TcSizes tz;
  size_t oTc[7] = {0, 0, 0, 0, 0, 0, 0};  // T, Gb, Zw, Zc, OFF2, err, Nw
  std::vector<uint32_t> hOff2;
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
  R.tc = tc_numerators(R.nc, mp);
  if (R.tc) {
    R.tz = tc_sizes(LG);
    tc_layout_add(L, R.nc, mp, R.W, R.tz, R.oTc);
    // OFF2 = m' ((P' + 1) / 2) Q > |sum_i x_i G_i|, a multiple of Q
    const Nat off2 = big::mul(big::mul(big::from_u64((uint64_t)mp), big::add(R.ps.half, big::from_u64(1))), Q);
    if ((int64_t)((big::bitlen(off2) + 32) / 32) > R.tz.LZ2 - 1) return ES_ERR_INTERNAL;
    R.hOff2.assign((size_t)R.tz.LZ2, 0u);
    to_words(off2, R.tz.LZ2, R.hOff2.data());
  }
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
  R.dyn = (int)numerator_smem(LG, mp);
  *out = rp.release();
  return ES_OK;
}

// One numerator pass on the tensor cores: the balanced bytes of every G_i
// (host), their T units, the product of all components' digit bytes by them,
// and the per-component finish.
static es_status tc_numerator_pass(const ReconPlan& R, const std::vector<uint32_t>& hG, int64_t GS,
                                   const uint64_t* D_dev, char* scratch, const RParams& rp, std::vector<int8_t>& hGb,
                                   uint64_t* host_out, int host_threads, cudaStream_t st) {
  const TcSizes& z = R.tz;
  const int32_t mp = R.mp;
  const int64_t LG = R.LG, nc = R.nc;
  // balanced bytes: G = sum_u gb_u 256^u, gb_u in [-128, 127] (carry up)
  parallel_for(mp, 0, [&](int64_t i) {
    const uint32_t* gw = hG.data() + (size_t)i * GS + kGPad;
    int8_t* out = hGb.data() + (size_t)i * z.LGB1;
    int carry = 0;
    for (int64_t u = 0; u < z.LGB1; ++u) {
      const int64_t w = u >> 2;
      int v = (w < LG ? (int)((gw[w] >> (8 * (u & 3))) & 0xFFu) : 0) + carry;
      carry = v > 127 ? 1 : 0;
      out[u] = (int8_t)(v - 256 * carry);
    }
  });
  uint8_t* T = reinterpret_cast<uint8_t*>(scratch + R.oTc[0]);
  int8_t* Gb = reinterpret_cast<int8_t*>(scratch + R.oTc[1]);
  int* err = reinterpret_cast<int*>(scratch + R.oTc[5]);
  ES_CHECK(cuda_status(cudaMemcpyAsync(Gb, hGb.data(), hGb.size(), cudaMemcpyHostToDevice, st), "recon Gb H2D"));
  ES_CHECK(cuda_status(cudaMemsetAsync(err, 0, sizeof(int), st), "recon err memset"));
  const int64_t rows = (int64_t)mp * z.NU * 8;
  k_recon_tbuild<<<(unsigned)((rows + 255) / 256), 256, 0, st>>>(Gb, z.LGB1, z.NU, mp, T);
  ES_CHECK(cuda_status(cudaGetLastError(), "k_recon_tbuild"));
  GParams gp;
  gp.X = reinterpret_cast<const uint8_t*>(D_dev);
  gp.T = T;
  gp.nc = nc;
  gp.mp = mp;
  gp.NP = z.NP;
  gp.NU = z.NU;
  gp.tiles = (int)(((nc + rg::kM - 1) / rg::kM) * z.NP);
  gp.Zw = reinterpret_cast<uint32_t*>(scratch + R.oTc[2]);
  gp.Zc = reinterpret_cast<int32_t*>(scratch + R.oTc[3]);
  gp.err = err;
  ES_CHECK(cuda_status(cudaFuncSetAttribute(k_recon_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)rg::kSmem),
                       "recon gemm smem attribute"));
  const int grid = std::min(gp.tiles, sm_count());
  k_recon_gemm<<<grid, rg::kThreads, rg::kSmem, st>>>(gp);
  ES_CHECK(cuda_status(cudaGetLastError(), "k_recon_gemm"));
  FParams fp;
  fp.Zw = gp.Zw;
  fp.Zc = gp.Zc;
  fp.OFF2 = reinterpret_cast<const uint32_t*>(scratch + R.oTc[4]);
  fp.Q = rp.Q;
  fp.Qhalf = rp.Qhalf;
  fp.MU = rp.MU;
  fp.nc = nc;
  fp.nb = rp.nb;
  fp.LG = (int)LG;
  fp.NP = z.NP;
  fp.LZ2 = z.LZ2;
  fp.W = rp.W;
  fp.Nw = reinterpret_cast<uint64_t*>(scratch + R.oTc[6]);
  fp.ok = rp.ok;
  k_recon_finish<<<(unsigned)((nc + 127) / 128), 128, 0, st>>>(fp);
  ES_CHECK(cuda_status(cudaGetLastError(), "k_recon_finish"));
  k_recon_transpose<<<dim3((unsigned)((nc + 31) / 32), (unsigned)((rp.W + 31) / 32)), dim3(32, 8), 0, st>>>(
      fp.Nw, nc, rp.W, rp.N);
  count_launch(4);
  ES_CHECK(cuda_status(cudaGetLastError(), "k_recon_transpose"));
  int herr = 0;
  ES_CHECK(cuda_status(cudaMemcpyAsync(&herr, err, sizeof(int), cudaMemcpyDeviceToHost, st), "recon err D2H"));
  // While the GPU works: the host threads write the result buffer once, which
  // makes the copy into it that follows several times faster on this host
  // (measured: a copy into a page-locked buffer the host has not just written
  // ran at a fraction of the copy engine's rate).
  {
    const size_t words = (size_t)nc * (size_t)rp.W, chunk = size_t(1) << 20;
    parallel_for((int64_t)((words + chunk - 1) / chunk), host_threads, [&](int64_t t) {
      const size_t a = (size_t)t * chunk, b = std::min(words, a + chunk);
      std::memset(host_out + a, 0, (b - a) * 8);
    });
  }
  ES_CHECK(cuda_status(cudaStreamSynchronize(st), "recon gemm sync"));
  if (herr) {
    set_last_error("numerator product: bounded wait expired (code " + std::to_string(herr) + ")");
    return ES_ERR_TIMEOUT;
  }
  return ES_OK;
}

std::vector<int64_t> recon_samples(int64_t n, int64_t c, int threads) {
  const int width = threads > 0 ? threads : std::max(1, (int)std::thread::hardware_concurrency());
  return sample_components(n, c, sample_count(c, width));
}

es_status recon_prepare_overlapped(int64_t n, int64_t c, int32_t m, int32_t mp, const uint8_t* good,
                                   int64_t num_bits, int64_t den_bits, const Stats& stats, int threads,
                                   const DigitStream* ds, int ns, void* lift_done, ReconPlan** out,
                                   std::vector<std::vector<uint64_t>>* pre) {
  const int width = threads > 0 ? threads : std::max(1, (int)std::thread::hardware_concurrency());
  const int nsamp = ds && ds->host ? ns : 0;
  std::vector<Nat> sums((size_t)nsamp);
  std::atomic<int> missing(0);
  es_status ps = ES_OK;
  const PrimeSet pset = make_prime_set(good);
  auto lift_over = [&]() {
    const cudaError_t q = cudaEventQuery((cudaEvent_t)lift_done);
    if (q == cudaErrorNotReady) return false;
    if (q != cudaSuccess) cudaGetLastError();
    return true;
  };
  parallel_for(1 + nsamp, width, [&](int64_t t) {
    if (t == 0) {
      ps = recon_device_prepare(n, c, m, mp, good, num_bits, den_bits, stats, out);
    } else if (!assemble_streamed(pset, ds->host, (int)t - 1, kStreamRows, kStreamWords, m, lift_over,
                                  &sums[(size_t)t - 1])) {
      missing = 1;
    }
  });
  pre->clear();
  if (nsamp && !missing) pre->assign(sums.begin(), sums.end());
  return ps;
}

es_status reconstruct_device(ReconPlan* plan, const uint64_t* D_dev, int threads, char* scratch,
                             size_t scratch_bytes, void* stream, Solution* out,
                             const std::vector<std::vector<uint64_t>>* pre) {
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
    denominators_parallel((int64_t)ks.size(), hw_threads, [&](int64_t t, const big::ReconOpts& ro) {
      const Nat u = shifted_to_residue(
          assemble_shifted_dc(ps, R.ap, hd.data() + (size_t)t * m * kDigitLimbs, kDigitLimbs), Mhalf, Mhalf1);
      if (!component_denominator(M, u, num_bits, den_bits, &(*dens)[(size_t)t], ro)) fail = 1;
    });
    return fail ? ES_ERR_INTERNAL : ES_OK;
  };
  const int64_t per_round = sample_count(c, hw_threads);
  const std::vector<int64_t> sk = sample_components(n, c, per_round);
  std::vector<Nat> sden;
  if (pre && pre->size() == sk.size()) {
    // the samples' shifted sums came in while the lift ran
    sden.assign(sk.size(), Nat{});
    std::atomic<int> fail(0);
    denominators_parallel((int64_t)sk.size(), hw_threads, [&](int64_t t, const big::ReconOpts& ro) {
      const Nat u = shifted_to_residue((*pre)[(size_t)t], Mhalf, Mhalf1);
      if (!component_denominator(M, u, num_bits, den_bits, &sden[(size_t)t], ro)) fail = 1;
    });
    if (fail) return ES_ERR_INTERNAL;
  } else {
    ES_CHECK(denominators(sk, &sden));
  }
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
  // The tensor-core path's transpose writes device memory, and one copy then
  // moves the limbs (the copy engine outruns kernel stores to host memory).
  uint64_t* Nout = reinterpret_cast<uint64_t*>(scratch + oN);
  bool direct = false;
  if (out->num.pinned() && !R.tc) {
    void* dp = nullptr;
    if (cudaHostGetDevicePointer(&dp, out->num.data(), 0) == cudaSuccess) {
      Nout = static_cast<uint64_t*>(dp);
      direct = true;
    } else {
      cudaGetLastError();
    }
  }
  if (!out->num.pinned() && !R.tc) std::memset(out->num.data(), 0, out->num.size() * 8);
  std::vector<uint8_t> okh((size_t)nc);
  const int64_t GS = g_stride(LG);
  std::vector<uint32_t> hG((size_t)mp * GS, 0u);
  std::vector<int8_t> hGb(R.tc ? (size_t)mp * R.tz.LGB1 : 0);
  if (R.tc)
    ES_CHECK(cuda_status(cudaMemcpyAsync(scratch + R.oTc[4], R.hOff2.data(), R.hOff2.size() * 4,
                                         cudaMemcpyHostToDevice, st),
                         "recon OFF2 H2D"));
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
    if (!R.tc)
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
    if (R.tc) {
      ES_CHECK(tc_numerator_pass(R, hG, GS, D_dev, scratch, rp, hGb, out->num.data(), hw_threads, st));
    } else {
      k_recon_numerators<<<(unsigned)nc, 256, dyn, st>>>(rp);
      count_launch();
      ES_CHECK(cuda_status(cudaGetLastError(), "k_recon_numerators"));
    }
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
