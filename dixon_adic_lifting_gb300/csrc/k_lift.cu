// The Dixon lift: m steps of
//     x_i = B r_i mod P      (per prime: Y_j = B_j R_j, exact int32, then mod q_j)
//     balanced CRT of the E' residues into one base-P digit x_i
//     r_{i+1} = (r_i - A x_i) P^{-1} mod 2^64   (one signed 64-bit limb)
// exact-solve card, §Method: each lift step forms the products of every
// prime's inverse with the residual's residues as one batched int8 matrix
// product, combines the residues into the wide digit by CRT, and updates the
// residual in a single 64-bit limb as (r_i - A x_i) P^{-1} mod 2^64 (P odd).
// The range n * max|A_ij| < 2^63 keeps the residual in one limb and K = n <=
// 2^17 keeps the int32 accumulator exact (2^17 * 125^2 < 2^31).
//
// Device buffers of one lift:
//   B     int8   [53][n][ld]       inverses (ld = n rounded up to 16), only good primes read
//   R     int8   [E'][c][ld]       balanced residues of r_i, column-major per prime, zero padded
//   V     int8   [E'][n*c]         balanced residues of x_i
//   r     int64  [2][n*c]          residual (double buffer; [c][n] with the tensor-core residual update)
//   xl    uint64 [n*c]             x_i mod 2^64
//   D     uint64 [m][n*c][6]       the digits
//   A32   int32  [n][n]            A narrowed when max|A| < 2^31 (else A int64 is read)
//   K     LiftConst                CRT / residual constants of the good prime set
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstring>
#include <string>
#include <vector>

#include "es_common.cuh"
#include "es_internal.h"
#include "lift_internal.h"
#include "lift_device.cuh"

namespace es {



// ------------------------------------------------------------ host constants
namespace {
// little-endian 32-bit word arithmetic on kCrtWords words
void w_mul_small(uint32_t* x, uint32_t s) {
  uint64_t carry = 0;
  for (int l = 0; l < kCrtWords; ++l) {
    uint64_t t = (uint64_t)x[l] * s + carry;
    x[l] = (uint32_t)t;
    carry = t >> 32;
  }
}
uint32_t w_mod_small(const uint32_t* x, uint32_t q) {
  uint64_t r = 0;
  for (int l = kCrtWords - 1; l >= 0; --l) r = ((r << 32) | x[l]) % q;
  return (uint32_t)r;
}
uint32_t inv_small(uint32_t a, uint32_t q) {  // extended Euclid, a != 0 mod q
  int64_t t0 = 0, t1 = 1, r0 = q, r1 = a % q;
  while (r1) {
    int64_t qq = r0 / r1, tmp = r0 - qq * r1;
    r0 = r1;
    r1 = tmp;
    tmp = t0 - qq * t1;
    t0 = t1;
    t1 = tmp;
  }
  return (uint32_t)((t0 % (int64_t)q + q) % q);
}
}  // namespace

void build_lift_const(const uint8_t* good, LiftConst* K) {
  std::memset(K, 0, sizeof(*K));
  int E = 0;
  for (int j = 0; j < kNumPrimes; ++j)
    if (good[j]) K->pidx[E++] = j;
  K->E = E;
  uint32_t P[kCrtWords] = {1};
  for (int e = 0; e < E; ++e) w_mul_small(P, kPrimes[K->pidx[e]]);
  std::memcpy(K->P, P, sizeof(P));
  // (P - 1) / 2 (P odd)
  uint32_t h[kCrtWords];
  std::memcpy(h, P, sizeof(P));
  h[0] -= 1;
  for (int l = 0; l < kCrtWords; ++l) h[l] = (h[l] >> 1) | (l + 1 < kCrtWords ? (h[l + 1] << 31) : 0);
  std::memcpy(K->Phalf, h, sizeof(h));
  for (int e = 0; e < E; ++e) {
    uint32_t q = kPrimes[K->pidx[e]];
    K->mq[e] = make_modq(q);
    uint32_t Mq[kCrtWords] = {1};
    for (int f = 0; f < E; ++f)
      if (f != e) w_mul_small(Mq, kPrimes[K->pidx[f]]);
    std::memcpy(K->Mq[e], Mq, sizeof(Mq));
    K->w[e] = inv_small(w_mod_small(Mq, q), q);
    K->tfix[e] = (1ull << 50) / q;
    K->t56[e] = (1ull << 56) / q;
  }
  // P^{-1} mod 2^64 by Newton's iteration x <- x (2 - P x) (P x = 1 mod 8 for x = P)
  uint64_t p64 = (uint64_t)P[0] | ((uint64_t)P[1] << 32), x = p64;
  for (int it = 0; it < 6; ++it) x *= 2 - p64 * x;
  K->Pinv64 = x;
  // byte matrix of the CRT product, row e (prime), column b (byte), as the B
  // fragments of mma.sync m16n8k16: lane = 4 g + t, register 0 holds rows
  // 16 ks + 2 t, + 1 and register 1 rows 16 ks + 2 t + 8, + 9, column 8 nt + g
  auto mbyte = [&](int e, int b) -> uint32_t {
    if (e >= E) return 0;
    if (b < 42) return (K->Mq[e][b / 4] >> (8 * (b % 4))) & 0xFFu;
    if (b < 49) return (uint32_t)((K->tfix[e] >> (8 * (b - 42))) & 0xFFu);
    return 0;
  };
  auto f16bits = [](uint32_t v) -> uint32_t {  // exact f16 of an integer 0 <= v <= 255
    if (v == 0) return 0;
    int ex = 0;
    while ((v >> ex) > 1) ++ex;                        // 2^ex <= v < 2^(ex+1)
    const uint32_t mant = (v << (10 - ex)) & 0x3FFu;  // ex <= 7: exact
    return ((uint32_t)(ex + 15) << 10) | mant;
  };
  for (int nt = 0; nt < kCrtNTiles; ++nt)
    for (int ks = 0; ks < 4; ++ks)
      for (int lane = 0; lane < 32; ++lane) {
        const int g = lane >> 2, t = lane & 3, col = 8 * nt + g;
        for (int rg = 0; rg < 2; ++rg) {
          const int e0 = 16 * ks + 2 * t + 8 * rg;
          K->crt_bfrag[nt][ks][lane][rg] = f16bits(mbyte(e0, col)) | (f16bits(mbyte(e0 + 1, col)) << 16);
        }
      }
}

// ------------------------------------------------------------ kernels
// r0 = b, R = residues of b.  Thread per entry, row fastest.
// r_0 = b and its residues: one thread per entry and prime (the primes'
// reductions are independent, so they run side by side rather than 53 in a
// row); the threads of prime 0 also copy the entry.
__global__ void k_lift_init(const int64_t* __restrict__ b, int64_t n, int64_t c, int64_t ld,
                            const LiftConst* __restrict__ K, int64_t* __restrict__ r, int8_t* __restrict__ R,
                            int col_major) {
  const int64_t nc = n * c;
  const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= nc * K->E) return;
  const int e = (int)(u / nc);
  const int64_t t = u - (int64_t)e * nc, row = t % n, col = t / n;
  const int64_t v = b[row * c + col];
  if (e == 0) r[col_major ? t : row * c + col] = v;
  R[((int64_t)e * c + col) * ld + row] = (int8_t)reduce_i64_bal(v, K->mq[e]);
}

// 16-byte load with an L2 cache-hint policy (createpolicy).
__device__ __forceinline__ int4 ld_hint(const int4* ptr, uint64_t pol) {
  int4 r;
  asm volatile("ld.global.L2::cache_hint.v4.s32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(ptr), "l"(pol));
  return r;
}
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// c == 1: V[e][i] = bal(sum_k B_j[i][k] R_e[k]).  Grid (n / (8 RPW), E'): each
// of the 8 warps takes RPW rows and walks them in rounds of 64 16-byte chunks
// (two per lane), issuing all of a round's loads before any dp4a so that
// 2 (RPW + 1) 16-byte loads per lane are in flight.  B is read every step:
// its loads carry an L2 evict-last hint so that, when it fits, it stays in L2
// across the steps instead of being streamed from HBM each time.
template <int RPW>
__global__ void __launch_bounds__(256) k_lift_gemv(const int8_t* __restrict__ B, const int8_t* __restrict__ R,
                                                   int64_t n, int64_t ld, const LiftConst* __restrict__ K,
                                                   int8_t* __restrict__ V) {
  const int e = blockIdx.y;
  const int j = K->pidx[e];
  const ModQ m = K->mq[e];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t row0 = (int64_t)blockIdx.x * (8 * RPW) + warp * RPW;
  const int4* Bj = reinterpret_cast<const int4*>(B + (int64_t)j * n * ld);
  const int4* Re = reinterpret_cast<const int4*>(R + (int64_t)e * ld);
  const int64_t chunks = ld / 16;
  int64_t roff[RPW];
#pragma unroll
  for (int u = 0; u < RPW; ++u) roff[u] = (row0 + u < n ? row0 + u : n - 1) * chunks;  // clamp; discarded
  int32_t acc[RPW];
#pragma unroll
  for (int u = 0; u < RPW; ++u) acc[u] = 0;
  const uint64_t keep = l2_evict_last_policy();
  for (int64_t k0 = 0; k0 < chunks; k0 += 64) {
    const int64_t ka = k0 + lane, kb = k0 + 32 + lane;
    const bool va = ka < chunks, vb = kb < chunks;
    const int4 z = make_int4(0, 0, 0, 0);
    const int4 ra = va ? __ldg(Re + ka) : z, rb = vb ? __ldg(Re + kb) : z;
    int4 ba[RPW], bb[RPW];
#pragma unroll
    for (int u = 0; u < RPW; ++u) {
      ba[u] = va ? ld_hint(Bj + roff[u] + ka, keep) : z;
      bb[u] = vb ? ld_hint(Bj + roff[u] + kb, keep) : z;
    }
#pragma unroll
    for (int u = 0; u < RPW; ++u) {
      acc[u] = __dp4a(ba[u].x, ra.x, acc[u]);
      acc[u] = __dp4a(ba[u].y, ra.y, acc[u]);
      acc[u] = __dp4a(ba[u].z, ra.z, acc[u]);
      acc[u] = __dp4a(ba[u].w, ra.w, acc[u]);
      acc[u] = __dp4a(bb[u].x, rb.x, acc[u]);
      acc[u] = __dp4a(bb[u].y, rb.y, acc[u]);
      acc[u] = __dp4a(bb[u].z, rb.z, acc[u]);
      acc[u] = __dp4a(bb[u].w, rb.w, acc[u]);
    }
  }
  int32_t mine = 0;
#pragma unroll
  for (int u = 0; u < RPW; ++u) {
    int32_t a = acc[u];
#pragma unroll
    for (int o = 16; o; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    if (lane == u) mine = a;
  }
  if (lane < RPW) {
    const int64_t i = row0 + lane;
    if (i < n) V[(int64_t)e * n + i] = (int8_t)reduce_bal(mine, m);
  }
}

// general c: V[e][i*c + col] = bal(sum_k B_j[i][k] R_e[col][k]).
// CTA tile 64 rows x 64 columns, K in chunks of 64 bytes, dp4a.
__global__ void __launch_bounds__(256) k_lift_gemm(const int8_t* __restrict__ B, const int8_t* __restrict__ R,
                                                   int64_t n, int64_t c, int64_t ld,
                                                   const LiftConst* __restrict__ K, int8_t* __restrict__ V) {
  const int e = blockIdx.z;
  const int j = K->pidx[e];
  const ModQ m = K->mq[e];
  const int64_t row0 = (int64_t)blockIdx.y * 64, col0 = (int64_t)blockIdx.x * 64;
  const int8_t* Bj = B + (int64_t)j * n * ld;
  const int8_t* Re = R + (int64_t)e * c * ld;
  __shared__ int32_t As[64][17];
  __shared__ int32_t Bs[64][17];
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  int32_t acc[4][4] = {};
  for (int64_t k0 = 0; k0 < ld; k0 += 64) {
    {
      int r = tid >> 2, cch = tid & 3;
      int64_t i = row0 + r, kk = k0 + 16 * cch;
      int4 v = make_int4(0, 0, 0, 0);
      if (i < n && kk < ld) v = *reinterpret_cast<const int4*>(Bj + i * ld + kk);
      As[r][cch * 4 + 0] = v.x;
      As[r][cch * 4 + 1] = v.y;
      As[r][cch * 4 + 2] = v.z;
      As[r][cch * 4 + 3] = v.w;
      int64_t col = col0 + r;
      int4 u = make_int4(0, 0, 0, 0);
      if (col < c && kk < ld) u = *reinterpret_cast<const int4*>(Re + col * ld + kk);
      Bs[r][cch * 4 + 0] = u.x;
      Bs[r][cch * 4 + 1] = u.y;
      Bs[r][cch * 4 + 2] = u.z;
      Bs[r][cch * 4 + 3] = u.w;
    }
    __syncthreads();
#pragma unroll
    for (int w = 0; w < 16; ++w) {
      int32_t a[4], bb[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) a[r] = As[ty * 4 + r][w];
#pragma unroll
      for (int u = 0; u < 4; ++u) bb[u] = Bs[tx + 16 * u][w];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[r][u] = __dp4a(a[r], bb[u], acc[r][u]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    int64_t i = row0 + ty * 4 + r;
    if (i >= n) continue;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      int64_t col = col0 + tx + 16 * u;
      if (col < c) V[(int64_t)e * n * c + i * c + col] = (int8_t)reduce_bal(acc[r][u], m);
    }
  }
}

// Limb s of x mod 2^64 in balanced base 256: x = sum_s d_s 256^s (mod 2^64)
// with d_s in [-128, 127] is byte s of x + 0x80...80, less 128.
__device__ __forceinline__ __half x_limb(uint64_t x, int s) {
  const uint64_t u = x + 0x8080808080808080ull;
  return __int2half_rn((int)((u >> (8 * s)) & 255u) - 128);
}

// Where the tcgen05 residual update runs, the CRT also writes the limbs of
// x_i mod 2^64 as f16 planes XL[na - 1 + s][col][i] (limb s, entry t = i c + col).
struct XLimbs {
  __half* XL;  // null: not written
  int64_t c, ld;
  int na;
};

// Same digit, one thread per entry (for many entries: no cross-lane work).
// The per-prime constants are staged in shared memory once per CTA, so the
// inner loop reads P'/q_e as three 16-byte broadcasts instead of twelve
// global loads.
__global__ void __launch_bounds__(128) k_lift_crt_thread(const int8_t* __restrict__ V, int64_t nc,
                                                         const LiftConst* __restrict__ K, uint64_t* __restrict__ D,
                                                         uint64_t* __restrict__ xl, XLimbs xo) {
  __shared__ __align__(16) uint32_t sMq[kNumPrimes * kCrtWords];
  __shared__ uint64_t sTf[kNumPrimes];
  __shared__ uint32_t sW[kNumPrimes], sQ[kNumPrimes], sMu[kNumPrimes];
  const int E = K->E;
  for (int i = threadIdx.x; i < E * kCrtWords; i += blockDim.x) sMq[i] = K->Mq[i / kCrtWords][i % kCrtWords];
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    sTf[e] = K->tfix[e];
    sW[e] = K->w[e];
    sQ[e] = K->mq[e].q;
    sMu[e] = K->mq[e].mu;
  }
  __syncthreads();
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= nc) return;
  uint64_t acc[kCrtWords];
#pragma unroll
  for (int l = 0; l < kCrtWords; ++l) acc[l] = 0;
  uint64_t tf = 0;
  // eight primes' residues are loaded before any is used, so that their
  // latencies overlap
#pragma unroll 1
  for (int e0 = 0; e0 < E; e0 += 8) {
    int32_t vv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) vv[u] = e0 + u < E ? V[(int64_t)(e0 + u) * nc + t] : 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = e0 + u;
      if (e >= E) break;
      ModQ m{};
      m.q = sQ[e];
      m.mu = sMu[e];
      const int32_t v = vv[u];
      const uint32_t ce = barrett((uint32_t)(v < 0 ? v + (int32_t)m.q : v) * sW[e], m);
      tf += (uint64_t)ce * sTf[e];
      const uint4* mq4 = reinterpret_cast<const uint4*>(sMq + e * kCrtWords);
#pragma unroll
      for (int h = 0; h < kCrtWords / 4; ++h) {
        const uint4 w = mq4[h];
        acc[4 * h] += (uint64_t)ce * w.x;
        acc[4 * h + 1] += (uint64_t)ce * w.y;
        acc[4 * h + 2] += (uint64_t)ce * w.z;
        acc[4 * h + 3] += (uint64_t)ce * w.w;
      }
    }
  }
  uint32_t S[kCrtWords];
  crt_finish(acc, tf, K, S);
  uint64_t* out = D + t * kDigitLimbs;
#pragma unroll
  for (int l = 0; l < kDigitLimbs; ++l) out[l] = (uint64_t)S[2 * l] | ((uint64_t)S[2 * l + 1] << 32);
  const uint64_t x = (uint64_t)S[0] | ((uint64_t)S[1] << 32);
  xl[t] = x;
  if (xo.XL) {
    const int64_t i = t / xo.c, col = t - i * xo.c;
#pragma unroll
    for (int s = 0; s < 8; ++s) xo.XL[((int64_t)(xo.na - 1 + s) * xo.c + col) * xo.ld + i] = x_limb(x, s);
  }
}

// The same digit from c_e = v_e w_e mod q_e in [0, q_e) (V holds c_e as bytes,
// as the tensor-core product writes them), with the word sums on the tensor
// cores: the byte columns S_b = sum_e c_e byte_b(P'/q_e) (and of floor(2^50/q_e))
// are one mma.sync m16n8k16 product of the [entries x primes] matrix of c_e by
// the constant [primes x 56] byte matrix, exact in the FP32 accumulator (each
// product < 2^16, 53 of them < 2^22).  CTA = 4 warps over four sub-tiles of
// 128 consecutive entries: per sub-tile the c_e tile is staged in shared
// memory, each warp forms the column sums of its 32 entries (two 16-row tiles
// x 7 column tiles x 4 k-steps), parks them in shared memory, and each lane
// assembles and finishes the digit of one entry.  The limb planes of x_i mod
// 2^64 (for the tensor-core residual) are written at the end, rows fastest.
__device__ __forceinline__ uint32_t u8pair_f16(uint32_t lo, uint32_t hi) {
  // 0x64uu is the f16 1024 + u; subtracting 1024 leaves u exactly
  uint32_t r = (lo & 0xFFu) | ((hi & 0xFFu) << 16) | 0x64006400u;
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(r) : "r"(0x64006400u));
  return r;
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
constexpr int kCrtDStride = 49;  // words per entry row of the parked sums (odd: no bank conflicts)
constexpr int kCrtSub = 2;       // 128-entry sub-tiles per CTA
__global__ void __launch_bounds__(128) k_lift_crt_mma(const uint8_t* __restrict__ V, int64_t nc,
                                                      const LiftConst* __restrict__ K, uint64_t* __restrict__ D,
                                                      uint64_t* __restrict__ xl, XLimbs xo) {
  __shared__ __align__(16) uint8_t sV[64][144];  // rows of 144 bytes: the fragment loads hit distinct banks
  __shared__ uint32_t sD[128 * kCrtDStride];
  __shared__ __align__(16) uint32_t sB[kCrtNTiles * 4 * 32 * 2];
  __shared__ uint64_t sX[kCrtSub * 128];
  __shared__ uint32_t sP[kCrtWords], sPh[kCrtWords];
  const int E = K->E;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
  const int64_t tcta = (int64_t)blockIdx.x * (128 * kCrtSub);
  {
    const uint4* src = reinterpret_cast<const uint4*>(&K->crt_bfrag[0][0][0][0]);
    for (int i = tid; i < kCrtNTiles * 4 * 32 * 2 / 4; i += 128) reinterpret_cast<uint4*>(sB)[i] = src[i];
    if (tid < kCrtWords) {
      sP[tid] = K->P[tid];
      sPh[tid] = K->Phalf[tid];
    }
  }
  // 16-byte pieces of the rows (all four of a thread's loads in flight at once);
  // the next sub-tile's pieces are loaded while this one is worked on
  const bool wide = (nc & 15) == 0;
  auto load_tile = [&](int64_t t0, uint4 (&v)[4]) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = tid + 128 * u, e = idx >> 3, q = idx & 7;
      v[u] = e < E ? *reinterpret_cast<const uint4*>(V + (int64_t)e * nc + t0 + 16 * q) : make_uint4(0, 0, 0, 0);
    }
  };
  uint4 pre[4];
  if (wide && tcta + 128 <= nc) load_tile(tcta, pre);
  for (int sub = 0; sub < kCrtSub; ++sub) {
    const int64_t t0 = tcta + 128 * sub, tt = t0 + tid;
    if (t0 >= nc) break;
    __syncthreads();  // the previous sub-tile's reads of sV are done (and the constants are in place)
    if (wide && t0 + 128 <= nc) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int idx = tid + 128 * u;
        *reinterpret_cast<uint4*>(&sV[idx >> 3][16 * (idx & 7)]) = pre[u];
      }
      if (sub + 1 < kCrtSub && wide && t0 + 256 <= nc) load_tile(t0 + 128, pre);
    } else {
#pragma unroll 8
      for (int e = 0; e < 64; ++e) sV[e][tid] = (e < E && tt < nc) ? V[(int64_t)e * nc + tt] : 0;
    }
    __syncthreads();
    // A fragments of this warp's two 16-entry tiles
    uint32_t a[2][4][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const int r0 = 32 * warp + 16 * mt + g;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const int e0 = 16 * ks + 2 * t4;
        a[mt][ks][0] = u8pair_f16(sV[e0][r0], sV[e0 + 1][r0]);
        a[mt][ks][1] = u8pair_f16(sV[e0][r0 + 8], sV[e0 + 1][r0 + 8]);
        a[mt][ks][2] = u8pair_f16(sV[e0 + 8][r0], sV[e0 + 9][r0]);
        a[mt][ks][3] = u8pair_f16(sV[e0 + 8][r0 + 8], sV[e0 + 9][r0 + 8]);
      }
    }
#pragma unroll
    for (int nt = 0; nt < kCrtNTiles; ++nt) {
      float d[2][4] = {};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint2 bb = *reinterpret_cast<const uint2*>(&sB[((nt * 4 + ks) * 32 + lane) * 2]);
        mma16816(d[0], a[0][ks], bb.x, bb.y);
        mma16816(d[1], a[1][ks], bb.x, bb.y);
      }
      const int c0 = 8 * nt + 2 * t4;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const int r0 = 32 * warp + 16 * mt + g;
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // columns c0, c0 + 1 (only the first 49 are used)
          if (c0 + h < kCrtDStride) {
            sD[r0 * kCrtDStride + c0 + h] = (uint32_t)d[mt][h];
            sD[(r0 + 8) * kCrtDStride + c0 + h] = (uint32_t)d[mt][2 + h];
          }
        }
      }
    }
    __syncwarp();
    if (tt < nc) {
      const uint32_t* col = sD + tid * kCrtDStride;  // this lane's entry: row 32 warp + lane = tid
      uint64_t acc[kCrtWords];
#pragma unroll
      for (int l = 0; l < kCrtWords; ++l) {
        uint64_t w = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (4 * l + j < 42) w += (uint64_t)col[4 * l + j] << (8 * j);
        acc[l] = w;
      }
      uint64_t tf = 0;
#pragma unroll
      for (int j = 0; j < 7; ++j) tf += (uint64_t)col[42 + j] << (8 * j);
      uint32_t S[kCrtWords];
      crt_finish(acc, tf, sP, sPh, S);
      // the digit's words go back into this entry's own row, for a coalesced store below
#pragma unroll
      for (int l = 0; l < kCrtWords; ++l) sD[tid * kCrtDStride + l] = S[l];
      const uint64_t x = (uint64_t)S[0] | ((uint64_t)S[1] << 32);
      xl[tt] = x;
      sX[128 * sub + tid] = x;
    }
    __syncthreads();
    {  // the sub-tile's digits are 48 contiguous bytes per entry: 16-byte stores
      const int cnt = (int)(nc - t0 < 128 ? nc - t0 : 128);
      uint8_t* dst = reinterpret_cast<uint8_t*>(D + t0 * kDigitLimbs);
      for (int ch = tid; ch < 3 * cnt; ch += 128) {
        const int en = ch / 3, part = ch - 3 * en;
        const uint32_t* w = sD + en * kCrtDStride + 4 * part;
        *reinterpret_cast<uint4*>(dst + 16 * ch) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
  if (!xo.XL) return;
  __syncthreads();
  // limb planes XL[na - 1 + s][col][i] of this CTA's entries [tcta, tcta + cnt):
  // walked with i fastest, so that consecutive threads store consecutive i
  const int64_t cnt = (nc - tcta) < 128 * kCrtSub ? (nc - tcta) : 128 * kCrtSub;
  const int64_t c = xo.c, i0 = tcta / c;
  const int nr = (int)((tcta + cnt - 1) / c - i0 + 1);  // rows touched (at most 512 / c + 2)
  const int cnr = (int)c * nr, total = 8 * cnr;          // c <= 2^24: fits 32 bits
  for (int idx = tid; idx < total; idx += 128) {
    const int s8 = idx / cnr, rem = idx - s8 * cnr, cl = rem / nr;
    const int64_t i = i0 + (rem - cl * nr), t = i * c + cl;
    if (t < tcta || t >= tcta + cnt) continue;
    xo.XL[((int64_t)(xo.na - 1 + s8) * c + cl) * xo.ld + i] = x_limb(sX[t - tcta], s8);
  }
}

// Balanced CRT of one entry: x = sum_e c_e (P'/q_e) - t P', c_e = v_e w_e mod q_e,
// t = floor(sum_e c_e / q_e) estimated in 2^-50 fixed point (exact or one too
// small), one conditional subtraction of P', then the balanced shift.
// One warp per entry: lane l takes primes l and l + 32, the 12 word sums and
// the fixed-point sum are reduced across the warp, and every lane finishes the
// (identical) digit; lanes 0..5 store its six limbs.
// kWeights: V holds the CRT weights c_e in [0, q_e) (as the tensor-core
// product writes them) instead of balanced residues.
template <bool kWeights>
__global__ void __launch_bounds__(256) k_lift_crt(const int8_t* __restrict__ V, int64_t nc,
                                                  const LiftConst* __restrict__ K, uint64_t* __restrict__ D,
                                                  uint64_t* __restrict__ xl, XLimbs xo) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= nc) return;
  const int E = K->E;
  const int32_t v0 = lane < E ? (kWeights ? (int32_t)(uint8_t)V[(int64_t)lane * nc + t] : V[(int64_t)lane * nc + t]) : 0;
  const int32_t v1 =
      lane + 32 < E ? (kWeights ? (int32_t)(uint8_t)V[(int64_t)(lane + 32) * nc + t] : V[(int64_t)(lane + 32) * nc + t])
                    : 0;
  uint32_t S[kCrtWords];
  crt_warp<kWeights>(v0, v1, lane, K, S);
  uint64_t limb = 0;
#pragma unroll
  for (int l = 0; l < kDigitLimbs; ++l)
    if (lane == l) limb = (uint64_t)S[2 * l] | ((uint64_t)S[2 * l + 1] << 32);
  if (lane < kDigitLimbs) D[t * kDigitLimbs + lane] = limb;
  if (lane == 0) xl[t] = limb;
  if (xo.XL && lane < 8) {
    const int64_t i = t / xo.c, col = t - i * xo.c;
    const uint64_t x = (uint64_t)S[0] | ((uint64_t)S[1] << 32);
    xo.XL[((int64_t)(xo.na - 1 + lane) * xo.c + col) * xo.ld + i] = x_limb(x, lane);
  }
}

template <typename AT>
__device__ __forceinline__ uint64_t mac64(uint64_t acc, AT a, uint64_t x) {
  return acc + (uint64_t)(int64_t)a * x;
}

// c == 1: r'[i] = (r[i] - sum_k A[i][k] xl[k]) Pinv mod 2^64 and its residues.
// Warp per row, 4 warps per CTA.  A is read through rows of stride lda
// (lda = 4-aligned with zero padding for the int32 copy, so 16-byte loads),
// xl is zero beyond n.
template <typename AT>
__device__ __forceinline__ uint64_t row_dot(const AT* __restrict__ Ai, const uint64_t* __restrict__ xl, int64_t n,
                                            int lane);
template <>
__device__ __forceinline__ uint64_t row_dot<int32_t>(const int32_t* __restrict__ Ai,
                                                     const uint64_t* __restrict__ xl, int64_t n, int lane) {
  const int4* A4 = reinterpret_cast<const int4*>(Ai);
  const ulonglong2* X2 = reinterpret_cast<const ulonglong2*>(xl);
  const int64_t q = (n + 3) / 4;
  uint64_t s0 = 0, s1 = 0;
  int64_t k = lane;
  for (; k + 32 < q; k += 64) {
    const int4 a0 = __ldg(A4 + k), a1 = __ldg(A4 + k + 32);
    const ulonglong2 x0 = __ldg(X2 + 2 * k), x1 = __ldg(X2 + 2 * k + 1);
    const ulonglong2 y0 = __ldg(X2 + 2 * (k + 32)), y1 = __ldg(X2 + 2 * (k + 32) + 1);
    s0 += (uint64_t)(int64_t)a0.x * x0.x + (uint64_t)(int64_t)a0.y * x0.y + (uint64_t)(int64_t)a0.z * x1.x +
          (uint64_t)(int64_t)a0.w * x1.y;
    s1 += (uint64_t)(int64_t)a1.x * y0.x + (uint64_t)(int64_t)a1.y * y0.y + (uint64_t)(int64_t)a1.z * y1.x +
          (uint64_t)(int64_t)a1.w * y1.y;
  }
  for (; k < q; k += 32) {
    const int4 a0 = __ldg(A4 + k);
    const ulonglong2 x0 = __ldg(X2 + 2 * k), x1 = __ldg(X2 + 2 * k + 1);
    s0 += (uint64_t)(int64_t)a0.x * x0.x + (uint64_t)(int64_t)a0.y * x0.y + (uint64_t)(int64_t)a0.z * x1.x +
          (uint64_t)(int64_t)a0.w * x1.y;
  }
  return s0 + s1;
}
template <>
__device__ __forceinline__ uint64_t row_dot<int64_t>(const int64_t* __restrict__ Ai,
                                                     const uint64_t* __restrict__ xl, int64_t n, int lane) {
  uint64_t s = 0;
  for (int64_t k = lane; k < n; k += 32) s += (uint64_t)__ldg(Ai + k) * __ldg(xl + k);
  return s;
}

template <typename AT>
__global__ void __launch_bounds__(128) k_lift_resid_gemv(const AT* __restrict__ A, int64_t lda,
                                                         const uint64_t* __restrict__ xl,
                                                         const int64_t* __restrict__ r, int64_t n, int64_t ld,
                                                         const LiftConst* __restrict__ K,
                                                         int64_t* __restrict__ rn, int8_t* __restrict__ R) {
  const int lane = threadIdx.x & 31;
  const int64_t i = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (i >= n) return;
  uint64_t s = row_dot<AT>(A + i * lda, xl, n, lane);
#pragma unroll
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const int64_t v = (int64_t)(((uint64_t)r[i] - s) * K->Pinv64);
  if (lane == 0) rn[i] = v;
  const int E = K->E;
  for (int e = lane; e < E; e += 32) R[(int64_t)e * ld + i] = (int8_t)reduce_i64_bal(v, K->mq[e]);
}

// general c: r'[i][col] = (r[i][col] - sum_k A[i][k] x[k][col]) Pinv mod 2^64
// and its residues.  CTA tile TR rows (16, or 8 for small grids) x 16
// columns.  Its 256 threads are TR thread tiles of 4 x 4 outputs times
// 256 / TR slices of K (slice s takes the groups k = 4s + 4 S t .. 4s + 4 S t + 3
// for S slices); the slices' partial sums meet in shared memory, one thread per
// output adds them, and all threads then share the E residues of the tile's
// 16 TR new residual entries (four rows, one 32-bit store, per task).
// For int32 A the product uses x = x_lo + 2^32 x_hi with x_lo read as a
// signed int32 and its borrow folded into the high word (x_hi' = x_hi +
// (x_lo >> 31)):
//   A x mod 2^64 = sum_k A x_lo_s (exact int64) + 2^32 (sum_k A x_hi' mod 2^32),
// one 32 x 32 -> 64 multiply-add and one 32-bit multiply-add per term; A is
// the zero-padded int32 copy (lda = padded row length, a multiple of 16) and
// x is zero for k >= n, so whole groups of four run to lda.  For int64 A
// (entries of 2^31 or more, lda = n) the terms are full 64-bit products and
// the groups stop at n.
constexpr int kResidTile = 16;           // columns per CTA of the tiled residual update
constexpr int64_t kResidSmallGrid = 152;  // below 2 x this many 16-row CTAs: 8-row tiles

template <typename AT, bool VecX>
__device__ __forceinline__ void resid_group(const AT* __restrict__ A, int64_t lda, const uint64_t* __restrict__ xl,
                                            int64_t n, int64_t c, const int64_t (&arow)[4], int64_t col,
                                            int64_t k, uint64_t (&acc)[4][4], uint32_t (&hi)[4][4]);

// int32 A: four k at once (int4 of each row), x for four columns per k
template <>
__device__ __forceinline__ void resid_group<int32_t, true>(const int32_t* __restrict__ A, int64_t lda,
                                                           const uint64_t* __restrict__ xl, int64_t n, int64_t c,
                                                           const int64_t (&arow)[4], int64_t col, int64_t k,
                                                           uint64_t (&acc)[4][4], uint32_t (&hi)[4][4]) {
  int32_t a[4][4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int4 v = __ldg(reinterpret_cast<const int4*>(A + arow[q] * lda + k));
    a[q][0] = v.x;
    a[q][1] = v.y;
    a[q][2] = v.z;
    a[q][3] = v.w;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // c is a multiple of four: a column group lies wholly inside or outside [0, c)
    const ulonglong2* X2 = reinterpret_cast<const ulonglong2*>(xl + (k + j) * c + col);
    const ulonglong2 z = make_ulonglong2(0, 0);
    const ulonglong2 x01 = col < c ? __ldg(X2) : z, x23 = col < c ? __ldg(X2 + 1) : z;
    const uint64_t x[4] = {x01.x, x01.y, x23.x, x23.y};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t lo = (uint32_t)x[u];
      const int64_t los = (int64_t)(int32_t)lo;
      const uint32_t hw = (uint32_t)(x[u] >> 32) + (lo >> 31);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[q][u] += (uint64_t)((int64_t)a[q][j] * los);
        hi[q][u] += (uint32_t)a[q][j] * hw;
      }
    }
  }
}

// int32 A, c not a multiple of four: x read one column at a time
template <>
__device__ __forceinline__ void resid_group<int32_t, false>(const int32_t* __restrict__ A, int64_t lda,
                                                            const uint64_t* __restrict__ xl, int64_t n, int64_t c,
                                                            const int64_t (&arow)[4], int64_t col, int64_t k,
                                                            uint64_t (&acc)[4][4], uint32_t (&hi)[4][4]) {
  int32_t a[4][4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int4 v = __ldg(reinterpret_cast<const int4*>(A + arow[q] * lda + k));
    a[q][0] = v.x;
    a[q][1] = v.y;
    a[q][2] = v.z;
    a[q][3] = v.w;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint64_t x = col + u < c ? __ldg(xl + (k + j) * c + col + u) : 0;
      const uint32_t lo = (uint32_t)x;
      const int64_t los = (int64_t)(int32_t)lo;
      const uint32_t hw = (uint32_t)(x >> 32) + (lo >> 31);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[q][u] += (uint64_t)((int64_t)a[q][j] * los);
        hi[q][u] += (uint32_t)a[q][j] * hw;
      }
    }
  }
}

// int64 A: plain 64-bit products, k < n
template <>
__device__ __forceinline__ void resid_group<int64_t, false>(const int64_t* __restrict__ A, int64_t lda,
                                                            const uint64_t* __restrict__ xl, int64_t n, int64_t c,
                                                            const int64_t (&arow)[4], int64_t col, int64_t k,
                                                            uint64_t (&acc)[4][4], uint32_t (&)[4][4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (k + j >= n) break;
    uint64_t x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) x[u] = col + u < c ? __ldg(xl + (k + j) * c + col + u) : 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint64_t a = (uint64_t)__ldg(A + arow[q] * lda + k + j);
#pragma unroll
      for (int u = 0; u < 4; ++u) acc[q][u] += a * x[u];
    }
  }
}

template <typename AT, bool VecX, int TR>
__global__ void __launch_bounds__(256) k_lift_resid_tile(const AT* __restrict__ A, int64_t lda,
                                                         const uint64_t* __restrict__ xl,
                                                         const int64_t* __restrict__ r, int64_t n, int64_t c,
                                                         int64_t ld, const LiftConst* __restrict__ K,
                                                         int64_t* __restrict__ rn, int8_t* __restrict__ R) {
  constexpr int T = kResidTile;      // columns per CTA
  constexpr int G4 = TR / 4;         // groups of four rows
  constexpr int SUBS = G4 * 4;       // 4 x 4 thread tiles
  constexpr int SL = 256 / SUBS;     // K slices
  static_assert(TR == 8 || TR == 16, "row tile");
  __shared__ uint64_t part[SL][TR * T];
  __shared__ int64_t vs[T][TR + 1];  // [column][row]
  const int tid = threadIdx.x, sub = tid % SUBS, s = tid / SUBS;
  const int rg = sub >> 2, cg = sub & 3;
  const int64_t row0 = (int64_t)blockIdx.x * TR, col0 = (int64_t)blockIdx.y * T;
  const int64_t col = col0 + 4 * cg;
  int64_t arow[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int64_t i = row0 + 4 * rg + q;
    arow[q] = i < n ? i : n - 1;  // clamped; its result is discarded
  }
  uint64_t acc[4][4];
  uint32_t hi[4][4];
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      acc[q][u] = 0;
      hi[q][u] = 0;
    }
  const int64_t kend = sizeof(AT) == 4 ? lda : n;
  for (int64_t k = 4 * s; k < kend; k += 4 * SL) resid_group<AT, VecX>(A, lda, xl, n, c, arow, col, k, acc, hi);
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int u = 0; u < 4; ++u)
      part[s][(4 * rg + q) * T + 4 * cg + u] = acc[q][u] + ((uint64_t)hi[q][u] << 32);
  __syncthreads();
  if (tid < TR * T) {
    const int rl = tid / T, cl = tid % T;
    const int64_t i = row0 + rl, cc = col0 + cl;
    uint64_t sum = 0;
#pragma unroll
    for (int t = 0; t < SL; ++t) sum += part[t][tid];
    int64_t v = 0;
    if (i < n && cc < c) {
      v = (int64_t)(((uint64_t)r[i * c + cc] - sum) * K->Pinv64);
      rn[i * c + cc] = v;
    }
    vs[cl][rl] = v;
  }
  __syncthreads();
  const int E = K->E;
  for (int t = tid; t < E * T * G4; t += 256) {
    const int e = t / (T * G4), cl = (t / G4) % T, g = t % G4;
    const int64_t cc = col0 + cl;
    if (cc >= c) continue;
    const ModQ m = K->mq[e];
    uint32_t w = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) w |= (uint32_t)(uint8_t)(int8_t)reduce_i64_bal(vs[cl][4 * g + b], m) << (8 * b);
    *reinterpret_cast<uint32_t*>(R + ((int64_t)e * c + cc) * ld + row0 + 4 * g) = w;
  }
}

// A32[i][k] = A[i][k] for k < n, 0 for n <= k < lda.
__global__ void k_narrow_a(const int64_t* __restrict__ A, int64_t n, int64_t lda, int32_t* __restrict__ A32) {
  int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n * lda) return;
  int64_t i = t / lda, k = t - i * lda;
  A32[t] = k < n ? (int32_t)A[i * n + k] : 0;
}

// ------------------------------------------------------------ driver
namespace {
constexpr int64_t kTcMinCols = 16;       // c >= 16: product on tcgen05 (k_lift_tc.cu)
constexpr int64_t kResidTcMinN = 1024;   // from this n: the residual update on tcgen05 (k_lift_tc.cu)
constexpr int64_t kCrtThreadMin = 32768;  // from this many entries: one thread per entry
constexpr int64_t kCrtMmaMin = 32768;     // tensor-core product path: from this many entries the CRT on mma.sync
struct LiftLayout {
  size_t K, R, V, r, xl, A32, R16, A16, X16, Sacc, Bf, Bt, err, bar, total;
};
LiftLayout lift_layout(int64_t n, int64_t c, int E, bool a32) {
  int64_t ld = padded_ld(n);
  const bool tc = c >= kTcMinCols;
  Layout L;
  LiftLayout o;
  o.K = L.add(sizeof(LiftConst));
  o.R = L.add((size_t)E * c * ld);
  o.V = L.add((size_t)E * n * c);
  o.r = L.add((size_t)2 * n * c * 8);
  o.xl = L.add((size_t)padded_ld(n) * c * 8);
  o.A32 = a32 ? L.add((size_t)n * padded_ld(n) * 4) : 0;
  o.R16 = tc ? L.add((size_t)E * c * ld * 2) : 0;
  o.A16 = tc && a32 ? L.add((size_t)kResidLimbsMax * n * ld * 2) : 0;
  o.X16 = tc && a32 ? L.add((size_t)(kResidLimbsMax + 7) * c * ld * 2) : 0;
  o.Sacc = tc && a32 ? L.add((size_t)n * c * 8) : 0;
  o.Bf = (c == 1 && ld <= kFusedMaxLd) ? L.add((size_t)E * n * ld) : 0;
  o.Bt = tc ? L.add(tc_tiled_b_bytes(n, E)) : 0;
  o.err = L.add(sizeof(int));
  o.bar = L.add(sizeof(unsigned));
  o.total = L.total;
  return o;
}
}  // namespace

size_t lift_scratch_bytes(int64_t n, int64_t c, int E, bool a32) { return lift_layout(n, c, E, a32).total; }

LiftRun::~LiftRun() {
  for (void* e : ev)
    if (e) cudaEventDestroy((cudaEvent_t)e);
}

namespace {
es_status create_events(LiftRun* run, size_t count) {
  for (void* e : run->ev)
    if (e) cudaEventDestroy((cudaEvent_t)e);
  run->ev.assign(count, nullptr);
  for (auto& e : run->ev) {
    cudaEvent_t x = nullptr;
    ES_CHECK(cuda_status(cudaEventCreate(&x), "event create"));
    e = x;
  }
  return ES_OK;
}
}  // namespace

es_status run_lift_start(const int64_t* A_dev, const int64_t* b_dev, int64_t n, int64_t c, const int8_t* B_dev,
                         const uint8_t* good_host, int32_t m, uint64_t* digits_dev, uint64_t max_abs_a,
                         char* scratch, void* stream, KernelTiming* kt, bool allow_fused, LiftRun* run,
                         bool stall_barrier, const DigitStream* stream_digits) {
  cudaStream_t st = (cudaStream_t)stream;
  const bool a32 = max_abs_a < (uint64_t(1) << 31);
  LiftConst hK;
  build_lift_const(good_host, &hK);
  if (hK.E == 0) return ES_ERR_ARG;
  const int E = hK.E;
  const int64_t ld = padded_ld(n), nc = n * c;
  LiftLayout L = lift_layout(n, c, E, a32);
  LiftConst* K = reinterpret_cast<LiftConst*>(scratch + L.K);
  int8_t* R = reinterpret_cast<int8_t*>(scratch + L.R);
  int8_t* V = reinterpret_cast<int8_t*>(scratch + L.V);
  int64_t* r[2] = {reinterpret_cast<int64_t*>(scratch + L.r), reinterpret_cast<int64_t*>(scratch + L.r) + nc};
  uint64_t* xl = reinterpret_cast<uint64_t*>(scratch + L.xl);
  int32_t* A32 = a32 ? reinterpret_cast<int32_t*>(scratch + L.A32) : nullptr;
  const bool tc = c >= kTcMinCols;
  void* R16 = tc ? (void*)(scratch + L.R16) : nullptr;
  // tcgen05 residual update with the tcgen05 product (entries below 2^31,
  // n >= kResidTcMinN: below that its few CTAs, each forming the residues of
  // 128 x 8 entries, lose to the CUDA-core update)
  int na = tc && a32 && n >= kResidTcMinN ? resid_limbs(max_abs_a) : 0;
  if ((int64_t)na * n > kResidTcMaxK) na = 0;
  TcResid tcr;
  XLimbs xo{nullptr, c, ld, na};
  if (na) xo.XL = reinterpret_cast<__half*>(scratch + L.X16);
  int* err = reinterpret_cast<int*>(scratch + L.err);
  unsigned* bar = reinterpret_cast<unsigned*>(scratch + L.bar);
  TcLift tcl;
  int device = 0;
  ES_CHECK(cuda_status(cudaGetDevice(&device), "get device"));
  FusedPlan fp;
  bool fused = allow_fused && L.Bf && fused_lift_plan(n, c, E, device, &fp);
  int8_t* Bf = fused ? reinterpret_cast<int8_t*>(scratch + L.Bf) : nullptr;

  // LiftConst lives in pageable host memory on this thread's stack: copy it
  // synchronously with respect to the host before returning.
  ES_CHECK(cuda_status(cudaMemcpyAsync(K, &hK, sizeof(hK), cudaMemcpyHostToDevice, st), "lift const H2D"));
  ES_CHECK(cuda_status(cudaMemsetAsync(R, 0, (size_t)E * c * ld, st), "memset R"));
  ES_CHECK(cuda_status(cudaMemsetAsync(xl, 0, (size_t)padded_ld(n) * c * 8, st), "memset xl"));
  ES_CHECK(cuda_status(cudaMemsetAsync(err, 0, sizeof(int), st), "memset err"));
  if (stall_barrier) {
    // arrivals wrap the counter to G - 11 < G: the first barrier never completes
    static const unsigned kStalled = 0u - 11u;
    ES_CHECK(cuda_status(cudaMemcpyAsync(bar, &kStalled, sizeof(unsigned), cudaMemcpyHostToDevice, st),
                         "barrier init"));
  } else {
    ES_CHECK(cuda_status(cudaMemsetAsync(bar, 0, sizeof(unsigned), st), "memset barrier"));
  }
  if (tc) {
    int8_t* Bt = reinterpret_cast<int8_t*>(scratch + L.Bt);
    ES_CHECK(tc_prepare(&tcl, Bt, R16, n, c, ld, E));
    ES_CHECK(tc_tile_b(B_dev, K, Bt, n, ld, E, st));
  }
  uint64_t* Sacc = na ? reinterpret_cast<uint64_t*>(scratch + L.Sacc) : nullptr;
  if (na) {
    ES_CHECK(tc_resid_prepare(&tcr, A_dev, scratch + L.A16, xo.XL, n, c, ld, na, st));
    ES_CHECK(cuda_status(cudaMemsetAsync(Sacc, 0, (size_t)nc * 8, st), "memset Sacc"));
  }
  if (a32 && !na) {
    k_narrow_a<<<(unsigned)((n * ld + 255) / 256), 256, 0, st>>>(A_dev, n, ld, A32);
    ES_CHECK(cuda_status(cudaGetLastError(), "k_narrow_a"));
  }
  // the tensor-core residual keeps r column by column ([c][n]), so that forming
  // r_{i+1} and its residues reads and writes whole columns
  k_lift_init<<<(unsigned)((nc * E + 255) / 256), 256, 0, st>>>(b_dev, n, c, ld, K, r[0], R, na ? 1 : 0);
  ES_CHECK(cuda_status(cudaGetLastError(), "k_lift_init"));
  count_launch(a32 && !na ? 2 : 1);
  run->stream = stream;
  run->kt = kt;
  if (kt && kt->events) ES_CHECK(create_events(run, fused ? 2 : 2 * (size_t)m));
  auto ev = [&](size_t i) { return (cudaEvent_t)run->ev[i]; };
  if (fused) {
    ES_CHECK(fused_lift_relayout(fp, B_dev, K, Bf, n, st));
    count_launch();
    if (!run->ev.empty()) cudaEventRecord(ev(0), st);
    es_status fs = fused_lift_launch(fp, Bf, A32, a32 ? nullptr : A_dev, b_dev, K, R, xl, digits_dev, bar, err,
                                     n, E, m, st, stream_digits);
    if (fs == ES_OK) {
      if (!run->ev.empty()) cudaEventRecord(ev(1), st);
      count_launch();
    } else if (fs == ES_ERR_RANGE) {
      fused = false;  // co-residency refused: per-step kernels below
      if (kt && kt->events) ES_CHECK(create_events(run, 2 * (size_t)m));
    } else {
      return fs;
    }
  }
  for (int32_t i = 0; i < m && !fused; ++i) {
    // the tcgen05 residual update writes R16 itself; step 0 converts the residues of b
    if (tc && (i == 0 || !na)) ES_CHECK(tc_convert_f16(R, R16, (int64_t)E * c * ld, st));
    if (!run->ev.empty()) cudaEventRecord(ev(2 * i), st);
    if (c == 1) {
      k_lift_gemv<4><<<dim3((unsigned)((n + 31) / 32), E), 256, 0, st>>>(B_dev, R, n, ld, K, V);
      count_launch();
    } else if (tc) {
      ES_CHECK(tc_launch(tcl, K, V, n, c, ld, E, err, st));
    } else {
      k_lift_gemm<<<dim3((unsigned)((c + 63) / 64), (unsigned)((n + 63) / 64), E), 256, 0, st>>>(B_dev, R, n, c,
                                                                                                ld, K, V);
      count_launch();
    }
    if (!run->ev.empty()) cudaEventRecord(ev(2 * i + 1), st);
    count_launch();
    if (tc && nc >= kCrtMmaMin)
      k_lift_crt_mma<<<(unsigned)((nc + 128 * kCrtSub - 1) / (128 * kCrtSub)), 128, 0, st>>>(
          reinterpret_cast<const uint8_t*>(V), nc, K, digits_dev + (size_t)i * nc * kDigitLimbs, xl, xo);
    else if (tc)  // few entries: one warp each, from the CRT weights
      k_lift_crt<true><<<(unsigned)((nc + 7) / 8), 256, 0, st>>>(V, nc, K, digits_dev + (size_t)i * nc * kDigitLimbs,
                                                                 xl, xo);
    else if (nc >= kCrtThreadMin)
      k_lift_crt_thread<<<(unsigned)((nc + 127) / 128), 128, 0, st>>>(V, nc, K, digits_dev + (size_t)i * nc * kDigitLimbs,
                                                                      xl, xo);
    else
      k_lift_crt<false><<<(unsigned)((nc + 7) / 8), 256, 0, st>>>(V, nc, K, digits_dev + (size_t)i * nc * kDigitLimbs,
                                                                  xl, xo);
    if (i + 1 < m) {
      const int64_t* rc = r[i & 1];
      int64_t* rn = r[(i + 1) & 1];
      if (na) {
        ES_CHECK(tc_resid_launch(tcr, K, rc, rn, Sacc, R16, n, c, ld, err, st));
        continue;
      }
      count_launch(1);
      if (c == 1) {
        if (a32)
          k_lift_resid_gemv<int32_t><<<(unsigned)((n + 3) / 4), 128, 0, st>>>(A32, ld, xl, rc, n, ld, K, rn, R);
        else
          k_lift_resid_gemv<int64_t><<<(unsigned)((n + 3) / 4), 128, 0, st>>>(A_dev, n, xl, rc, n, ld, K, rn, R);
      } else {
        // 16-row tiles, or 8-row ones (twice the CTAs, K in 32 slices) while
        // there would be fewer than two per SM
        const unsigned gy = (unsigned)((c + kResidTile - 1) / kResidTile);
        const bool small = ((n + 15) / 16) * (int64_t)gy < 2 * kResidSmallGrid;
        const dim3 g((unsigned)((n + (small ? 7 : 15)) / (small ? 8 : 16)), gy);
        if (a32 && c % 4 == 0) {
          if (small)
            k_lift_resid_tile<int32_t, true, 8><<<g, 256, 0, st>>>(A32, ld, xl, rc, n, c, ld, K, rn, R);
          else
            k_lift_resid_tile<int32_t, true, 16><<<g, 256, 0, st>>>(A32, ld, xl, rc, n, c, ld, K, rn, R);
        } else if (a32) {
          if (small)
            k_lift_resid_tile<int32_t, false, 8><<<g, 256, 0, st>>>(A32, ld, xl, rc, n, c, ld, K, rn, R);
          else
            k_lift_resid_tile<int32_t, false, 16><<<g, 256, 0, st>>>(A32, ld, xl, rc, n, c, ld, K, rn, R);
        } else {
          if (small)
            k_lift_resid_tile<int64_t, false, 8><<<g, 256, 0, st>>>(A_dev, n, xl, rc, n, c, ld, K, rn, R);
          else
            k_lift_resid_tile<int64_t, false, 16><<<g, 256, 0, st>>>(A_dev, n, xl, rc, n, c, ld, K, rn, R);
        }
      }
    }
  }
  ES_CHECK(cuda_status(cudaGetLastError(), "lift steps"));
  run->err = err;
  run->fused = fused;
  run->tc = tc;
  run->a32 = a32;
  run->E = E;
  run->n = n;
  run->c = c;
  run->m = m;
  return ES_OK;
}

es_status run_lift_finish(LiftRun* run) {
  cudaStream_t st = (cudaStream_t)run->stream;
  int herr = 0;
  ES_CHECK(cuda_status(cudaMemcpyAsync(&herr, run->err, sizeof(int), cudaMemcpyDeviceToHost, st), "lift err D2H"));
  es_status sst = cuda_status(cudaStreamSynchronize(st), "lift sync");
  const bool fused = run->fused;
  if (sst == ES_OK && herr == kFusedErrDigit) {
    set_last_error("fused lift kernel: the short-path digit disagreed with the full digit");
    sst = ES_ERR_INTERNAL;
  } else if (sst == ES_OK && herr) {
    set_last_error(std::string(fused ? "fused lift kernel" : "lift step kernels") +
                   ": bounded wait expired (code " + std::to_string(herr) + ")");
    sst = ES_ERR_TIMEOUT;
  }
  if (KernelTiming* kt = run->kt) {
    const int64_t n = run->n, c = run->c;
    const int E = run->E;
    kt->launches += fused ? 1 : run->m;
    // algorithmic bytes: per step E' n^2 of B, w_A n^2 of A and n (8 + E' + 48)
    // for the residual, its residues and the digit (fused: all m steps);
    // per-step product kernels: E' (n^2 + 2 n c)
    const double nn = (double)n * (double)n;
    kt->bytes_per_launch = fused ? (double)run->m * (E * nn + (run->a32 ? 4.0 : 8.0) * nn + (double)n * (8.0 + E + 48.0))
                                 : (double)E * (nn + 2.0 * (double)n * (double)c);
    kt->fused = fused;
    kt->name = fused ? "k_lift_fused" : c == 1 ? "k_lift_gemv" : run->tc ? "k_lift_gemm_tc" : "k_lift_gemm";
    for (size_t i = 0; i + 1 < run->ev.size(); i += 2) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, (cudaEvent_t)run->ev[i], (cudaEvent_t)run->ev[i + 1]) == cudaSuccess) kt->ms += ms;
    }
  }
  return sst;
}

es_status run_lift(const int64_t* A_dev, const int64_t* b_dev, int64_t n, int64_t c, const int8_t* B_dev,
                   const uint8_t* good_host, int32_t m, uint64_t* digits_dev, uint64_t max_abs_a, char* scratch,
                   void* stream, KernelTiming* kt, bool allow_fused) {
  LiftRun run;
  ES_CHECK(run_lift_start(A_dev, b_dev, n, c, B_dev, good_host, m, digits_dev, max_abs_a, scratch, stream, kt,
                          allow_fused, &run));
  return run_lift_finish(&run);
}

}  // namespace es
