// Internal declarations shared by the lift translation units.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "es_common.cuh"
#include "es_internal.h"

namespace es {

constexpr int kCrtNTiles = 7;  // 56 byte columns of the CRT product

struct LiftConst {
  int32_t E;                      // number of good primes
  int32_t pidx[kNumPrimes];       // their indices in the prime table, ascending
  ModQ mq[kNumPrimes];            // reduction constants, compact order
  uint32_t w[kNumPrimes];         // (P'/q)^{-1} mod q
  uint64_t tfix[kNumPrimes];      // floor(2^50 / q)
  uint64_t t56[kNumPrimes];       // floor(2^56 / q)
  uint32_t Mq[kNumPrimes][kCrtWords];  // P'/q, 32-bit little-endian words
  uint32_t P[kCrtWords];          // P'
  uint32_t Phalf[kCrtWords];      // (P' - 1) / 2
  uint64_t Pinv64;                // P'^{-1} mod 2^64
  // The CRT as one small matrix product (k_lift_crt_mma): with c_e in [0, q_e)
  // the digit's word sums are sum_e c_e P'/q_e, and the fixed-point quotient
  // estimate is sum_e c_e floor(2^50/q_e).  Byte columns 0..41 hold the bytes
  // of P'/q_e, columns 42..48 those of floor(2^50/q_e), 49..55 are zero; rows
  // are the primes (zero from E').  Stored as the B fragments of mma.sync
  // m16n8k16 (f16 pairs): [n-tile 7][k-step 4][lane 32][register 2].
  uint32_t crt_bfrag[kCrtNTiles][4][32][2];
};

// tcgen05 lift product (k_lift_tc.cu), used for c >= 16.  It reads the
// inverses of the good primes from a tiled copy Bt [E'][n / 128][ld / 128]
// [128][128] (rounded up, zero padded): each 128 x 128 tile one contiguous
// 16 KB block, so that every copy streams whole DRAM pages.
struct TcLift {
  CUtensorMap mapB;  // int8 Bt, one 128 x 128 tile per plane
  CUtensorMap mapR;  // f16 [E'][c][ld] residues of r_i
  int nt = 64;       // MMA N tile
  int tiles_m = 0, kstages = 0;
};
size_t tc_tiled_b_bytes(int64_t n, int E);
es_status tc_convert_f16(const int8_t* src, void* dst, int64_t count, void* stream);
es_status tc_prepare(TcLift* t, const int8_t* Bt, const void* R16, int64_t n, int64_t c, int64_t ld, int E);
// B [53][n][ld] (good primes via K->pidx) -> Bt, once per lift.
es_status tc_tile_b(const int8_t* B, const LiftConst* K, int8_t* Bt, int64_t n, int64_t ld, int E, void* stream);
es_status tc_launch(const TcLift& t, const LiftConst* K, int8_t* V, int64_t n, int64_t c, int64_t ld, int E,
                    int* err, void* stream);

// tcgen05 residual update (k_lift_tc.cu), used with the tcgen05 product when
// max|A| < 2^31: A and x_i mod 2^64 in balanced 8-bit limbs, A x_i mod 2^64
// as f16 GEMMs (one per limb plane of A) summed into Sacc [c][n] (zero on
// entry, cleared again once r_{i+1} is formed; r and r_{i+1} are [c][n] too).
constexpr int kResidLimbsMax = 4;      // limbs of A (|A| < 2^31)
constexpr int64_t kResidTcMaxK = 65536;  // na n at most this: int32 sums stay exact
struct TcResid {
  CUtensorMap mapA;  // f16 [na][n][ld]      limbs of A, zero for k >= n
  CUtensorMap mapX;  // f16 [na + 7][c][ld]  limbs of x_i mod 2^64 on planes na - 1 .. na + 6, the rest zero
  int na = 0;        // limbs of A
  int kbp = 0;       // 64-wide K blocks per limb plane
  int nc = 32;       // columns per CTA (MMA N = 8 nc)
};
int resid_limbs(uint64_t max_abs_a);  // na for entries up to max_abs_a (0: not representable)
es_status tc_resid_prepare(TcResid* t, const int64_t* A_dev, void* A16, void* X16, int64_t n, int64_t c, int64_t ld,
                           int na, void* stream);
es_status tc_resid_launch(const TcResid& t, const LiftConst* K, const int64_t* r, int64_t* rn, uint64_t* Sacc,
                          void* R16, int64_t n, int64_t c, int64_t ld, int* err, void* stream);

constexpr int kFusedErrDigit = 15;  // error code: the fused lift's two digit paths disagreed

// Fused single-launch lift for c == 1 (k_lift_fused.cu), for n <= kFusedMaxLd:
// each consumer warp keeps its row of A (int32) in registers.
constexpr int64_t kFusedMaxLd = 1024;
struct FusedPlan {
  int G = 0;         // CTAs (one per SM, at most n)
  int slots = 0;     // ring slots per CTA
  int slot_bytes = 0;  // bytes per ring slot (two primes x the most owned rows)
  size_t smem = 0;   // dynamic shared memory per CTA
  size_t relayout_bytes = 0;  // B in the order of ownership (E' n ld bytes)
};
bool fused_lift_plan(int64_t n, int64_t c, int E, int device, FusedPlan* p);
// B [53][n][ld] -> Bf [n][E'][ld] in the order of row ownership.
es_status fused_lift_relayout(const FusedPlan& p, const int8_t* B, const LiftConst* K, int8_t* Bf, int64_t n,
                              void* stream);
// ES_ERR_RANGE when the cooperative launch is refused (then nothing ran).
es_status fused_lift_launch(const FusedPlan& p, const int8_t* Bf, const int32_t* A32, const int64_t* A64,
                            const int64_t* b, const LiftConst* K, int8_t* R, uint64_t* xl, uint64_t* D,
                            unsigned* bar, int* err, int64_t n, int E, int32_t m, void* stream,
                            const DigitStream* ds = nullptr);

}  // namespace es
