// Internal declarations shared by the lift translation units.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "es_common.cuh"
#include "es_internal.h"

namespace es {

struct LiftConst {
  int32_t E;                      // number of good primes
  int32_t pidx[kNumPrimes];       // their indices in the prime table, ascending
  ModQ mq[kNumPrimes];            // reduction constants, compact order
  uint32_t w[kNumPrimes];         // (P'/q)^{-1} mod q
  uint64_t tfix[kNumPrimes];      // floor(2^50 / q)
  uint32_t Mq[kNumPrimes][kCrtWords];  // P'/q, 32-bit little-endian words
  uint32_t P[kCrtWords];          // P'
  uint32_t Phalf[kCrtWords];      // (P' - 1) / 2
  uint64_t Pinv64;                // P'^{-1} mod 2^64
};

// tcgen05 lift product (k_lift_tc.cu), used for c >= 16.
struct TcLift {
  CUtensorMap mapB;  // f16 [53][n][ld] inverses
  CUtensorMap mapR;  // f16 [E'][c][ld] residues of r_i
  int nt = 64;       // MMA N tile
};
es_status tc_convert_f16(const int8_t* src, void* dst, int64_t count, void* stream);
es_status tc_prepare(TcLift* t, const void* B16, const void* R16, int64_t n, int64_t c, int64_t ld, int E);
es_status tc_launch(const TcLift& t, const LiftConst* K, int8_t* V, int64_t n, int64_t c, int64_t ld, int E,
                    int* err, void* stream);

}  // namespace es
