// Device helpers shared by the lift translation units.
#pragma once

#include "es_common.cuh"
#include "lift_internal.h"

namespace es {

// The digit from the word sums acc (S = sum_e c_e P'/q_e as 12 base-2^32
// columns) and the fixed-point estimate tf of floor(S / P'): normalise,
// subtract t P', one conditional subtraction of P', then the balanced shift.
__device__ __forceinline__ void crt_finish(const uint64_t (&acc)[kCrtWords], uint64_t tf, const uint32_t* Pw,
                                           const uint32_t* Phw, uint32_t (&S)[kCrtWords]);
__device__ __forceinline__ void crt_finish(const uint64_t (&acc)[kCrtWords], uint64_t tf,
                                           const LiftConst* __restrict__ K, uint32_t (&S)[kCrtWords]) {
  crt_finish(acc, tf, K->P, K->Phalf, S);
}
// P' and (P' - 1) / 2 as 32-bit words, read from Pw and Phw (global or shared).
__device__ __forceinline__ void crt_finish(const uint64_t (&acc)[kCrtWords], uint64_t tf, const uint32_t* Pw,
                                           const uint32_t* Phw, uint32_t (&S)[kCrtWords]) {
  uint64_t carry = 0;
#pragma unroll
  for (int l = 0; l < kCrtWords; ++l) {
    uint64_t s = acc[l] + carry;
    S[l] = (uint32_t)s;
    carry = s >> 32;
  }
  // x = S - tq P'
  const uint32_t tq = (uint32_t)(tf >> 50);
  uint64_t mc = 0;
  int64_t borrow = 0;
#pragma unroll
  for (int l = 0; l < kCrtWords; ++l) {
    uint64_t prod = (uint64_t)tq * Pw[l] + mc;
    mc = prod >> 32;
    int64_t d = (int64_t)S[l] - (int64_t)(uint32_t)prod + borrow;
    S[l] = (uint32_t)d;
    borrow = d >> 32;  // 0 or -1
  }
  // if S >= P' subtract once
  bool ge = true;
#pragma unroll
  for (int l = kCrtWords - 1; l >= 0; --l) {
    if (S[l] != Pw[l]) {
      ge = S[l] > Pw[l];
      break;
    }
  }
  if (ge) {
    borrow = 0;
#pragma unroll
    for (int l = 0; l < kCrtWords; ++l) {
      int64_t d = (int64_t)S[l] - (int64_t)Pw[l] + borrow;
      S[l] = (uint32_t)d;
      borrow = d >> 32;
    }
  }
  // balanced: if S > (P'-1)/2 then S -= P' (mod 2^384)
  bool gt = false;
#pragma unroll
  for (int l = kCrtWords - 1; l >= 0; --l) {
    if (S[l] != Phw[l]) {
      gt = S[l] > Phw[l];
      break;
    }
  }
  if (gt) {
    borrow = 0;
#pragma unroll
    for (int l = 0; l < kCrtWords; ++l) {
      int64_t d = (int64_t)S[l] - (int64_t)Pw[l] + borrow;
      S[l] = (uint32_t)d;
      borrow = d >> 32;
    }
  }
}

// Balanced CRT digit of one entry, one warp: lane l contributes the residues
// v_e of primes e = l and l + 32 (v0, v1; ignored where e >= E'), or with
// kWeights their CRT weights c_e = v_e w_e mod q_e.
//   c_e = v_e w_e mod q_e,  S = sum_e c_e P'/q_e  (12 word columns),
//   t estimated as floor(sum_e c_e floor(2^50/q_e) / 2^50)
// The word sums and the estimate are reduced across the warp; every lane
// finishes the same digit and returns its 12 words in S.
template <bool kWeights = false>
__device__ __forceinline__ void crt_warp(int32_t v0, int32_t v1, int lane, const LiftConst* __restrict__ K,
                                         uint32_t (&S)[kCrtWords]) {
  const int E = K->E;
  uint64_t acc[kCrtWords];
#pragma unroll
  for (int l = 0; l < kCrtWords; ++l) acc[l] = 0;
  uint64_t tf = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int e = lane + 32 * h;
    if (e < E) {
      const ModQ m = K->mq[e];
      const int32_t v = h ? v1 : v0;
      const uint32_t vu = (uint32_t)(v < 0 ? v + (int32_t)m.q : v);
      // kWeights: the inputs are the CRT weights c_e in [0, q_e) already
      const uint32_t ce = kWeights ? (uint32_t)v : barrett(vu * K->w[e], m);
      tf += (uint64_t)ce * K->tfix[e];
#pragma unroll
      for (int l = 0; l < kCrtWords; ++l) acc[l] += (uint64_t)ce * K->Mq[e][l];
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    tf += __shfl_xor_sync(0xffffffffu, tf, o);
#pragma unroll
    for (int l = 0; l < kCrtWords; ++l) acc[l] += __shfl_xor_sync(0xffffffffu, acc[l], o);
  }
  crt_finish(acc, tf, K, S);
}

}  // namespace es
