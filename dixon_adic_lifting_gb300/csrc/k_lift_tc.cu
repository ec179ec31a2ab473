// Lift product on the 5th-generation tensor cores, for c >= 16 columns:
//     V[e][i][col] = bal( sum_k B_j[i][k] R_e[col][k]  mod q_j )
// (exact-solve card, §Method: the per-step per-prime products as one batched
// GEMM on balanced residues, exact in the integer accumulator).
//
// sm_103a has no integer tcgen05 MMA kind, so residues are kept as f16
// (every |v| <= 125 is exact in f16) and multiplied with tcgen05.mma
// .kind::f16 into an FP32 accumulator in tensor memory.  FP32 is exact for
// integers below 2^24; the accumulator is folded into int32 registers every
// kFoldBlocks K-blocks (K = 512: |partial| <= 512 * 125^2 < 2^23) and then
// restarted, so the product is exact for any n <= 2^17.
//
// CTA = one prime e, 128 rows of B_j (MMA M = 128) and NT columns (N = NT):
//   warp 0      one thread: TMA producer, 4-stage ring of 128B-swizzled
//               K-major tiles (A: 128 x 64 f16 of B_j, B: NT x 64 f16 of R_e)
//   warp 1      one thread: issues 4 MMAs (K = 16 each) per stage; commits
//               free the stage and, at chunk ends, publish the accumulator
//   warps 2..5  epilogue: fold each finished chunk from TMEM (tcgen05.ld,
//               lane quarter = warp % 4) into int32, Barrett at the end.
// The TMEM accumulator is double-buffered (2 NT columns) so MMAs of the next
// chunk overlap the fold of the previous one.  Every mbarrier wait is bounded:
// on expiry the kernel records an error code, stops issuing work and returns.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "es_common.cuh"
#include "es_internal.h"
#include "lift_internal.h"
#include "tc_common.cuh"

namespace es {
namespace {
using namespace tc;

constexpr int kBM = 128;           // MMA M (rows of B_j per CTA)
constexpr int kBK = 64;            // K per stage: one 128-byte row of f16
constexpr int kStages = 4;
constexpr int kFoldBlocks = 8;     // fold every 8 stages (K = 512)
constexpr int kThreads = 192;
constexpr int kATileBytes = kBM * kBK * 2;  // 16 KB

template <int NT>
__global__ void __launch_bounds__(kThreads, 1)
    k_lift_gemm_tc(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmR,
                   const LiftConst* __restrict__ K, int8_t* __restrict__ V, int n, int c, int kblocks,
                   int* __restrict__ err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kATileBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + kStages * NT * 128);
  uint64_t* empty = full + kStages;
  uint64_t* accfull = empty + kStages;
  uint64_t* accempty = accfull + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(accempty + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.z, j = K->pidx[e];
  const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * NT;
  const int nchunks = (kblocks + kFoldBlocks - 1) / kFoldBlocks;
  constexpr uint32_t kCols = 2 * NT < 32 ? 32 : 2 * NT;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accfull + b, 1);
      mbar_init(accempty + b, 128);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(s_tmem)),
                 "r"(kCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      for (int kb = 0; kb < kblocks; ++kb) {
        const int s = kb % kStages;
        if (kb >= kStages && !mbar_wait(empty + s, ((kb / kStages) & 1) ^ 1, err, 1)) break;
        mbar_expect_tx(full + s, kATileBytes + NT * 128);
        tma_load_3d(sA + s * kATileBytes, &tmB, full + s, kb * kBK, m0, j);
        tma_load_3d(sB + s * NT * 128, &tmR, full + s, kb * kBK, n0, e);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      const uint32_t idesc = (1u << 4) | ((uint32_t)(NT >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
      for (int kb = 0; kb < kblocks; ++kb) {
        const int s = kb % kStages, ch = kb / kFoldBlocks, buf = ch & 1;
        const bool first = (kb % kFoldBlocks) == 0;
        if (first && ch >= 2 && !mbar_wait(accempty + buf, ((ch - 2) >> 1) & 1, err, 2)) break;
        if (!mbar_wait(full + s, (kb / kStages) & 1, err, 3)) break;
        tc_fence_after();
        const uint64_t ad = desc_sw128(sA + s * kATileBytes), bd = desc_sw128(sB + s * NT * 128);
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          mma_f16(tmem + buf * NT, ad + 2 * k, bd + 2 * k, idesc, (first && k == 0) ? 0u : 1u);
        mma_commit(empty + s);
        if ((kb % kFoldBlocks) == kFoldBlocks - 1 || kb == kblocks - 1) mma_commit(accfull + buf);
      }
    }
  } else {  // epilogue warpgroup
    const int quarter = warp & 3;
    const int row = m0 + 32 * quarter + lane;
    const ModQ m = K->mq[e];
    int32_t acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0;
    bool ok = true;
    for (int ch = 0; ch < nchunks; ++ch) {
      const int buf = ch & 1;
      if (!mbar_wait(accfull + buf, (ch >> 1) & 1, err, 4)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c16 = 0; c16 < NT / 16; ++c16) {
        float f[16];
        tmem_ld<16>(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(buf * NT + 16 * c16), f);
#pragma unroll
        for (int t = 0; t < 16; ++t) acc[16 * c16 + t] += __float2int_rn(f[t]);
      }
      tc_fence_before();
      mbar_arrive(accempty + buf);
    }
    if (ok && row < n) {
      int8_t* out = V + ((int64_t)e * n + row) * c;
#pragma unroll
      for (int t = 0; t < NT; ++t)
        if (n0 + t < c) out[n0 + t] = (int8_t)reduce_bal(acc[t], m);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols));
  }
}

__global__ void k_to_f16(const int8_t* __restrict__ src, __half* __restrict__ dst, int64_t count) {
  int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (t + 4 <= count) {
    const char4 v = *reinterpret_cast<const char4*>(src + t);
    __half2* d = reinterpret_cast<__half2*>(dst + t);
    d[0] = __halves2half2(__int2half_rn(v.x), __int2half_rn(v.y));
    d[1] = __halves2half2(__int2half_rn(v.z), __int2half_rn(v.w));
  } else {
    for (; t < count; ++t) dst[t] = __int2half_rn(src[t]);
  }
}

template <int NT>
es_status launch_nt(const CUtensorMap& mB, const CUtensorMap& mR, const LiftConst* K, int8_t* V, int64_t n,
                    int64_t c, int64_t ld, int E, int* err, cudaStream_t st) {
  const size_t smem = 1024 + (size_t)kStages * (kATileBytes + NT * 128) + 256;
  static_assert(NT % 16 == 0 && NT <= 64, "N tile");
  ES_CHECK(cuda_status(cudaFuncSetAttribute(k_lift_gemm_tc<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)smem),
                       "tc smem attribute"));
  dim3 grid((unsigned)((n + kBM - 1) / kBM), (unsigned)((c + NT - 1) / NT), (unsigned)E);
  const int kblocks = (int)((ld + kBK - 1) / kBK);
  k_lift_gemm_tc<NT><<<grid, kThreads, smem, st>>>(mB, mR, K, V, (int)n, (int)c, kblocks, err);
  return cuda_status(cudaGetLastError(), "k_lift_gemm_tc");
}

}  // namespace

es_status tc_convert_f16(const int8_t* src, void* dst, int64_t count, void* stream) {
  const int64_t threads = (count + 3) / 4;
  k_to_f16<<<(unsigned)((threads + 255) / 256), 256, 0, (cudaStream_t)stream>>>(src, (__half*)dst, count);
  count_launch();
  return cuda_status(cudaGetLastError(), "k_to_f16");
}

es_status tc_prepare(TcLift* t, const void* B16, const void* R16, int64_t n, int64_t c, int64_t ld, int E) {
  t->nt = c <= 16 ? 16 : c <= 32 ? 32 : 64;
  ES_CHECK(make_map(&t->mapB, B16, ld, n, kNumPrimes, kBM));
  ES_CHECK(make_map(&t->mapR, R16, ld, c, E, t->nt));
  return ES_OK;
}

es_status tc_launch(const TcLift& t, const LiftConst* K, int8_t* V, int64_t n, int64_t c, int64_t ld, int E,
                    int* err, void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  count_launch();
  if (t.nt == 16) return launch_nt<16>(t.mapB, t.mapR, K, V, n, c, ld, E, err, st);
  if (t.nt == 32) return launch_nt<32>(t.mapB, t.mapR, K, V, n, c, ld, E, err, st);
  return launch_nt<64>(t.mapB, t.mapR, K, V, n, c, ld, E, err, st);
}

}  // namespace es
