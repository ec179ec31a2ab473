// Lift product on the 5th-generation tensor cores, for c >= 16 columns:
//     V[e][i][col] = w_e bal( sum_k B_j[i][k] R_e[col][k] ) mod q_j   in [0, q_j)
// (w_e = (P'/q_e)^{-1} mod q_e: the CRT's weight, so that the digit is
// sum_e V[e] P'/q_e reduced mod P', formed by k_lift_crt_mma)
// (exact-solve card, §Method: the per-step per-prime products as one batched
// GEMM on balanced residues, exact in the integer accumulator).
//
// sm_103a has no integer tcgen05 MMA kind, so residues are multiplied as f16
// (every |v| <= 125 is exact in f16) with tcgen05.mma .kind::f16 into an FP32
// accumulator in tensor memory.  FP32 is exact for integers below 2^24; the
// accumulator is folded into int32 registers every 512 K (|partial| <= 512 *
// 125^2 < 2^23) and then restarted, so the product is exact for any n <= 2^17.
// B_j stays int8 in HBM (the product is bound by reading it once per step):
// TMA brings 128 x 128 int8 tiles into shared memory and eight converter warps
// widen them to f16 straight into tensor memory, where the MMA reads its A
// operand.  Shared memory then carries only the int8 tile (written by TMA,
// read once by the converters) and the f16 residue tile of R_e (the B
// operand), a third of the traffic of widening into shared memory, so that
// reading B_j from HBM is the bound rather than shared-memory bandwidth.
//
// CTA = one prime e, 128 rows of B_j (MMA M = 128) and NT columns (N = NT):
//   warp 0      one thread: TMA producer, 6-stage ring; a stage is K = 128:
//               the int8 tile of B_j and two NT x 64 f16 tiles of R_e
//               (128-byte swizzled, K-major)
//   warps 6..13 converters: warp w may touch tensor-memory lanes 32 (w % 4)
//               .. + 31, so thread (w, lane) widens half (w - 6) / 4 of row
//               32 (w % 4) + lane of the int8 tile into 32 columns of the
//               stage's A slot (tcgen05.st), waits for its stores and
//               arrives on the stage's `conv` barrier
//   warp 1      one thread: 8 MMAs (K = 16 each, A from tensor memory) per
//               stage; a commit frees the stage's shared memory and A slot
//               and, at 512-K chunk ends, publishes the accumulator
//   warps 2..5  epilogue: fold each finished chunk from TMEM (tcgen05.ld,
//               lane quarter = warp % 4) into int32, Barrett at the end.
// Tensor memory (512 columns, one CTA per SM): the accumulator double-buffered
// in columns 0 .. 2 NT (MMAs of the next chunk overlap the fold of the
// previous one) and six 64-column A slots from column 128.  Every mbarrier
// wait is bounded: on expiry the kernel records an error code, stops issuing
// work, lets the copies and MMAs in flight land and returns.
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

constexpr int kBM = 128;           // MMA M (rows per CTA)
constexpr int kBK = 64;            // f16 tile K: one 128-byte row
constexpr int kATileBytes = kBM * kBK * 2;  // 16 KB

// product kernel
constexpr int kPStages = 6;
constexpr int kPK = 128;                    // K per stage: one 128-byte int8 row
constexpr int kPTileI8 = kBM * kPK;         // 16 KB
constexpr int kPFoldStages = 4;             // fold every 4 stages (K = 512)
constexpr int kPThreads = 448;             // producer, MMA, 4 epilogue and 8 converter warps
// tensor memory: two accumulator buffers (2 NT <= 128 columns) from column 0,
// then one f16 A slot of 64 columns (128 rows x 128 K) per stage
constexpr uint32_t kPColA = 128;
constexpr uint32_t kPTmemCols = 512;
static_assert(kPColA + 64 * kPStages <= kPTmemCols, "tensor memory A slots");


// The producer's exit: wait (bounded, whatever the error flag) for the copies
// of the last `depth` stages it issued, so that none is still writing shared
// memory when the CTA ends.
__device__ __forceinline__ void drain_loads(uint64_t* full, int issued, int depth) {
  for (int kb = issued > depth ? issued - depth : 0; kb < issued; ++kb)
    mbar_wait_drain(full + kb % depth, (kb / depth) & 1);
}

// Persistent: one CTA per SM walks the tiles t = blockIdx.x, + gridDim.x, ...
// (tile t = (row tile, column tile, prime), row tile fastest); the copy ring,
// the f16 slots and the two TMEM buffers run on across tiles, so a CTA's set-up
// and its pipeline fill are paid once rather than per tile.
struct ProdTile {
  int m0, n0, e;
};
__device__ __forceinline__ ProdTile prod_tile(int t, int tiles_m, int tiles_n, int nt) {
  const int mt = t % tiles_m, rest = t / tiles_m;
  return ProdTile{mt * kBM, (rest % tiles_n) * nt, rest / tiles_n};
}

template <int NT>
__global__ void __launch_bounds__(kPThreads, 1)
    k_lift_gemm_tc(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmR,
                   const LiftConst* __restrict__ K, int8_t* __restrict__ V, int n, int c, int kstages, int tiles_m,
                   int tiles_n, int ntiles, int* __restrict__ err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sI = smem;                               // [S] 128 x 128 int8
  uint8_t* sR = sI + kPStages * kPTileI8;           // [S][2] NT x 64 f16
  uint64_t* full = reinterpret_cast<uint64_t*>(sR + kPStages * 2 * NT * 128);
  uint64_t* conv = full + kPStages;
  uint64_t* empty = conv + kPStages;
  uint64_t* accfull = empty + kPStages;
  uint64_t* accempty = accfull + 2;
  uint64_t* drained = accempty + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drained + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunks = (kstages + kPFoldStages - 1) / kPFoldStages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(conv + s, 256);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accfull + b, 1);
      mbar_init(accempty + b, 128);
    }
    mbar_init(drained, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(s_tmem)),
                 "r"(kPTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // broadcast: the compiler then knows the base is the same in every lane
  const uint32_t tmem = __shfl_sync(0xffffffffu, *s_tmem, 0);

  if (warp == 0) {  // TMA producer: the warp runs the loop, one elected lane issues
    int g = 0;      // stages issued by this CTA
    bool stop = false;
    // B_j is streamed once per step: evict-first, so that the residues, the
    // residual's operands and the CRT weights stay in L2
    const uint64_t stream_pol = l2_evict_first();
    for (int t = blockIdx.x; t < ntiles && !stop; t += gridDim.x) {
      const ProdTile T = prod_tile(t, tiles_m, tiles_n, NT);
      for (int st = 0; st < kstages; ++st, ++g) {
        const int s = g % kPStages;
        if (g >= kPStages && !mbar_wait_warp(empty + s, ((g / kPStages) & 1) ^ 1, err, 1)) {
          stop = true;
          break;
        }
        if (elect_one()) {
          mbar_expect_tx(full + s, kPTileI8 + 2 * NT * 128);
          tma_load_3d_hint(sI + s * kPTileI8, &tmB, full + s, 0, 0, (T.e * tiles_m + T.m0 / kBM) * kstages + st,
                           stream_pol);
          tma_load_3d(sR + (2 * s) * NT * 128, &tmR, full + s, st * kPK, T.n0, T.e);
          tma_load_3d(sR + (2 * s + 1) * NT * 128, &tmR, full + s, st * kPK + kBK, T.n0, T.e);
        }
        __syncwarp();
      }
    }
    drain_loads(full, g, kPStages);
  } else if (warp >= 6) {
    // converters: warp w may touch tensor-memory lanes 32 (w % 4) .. + 31, so
    // thread u of the eight warps widens half h of row r of the int8 tile
    // (64 K) into 32 columns of the stage's A slot in tensor memory
    const int quarter = warp & 3, h = (warp - 6) >> 2, r = 32 * quarter + lane, sw = r & 7;
    const uint32_t trow = tmem + ((uint32_t)(32 * quarter) << 16);
    int g = 0;
    bool stop = false;
    for (int t = blockIdx.x; t < ntiles && !stop; t += gridDim.x) {
      for (int st = 0; st < kstages; ++st, ++g) {
        const int s = g % kPStages;
        // the slot's previous MMAs completed before its copy was issued (empty -> full)
        if (!mbar_wait(full + s, (g / kPStages) & 1, err, 5)) {
          stop = true;
          break;
        }
        tc_fence_after();
        const uint8_t* src = sI + s * kPTileI8 + r * 128;
        uint32_t wv[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // 16-byte chunk 4 h + q of the row: k = 64 h + 16 q .. + 15
          const uint4 w = *reinterpret_cast<const uint4*>(src + (((4 * h + q) ^ sw) << 4));
          s8x4_to_f16(w.x, wv[8 * q + 0], wv[8 * q + 1]);
          s8x4_to_f16(w.y, wv[8 * q + 2], wv[8 * q + 3]);
          s8x4_to_f16(w.z, wv[8 * q + 4], wv[8 * q + 5]);
          s8x4_to_f16(w.w, wv[8 * q + 6], wv[8 * q + 7]);
        }
        tmem_st32(trow + (uint32_t)(kPColA + s * 64 + 32 * h), wv);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(conv + s);
      }
    }
  } else if (warp == 1) {  // MMA issuer: the warp runs the loop, one elected lane issues
    const uint32_t idesc = (1u << 4) | ((uint32_t)(NT >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
    int g = 0, gc0 = 0;  // stages and accumulator chunks of earlier tiles
    bool stop = false;
    for (int t = blockIdx.x; t < ntiles && !stop; t += gridDim.x, gc0 += nchunks) {
      for (int st = 0; st < kstages; ++st, ++g) {
        const int s = g % kPStages, gc = gc0 + st / kPFoldStages, buf = gc & 1;
        const bool first = (st % kPFoldStages) == 0;
        if (first && gc >= 2 && !mbar_wait_warp(accempty + buf, ((gc - 2) >> 1) & 1, err, 2)) {
          stop = true;
          break;
        }
        if (!mbar_wait_warp(conv + s, (g / kPStages) & 1, err, 3)) {
          stop = true;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const uint64_t bd = desc_sw128(sR + (2 * s + hh) * NT * 128);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              mma_f16_ta(tmem + buf * NT, tmem + (uint32_t)(kPColA + s * 64 + 32 * hh + 8 * k), bd + 2 * k, idesc,
                         (first && hh == 0 && k == 0) ? 0u : 1u);
          }
          mma_commit(empty + s);
          if ((st % kPFoldStages) == kPFoldStages - 1 || st == kstages - 1) mma_commit(accfull + buf);
        }
        __syncwarp();
      }
    }
    // every MMA issued has completed before tensor memory is released
    if (elect_one()) mma_commit(drained);
    __syncwarp();
    mbar_wait_drain(drained, 0);
  } else {  // epilogue warpgroup (warps 2..5)
    const int quarter = warp & 3;
    int gc0 = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, gc0 += nchunks) {
      const ProdTile T = prod_tile(t, tiles_m, tiles_n, NT);
      const int row = T.m0 + 32 * quarter + lane;
      int32_t acc[NT];
#pragma unroll
      for (int i = 0; i < NT; ++i) acc[i] = 0;
      for (int ch = 0; ch < nchunks; ++ch) {
        const int gc = gc0 + ch, buf = gc & 1;
        if (!mbar_wait(accfull + buf, (gc >> 1) & 1, err, 4)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c16 = 0; c16 < NT / 16; ++c16) {
          float f[16];
          tmem_ld<16>(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(buf * NT + 16 * c16), f);
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[16 * c16 + i] += __float2int_rn(f[i]);
        }
        tc_fence_before();
        mbar_arrive(accempty + buf);
      }
      if (ok && row < n) {
        // the CRT's weight of this prime applied here: c_e = y w_e mod q_e in [0, q_e)
        const ModQ m = K->mq[T.e];
        const uint32_t we = K->w[T.e];
        auto ce = [&](int32_t y) -> uint32_t { return barrett(barrett((uint32_t)y + m.off, m) * we, m); };
        uint8_t* out = reinterpret_cast<uint8_t*>(V) + ((int64_t)T.e * n + row) * c + T.n0;
        if (c % 16 == 0 && T.n0 + NT <= c) {
          // the row's NT bytes are contiguous and 16-byte aligned: 16-byte stores
#pragma unroll
          for (int i = 0; i < NT; i += 16) {
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
              w[q] = ce(acc[i + 4 * q]) | ce(acc[i + 4 * q + 1]) << 8 | ce(acc[i + 4 * q + 2]) << 16 |
                     ce(acc[i + 4 * q + 3]) << 24;
            *reinterpret_cast<uint4*>(out + i) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < NT; ++i)
            if (T.n0 + i < c) out[i] = (uint8_t)ce(acc[i]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kPTmemCols));
  }
}

// ---------------------------------------------------------------- residual
// A x_i mod 2^64 on the tensor cores, for r_{i+1} = (r_i - A x_i) P'^{-1} mod
// 2^64 (exact-solve card, §Method: the residual kept in one 64-bit limb).
// With A = sum_a A_a 256^a and x_i = sum_t X_t 256^t (mod 2^64) in balanced
// 8-bit limbs (|A_a|, |X_t| <= 128, exact in f16),
//     A x_i = sum_a S_a (mod 2^64),   S_a = sum_{s < 8} 256^s A_a X_{s-a},
// and each plane's S_a is one GEMM whose B operand rows (s, col) are
// X_{s-a}[col]: one 3-D TMA box of 8 limb planes x NC columns from the X
// planes, stored after na - 1 zero planes (X_{s-a} is plane s - a + na - 1).
// CTA = (128 rows, NC columns, plane a): MMA M = 128, N = 8 NC (limb-major),
// K = one plane (split K: the planes run in parallel).  Products are at most
// 2^14, so 1024-term FP32 partial sums are exact (at most 2^24); every such
// chunk the epilogue folds the accumulator into one 64-bit word per column,
// S += sum_s 256^s y_s (mod 2^64), double-buffered in tensor memory so the
// MMAs of the next chunk overlap the fold.  At the end each plane's S_a is
// added into Sacc [c][n] (64-bit atomics: addition mod 2^64), which
// k_lift_r16 turns into r_{i+1} and its residues and clears.
constexpr int kR2Fold = 16;  // fold every 16 K-blocks (K = 1024)
constexpr int kR2Threads = 192;

template <int NC>
struct R2Cfg {
  static constexpr int N = 8 * NC;                  // MMA N
  static constexpr int Stages = NC == 32 ? 4 : 3;   // 48 KB or 32 KB per stage
  static constexpr int CtasPerSm = NC == 32 ? 1 : 2;
  static constexpr uint32_t Cols = 2 * N;           // double-buffered accumulator
  static constexpr size_t Smem = 1024 + (size_t)Stages * (kATileBytes + N * 128) + 256;
};

template <int NC>
__global__ void __launch_bounds__(kR2Threads, R2Cfg<NC>::CtasPerSm)
    k_lift_resid_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmX, int n, int c,
                    int na, int kbp, uint64_t* __restrict__ Sacc, int* __restrict__ err) {
  using Cfg = R2Cfg<NC>;
  constexpr int N = Cfg::N, S_ = Cfg::Stages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + S_ * kATileBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + S_ * N * 128);
  uint64_t* empty = full + S_;
  uint64_t* accfull = empty + S_;
  uint64_t* accempty = accfull + 2;
  uint64_t* drained = accempty + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drained + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kBM, col0 = blockIdx.y * NC, a = blockIdx.z;
  const int nchunks = (kbp + kR2Fold - 1) / kR2Fold;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S_; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accfull + b, 1);
      mbar_init(accempty + b, 128);
    }
    mbar_init(drained, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(s_tmem)),
                 "r"(Cfg::Cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = __shfl_sync(0xffffffffu, *s_tmem, 0);

  if (warp == 0) {  // TMA producer: the warp runs the loop, one elected lane issues
    int issued = 0;
    for (int kb = 0; kb < kbp; ++kb) {
      const int s = kb % S_;
      if (kb >= S_ && !mbar_wait_warp(empty + s, ((kb / S_) & 1) ^ 1, err, 1)) break;
      if (elect_one()) {
        mbar_expect_tx(full + s, kATileBytes + N * 128);
        tma_load_3d(sA + s * kATileBytes, &tmA, full + s, kb * kBK, m0, a);
        tma_load_3d(sB + s * N * 128, &tmX, full + s, kb * kBK, col0, na - 1 - a);
      }
      __syncwarp();
      issued = kb + 1;
    }
    drain_loads(full, issued, S_);
  } else if (warp == 1) {  // MMA issuer: the warp runs the loop, one elected lane issues
    const uint32_t idesc = (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
    for (int kb = 0; kb < kbp; ++kb) {
      const int s = kb % S_, ch = kb / kR2Fold, buf = ch & 1;
      const bool first = (kb % kR2Fold) == 0;
      if (first && ch >= 2 && !mbar_wait_warp(accempty + buf, ((ch - 2) >> 1) & 1, err, 2)) break;
      if (!mbar_wait_warp(full + s, (kb / S_) & 1, err, 3)) break;
      tc_fence_after();
      if (elect_one()) {
        const uint64_t ad = desc_sw128(sA + s * kATileBytes), bd = desc_sw128(sB + s * N * 128);
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          mma_f16(tmem + buf * N, ad + 2 * k, bd + 2 * k, idesc, (first && k == 0) ? 0u : 1u);
        mma_commit(empty + s);
        if ((kb % kR2Fold) == kR2Fold - 1 || kb == kbp - 1) mma_commit(accfull + buf);
      }
      __syncwarp();
    }
    // every MMA issued has completed before tensor memory is released
    if (elect_one()) mma_commit(drained);
    __syncwarp();
    mbar_wait_drain(drained, 0);
  } else {  // epilogue warpgroup (warps 2..5)
    const int quarter = warp & 3;
    const int row = m0 + 32 * quarter + lane;
    uint64_t S[NC];
#pragma unroll
    for (int t = 0; t < NC; ++t) S[t] = 0;
    bool ok = true;
    for (int ch = 0; ch < nchunks; ++ch) {
      const int buf = ch & 1;
      if (!mbar_wait(accfull + buf, (ch >> 1) & 1, err, 4)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int s8 = 0; s8 < 8; ++s8) {
        float f[NC];
        tmem_ld<NC>(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(buf * N + s8 * NC), f);
#pragma unroll
        for (int t = 0; t < NC; ++t) S[t] += (uint64_t)(int64_t)__float2int_rn(f[t]) << (8 * s8);
      }
      tc_fence_before();
      mbar_arrive(accempty + buf);
    }
    if (ok && row < n) {
#pragma unroll
      for (int cl = 0; cl < NC; ++cl) {
        const int col = col0 + cl;
        if (col >= c) break;
        atomicAdd(reinterpret_cast<unsigned long long*>(Sacc + (int64_t)col * n + row), (unsigned long long)S[cl]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(Cfg::Cols));
  }
}

// r_{i+1} = (r_i - A x_i) P'^{-1} mod 2^64 from Sacc = A x_i mod 2^64 (which is
// cleared for the next step), and R16[e][col][i] = its balanced residue mod
// q_e as f16; one thread per entry, rows fastest so that the stores of a prime
// are coalesced (r, r_{i+1} and Sacc are stored [c][n]).  The residual is usually far inside the int32 range
// (|r_{i+1}| < n max|A| / 2 + 1 once the first step is done), so a CTA whose
// entries all fit takes the one-Barrett path; the reduction constants come
// from shared memory.
__global__ void __launch_bounds__(256) k_lift_r16(const int64_t* __restrict__ r, uint64_t* __restrict__ Sacc,
                                                  int64_t* __restrict__ rn, int64_t n, int64_t c, int64_t ld,
                                                  const LiftConst* __restrict__ K, __half* __restrict__ R16) {
  __shared__ ModQ sm[kNumPrimes];
  const int E = K->E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) sm[e] = K->mq[e];
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool live = t < n * c;
  const int64_t col = live ? t / n : 0, i = live ? t - col * n : 0;
  int64_t v = 0;
  if (live) {  // r, r_{i+1} and Sacc are [c][n]: entry t
    v = (int64_t)(((uint64_t)r[t] - Sacc[t]) * K->Pinv64);
    rn[t] = v;
    Sacc[t] = 0;
  }
  // -2^31 < v < 2^31 - 256: the signed 32-bit reduction applies
  const bool narrow = __syncthreads_and(v > -(int64_t(1) << 31) && v < (int64_t(1) << 31) - 256);
  if (!live) return;
  __half* out = R16 + col * ld + i;
  if (narrow) {
    const int32_t v32 = (int32_t)v;
#pragma unroll 4
    for (int e = 0; e < E; ++e) out[(int64_t)e * c * ld] = __int2half_rn(reduce_bal(v32, sm[e]));
  } else {
    for (int e = 0; e < E; ++e) out[(int64_t)e * c * ld] = __int2half_rn(reduce_i64_bal(v, sm[e]));
  }
}

// A16[a][i][k] = limb a of A[i][k] in balanced base 256 (k < n), 0 for n <= k < ld.
__global__ void k_a_limbs(const int64_t* __restrict__ A, int64_t n, int64_t ld, int na, __half* __restrict__ A16) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n * ld) return;
  const int64_t i = t / ld, k = t - i * ld;
  int64_t v = k < n ? A[i * n + k] : 0;
  for (int a = 0; a < na - 1; ++a) {
    const int64_t d = ((v + 128) & 255) - 128;
    A16[((int64_t)a * n + i) * ld + k] = __int2half_rn((int)d);
    v = (v - d) >> 8;
  }
  A16[((int64_t)(na - 1) * n + i) * ld + k] = __int2half_rn((int)v);
}

// Bt[e][mt][kb][r][k'] = B_j[128 mt + r][128 kb + k'] (j = K->pidx[e]), zero
// outside n rows and ld columns; one thread per 16-byte chunk, in Bt order.
__global__ void k_tile_b(const int8_t* __restrict__ B, const LiftConst* __restrict__ K, int8_t* __restrict__ Bt,
                         int64_t n, int64_t ld, int64_t tiles_m, int64_t kst, int64_t chunks) {
  const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= chunks) return;
  const int q = (int)(u & 7);
  int64_t rest = u >> 3;
  const int r = (int)(rest % kBM);
  rest /= kBM;
  const int64_t kb = rest % kst;
  rest /= kst;
  const int64_t mt = rest % tiles_m, e = rest / tiles_m;
  const int64_t i = mt * kBM + r, k = kb * kPK + 16 * q;
  int4 v = make_int4(0, 0, 0, 0);
  if (i < n && k < ld) v = *reinterpret_cast<const int4*>(B + ((int64_t)K->pidx[e] * n + i) * ld + k);
  reinterpret_cast<int4*>(Bt)[u] = v;
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
  const size_t smem = 1024 + (size_t)kPStages * (kPTileI8 + 2 * NT * 128) + 256;
  static_assert(NT % 16 == 0 && NT <= 64, "N tile");
  ES_CHECK(cuda_status(cudaFuncSetAttribute(k_lift_gemm_tc<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)smem),
                       "tc smem attribute"));
  const int tiles_m = (int)((n + kBM - 1) / kBM), tiles_n = (int)((c + NT - 1) / NT);
  const int ntiles = tiles_m * tiles_n * E;
  const int kstages = (int)((ld + kPK - 1) / kPK);
  const int grid = ntiles < sm_count() ? ntiles : sm_count();
  k_lift_gemm_tc<NT><<<grid, kPThreads, smem, st>>>(mB, mR, K, V, (int)n, (int)c, kstages, tiles_m, tiles_n, ntiles,
                                                    err);
  return cuda_status(cudaGetLastError(), "k_lift_gemm_tc");
}

}  // namespace

es_status tc_convert_f16(const int8_t* src, void* dst, int64_t count, void* stream) {
  const int64_t threads = (count + 3) / 4;
  k_to_f16<<<(unsigned)((threads + 255) / 256), 256, 0, (cudaStream_t)stream>>>(src, (__half*)dst, count);
  count_launch();
  return cuda_status(cudaGetLastError(), "k_to_f16");
}

size_t tc_tiled_b_bytes(int64_t n, int E) {
  const int64_t tiles_m = (n + kBM - 1) / kBM, kst = (padded_ld(n) + kPK - 1) / kPK;
  return (size_t)E * tiles_m * kst * kPTileI8;
}

es_status tc_prepare(TcLift* t, const int8_t* Bt, const void* R16, int64_t n, int64_t c, int64_t ld, int E) {
  t->nt = c <= 16 ? 16 : c <= 32 ? 32 : 64;
  t->tiles_m = (int)((n + kBM - 1) / kBM);
  t->kstages = (int)((ld + kPK - 1) / kPK);
  ES_CHECK(make_map_u8(&t->mapB, Bt, kPK, kBM, (int64_t)E * t->tiles_m * t->kstages, kBM));
  ES_CHECK(make_map(&t->mapR, R16, ld, c, E, t->nt));
  return ES_OK;
}

es_status tc_tile_b(const int8_t* B, const LiftConst* K, int8_t* Bt, int64_t n, int64_t ld, int E, void* stream) {
  const int64_t tiles_m = (n + kBM - 1) / kBM, kst = (ld + kPK - 1) / kPK;
  const int64_t chunks = (int64_t)E * tiles_m * kst * (kPTileI8 / 16);
  k_tile_b<<<(unsigned)((chunks + 255) / 256), 256, 0, (cudaStream_t)stream>>>(B, K, Bt, n, ld, tiles_m, kst, chunks);
  count_launch();
  return cuda_status(cudaGetLastError(), "k_tile_b");
}

int resid_limbs(uint64_t max_abs_a) {
  // After na - 1 balanced peels |top| <= (|A| + 128 (256^(na-1) - 1) / 255) / 256^(na-1),
  // which stays within 128 when |A| + 128 (256^(na-1) - 1) / 255 < 129 256^(na-1).
  for (int na = 1; na <= kResidLimbsMax; ++na) {
    const uint64_t w = uint64_t(1) << (8 * (na - 1));
    if (max_abs_a + 128 * ((w - 1) / 255) < 129 * w) return na;
  }
  return 0;
}

es_status tc_resid_prepare(TcResid* t, const int64_t* A_dev, void* A16, void* X16, int64_t n, int64_t c, int64_t ld,
                           int na, void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  if (na < 1 || na > kResidLimbsMax) return ES_ERR_INTERNAL;
  t->na = na;
  t->kbp = (int)((ld + kBK - 1) / kBK);
  k_a_limbs<<<(unsigned)((n * ld + 255) / 256), 256, 0, st>>>(A_dev, n, ld, na, (__half*)A16);
  count_launch();
  ES_CHECK(cuda_status(cudaGetLastError(), "k_a_limbs"));
  ES_CHECK(cuda_status(cudaMemsetAsync(X16, 0, (size_t)(na + 7) * c * ld * 2, st), "memset x limbs"));
  // 32 columns per CTA (MMA N = 256) while that still gives at least one CTA
  // per SM, else 16 (N = 128, two CTAs per SM)
  const int64_t tiles_m = (n + kBM - 1) / kBM;
  t->nc = tiles_m * ((c + 31) / 32) * na >= sm_count() ? 32 : 16;
  ES_CHECK(make_map(&t->mapA, A16, ld, n, na, kBM));
  ES_CHECK(make_map(&t->mapX, X16, ld, c, na + 7, t->nc, 8));
  return ES_OK;
}

namespace {
template <int NC>
es_status launch_resid(const TcResid& t, uint64_t* Sacc, int64_t n, int64_t c, int* err, cudaStream_t st) {
  const size_t smem = R2Cfg<NC>::Smem;
  ES_CHECK(cuda_status(cudaFuncSetAttribute(k_lift_resid_tc<NC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)smem),
                       "tc resid smem attribute"));
  dim3 grid((unsigned)((n + kBM - 1) / kBM), (unsigned)((c + NC - 1) / NC), (unsigned)t.na);
  k_lift_resid_tc<NC><<<grid, kR2Threads, smem, st>>>(t.mapA, t.mapX, (int)n, (int)c, t.na, t.kbp, Sacc, err);
  return cuda_status(cudaGetLastError(), "k_lift_resid_tc");
}
}  // namespace

es_status tc_resid_launch(const TcResid& t, const LiftConst* K, const int64_t* r, int64_t* rn, uint64_t* Sacc,
                          void* R16, int64_t n, int64_t c, int64_t ld, int* err, void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  if (t.nc == 32)
    ES_CHECK(launch_resid<32>(t, Sacc, n, c, err, st));
  else
    ES_CHECK(launch_resid<16>(t, Sacc, n, c, err, st));
  k_lift_r16<<<(unsigned)((n * c + 255) / 256), 256, 0, st>>>(r, Sacc, rn, n, c, ld, K, (__half*)R16);
  count_launch(2);
  return cuda_status(cudaGetLastError(), "k_lift_r16");
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
