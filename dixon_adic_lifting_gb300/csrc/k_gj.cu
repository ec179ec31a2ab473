// Batched modular inverse B_j = A^{-1} mod q_j for all 53 primes at once.
//
// exact-solve card, §Method: A^{-1} mod q_j is formed for every prime at
// once by Gauss-Jordan elimination, each elimination step one launch over
// all primes, with Barrett reduction instead of the hardware remainder;
// §Requirements: working memory grows with the prime count and n.
//
// GB300 design.  Gauss-Jordan is run in place (no augmented half: the
// exchange form of Gauss-Jordan stores the inverse's columns where the
// eliminated columns were), on balanced int8 residues (1 byte per entry,
// [53][n][ld], ld = n rounded up to 16), and blocked by panels of NB
// columns:
//   1. k_gj_panel   one CTA per prime: the NB exchange steps of the panel,
//                   restricted to the panel's columns, in shared memory
//                   (pivot search = lowest-index unused row with a nonzero
//                   entry; no rows are moved, the pivot row of every column
//                   is recorded).  It also stages the pivot rows' other
//                   columns (U, transposed) and zeroes them in place.
//   2. k_gj_update  one grid over all primes: every other column receives
//                   the block exchange  W[:, t] += F U[:, t]  (mod q_j),
//                   F = the panel just computed: an int8 x int8 -> int32
//                   contraction of depth NB (dp4a), exact since
//                   NB * 125^2 + 125 < 2^31, reduced by Barrett.
//   3. k_gj_permute undoes the pivot order: with p_k the pivot row of
//                   column k and pinv its inverse permutation,
//                   (A^{-1})[k][t] = W[p_k][pinv[t]].
// A prime with no pivot in some column divides det A; it is flagged bad and
// its CTAs exit early in every later launch.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>

#include "es_common.cuh"
#include "es_internal.h"

namespace es {

struct GJParams {
  int8_t* W;       // [53][n][ld] working matrices
  int64_t n, ld;
  int32_t* piv;    // [53][n] pivot row of each column
  int32_t* pinv;   // [53][n] inverse permutation
  uint8_t* used;   // [53][n] row already a pivot
  int32_t* bad;    // [53] prime divides det A
  int8_t* UT;      // [53][ld][utw] pivot rows' values, transposed, zero for a >= kb
  int utw;         // bytes per U^T row (NB = 16: 16; NB = 32: 64, two panels side by side)
  int8_t* gpanel;  // [53][n][NBP] panel in global memory when shared memory is too small
};

__device__ __forceinline__ int32_t sbyte(uint32_t w, int u) { return (int32_t)(w << (24 - 8 * u)) >> 24; }

// fl(1/q) per prime (correctly rounded)
struct QInvTable {
  float v[kNumPrimes];
};
constexpr QInvTable make_qinv_table() {
  QInvTable t{};
  for (int i = 0; i < kNumPrimes; ++i) t.v[i] = 1.0f / (float)kPrimes[i];
  return t;
}
__constant__ QInvTable c_qinv = make_qinv_table();

// Exact residue arithmetic in f32 for |x| < 2^22: bal(x) = x - q rint(x fl(1/q))
// (the quotient estimate errs by less than |x| 2^-24 / q < 1/(4 q), and x / q
// is never within 1/(2 q) of a half-integer since q is odd); the updates keep
// |x| below 2^21 + 2^10, the range es_selftest_gj_reduction checks.
struct ModF {
  float q, qinv;
};
// The host branch performs the same three IEEE operations (fused multiply-add,
// add, fused multiply-add, round to nearest) so that es_selftest_gj_reduction
// can check this function exhaustively on the CPU.
ES_HD float fred(float x, const ModF& mf) {
  const float kM = 12582912.0f;  // 1.5 * 2^23
#if defined(__CUDA_ARCH__)
  const float k = __fadd_rn(__fmaf_rn(x, mf.qinv, kM), -kM);
  return __fmaf_rn(-k, mf.q, x);
#else
  const float k = std::fmaf(x, mf.qinv, kM) + (-kM);
  return std::fmaf(-k, mf.q, x);
#endif
}
// 2^23 + 128 + x for the signed byte x = byte u of w: the f32 with bits 0x4B0000uu, uu = x + 128
__device__ __forceinline__ float sbyte_fb(uint32_t w, int u) {
  return __int_as_float((int)__byte_perm(w ^ 0x80808080u, 0x4B000000u, 0x7540 + u));
}
// signed byte u of w as f32
__device__ __forceinline__ float sbyte_f(uint32_t w, int u) { return __fadd_rn(sbyte_fb(w, u), -8388736.0f); }
// low byte of an exact integer-valued f32 in (-2^22, 2^22), two's complement
ES_HD uint32_t fbyte(float x) {
#if defined(__CUDA_ARCH__)
  return (uint32_t)__float_as_int(__fadd_rn(x, 12582912.0f)) & 0xFFu;
#else
  const float t = x + 12582912.0f;
  uint32_t u;
  std::memcpy(&u, &t, 4);
  return u & 0xFFu;
#endif
}

__device__ __forceinline__ void mma_f16_16x8x16(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}

// 16-byte global -> shared copy (zero fill when !valid), its group commit and wait
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}






// ------------------------------------------------------------------ panel
template <int NBP>
__global__ void __launch_bounds__(1024) k_gj_panel(GJParams p, int64_t k0, int kb, int use_smem) {
  const int j = blockIdx.x;
  if (p.bad[j]) return;
  const ModQ m = c_modq.v[j];
  const int64_t n = p.n, ld = p.ld;
  int8_t* Wj = p.W + (int64_t)j * n * ld;
  extern __shared__ __align__(16) unsigned char smem[];
  int8_t* panel = use_smem ? reinterpret_cast<int8_t*>(smem) : p.gpanel + (int64_t)j * n * NBP;
  uint8_t* usedS = use_smem ? reinterpret_cast<uint8_t*>(smem + n * NBP) : p.used + (int64_t)j * n;
  __shared__ int s_red[32];
  __shared__ int s_piv[NBP];
  __shared__ int32_t s_prow[NBP];
  __shared__ int s_p;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;

  // panel columns k0 .. k0+NBP-1 (16-byte chunks; chunks past ld read as zero)
  for (int64_t idx = tid; idx < n * (NBP / 16); idx += blockDim.x) {
    int64_t i = idx / (NBP / 16);
    int cch = (int)(idx - i * (NBP / 16));
    int4 v = make_int4(0, 0, 0, 0);
    if (k0 + 16 * cch < ld) v = *reinterpret_cast<const int4*>(Wj + i * ld + k0 + 16 * cch);
    *reinterpret_cast<int4*>(panel + i * NBP + 16 * cch) = v;
  }
  if (use_smem)
    for (int64_t i = tid; i < n; i += blockDim.x) usedS[i] = p.used[(int64_t)j * n + i];
  __syncthreads();

  for (int a = 0; a < kb; ++a) {
    // pivot: lowest-index row not yet used with a nonzero entry in column a
    int best = INT_MAX;
    for (int64_t i = tid; i < n; i += blockDim.x)
      if (!usedS[i] && panel[i * NBP + a] != 0) {
        best = (int)i;
        break;
      }
    best = __reduce_min_sync(0xffffffffu, best);
    if (lane == 0) s_red[warp] = best;
    __syncthreads();
    if (warp == 0) {
      int v = lane < nwarps ? s_red[lane] : INT_MAX;
      v = __reduce_min_sync(0xffffffffu, v);
      if (lane == 0) s_p = v;
    }
    __syncthreads();
    const int pr = s_p;
    if (pr == INT_MAX) {  // no pivot: q_j | det A
      if (tid == 0) p.bad[j] = 1;
      return;
    }
    const int32_t pvs = panel[(int64_t)pr * NBP + a];
    const uint32_t inv = inv_mod((uint32_t)(pvs < 0 ? pvs + (int32_t)m.q : pvs), m);
    if (tid < NBP) {
      int32_t v = panel[(int64_t)pr * NBP + tid];
      s_prow[tid] = (tid == a) ? bal_from_unsigned(inv, m) : reduce_bal(v * (int32_t)inv, m);
    }
    __syncthreads();
    for (int64_t i = tid; i < n; i += blockDim.x) {
      int8_t* row = panel + i * NBP;
      if (i == pr) {
#pragma unroll
        for (int c4 = 0; c4 < NBP / 16; ++c4) {
          uint32_t w[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t x = 0;
#pragma unroll
            for (int u = 0; u < 4; ++u) x |= ((uint32_t)(uint8_t)(int8_t)s_prow[c4 * 16 + q4 * 4 + u]) << (8 * u);
            w[q4] = x;
          }
          *reinterpret_cast<int4*>(row + 16 * c4) = make_int4(w[0], w[1], w[2], w[3]);
        }
        continue;
      }
      const int32_t f = row[a];
      if (f == 0) continue;
#pragma unroll
      for (int c4 = 0; c4 < NBP / 16; ++c4) {
        int4 v = *reinterpret_cast<const int4*>(row + 16 * c4);
        uint32_t w[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t x = 0;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int t = c4 * 16 + q4 * 4 + u;
            int32_t old = (t == a) ? 0 : sbyte(w[q4], u);
            int32_t r = reduce_bal(old - f * s_prow[t], m);
            x |= ((uint32_t)(uint8_t)(int8_t)r) << (8 * u);
          }
          w[q4] = x;
        }
        *reinterpret_cast<int4*>(row + 16 * c4) = make_int4(w[0], w[1], w[2], w[3]);
      }
    }
    if (tid == 0) {
      usedS[pr] = 1;
      s_piv[a] = pr;
      p.piv[(int64_t)j * n + k0 + a] = pr;
    }
    __syncthreads();
  }

  // write the panel back (only its kb real columns)
  for (int64_t idx = tid; idx < n * kb; idx += blockDim.x) {
    int64_t i = idx / kb;
    int a = (int)(idx - i * kb);
    Wj[i * ld + k0 + a] = panel[i * NBP + a];
  }
  if (use_smem)
    for (int64_t i = tid; i < n; i += blockDim.x) p.used[(int64_t)j * n + i] = usedS[i];
  // stage U^T (pivot rows outside the panel) and zero those entries in place
  int8_t* UTj = p.UT + (int64_t)j * ld * p.utw;
  for (int64_t idx = tid; idx < (int64_t)NBP * ld; idx += blockDim.x) {
    int a = (int)(idx / ld);
    int64_t col = idx - (int64_t)a * ld;
    int8_t v = 0;
    if (a < kb && (col < k0 || col >= k0 + kb)) {
      int64_t off = (int64_t)s_piv[a] * ld + col;
      v = Wj[off];
      Wj[off] = 0;
    }
    UTj[col * p.utw + a] = v;
  }
}

// ------------------------------------------------------------------ cluster panel
// The NB = 32 panel for 1024 < n <= 4096, spread over a thread-block cluster of
// kClCtas CTAs per prime, so that the rows fit in registers and 424 CTAs share
// the SMs instead of 53.  CTA c of the cluster owns rows c kClRows + tid +
// kClThreads i (i < kClR) as exact f32 in a rotating frame: at step a the
// entry of panel column (a + t) mod 32 sits in v[t], so the pivot column is
// always v[0] and no register is indexed at run time.  Entries are reduced
// lazily: each step adds at most |f p_t| <= 125^2, so after 32 steps they
// stay below 2^19 (exact in f32 and in fred's range).  One cluster barrier
// per step: every warp broadcasts (distributed shared memory) its lowest
// unused row with a nonzero reduced pivot entry and that row's reduced
// entries to all CTAs of the cluster; after the barrier every thread takes
// the lowest of the cluster's 32 candidates as the pivot row, scales it by
// the pivot's inverse, and updates its rows (exchange form: the pivot
// column becomes -f p^-1, as in k_gj_panel).  Every decision is taken from
// the same broadcast data in every CTA, so the control flow (including a
// prime without a pivot) is uniform over the cluster.  Then the panel is
// written back, and the CTAs stage U^T and zero the pivot rows column-wise.
constexpr int kClCtas = 8, kClThreads = 128, kClR = 4, kClRows = kClThreads * kClR;
constexpr int64_t kClMaxN = (int64_t)kClCtas * kClRows;  // 4096
constexpr int kClWarps = kClCtas * kClThreads / 32;      // 32 candidates per step

__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cl_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cl_map(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"((uint32_t)__cvta_generic_to_shared(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void cl_st_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void cl_st_s32(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__global__ void __launch_bounds__(kClThreads) k_gj_panel_cl(GJParams p, int64_t k0, int kb) {
  constexpr int NBP = 32;
  const int j = blockIdx.x / kClCtas;
  if (p.bad[j]) return;  // the same for every CTA of the cluster
  const uint32_t crank = cl_rank();
  const ModQ m = c_modq.v[j];
  const ModF mf{(float)m.q, c_qinv.v[j]};
  const int n = (int)p.n, ld = (int)p.ld;
  int8_t* Wj = p.W + (int64_t)j * n * ld;
  __shared__ uint8_t s_inv[256];
  __shared__ int s_wmin[2][kClWarps];
  __shared__ __align__(16) float s_cand[2][kClWarps][NBP];
  __shared__ int s_piv[NBP];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gw = (int)crank * (kClThreads / 32) + warp;
  for (int v = tid; v < (int)m.q; v += kClThreads) s_inv[v] = v ? (uint8_t)inv_mod((uint32_t)v, m) : 0;
  float v[kClR][NBP];
  bool used[kClR];
  int rowi[kClR];
#pragma unroll
  for (int i = 0; i < kClR; ++i) {
    const int row = (int)crank * kClRows + tid + kClThreads * i;
    rowi[i] = row;
    const bool active = row < n;
#pragma unroll
    for (int c4 = 0; c4 < NBP / 16; ++c4) {
      int4 w = make_int4(0, 0, 0, 0);
      if (active && k0 + 16 * c4 < ld) w = *reinterpret_cast<const int4*>(Wj + (int64_t)row * ld + k0 + 16 * c4);
      const uint32_t ww[4] = {(uint32_t)w.x, (uint32_t)w.y, (uint32_t)w.z, (uint32_t)w.w};
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
        for (int u = 0; u < 4; ++u) v[i][c4 * 16 + q4 * 4 + u] = (float)sbyte(ww[q4], u);
    }
    used[i] = active ? p.used[(int64_t)j * n + row] != 0 : true;
  }
  cl_sync();  // every CTA of the cluster runs before any broadcast reaches it
#pragma unroll 1
  for (int a = 0; a < kb; ++a) {
    const int par = a & 1;
    // this thread's lowest candidate row (its rows ascend with i)
    float f[kClR];
    int cand = INT_MAX, ci = 0;
#pragma unroll
    for (int i = kClR - 1; i >= 0; --i) {
      f[i] = fred(v[i][0], mf);
      if (!used[i] && f[i] != 0.0f) {
        cand = rowi[i];
        ci = i;
      }
    }
    const int wc = __reduce_min_sync(0xffffffffu, cand);
    const unsigned own = __ballot_sync(0xffffffffu, cand == wc && wc != INT_MAX);
    float mine = 0.0f;
    if (wc != INT_MAX) {
      const int owner = __ffs(own) - 1;
#pragma unroll
      for (int t = 0; t < NBP; ++t) {
        float x = v[0][t];
#pragma unroll
        for (int i = 1; i < kClR; ++i) x = ci == i ? v[i][t] : x;
        x = __shfl_sync(0xffffffffu, x, owner);
        if (lane == t) mine = fred(x, mf);
      }
    }
#pragma unroll 1
    for (uint32_t dst = 0; dst < (uint32_t)kClCtas; ++dst) {
      if (wc != INT_MAX) cl_st_f32(cl_map(&s_cand[par][gw][lane], dst), mine);
      if (lane == 0) cl_st_s32(cl_map(&s_wmin[par][gw], dst), wc);
    }
    cl_sync();
    int pr = INT_MAX, pw = 0;
#pragma unroll 4
    for (int w = 0; w < kClWarps; ++w) {
      const int x = s_wmin[par][w];
      if (x < pr) {
        pr = x;
        pw = w;
      }
    }
    if (pr == INT_MAX) {  // no pivot in this column: q_j | det A (every CTA sees it)
      if (crank == 0 && tid == 0) p.bad[j] = 1;
      cl_sync();
      return;
    }
    // the pivot row scaled by its inverse (rotated frame; entry 0 = the pivot
    // entry): lane t holds entry t, handed to the update by shuffles
    float pl;
    {
      const float p0 = s_cand[par][pw][0];
      const int p0i = (int)p0;
      const float inv = (float)bal_from_unsigned(s_inv[p0i < 0 ? p0i + (int)m.q : p0i], m);
      pl = lane == 0 ? inv : fred(s_cand[par][pw][lane] * inv, mf);
    }
    if (tid == 0) s_piv[a] = pr;
    if (crank == 0 && tid == 0) p.piv[(int64_t)j * n + k0 + a] = pr;
    float fe[kClR];  // multiplier per row: -f, 0 for an untouched row; the pivot row takes the scaled row
    bool isp[kClR];
#pragma unroll
    for (int i = 0; i < kClR; ++i) {
      isp[i] = rowi[i] == pr;
      fe[i] = isp[i] ? 0.0f : -f[i];
      if (isp[i]) used[i] = true;
    }
    // update and rotate by one in place (column a + 1 becomes entry 0): entry
    // t - 1 takes the new value of entry t, the last one the new pivot column
    // (-f p^-1, the scaled pivot entry for the pivot row, the old entry when f = 0)
    const float p0s = __shfl_sync(0xffffffffu, pl, 0);
    float last[kClR];
#pragma unroll
    for (int i = 0; i < kClR; ++i) last[i] = isp[i] ? p0s : (fe[i] != 0.0f ? fe[i] * p0s : v[i][0]);
#pragma unroll
    for (int t = 1; t < NBP; ++t) {
      const float pt = __shfl_sync(0xffffffffu, pl, t);
#pragma unroll
      for (int i = 0; i < kClR; ++i) v[i][t - 1] = isp[i] ? pt : __fmaf_rn(fe[i], pt, v[i][t]);
    }
#pragma unroll
    for (int i = 0; i < kClR; ++i) v[i][NBP - 1] = last[i];
  }
  // rotate the frame back: column c at v[c] (kb < 32 only on the last panel)
  for (int a = kb; a < NBP; ++a)
#pragma unroll
    for (int i = 0; i < kClR; ++i) {
      const float v0 = v[i][0];
#pragma unroll
      for (int t = 1; t < NBP; ++t) v[i][t - 1] = v[i][t];
      v[i][NBP - 1] = v0;
    }
  // write back the panel's kb real columns and the used flags
#pragma unroll
  for (int i = 0; i < kClR; ++i) {
    const int row = rowi[i];
    if (row >= n) continue;
#pragma unroll
    for (int c4 = 0; c4 < NBP / 16; ++c4) {
      if (k0 + 16 * c4 >= ld) continue;
      uint32_t ww[4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t x = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = c4 * 16 + q4 * 4 + u;
          const uint32_t b = c < kb ? fbyte(fred(v[i][c], mf)) : (uint32_t)(uint8_t)Wj[(int64_t)row * ld + k0 + c];
          x |= b << (8 * u);
        }
        ww[q4] = x;
      }
      *reinterpret_cast<int4*>(Wj + (int64_t)row * ld + k0 + 16 * c4) = make_int4(ww[0], ww[1], ww[2], ww[3]);
    }
    p.used[(int64_t)j * n + row] = used[i] ? 1 : 0;
  }
  __syncthreads();
  // stage U^T (pivot rows outside the panel) and zero those entries in place;
  // the cluster's CTAs take interleaved columns
  int8_t* UTj = p.UT + (int64_t)j * ld * p.utw;
  for (int col = (int)crank * kClThreads + tid; col < ld; col += kClCtas * kClThreads) {
    const bool outside = col < k0 || col >= k0 + kb;
    uint32_t w[NBP / 4];
#pragma unroll
    for (int q = 0; q < NBP / 4; ++q) {
      uint32_t x = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int a = 4 * q + u;
        const uint8_t b = (a < kb && outside) ? (uint8_t)Wj[(int64_t)s_piv[a] * ld + col] : (uint8_t)0;
        x |= (uint32_t)b << (8 * u);
      }
      w[q] = x;
    }
#pragma unroll
    for (int c4 = 0; c4 < NBP / 16; ++c4)
      *reinterpret_cast<int4*>(UTj + (int64_t)col * p.utw + 16 * c4) =
          make_int4(w[4 * c4], w[4 * c4 + 1], w[4 * c4 + 2], w[4 * c4 + 3]);
    if (outside)
      for (int a = 0; a < kb; ++a) Wj[(int64_t)s_piv[a] * ld + col] = 0;
  }
  cl_sync();  // no CTA leaves while another could still address its shared memory
}

// Panel in registers (n <= blockDim = 1024): thread i holds row i's NBP panel
// entries as int32 and applies each exchange step with one multiply-add per
// entry, without reducing: the pivot column is reduced when it becomes the
// pivot column (to find the pivot and the multipliers f, |f| <= 125) and the
// pivot row when it is scaled, so every other entry grows by at most
// |f p_t| <= 125^2 per step: below 125 + NBP 125^2 < 2^31.  Entries are
// reduced once, when the panel is written back.  The step loop is not
// unrolled (the register row is read and written through selects on the
// step index) so its code stays resident in the instruction cache; the pivot
// row is scaled by warp 0, one entry per lane, with inverses from a per-prime
// table in shared memory.  Same result as k_gj_panel.
template <int NBP>
__device__ __forceinline__ int32_t sel(const int32_t (&v)[NBP], int a) {
  int32_t r = 0;
#pragma unroll
  for (int t = 0; t < NBP; ++t) r = (t == a) ? v[t] : r;
  return r;
}

template <int NBP>
__global__ void __launch_bounds__(1024, 1) k_gj_panel_reg(GJParams p, int64_t k0, int kb) {
  const int j = blockIdx.x;
  if (p.bad[j]) return;
  const ModQ m = c_modq.v[j];
  const int n = (int)p.n, ld = (int)p.ld;
  int8_t* Wj = p.W + (int64_t)j * n * ld;
  __shared__ uint8_t s_inv[256];
  __shared__ __align__(16) int s_wmin[32];
  __shared__ __align__(16) int32_t s_raw[NBP];
  __shared__ __align__(16) int32_t s_prow[NBP];
  __shared__ __align__(16) int32_t s_pupd[NBP];
  __shared__ int s_piv[NBP];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int row = tid;
  const bool active = row < n;
  for (int v = tid; v < (int)m.q; v += blockDim.x) s_inv[v] = v ? (uint8_t)inv_mod((uint32_t)v, m) : 0;
  if (tid < 32) s_wmin[tid] = INT_MAX;
  int32_t v[NBP];
#pragma unroll
  for (int c4 = 0; c4 < NBP / 16; ++c4) {
    int4 w = make_int4(0, 0, 0, 0);
    if (active && k0 + 16 * c4 < ld) w = *reinterpret_cast<const int4*>(Wj + (int64_t)row * ld + k0 + 16 * c4);
    const uint32_t ww[4] = {(uint32_t)w.x, (uint32_t)w.y, (uint32_t)w.z, (uint32_t)w.w};
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
      for (int u = 0; u < 4; ++u) v[c4 * 16 + q4 * 4 + u] = sbyte(ww[q4], u);
  }
  bool used = active ? p.used[(int64_t)j * n + row] != 0 : true;
  __syncthreads();
#pragma unroll 1
  for (int a = 0; a < kb; ++a) {
    const int32_t f = reduce_bal(sel<NBP>(v, a), m);
    int cand = (!used && f != 0) ? row : INT_MAX;
    cand = __reduce_min_sync(0xffffffffu, cand);
    if (lane == 0) s_wmin[warp] = cand;
    __syncthreads();  // (1) candidates of every warp
    int pr = INT_MAX;
#pragma unroll
    for (int w4 = 0; w4 < 8; ++w4) {
      const int4 c = *reinterpret_cast<const int4*>(s_wmin + 4 * w4);
      pr = min(pr, min(min(c.x, c.y), min(c.z, c.w)));
    }
    if (pr == INT_MAX) {  // no pivot: q_j | det A
      if (tid == 0) p.bad[j] = 1;
      return;
    }
    if (row == pr) {
#pragma unroll
      for (int t = 0; t < NBP; ++t) s_raw[t] = (t == a) ? f : v[t];
      used = true;
      s_piv[a] = pr;
      p.piv[(int64_t)j * n + k0 + a] = pr;
    }
    __syncthreads();  // (2) raw pivot row
    if (warp == 0) {
      const int32_t pf = s_raw[a];
      const uint32_t inv = s_inv[pf < 0 ? pf + (int32_t)m.q : pf];
      for (int t = lane; t < NBP; t += 32) {
        const int32_t pt =
            (t == a) ? bal_from_unsigned(inv, m) : reduce_bal(reduce_bal(s_raw[t], m) * (int32_t)inv, m);
        s_prow[t] = pt;
        s_pupd[t] = (t == a) ? pt + 1 : pt;
      }
    }
    __syncthreads();  // (3) scaled pivot row
    if (row == pr) {
#pragma unroll
      for (int t4 = 0; t4 < NBP / 4; ++t4) {
        const int4 pv = *reinterpret_cast<const int4*>(s_prow + 4 * t4);
        v[4 * t4] = pv.x;
        v[4 * t4 + 1] = pv.y;
        v[4 * t4 + 2] = pv.z;
        v[4 * t4 + 3] = pv.w;
      }
    } else if (f != 0) {
      // v[t] -= f p_t for every t, with p_a taken as inv + 1: the pivot column
      // then becomes v[a] - f inv - f = -f inv (mod q), since v[a] = f (mod q).
#pragma unroll
      for (int t4 = 0; t4 < NBP / 4; ++t4) {
        const int4 pv = *reinterpret_cast<const int4*>(s_pupd + 4 * t4);
        v[4 * t4] -= f * pv.x;
        v[4 * t4 + 1] -= f * pv.y;
        v[4 * t4 + 2] -= f * pv.z;
        v[4 * t4 + 3] -= f * pv.w;
      }
    }
  }
  // reduce and write the panel back (padding columns stay zero: their pivot-row entries are zero)
  if (active) {
#pragma unroll
    for (int c4 = 0; c4 < NBP / 16; ++c4) {
      if (k0 + 16 * c4 >= ld) continue;
      uint32_t ww[4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t x = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          x |= ((uint32_t)(uint8_t)(int8_t)reduce_bal(v[c4 * 16 + q4 * 4 + u], m)) << (8 * u);
        ww[q4] = x;
      }
      *reinterpret_cast<int4*>(Wj + (int64_t)row * ld + k0 + 16 * c4) = make_int4(ww[0], ww[1], ww[2], ww[3]);
    }
    p.used[(int64_t)j * n + row] = used ? 1 : 0;
  }
  __syncthreads();
  // stage U^T (pivot rows outside the panel) and zero those entries in place:
  // thread = column; all kb loads are issued before any store
  int8_t* UTj = p.UT + (int64_t)j * ld * p.utw;
  for (int col = tid; col < ld; col += blockDim.x) {
    const bool outside = col < k0 || col >= k0 + kb;
    uint32_t w[NBP / 4];
#pragma unroll
    for (int q = 0; q < NBP / 4; ++q) {
      uint32_t x = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int a = 4 * q + u;
        const uint8_t b = (a < kb && outside) ? (uint8_t)Wj[(int64_t)s_piv[a] * ld + col] : (uint8_t)0;
        x |= (uint32_t)b << (8 * u);
      }
      w[q] = x;
    }
#pragma unroll
    for (int c4 = 0; c4 < NBP / 16; ++c4)
      *reinterpret_cast<int4*>(UTj + (int64_t)col * p.utw + 16 * c4) =
          make_int4(w[4 * c4], w[4 * c4 + 1], w[4 * c4 + 2], w[4 * c4 + 3]);
    if (outside)
      for (int a = 0; a < kb; ++a) Wj[(int64_t)s_piv[a] * ld + col] = 0;
  }
}

// Register panel with R rows per thread and T threads (n <= T R), one CTA
// per prime.  Exchange steps in a rotating frame: after each step a thread's
// row is rotated by one entry, so that at step a the entry of panel column c
// sits in v[(c - a) mod NBP] and the pivot column is always v[0] -- no
// runtime-indexed register access.  The update writes v[t] - f u_{t} into
// v[t - 1] (the rotation costs one move per row), with the pivot row scaled
// and stored already rotated by warp 0; the row is rotated back once, by kb,
// when the panel is written.  Rows of thread t: t, t + T, ..., t + T (R - 1).
struct PanelSmem {
  uint8_t inv[256];                   // inverses mod q
  __align__(16) int wmin[2][32];      // per-warp pivot candidate (row), by step parity
  __align__(16) float cand[2][32][32];  // per-warp candidate row's entries, reduced, rotated frame
  int piv[32];                        // the panel's pivot rows
  __align__(16) uint32_t u[32][8];    // a narrow update's U: column c, pivot rows 4w .. 4w + 3 in word w
};

// The kb exchange steps of the panel at k0; writes the reduced panel back to
// W and the used flags.  False when the prime has no pivot (it is flagged bad).
//
// Rows live in registers as exact f32 in a rotated frame (entry t of step a
// = column (a + t) mod NBP, so the pivot column is always entry 0).  One
// barrier per step: every warp publishes its own lowest unused row with a
// nonzero pivot-column entry, reduced by the warp's lanes, and after the
// barrier every thread takes the lowest of them, p = its pivot entry, and
// updates its rows with the multiplier f' = f p^-1:  v[t] <- v[t] - f' raw[t],
// pivot column <- -f'.  The pivot row itself is not scaled: it keeps raw with
// the pivot entry set to 1 and a scale p^-1 that multiplies the whole row on
// write-back (the multiplier of a scaled row's stored form is again its
// stored pivot entry times p^-1, so later steps treat it like any other row).
// Entries stay below 32 * 125^2 + 125 < 2^20 in magnitude.
template <int NBP, int R, int T>
__device__ __forceinline__ bool panel_factor(const GJParams& p, int j, const ModQ& m, int8_t* Wj, int64_t k0, int kb,
                                             PanelSmem& S) {
  static_assert(NBP == 32, "one reduced entry per lane");
  const int n = (int)p.n, ld = (int)p.ld;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const ModF mf{(float)m.q, c_qinv.v[j]};
  float v[R][NBP];
  int32_t sc[R];  // 0: row not yet a pivot (used rows of earlier panels stay 0 too), else its scale
  uint32_t usedm = 0;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int row = tid + T * i;
    const bool active = row < n;
#pragma unroll
    for (int c4 = 0; c4 < NBP / 16; ++c4) {
      int4 w = make_int4(0, 0, 0, 0);
      if (active && k0 + 16 * c4 < ld) w = *reinterpret_cast<const int4*>(Wj + (int64_t)row * ld + k0 + 16 * c4);
      const uint32_t ww[4] = {(uint32_t)w.x, (uint32_t)w.y, (uint32_t)w.z, (uint32_t)w.w};
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
        for (int u = 0; u < 4; ++u) v[i][c4 * 16 + q4 * 4 + u] = sbyte_f(ww[q4], u);
    }
    if (!active || p.used[(int64_t)j * n + row] != 0) usedm |= 1u << i;
    sc[i] = 0;
  }
  __syncthreads();
#pragma unroll 1
  for (int a = 0; a < kb; ++a) {
    const int par = a & 1;
    float f[R];
    int cand = INT_MAX;
#pragma unroll
    for (int i = R - 1; i >= 0; --i) {  // rows grow with i: the smallest i wins
      f[i] = fred(v[i][0], mf);
      if (!((usedm >> i) & 1) && f[i] != 0.0f) cand = tid + T * i;
    }
    const int wc = __reduce_min_sync(0xffffffffu, cand);
    if (wc != INT_MAX) {
      float* slot = S.cand[par][warp];
      if (cand == wc) {
#pragma unroll
        for (int i = 0; i < R; ++i)
          if (tid + T * i == wc) {
#pragma unroll
            for (int t4 = 0; t4 < NBP / 4; ++t4)
              *reinterpret_cast<float4*>(slot + 4 * t4) =
                  make_float4(v[i][4 * t4], v[i][4 * t4 + 1], v[i][4 * t4 + 2], v[i][4 * t4 + 3]);
          }
      }
      __syncwarp();
      slot[lane] = fred(slot[lane], mf);
    }
    if (lane == 0) S.wmin[par][warp] = wc;
    __syncthreads();  // the candidates of every warp
    int pr = INT_MAX;
#pragma unroll
    for (int w4 = 0; w4 < T / 128; ++w4) {
      const int4 c = *reinterpret_cast<const int4*>(&S.wmin[par][4 * w4]);
      pr = min(pr, min(min(c.x, c.y), min(c.z, c.w)));
    }
    if (pr == INT_MAX) {  // no pivot: q_j | det A
      if (tid == 0) p.bad[j] = 1;
      return false;
    }
    const float* raw = S.cand[par][(pr % T) >> 5];
    const int p0 = (int)raw[0];
    const int32_t inv = (int32_t)S.inv[p0 < 0 ? p0 + (int)m.q : p0];
    const float finv = (float)inv;
#pragma unroll
    for (int i = 0; i < R; ++i) {
      // the pivot row takes multiplier 0 and pivot entry 1 (its scale records p^-1)
      const bool is_piv = tid + T * i == pr;
      if (is_piv) {
        usedm |= 1u << i;
        sc[i] = inv;
        S.piv[a] = pr;
        p.piv[(int64_t)j * n + k0 + a] = pr;
      }
      const float fp = is_piv ? 0.0f : fred(f[i] * finv, mf);
#pragma unroll
      for (int t4 = 0; t4 < NBP / 4; ++t4) {
        const float4 r4 = *reinterpret_cast<const float4*>(raw + 4 * t4);
        const float rs[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int t = 4 * t4 + u;
          if (t > 0) v[i][t - 1] = __fmaf_rn(-fp, rs[u], v[i][t]);
        }
      }
      v[i][NBP - 1] = is_piv ? 1.0f : -fp;
    }
  }
  // rotate back by kb (entry t holds column (kb + t) mod NBP), log shifter
#pragma unroll
  for (int i = 0; i < R; ++i) {
#pragma unroll
    for (int sh = 1; sh < NBP; sh <<= 1) {
      if (kb & sh) {
        float tmp[NBP];
#pragma unroll
        for (int t = 0; t < NBP; ++t) tmp[(t + sh) & (NBP - 1)] = v[i][t];
#pragma unroll
        for (int t = 0; t < NBP; ++t) v[i][t] = tmp[t];
      }
    }
  }
  // reduce (times the row's scale, if it became a pivot here) and write the
  // panel back (padding columns stay zero: their pivot-row entries are zero)
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int row = tid + T * i;
    if (row >= n) continue;
    const float s = sc[i] ? (float)sc[i] : 1.0f;
#pragma unroll
    for (int c4 = 0; c4 < NBP / 16; ++c4) {
      uint32_t x[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        x[q] = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) x[q] |= fbyte(fred(fred(v[i][16 * c4 + 4 * q + u], mf) * s, mf)) << (8 * u);
      }
      if (k0 + 16 * c4 < ld)
        *reinterpret_cast<int4*>(Wj + (int64_t)row * ld + k0 + 16 * c4) = make_int4(x[0], x[1], x[2], x[3]);
    }
    p.used[(int64_t)j * n + row] = ((usedm >> i) & 1) ? 1 : 0;
  }
  return true;
}

// Stage U^T of the panel at k0 (pivot rows S.piv, kb of them) for the
// columns cb <= col < ce outside the panel into UT[col][0 .. NBP) (row width
// utw) and zero those entries in W.
template <int NBP, int T>
__device__ __forceinline__ void panel_stage(int64_t cb, int64_t ce, int8_t* Wj, int64_t ld, int64_t k0, int kb,
                                            const PanelSmem& S, int8_t* UTj, int utw) {
  for (int64_t col = cb + threadIdx.x; col < ce; col += T) {
    const bool outside = col < k0 || col >= k0 + kb;
    uint32_t w[NBP / 4];
#pragma unroll
    for (int q = 0; q < NBP / 4; ++q) {
      uint32_t x = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int aa = 4 * q + u;
        const uint8_t b = (aa < kb && outside) ? (uint8_t)Wj[(int64_t)S.piv[aa] * ld + col] : (uint8_t)0;
        x |= (uint32_t)b << (8 * u);
      }
      w[q] = x;
    }
#pragma unroll
    for (int c4 = 0; c4 < NBP / 16; ++c4)
      *reinterpret_cast<int4*>(UTj + col * utw + 16 * c4) =
          make_int4(w[4 * c4], w[4 * c4 + 1], w[4 * c4 + 2], w[4 * c4 + 3]);
    if (outside)
      for (int aa = 0; aa < kb; ++aa) Wj[(int64_t)S.piv[aa] * ld + col] = 0;
  }
}

// W[r][tc + c] = bal(W[r][tc + c] + sum_{a < K} W[r][fc + a] U[c][a]) for
// every row r < n and c < NC (columns at or past n keep their zero padding),
// with U staged in shared memory as Us[c][0 .. K) (row pitch K bytes).  f16
// tensor-core tiles, exact as in k_gj_update_mma (|sum| < 2^20): each warp
// takes 16-row tiles in turn with U's fragments held in registers, reading F
// as 32-bit words of m16n8k32 s8 layout and widening them to f16.  A tile's
// old entries come into the warp's own shared buffer by cp.async (double
// buffered, 16-byte copies), are updated there and leave with 16-byte stores.
// Buffer rows are NC bytes with chunk c of row r at c ^ f(r) (f = (r >> 1) & 3
// for 64-byte rows, (r >> 2) & 1 for 32-byte rows), conflict-free for the
// two-byte accesses of the C fragments.
constexpr int kBlkBuf = 2 * 16 * 64;  // bytes of a warp's two tile buffers
template <int K, int NC, int T>
__device__ __forceinline__ void block_mma_update(int8_t* Wj, int64_t ld, int n, int64_t fc, int64_t tc,
                                                 const uint8_t* Us, const ModF& mf, uint8_t* wbuf) {
  constexpr int NT = NC / 8, KK = K / 32, CPR = NC / 16;  // n-tiles, k chunks, 16-byte chunks per row
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t = lane & 3;
  auto swzo = [](int r, int c) { return r * NC + 16 * (c ^ (NC == 64 ? (r >> 1) & 3 : (r >> 2) & 1)); };
  uint32_t bf[NT][KK][2][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int kk = 0; kk < KK; ++kk)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(Us + (8 * nt + g) * K + 32 * kk + 16 * h + 4 * t);
        s8x4_to_f16(w, bf[nt][kk][h][0], bf[nt][kk][h][1]);
      }
  auto load_a = [&](int mt, uint32_t (&a8)[KK][4]) {
#pragma unroll
    for (int kk = 0; kk < KK; ++kk)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = 16 * mt + g + 8 * (r & 1);
        const int64_t col = fc + 32 * kk + 16 * (r >> 1) + 4 * t;
        a8[kk][r] = (row < n && col < ld) ? *reinterpret_cast<const uint32_t*>(Wj + (int64_t)row * ld + col) : 0u;
      }
  };
  auto issue_old = [&](int mt, uint8_t* buf) {  // 16 rows x NC bytes, 16 * CPR chunks
#pragma unroll
    for (int i = 0; i < (16 * CPR + 31) / 32; ++i) {
      const int idx = lane + 32 * i;
      if (idx < 16 * CPR) {
        const int r = idx / CPR, c = idx % CPR;
        const int row = 16 * mt + r;
        const int64_t col = tc + 16 * c;
        const bool ok = row < n && col < ld;
        cp_async16(buf + swzo(r, c), ok ? Wj + (int64_t)row * ld + col : Wj, ok);
      }
    }
    cp_async_commit();
  };
  const int ntiles = (n + 15) / 16;
  uint8_t* const obuf = wbuf + (size_t)warp * kBlkBuf;  // buffer i at obuf + 1024 i
  uint32_t a8[KK][4];
  if (warp < ntiles) {
    load_a(warp, a8);
    issue_old(warp, obuf);
  }
  const bool full = tc + NC <= n;  // no padding column among the NC
  int it = 0;
#pragma unroll 1
  for (int mt = warp; mt < ntiles; mt += T / 32, ++it) {
    uint8_t* buf = obuf + 1024 * (it & 1);
    const int mn = mt + T / 32;
    if (mn < ntiles) {
      issue_old(mn, obuf + 1024 * ((it + 1) & 1));
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncwarp();
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = -8388736.0f;
#pragma unroll
    for (int kk = 0; kk < KK; ++kk)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t af[4];
        s8x4_to_f16(a8[kk][2 * h], af[0], af[2]);
        s8x4_to_f16(a8[kk][2 * h + 1], af[1], af[3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_f16_16x8x16(acc[nt], af, bf[nt][kk][h]);
      }
    if (mn < ntiles) load_a(mn, a8);  // the next tile's F in flight during the epilogue
    // C reg r = row g + 8 (r >> 1), column 2 t + (r & 1); the accumulators
    // start at -(2^23 + 128) so that adding the old byte's 2^23 + (x + 128)
    // gives v = x + (F U) exactly
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int r = g + 8 * rr, c = 8 * nt + 2 * t;
        uint16_t* o = reinterpret_cast<uint16_t*>(buf + swzo(r, c >> 4) + (c & 15));
        const uint32_t ov = *o;
        const float v0 = __fadd_rn(acc[nt][2 * rr], sbyte_fb(ov, 0));
        const float v1 = __fadd_rn(acc[nt][2 * rr + 1], sbyte_fb(ov, 1));
        uint32_t nb = __byte_perm((uint32_t)__float_as_int(__fadd_rn(fred(v0, mf), 12582912.0f)),
                                  (uint32_t)__float_as_int(__fadd_rn(fred(v1, mf), 12582912.0f)), 0x0040);
        if (!full) {
          const int64_t gc = tc + c;
          if (gc + 1 >= n) nb = gc >= n ? ov : ((nb & 0xFFu) | (ov & 0xFF00u));
        }
        *o = (uint16_t)nb;
      }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < (16 * CPR + 31) / 32; ++i) {
      const int idx = lane + 32 * i;
      if (idx < 16 * CPR) {
        const int r = idx / CPR, c = idx % CPR;
        const int row = 16 * mt + r;
        const int64_t col = tc + 16 * c;
        if (row < n && col < ld)
          *reinterpret_cast<int4*>(Wj + (int64_t)row * ld + col) = *reinterpret_cast<const int4*>(buf + swzo(r, c));
      }
    }
    __syncwarp();  // the buffer is refilled two tiles on
  }
}

// One 64-column block (n <= 1024), one CTA per prime.  prev >= 0: first the
// previous block's update of this block's columns, F = W[:, prev .. prev + 64)
// (its final columns), U = its pivot rows in these columns (gathered and
// zeroed here; they must be current through the block before it).  Then
// for each 32-column half h: panel k0 + 32 h (kb1 or kb2 columns, kb2 = 0 =
// none), its U^T into UT[:, 32 h .. 32 h + 32) with the pivot rows zeroed,
// and the update of the block's other half by it (before the second panel
// is factored, after the first).
// own_only: stage only the block's own columns; the other columns read the
// pivot rows themselves (k_gj_update_strip, and the next block's catch-up),
// in the schedule that overlaps this kernel with the previous block's update.
template <int R, int T>
__global__ void __launch_bounds__(T, 1) k_gj_block64(GJParams p, int64_t k0, int kb1, int kb2, int own_only,
                                                     int64_t prev) {
  const int j = blockIdx.x;
  if (p.bad[j]) return;
  const ModQ m = c_modq.v[j];
  const ModF mf{(float)m.q, c_qinv.v[j]};
  const int n = (int)p.n;
  const int64_t ld = p.ld;
  int8_t* Wj = p.W + (int64_t)j * p.n * ld;
  int8_t* UTj = p.UT + (int64_t)j * ld * 64;
  __shared__ PanelSmem S;
  __shared__ __align__(16) uint8_t Us[64 * 64];
  __shared__ __align__(128) uint8_t wbuf[(T / 32) * kBlkBuf];
  for (int x = threadIdx.x; x < (int)m.q; x += T) S.inv[x] = x ? (uint8_t)inv_mod((uint32_t)x, m) : 0;
  if (prev >= 0) {
    // U of the previous block for this block's columns, gathered here from
    // its 64 pivot rows (a full block: every one is a pivot), which are
    // then zeroed in these columns: Us[c][a] = W[piv[prev + a]][k0 + c]
    uint8_t* Pr = wbuf;  // [64][64] staging, free until the block updates
    for (int idx = threadIdx.x; idx < 64 * 4; idx += T) {
      const int a = idx >> 2, h = idx & 3;
      const int64_t col = k0 + 16 * h;
      int4 x = make_int4(0, 0, 0, 0);
      if (col < ld) {
        int4* src = reinterpret_cast<int4*>(Wj + (int64_t)p.piv[(int64_t)j * p.n + prev + a] * ld + col);
        x = *src;
        *src = make_int4(0, 0, 0, 0);
      }
      *reinterpret_cast<int4*>(Pr + 64 * a + 16 * h) = x;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < 64 * 4; idx += T) {
      const int c = idx >> 2, a0 = 16 * (idx & 3);
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t x = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) x |= (uint32_t)Pr[64 * (a0 + 4 * q + u) + c] << (8 * u);
        w[q] = x;
      }
      *reinterpret_cast<int4*>(Us + 64 * c + a0) = make_int4(w[0], w[1], w[2], w[3]);
    }
    __syncthreads();
    block_mma_update<64, 64, T>(Wj, ld, n, prev, k0, Us, mf, wbuf);
  }
  __syncthreads();
  const int64_t cb = own_only ? k0 : 0, ce = own_only ? (k0 + 64 < ld ? k0 + 64 : ld) : ld;
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    const int64_t kp = k0 + 32 * h, other = k0 + 32 * (1 - h);
    const int kb = h ? kb2 : kb1;
    if (!panel_factor<32, R, T>(p, j, m, Wj, kp, kb, S)) return;
    __syncthreads();
    panel_stage<32, T>(cb, ce, Wj, ld, kp, kb, S, UTj + 32 * h, 64);
    if (kb2 == 0) return;
    __syncthreads();
    if (threadIdx.x < 64) {
      const int c = threadIdx.x >> 1, hh = threadIdx.x & 1;
      const int64_t col = other + c;
      const int4 x = col < ld ? *reinterpret_cast<const int4*>(UTj + 32 * h + col * 64 + 16 * hh) : make_int4(0, 0, 0, 0);
      *reinterpret_cast<int4*>(&S.u[c][4 * hh]) = x;
    }
    __syncthreads();
    block_mma_update<32, 32, T>(Wj, ld, n, kp, other, reinterpret_cast<const uint8_t*>(S.u), mf, wbuf);
    __syncthreads();
  }
}

// ------------------------------------------------------------------ update
// W[i][t] = bal(W[i][t] + sum_a F[i][a] U[a][t]) for all rows i and all
// columns t outside the panel; CTA tile 64 rows x 128 columns, one prime.
template <int NBP>
__global__ void __launch_bounds__(256) k_gj_update(GJParams p, int64_t k0, int kb) {
  const int j = blockIdx.z;
  if (p.bad[j]) return;
  const ModQ m = c_modq.v[j];
  const int64_t n = p.n, ld = p.ld;
  const int64_t row0 = (int64_t)blockIdx.y * 64, col0 = (int64_t)blockIdx.x * 128;
  int8_t* Wj = p.W + (int64_t)j * n * ld;
  const int8_t* UTj = p.UT + (int64_t)j * ld * p.utw;
  constexpr int KW = NBP / 4;  // 32-bit words along the panel
  __shared__ int32_t Fs[64][KW + 1];
  __shared__ int32_t Us[128][KW + 1];
  const int tid = threadIdx.x;
  for (int idx = tid; idx < 64 * (NBP / 16); idx += 256) {
    int r = idx / (NBP / 16), cch = idx % (NBP / 16);
    int64_t i = row0 + r;
    int4 v = make_int4(0, 0, 0, 0);
    if (i < n && k0 + 16 * cch < ld) v = *reinterpret_cast<const int4*>(Wj + i * ld + k0 + 16 * cch);
    Fs[r][cch * 4 + 0] = v.x;
    Fs[r][cch * 4 + 1] = v.y;
    Fs[r][cch * 4 + 2] = v.z;
    Fs[r][cch * 4 + 3] = v.w;
  }
  for (int idx = tid; idx < 128 * (NBP / 16); idx += 256) {
    int cc = idx / (NBP / 16), cch = idx % (NBP / 16);
    int64_t col = col0 + cc;
    int4 v = make_int4(0, 0, 0, 0);
    if (col < ld) v = *reinterpret_cast<const int4*>(UTj + col * p.utw + 16 * cch);
    Us[cc][cch * 4 + 0] = v.x;
    Us[cc][cch * 4 + 1] = v.y;
    Us[cc][cch * 4 + 2] = v.z;
    Us[cc][cch * 4 + 3] = v.w;
  }
  __syncthreads();
  const int ty = tid >> 4, tx = tid & 15;
  int32_t acc[4][8];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[r][u] = 0;
#pragma unroll
  for (int w = 0; w < KW; ++w) {
    int32_t f[4], uu[8];
#pragma unroll
    for (int r = 0; r < 4; ++r) f[r] = Fs[ty * 4 + r][w];
#pragma unroll
    for (int u = 0; u < 8; ++u) uu[u] = Us[tx + 16 * u][w];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int u = 0; u < 8; ++u) acc[r][u] = __dp4a(f[r], uu[u], acc[r][u]);
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    int64_t i = row0 + ty * 4 + r;
    if (i >= n) continue;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      int64_t col = col0 + tx + 16 * u;
      if (col >= n || (col >= k0 && col < k0 + kb)) continue;
      int8_t* w = Wj + i * ld + col;
      *w = (int8_t)reduce_bal((int32_t)*w + acc[r][u], m);
    }
  }
}

// Update on the tensor cores, f16 x f16 -> f32 (mma.sync.m16n8k16): a
// balanced residue (|x| <= 125) is exact in f16, and every depth-KW sum of
// products plus the old entry (|s| <= 64 * 125^2 + 125 < 2^20) is exact in
// the f32 accumulator, so the contraction F U (KW = 32 or 64) is exact.  On
// this part the f16 path has four times the rate of the s8 one.
//
// A CTA takes 128 columns of one prime and kUpdRowTiles tiles of 64 rows
// below each other; 8 warps, each 32 rows x 32 columns of a tile.  U^T (row
// width utw bytes, U^T[col][a] = pivot row a's entry of column col) is
// staged once and its fragments stay in registers; each tile's F =
// W[:, k0 .. k0 + KW) and old entries are brought in by cp.async, double
// buffered (the next tile loads while this one computes).  Shared-memory
// rows of the s8 F and U^T are 64 bytes with chunk c of row r at
// c ^ ((r >> 1) & 3).  U^T is read with ldmatrix as s8 fragments of m16n8k32
// shape and widened to f16 in registers: a 32-bit s8 fragment word holds four
// consecutive k; its low pair goes to the f16 register for k-slots 2t, 2t + 1
// and its high pair to 2t + 8, 2t + 9.  F is widened once per tile by all
// threads into an f16 tile laid out so that ldmatrix yields the same k-slot
// mapping, so the products pair up the same k.  The old tile
// (rows of 128 bytes, chunk c of row r at c ^ (r & 7)) is updated in place
// from the C fragments and written back with 16-byte stores.
//
// The residue is taken in f32 as in fred (exact for |v| < 2^20).  The
// accumulators start at -(2^23 + 128), so adding an old byte's float
// 2^23 + (x + 128) gives v = x + (F U) exactly.  Columns updated: 32-column
// segments col0 with cbase <= col0 < cend outside [xb, xe) (which holds at
// least the panel); other segments are neither read nor written.
constexpr int kUpdRowTiles = 4;


__device__ __forceinline__ int rot3(int r) { return ((r << 1) | ((r >> 2) & 1)) & 7; }
__device__ __forceinline__ int swz64(int r, int c) { return r * 64 + 16 * (c ^ ((r >> 1) & 3)); }
__device__ __forceinline__ int swz128(int r, int c) { return r * 128 + 16 * (c ^ (r & 7)); }

template <int KW>
__global__ void __launch_bounds__(256, 2) k_gj_update_mma(GJParams p, const int8_t* __restrict__ UT, int utw,
                                                          int64_t k0, int64_t cbase, int64_t cend, int64_t xb,
                                                          int64_t xe) {
  constexpr int KC = KW / 16;  // 16-byte chunks per operand row
  const int j = blockIdx.z;
  if (p.bad[j]) return;
  const int64_t n = p.n, ld = p.ld;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t colc = cbase + (int64_t)blockIdx.x * 128;
  const int64_t rowc0 = (int64_t)blockIdx.y * (64 * kUpdRowTiles);
  const int ntile = (int)min((int64_t)kUpdRowTiles, (n - rowc0 + 63) / 64);
  int8_t* Wj = p.W + (int64_t)j * n * ld;
  const int8_t* UTj = UT + (int64_t)j * ld * utw;
  __shared__ __align__(128) uint8_t Bs[128 * 64];
  __shared__ __align__(128) uint8_t As[2][64 * 64];
  __shared__ __align__(128) uint8_t Os[2][64 * 128];
  __shared__ __align__(128) uint8_t Af[64 * 2 * KW];  // the tile's F widened to f16, rows of 2 KW bytes
  // chunk c of an Af row r: 128-byte rows c ^ (r & 7), 64-byte rows c ^ ((r >> 1) & 3)
  auto swzA = [](int r, int c) { return KW == 64 ? swz128(r, c) : swz64(r, c); };
  auto seg_ok = [&](int s) {  // 32-column segment s of this CTA is updated
    const int64_t c0 = colc + 32 * s;
    return c0 < ld && c0 < cend && (c0 < xb || c0 >= xe);
  };
  auto issue_tile = [&](int k) {
    const int buf = k & 1;
    const int64_t rowc = rowc0 + 64 * k;
    for (int i = tid; i < 64 * KC; i += 256) {
      const int r = i / KC, c = i % KC;
      const int64_t row = rowc + r, col = k0 + 16 * c;
      const bool ok = row < n && col < ld;
      cp_async16(As[buf] + swz64(r, c), ok ? Wj + row * ld + col : Wj, ok);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int idx = tid + 256 * i, r = idx >> 3, c = idx & 7;
      const int64_t row = rowc + r, col = colc + 16 * c;
      const bool ok = row < n && col < ld && seg_ok(c >> 1);
      cp_async16(Os[buf] + swz128(r, c), ok ? Wj + row * ld + col : Wj, ok);
    }
    cp_async_commit();
  };
  for (int i = tid; i < 128 * KC; i += 256) {
    const int r = i / KC, c = i % KC;
    const int64_t col = colc + r;
    cp_async16(Bs + swz64(r, c), col < ld ? UTj + col * utw + 16 * c : UTj, col < ld);
  }
  issue_tile(0);
  if (ntile > 1) issue_tile(1);
  const int mi8 = lane >> 3, rr8 = lane & 7;  // ldmatrix: matrix and row this lane addresses
  const int g = lane >> 2, t = lane & 3;
  const int wr = (warp >> 2) * 32, wc = (warp & 3) * 32;  // the warp's rows in a tile, columns in the CTA
  const bool wok = seg_ok(warp & 3);
  const float qf = (float)c_modq.v[j].q, qinv = c_qinv.v[j];
  const ModF mf{qf, qinv};
  uint32_t bf[KW / 32][2][4][2];  // U's f16 fragments: [kk][h][ni][reg]
#pragma unroll 1
  for (int k = 0; k < ntile; ++k) {
    const int buf = k & 1;
    if (k + 1 < ntile)
      cp_async_wait<1>();
    else
      cp_async_wait<0>();
    __syncthreads();
    // widen F once for all warps: an s8 chunk (16 consecutive k, four words)
    // becomes the f16 chunk pair 2 c (the words' low halves, k-slots 2t, 2t+1)
    // and 2 c + 1 (their high halves, k-slots 2t + 8, 2t + 9), so ldmatrix
    // gives the fragments the s8 path would widen in registers
    for (int i = tid; i < 64 * KC; i += 256) {
      const int r = i / KC, c = i % KC;
      const int4 w = *reinterpret_cast<const int4*>(As[buf] + swz64(r, c));
      uint32_t lo[4], hi[4];
      s8x4_to_f16((uint32_t)w.x, lo[0], hi[0]);
      s8x4_to_f16((uint32_t)w.y, lo[1], hi[1]);
      s8x4_to_f16((uint32_t)w.z, lo[2], hi[2]);
      s8x4_to_f16((uint32_t)w.w, lo[3], hi[3]);
      *reinterpret_cast<int4*>(Af + swzA(r, 2 * c)) = make_int4(lo[0], lo[1], lo[2], lo[3]);
      *reinterpret_cast<int4*>(Af + swzA(r, 2 * c + 1)) = make_int4(hi[0], hi[1], hi[2], hi[3]);
    }
    __syncthreads();
    if (k == 0) {
#pragma unroll
      for (int kk = 0; kk < KW / 32; ++kk)
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          uint32_t b8[4];  // reg i: column tile 2 np + (i >> 1), k half i & 1
          ldsm_x4(b8, Bs + swz64(wc + 8 * (2 * np + (mi8 >> 1)) + rr8, 2 * kk + (mi8 & 1)));
#pragma unroll
          for (int i = 0; i < 4; ++i)
            s8x4_to_f16(b8[i], bf[kk][i & 1][2 * np + (i >> 1)][0], bf[kk][i & 1][2 * np + (i >> 1)][1]);
        }
    }
    if (wok) {
      float acc[2][4][4];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[mi][ni][r] = -8388736.0f;
#pragma unroll
      for (int G = 0; G < KW / 16; ++G) {  // 16-k group: k half G & 1 of s8 chunk pair G >> 1
        // f16 fragment reg r = rows g + 8 (r & 1), k-slots 2 t + 8 (r >> 1) + 0..1
        uint32_t af[2][4];
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
          ldsm_x4(af[mi], Af + swzA(wr + 16 * mi + rr8 + 8 * (mi8 & 1), 2 * G + (mi8 >> 1)));
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
          for (int ni = 0; ni < 4; ++ni) mma_f16_16x8x16(acc[mi][ni], af[mi], bf[G >> 1][G & 1][ni]);
      }
      // C reg r = row g + 8 (r >> 1), column 2 t + (r & 1); two bytes of the old tile per pair.
      // The low bytes of x + 1.5 2^23 (x the balanced residue) are x's two's complement byte.
      const bool full = colc + wc + 32 <= n;  // no padding column in the warp's 32
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int r = wr + 16 * mi + g + 8 * rr, c = wc + 8 * ni + 2 * t;
            uint16_t* o = reinterpret_cast<uint16_t*>(Os[buf] + swz128(r, c >> 4) + (c & 15));
            const uint32_t ov = *o;
            const float v0 = __fadd_rn(acc[mi][ni][2 * rr], sbyte_fb(ov, 0));
            const float v1 = __fadd_rn(acc[mi][ni][2 * rr + 1], sbyte_fb(ov, 1));
            uint32_t nb = __byte_perm((uint32_t)__float_as_int(__fadd_rn(fred(v0, mf), 12582912.0f)),
                                      (uint32_t)__float_as_int(__fadd_rn(fred(v1, mf), 12582912.0f)), 0x0040);
            if (!full) {
              const int64_t gc = colc + c;
              if (gc + 1 >= n) nb = gc >= n ? ov : ((nb & 0xFFu) | (ov & 0xFF00u));
            }
            *o = (uint16_t)nb;
          }
    }
    __syncthreads();
    const int64_t rowc = rowc0 + 64 * k;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int idx = tid + 256 * i, r = idx >> 3, c = idx & 7;
      const int64_t row = rowc + r, col = colc + 16 * c;
      if (row < n && col < ld && seg_ok(c >> 1))
        *reinterpret_cast<int4*>(Wj + row * ld + col) = *reinterpret_cast<const int4*>(Os[buf] + swz128(r, c));
    }
    if (k + 2 < ntile) {
      __syncthreads();  // every thread has read this buffer
      issue_tile(k + 2);
    }
  }
}

// Depth-128 update (blocks of 128 columns, 1024 < n): as k_gj_update_mma, with
// two changes.  The sums reach 128 * 125^2 + 125 < 2^21; the f32 accumulator
// (started at -(2^23 + 128)) stays an exact integer below 2^24 in magnitude,
// and the residue step is exact up to |v| < 2^22 (its quotient estimate errs
// by less than 1/(4q) there; es_selftest_gj_reduction checks it exhaustively
// to 2^21 + 2^10).  U^T's fragments (128 columns x 128 k) no longer fit in
// registers next to the accumulators at two CTAs per SM, so U^T is widened
// once into a shared f16 tile laid out like the widened F (256-byte rows,
// chunk c of row r at c ^ (r & 7)) and read with ldmatrix every tile.
constexpr int kUpd128Smem = 128 * 256 + 2 * 64 * 128 + 2 * 64 * 128 + 64 * 256;  // Bh, As, Os, Af
__device__ __forceinline__ int swz256(int r, int c) { return r * 256 + 16 * (c ^ (r & 7)); }
__global__ void __launch_bounds__(256, 2) k_gj_update_mma128(GJParams p, const int8_t* __restrict__ UT, int utw,
                                                            int64_t k0, int64_t cbase, int64_t cend, int64_t xb,
                                                            int64_t xe) {
  constexpr int KW = 128, KC = KW / 16;
  const int j = blockIdx.z;
  if (p.bad[j]) return;
  const int64_t n = p.n, ld = p.ld;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t colc = cbase + (int64_t)blockIdx.x * 128;
  const int64_t rowc0 = (int64_t)blockIdx.y * (64 * kUpdRowTiles);
  const int ntile = (int)min((int64_t)kUpdRowTiles, (n - rowc0 + 63) / 64);
  int8_t* Wj = p.W + (int64_t)j * n * ld;
  const int8_t* UTj = UT + (int64_t)j * ld * utw;
  extern __shared__ __align__(128) uint8_t upd_smem[];
  uint8_t* Bh = upd_smem;                    // [128][256]: U^T widened to f16
  uint8_t* As0 = Bh + 128 * 256;             // [2][64][128]: s8 F
  uint8_t* Os0 = As0 + 2 * 64 * 128;         // [2][64][128]: old tile
  uint8_t* Af = Os0 + 2 * 64 * 128;          // [64][256]: F widened to f16
  auto seg_ok = [&](int sg) {
    const int64_t c0 = colc + 32 * sg;
    return c0 < ld && c0 < cend && (c0 < xb || c0 >= xe);
  };
  auto issue_tile = [&](int k) {
    const int buf = k & 1;
    const int64_t rowc = rowc0 + 64 * k;
    for (int i = tid; i < 64 * KC; i += 256) {
      const int r = i / KC, c = i % KC;
      const int64_t row = rowc + r, col = k0 + 16 * c;
      const bool ok = row < n && col < ld;
      cp_async16(As0 + buf * 64 * 128 + swz128(r, c), ok ? Wj + row * ld + col : Wj, ok);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int idx = tid + 256 * i, r = idx >> 3, c = idx & 7;
      const int64_t row = rowc + r, col = colc + 16 * c;
      const bool ok = row < n && col < ld && seg_ok(c >> 1);
      cp_async16(Os0 + buf * 64 * 128 + swz128(r, c), ok ? Wj + row * ld + col : Wj, ok);
    }
    cp_async_commit();
  };
  // U^T as s8 into Af's space first, then widened into Bh
  for (int i = tid; i < 128 * KC; i += 256) {
    const int r = i / KC, c = i % KC;
    const int64_t col = colc + r;
    cp_async16(Af + r * 128 + 16 * c, col < ld ? UTj + col * utw + 16 * c : UTj, col < ld);
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  for (int i = tid; i < 128 * KC; i += 256) {
    const int r = i / KC, c = i % KC;
    const int4 w = *reinterpret_cast<const int4*>(Af + r * 128 + 16 * c);
    uint32_t lo[4], hi[4];
    s8x4_to_f16((uint32_t)w.x, lo[0], hi[0]);
    s8x4_to_f16((uint32_t)w.y, lo[1], hi[1]);
    s8x4_to_f16((uint32_t)w.z, lo[2], hi[2]);
    s8x4_to_f16((uint32_t)w.w, lo[3], hi[3]);
    *reinterpret_cast<int4*>(Bh + swz256(r, 2 * c)) = make_int4(lo[0], lo[1], lo[2], lo[3]);
    *reinterpret_cast<int4*>(Bh + swz256(r, 2 * c + 1)) = make_int4(hi[0], hi[1], hi[2], hi[3]);
  }
  __syncthreads();  // Af's space is free again
  issue_tile(0);
  if (ntile > 1) issue_tile(1);
  const int mi8 = lane >> 3, rr8 = lane & 7;
  const int g = lane >> 2, t = lane & 3;
  const int wr = (warp >> 2) * 32, wc = (warp & 3) * 32;
  const bool wok = seg_ok(warp & 3);
  const float qf = (float)c_modq.v[j].q, qinv = c_qinv.v[j];
  const ModF mf{qf, qinv};
#pragma unroll 1
  for (int k = 0; k < ntile; ++k) {
    const int buf = k & 1;
    uint8_t* As = As0 + buf * 64 * 128;
    uint8_t* Os = Os0 + buf * 64 * 128;
    if (k + 1 < ntile)
      cp_async_wait<1>();
    else
      cp_async_wait<0>();
    __syncthreads();
    for (int i = tid; i < 64 * KC; i += 256) {
      const int r = i / KC, c = i % KC;
      const int4 w = *reinterpret_cast<const int4*>(As + swz128(r, c));
      uint32_t lo[4], hi[4];
      s8x4_to_f16((uint32_t)w.x, lo[0], hi[0]);
      s8x4_to_f16((uint32_t)w.y, lo[1], hi[1]);
      s8x4_to_f16((uint32_t)w.z, lo[2], hi[2]);
      s8x4_to_f16((uint32_t)w.w, lo[3], hi[3]);
      *reinterpret_cast<int4*>(Af + swz256(r, 2 * c)) = make_int4(lo[0], lo[1], lo[2], lo[3]);
      *reinterpret_cast<int4*>(Af + swz256(r, 2 * c + 1)) = make_int4(hi[0], hi[1], hi[2], hi[3]);
    }
    __syncthreads();
    if (wok) {
      float acc[2][4][4];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[mi][ni][r] = -8388736.0f;
#pragma unroll 2
      for (int G = 0; G < KW / 16; ++G) {  // 16-k group G: f16 chunks 2G (low halves) and 2G + 1 (high halves)
        uint32_t af[2][4];
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
          ldsm_x4(af[mi], Af + swz256(wr + 16 * mi + rr8 + 8 * (mi8 & 1), 2 * G + (mi8 >> 1)));
        uint32_t bfr[4][2];
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          uint32_t b4[4];  // reg i: column tile 2 np + (i >> 1), chunk 2 G + (i & 1)
          ldsm_x4(b4, Bh + swz256(wc + 8 * (2 * np + (mi8 >> 1)) + rr8, 2 * G + (mi8 & 1)));
#pragma unroll
          for (int i = 0; i < 4; ++i) bfr[2 * np + (i >> 1)][i & 1] = b4[i];
        }
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
          for (int ni = 0; ni < 4; ++ni) mma_f16_16x8x16(acc[mi][ni], af[mi], bfr[ni]);
      }
      const bool full = colc + wc + 32 <= n;
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int r = wr + 16 * mi + g + 8 * rr, c = wc + 8 * ni + 2 * t;
            uint16_t* o = reinterpret_cast<uint16_t*>(Os + swz128(r, c >> 4) + (c & 15));
            const uint32_t ov = *o;
            const float v0 = __fadd_rn(acc[mi][ni][2 * rr], sbyte_fb(ov, 0));
            const float v1 = __fadd_rn(acc[mi][ni][2 * rr + 1], sbyte_fb(ov, 1));
            uint32_t nb = __byte_perm((uint32_t)__float_as_int(__fadd_rn(fred(v0, mf), 12582912.0f)),
                                      (uint32_t)__float_as_int(__fadd_rn(fred(v1, mf), 12582912.0f)), 0x0040);
            if (!full) {
              const int64_t gc = colc + c;
              if (gc + 1 >= n) nb = gc >= n ? ov : ((nb & 0xFFu) | (ov & 0xFF00u));
            }
            *o = (uint16_t)nb;
          }
    }
    __syncthreads();
    const int64_t rowc = rowc0 + 64 * k;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int idx = tid + 256 * i, r = idx >> 3, c = idx & 7;
      const int64_t row = rowc + r, col = colc + 16 * c;
      if (row < n && col < ld && seg_ok(c >> 1))
        *reinterpret_cast<int4*>(Wj + row * ld + col) = *reinterpret_cast<const int4*>(Os + swz128(r, c));
    }
    if (k + 2 < ntile) {
      __syncthreads();
      issue_tile(k + 2);
    }
  }
}

// The wide update of the two-partition schedule, with the staging of U folded
// in.  A CTA owns one 64-column strip of one prime for every row, so it can
// read U straight from the block's pivot rows before anything writes them:
// no other CTA touches the strip.  The pivot rows' old entries count as zero
// (exactly what staging leaves in W), so W[pr][t] becomes F[pr] U[:, t].
// Per iteration a tile of 128 rows x 64 columns: 8 warps of 32 x 32, F and
// the old tile brought in by cp.async (double buffered), F widened to f16
// once per tile, U's f16 fragments held in registers, the old tile updated
// in shared memory and written back with 16-byte stores; arithmetic as in
// k_gj_update_mma (f16 mma.sync, exact f32 epilogue).  Strips inside
// [k0, xe) (the block and the next one, left to the panel side) are skipped.
// The block's pivots are piv[k0 + a] for a < kb1 and 32 <= a < 32 + kb2.
constexpr int kStripRows = 128;
constexpr size_t kStripSmem = 64 * 64 + 64 * 64 + 2 * kStripRows * 64 + kStripRows * 128 + 2 * kStripRows * 64 + 64 * 4;
__global__ void __launch_bounds__(256, 2) k_gj_update_strip(GJParams p, int64_t k0, int kb1, int kb2, int64_t xe) {
  const int j = blockIdx.y;
  if (p.bad[j]) return;
  const int64_t n = p.n, ld = p.ld;
  const int64_t colc = (int64_t)blockIdx.x * 64;
  if (colc >= ld || (colc >= k0 && colc < xe)) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int8_t* Wj = p.W + (int64_t)j * n * ld;
  extern __shared__ __align__(128) uint8_t usm[];
  uint8_t* Bs = usm;                      // U^T [64 columns][64 pivots], swz64
  uint8_t* Pr = Bs + 64 * 64;             // the pivot rows' strip [64][64], swz64
  uint8_t* As = Pr + 64 * 64;             // [2][128][64] s8 F, swz64
  uint8_t* Af = As + 2 * kStripRows * 64; // [128][128] f16 F, swz128
  uint8_t* Os = Af + kStripRows * 128;    // [2][128][64] old tile, swz64
  int32_t* pv = reinterpret_cast<int32_t*>(Os + 2 * kStripRows * 64);  // the block's pivot rows, -1 = none
  if (tid < 64) pv[tid] = (tid < 32 ? tid < kb1 : tid - 32 < kb2) ? p.piv[(int64_t)j * n + k0 + tid] : -1;
  __syncthreads();
  const int ntile = (int)((n + kStripRows - 1) / kStripRows);
  // this thread's two rows of a tile (r0, r0 + 64) and 16-byte chunk c of F
  // and of the strip; offsets within the prime fit 32 bits (n <= 1024 here)
  const int r0 = tid >> 2, c16 = 16 * (tid & 3);
  const int ni32 = (int)n, ld32 = (int)ld;
  const bool cf = k0 + c16 < ld, co = colc + c16 < ld;
  const int offA = (int)k0 + c16, offO = (int)colc + c16;
  const int sA0 = swz64(r0, tid & 3), sA1 = swz64(r0 + 64, tid & 3);
  auto issue_tile = [&](int k) {
    const int row0 = k * kStripRows + r0, row1 = row0 + 64;
    uint8_t* A = As + (k & 1) * kStripRows * 64;
    uint8_t* O = Os + (k & 1) * kStripRows * 64;
    const bool ok0 = row0 < ni32, ok1 = row1 < ni32;
    cp_async16(A + sA0, Wj + (ok0 && cf ? row0 * ld32 + offA : 0), ok0 && cf);
    cp_async16(O + sA0, Wj + (ok0 && co ? row0 * ld32 + offO : 0), ok0 && co);
    cp_async16(A + sA1, Wj + (ok1 && cf ? row1 * ld32 + offA : 0), ok1 && cf);
    cp_async16(O + sA1, Wj + (ok1 && co ? row1 * ld32 + offO : 0), ok1 && co);
    cp_async_commit();
  };
  {  // the pivot rows' strip (before this CTA writes any of them)
    const int r = tid >> 2, c = tid & 3;
    const int pr = pv[r];
    const bool ok = pr >= 0 && colc + 16 * c < ld;
    cp_async16(Pr + swz64(r, c), ok ? Wj + (int64_t)pr * ld + colc + 16 * c : Wj, ok);
    cp_async_commit();
  }
  issue_tile(0);
  if (ntile > 1) {
    issue_tile(1);
    cp_async_wait<2>();  // the pivot strip (the two tiles may still be in flight)
  } else {
    cp_async_wait<1>();
  }
  __syncthreads();
  {  // transpose: U^T[col][a] = Pr[a][col]; thread: column tid >> 2, pivots 16 (tid & 3) .. + 16
    const int col = tid >> 2, a0 = 16 * (tid & 3);
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t x = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int a = a0 + 4 * q + u;
        x |= (uint32_t)Pr[swz64(a, col >> 4) + (col & 15)] << (8 * u);
      }
      w[q] = x;
    }
    *reinterpret_cast<int4*>(Bs + swz64(col, a0 >> 4)) = make_int4(w[0], w[1], w[2], w[3]);
  }
  __syncthreads();
  const int mi8 = lane >> 3, rr8 = lane & 7;
  const int g = lane >> 2, t = lane & 3;
  const int wr = (warp >> 1) * 32, wc = (warp & 1) * 32;  // warp's rows in a tile, columns in the strip
  const ModF mf{(float)c_modq.v[j].q, c_qinv.v[j]};
  uint32_t bf[2][2][4][2];  // U's f16 fragments: [kk][h][ni][reg]
#pragma unroll
  for (int kk = 0; kk < 2; ++kk)
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      uint32_t b8[4];  // reg i: column tile 2 np + (i >> 1), k half i & 1
      ldsm_x4(b8, Bs + swz64(wc + 8 * (2 * np + (mi8 >> 1)) + rr8, 2 * kk + (mi8 & 1)));
#pragma unroll
      for (int i = 0; i < 4; ++i)
        s8x4_to_f16(b8[i], bf[kk][i & 1][2 * np + (i >> 1)][0], bf[kk][i & 1][2 * np + (i >> 1)][1]);
    }
  const bool full = colc + wc + 32 <= n;  // no padding column in the warp's 32
#pragma unroll 1
  for (int k = 0; k < ntile; ++k) {
    const int64_t rowc = (int64_t)k * kStripRows;
    uint8_t* A = As + (k & 1) * kStripRows * 64;
    uint8_t* O = Os + (k & 1) * kStripRows * 64;
    if (k + 1 < ntile)
      cp_async_wait<1>();
    else
      cp_async_wait<0>();
    __syncthreads();
    // widen F (see k_gj_update_mma) and clear the tile's pivot rows in the old tile
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = r0 + 64 * i, c = tid & 3;
      const int4 w = *reinterpret_cast<const int4*>(A + (i ? sA1 : sA0));
      uint32_t lo[4], hi[4];
      s8x4_to_f16((uint32_t)w.x, lo[0], hi[0]);
      s8x4_to_f16((uint32_t)w.y, lo[1], hi[1]);
      s8x4_to_f16((uint32_t)w.z, lo[2], hi[2]);
      s8x4_to_f16((uint32_t)w.w, lo[3], hi[3]);
      *reinterpret_cast<int4*>(Af + swz128(r, 2 * c)) = make_int4(lo[0], lo[1], lo[2], lo[3]);
      *reinterpret_cast<int4*>(Af + swz128(r, 2 * c + 1)) = make_int4(hi[0], hi[1], hi[2], hi[3]);
    }
    if (tid < 64) {
      const int pr = pv[tid];
      if (pr >= rowc && pr < rowc + kStripRows) {
        const int r = (int)(pr - rowc);
#pragma unroll
        for (int c = 0; c < 4; ++c) *reinterpret_cast<int4*>(O + swz64(r, c)) = make_int4(0, 0, 0, 0);
      }
    }
    __syncthreads();
    float acc[2][4][4];
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int ni = 0; ni < 4; ++ni)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[mi][ni][r] = -8388736.0f;
#pragma unroll
    for (int G = 0; G < 4; ++G) {
      uint32_t af[2][4];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) ldsm_x4(af[mi], Af + swz128(wr + 16 * mi + rr8 + 8 * (mi8 & 1), 2 * G + (mi8 >> 1)));
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) mma_f16_16x8x16(acc[mi][ni], af[mi], bf[G >> 1][G & 1][ni]);
    }
    // C reg r = row g + 8 (r >> 1), column 2 t + (r & 1)
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int ni = 0; ni < 4; ++ni)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const int r = wr + 16 * mi + g + 8 * rr, c = wc + 8 * ni + 2 * t;
          uint16_t* o = reinterpret_cast<uint16_t*>(O + swz64(r, c >> 4) + (c & 15));
          const uint32_t ov = *o;
          const float v0 = __fadd_rn(acc[mi][ni][2 * rr], sbyte_fb(ov, 0));
          const float v1 = __fadd_rn(acc[mi][ni][2 * rr + 1], sbyte_fb(ov, 1));
          uint32_t nb = __byte_perm((uint32_t)__float_as_int(__fadd_rn(fred(v0, mf), 12582912.0f)),
                                    (uint32_t)__float_as_int(__fadd_rn(fred(v1, mf), 12582912.0f)), 0x0040);
          if (!full) {
            const int64_t gc = colc + c;
            if (gc + 1 >= n) nb = gc >= n ? ov : ((nb & 0xFFu) | (ov & 0xFF00u));
          }
          *o = (uint16_t)nb;
        }
    __syncthreads();
    {
      const int row0 = (int)rowc + r0, row1 = row0 + 64;
      if (co && row0 < ni32) *reinterpret_cast<int4*>(Wj + row0 * ld32 + offO) = *reinterpret_cast<const int4*>(O + sA0);
      if (co && row1 < ni32) *reinterpret_cast<int4*>(Wj + row1 * ld32 + offO) = *reinterpret_cast<const int4*>(O + sA1);
    }
    if (k + 2 < ntile) {
      __syncthreads();  // every thread has read this buffer
      issue_tile(k + 2);
    }
  }
}

// ------------------------------------------------------------------ permute
__global__ void k_gj_pinv(GJParams p) {
  const int j = blockIdx.y;
  if (p.bad[j]) return;
  int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= p.n) return;
  p.pinv[(int64_t)j * p.n + p.piv[(int64_t)j * p.n + k]] = (int32_t)k;
}

// B[j][k][t] = W[j][piv[k]][pinv[t]] (t < n), zero for n <= t < ld.  One CTA
// per row (any n).
__global__ void k_gj_permute(GJParams p, int8_t* __restrict__ B, uint8_t* __restrict__ good) {
  const int j = blockIdx.y;
  const int64_t n = p.n, ld = p.ld, k = blockIdx.x;
  if (k == 0 && threadIdx.x == 0) good[j] = p.bad[j] ? 0 : 1;
  if (p.bad[j]) return;
  extern __shared__ __align__(16) unsigned char rowS[];
  const int8_t* src = p.W + (int64_t)j * n * ld + (int64_t)p.piv[(int64_t)j * n + k] * ld;
  for (int64_t t = threadIdx.x * 16; t < ld; t += blockDim.x * 16)
    *reinterpret_cast<int4*>(rowS + t) = *reinterpret_cast<const int4*>(src + t);
  __syncthreads();
  const int32_t* pinv = p.pinv + (int64_t)j * n;
  int8_t* dst = B + (int64_t)j * n * ld + k * ld;
  for (int64_t t = threadIdx.x; t < ld; t += blockDim.x) dst[t] = t < n ? (int8_t)rowS[pinv[t]] : (int8_t)0;
}

// The same for n <= kPermuteMaxN, CTA per kPermuteRows rows and prime: the
// inverse permutation sits in shared memory as 16-bit indices, each warp
// takes rows in turn with its own shared row buffer (the next row's 16-byte
// loads in flight while this one is gathered) and writes 4 bytes per lane.
constexpr int kPermuteMaxN = 8192, kPermuteRows = 64;
template <int kMaxCh>  // 16-byte chunks per lane and row: ld <= 512 kMaxCh
__global__ void __launch_bounds__(256) k_gj_permute_rows(GJParams p, int8_t* __restrict__ B,
                                                         uint8_t* __restrict__ good) {
  const int j = blockIdx.y;
  const int64_t n = p.n, ld = p.ld;
  if (blockIdx.x == 0 && threadIdx.x == 0) good[j] = p.bad[j] ? 0 : 1;
  if (p.bad[j]) return;
  extern __shared__ __align__(16) unsigned char psm[];
  uint16_t* pinv = reinterpret_cast<uint16_t*>(psm);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned char* rowS = psm + ((2 * n + 15) / 16) * 16 + (int64_t)warp * ld;
  const int32_t* pj = p.pinv + (int64_t)j * n;
  for (int64_t t = threadIdx.x; t < n; t += blockDim.x) pinv[t] = (uint16_t)pj[t];
  __syncthreads();
  const int8_t* Wj = p.W + (int64_t)j * n * ld;
  const int32_t* piv = p.piv + (int64_t)j * n;
  const int64_t k0 = (int64_t)blockIdx.x * kPermuteRows, k1 = min(n, k0 + kPermuteRows);
  const int nch = (int)(ld / 16);  // 16-byte chunks per row
  int4 buf[kMaxCh];
  auto fetch = [&](int64_t k) {
    const int4* src = reinterpret_cast<const int4*>(Wj + (int64_t)piv[k] * ld);
#pragma unroll
    for (int i = 0; i < kMaxCh; ++i)
      if (lane + 32 * i < nch) buf[i] = src[lane + 32 * i];
  };
  int64_t k = k0 + warp;
  if (k < k1) fetch(k);
  for (; k < k1; k += 8) {
#pragma unroll
    for (int i = 0; i < kMaxCh; ++i)
      if (lane + 32 * i < nch) reinterpret_cast<int4*>(rowS)[lane + 32 * i] = buf[i];
    __syncwarp();
    if (k + 8 < k1) fetch(k + 8);
    uint32_t* dst = reinterpret_cast<uint32_t*>(B + (int64_t)j * n * ld + k * ld);
    for (int64_t t = 4 * lane; t < ld; t += 128) {
      uint32_t w = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (t + u < n) w |= (uint32_t)rowS[pinv[t + u]] << (8 * u);
      dst[t / 4] = w;
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------ driver
namespace {
constexpr size_t kPanelSmemLimit = 200 * 1024;
int choose_nbp(int64_t n, bool* use_smem) {
  if ((size_t)n * 32 + (size_t)n <= kPanelSmemLimit) {
    *use_smem = true;
    return 32;
  }
  if ((size_t)n * 16 + (size_t)n <= kPanelSmemLimit) {
    *use_smem = true;
    return 16;
  }
  *use_smem = false;
  return 32;
}

struct InvLayout {
  size_t W, UT, piv, pinv, used, bad, gpanel, total;
};
InvLayout inverse_layout(int64_t n) {
  bool sm;
  int nbp = choose_nbp(n, &sm);
  int64_t ld = padded_ld(n);
  Layout L;
  InvLayout r;
  r.W = L.add((size_t)kNumPrimes * n * ld);
  // NB = 32: two panels' U^T side by side (four beyond n = 1024: 128-column blocks)
  r.UT = L.add((size_t)kNumPrimes * ld * (nbp == 32 ? (n > 1024 ? 128 : 64) : nbp));
  r.piv = L.add((size_t)kNumPrimes * n * 4);
  r.pinv = L.add((size_t)kNumPrimes * n * 4);
  r.used = L.add((size_t)kNumPrimes * n);
  r.bad = L.add((size_t)kNumPrimes * 4);
  r.gpanel = sm ? 0 : L.add((size_t)kNumPrimes * n * nbp);
  r.total = L.total;
  return r;
}

// One NB-column panel: pivots, multipliers, and the pivot rows of every other
// column staged into U^T (at gp.UT, rows of gp.utw bytes) and zeroed in W.
template <int NBP>
void panel(GJParams& gp, int64_t n, int64_t k0, int kb, bool use_smem, cudaStream_t st) {
  if (NBP == 32 && n > 1024 && n <= kClMaxN) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(kNumPrimes * kClCtas));
    cfg.blockDim = dim3(kClThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kClCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, k_gj_panel_cl, gp, k0, kb);
  } else {
    k_gj_panel<NBP><<<kNumPrimes, 1024, use_smem ? (size_t)n * NBP + (size_t)n : 0, st>>>(gp, k0, kb,
                                                                                       use_smem ? 1 : 0);
  }
  count_launch();
}

// NB = 16: panel, then the dp4a update of every other column.
es_status run_blocks16(GJParams& gp, int64_t n, bool use_smem, cudaStream_t st) {
  ES_CHECK(cuda_status(cudaFuncSetAttribute(k_gj_panel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)kPanelSmemLimit + 1024),
                       "panel smem attribute"));
  gp.utw = 16;
  const dim3 ugrid((unsigned)((gp.ld + 127) / 128), (unsigned)((n + 63) / 64), kNumPrimes);
  for (int64_t k0 = 0; k0 < n; k0 += 16) {
    const int kb = (int)((n - k0) < 16 ? (n - k0) : 16);
    panel<16>(gp, n, k0, kb, use_smem, st);
    k_gj_update<16><<<ugrid, 256, 0, st>>>(gp, k0, kb);
    count_launch();
  }
  return cuda_status(cudaGetLastError(), "gauss-jordan blocks");
}

// NB = 32 panels in blocks of 64 columns.  The exchange steps of a block act
// on every column t outside it as W_t <- W_t[R -> 0] + F W_t[R] (R = the
// block's 64 pivot rows in order, F = the block's 64 columns after all its
// steps; by induction over the steps, since each step is
// I - e_p e_p^T + f e_p^T), so inside the block the two panels update each
// other's 32 columns, and every other column gets ONE depth-64 update:
//   panel k0        -> U^T[:, 0..32)   (pivot rows R1, all columns, zeroed)
//   update [k0+32, k0+64) by F1 U1
//   panel k0 + 32   -> U^T[:, 32..64)  (pivot rows R2, all columns, zeroed)
//   update [k0, k0+32) by F2 U2
//   update every column outside [k0, k0+64) by W[:, k0..k0+64) U^T
// R2's entries outside the block are staged before any update reached them,
// as the formula needs.  The number of full passes over W halves.
//
// Beyond n = 1024 the blocks are 128 columns wide, two such halves H0, H1 of
// 64 in turn: H0 as above (its U^T staged for every column outside each
// panel), then H1 brought up to date by F_H0 U_H0, H1 as above, then H0's
// columns by F_H1 U_H1 (H1's pivot rows staged from them after H0 was done),
// and every column outside the block gets ONE depth-128 update
// (k_gj_update_mma128): half the passes over W of 64-column blocks.
es_status run_blocks64(GJParams& gp, int64_t n, bool use_smem, cudaStream_t st) {
  ES_CHECK(cuda_status(cudaFuncSetAttribute(k_gj_panel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)kPanelSmemLimit + 1024),
                       "panel smem attribute"));
  int8_t* const UT = gp.UT;
  const int64_t ld = gp.ld;
  const unsigned rtiles = (unsigned)((n + 64 * kUpdRowTiles - 1) / (64 * kUpdRowTiles));
  const dim3 wide((unsigned)((ld + 127) / 128), rtiles, kNumPrimes);
  const dim3 narrow(1, rtiles, kNumPrimes);
  const bool reg_block = n <= 1024;  // the whole block in one launch, panel in registers
  int64_t kstart = 0;
  if (!reg_block) {
    ES_CHECK(cuda_status(cudaFuncSetAttribute(k_gj_update_mma128, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              kUpd128Smem),
                         "update128 smem attribute"));
    gp.utw = 128;
    for (; kstart + 128 <= n; kstart += 128) {
      const int64_t k0 = kstart, k1 = k0 + 32, k2 = k0 + 64, k3 = k0 + 96;
      gp.UT = UT;
      panel<32>(gp, n, k0, 32, use_smem, st);
      k_gj_update_mma<32><<<narrow, 256, 0, st>>>(gp, UT, 128, k0, k1, k1 + 32, k0, k1);
      gp.UT = UT + 32;
      panel<32>(gp, n, k1, 32, use_smem, st);
      k_gj_update_mma<32><<<narrow, 256, 0, st>>>(gp, UT + 32, 128, k1, k0, k0 + 32, k1, k1 + 32);
      k_gj_update_mma<64><<<narrow, 256, 0, st>>>(gp, UT, 128, k0, k2, k2 + 64, k0, k2);
      gp.UT = UT + 64;
      panel<32>(gp, n, k2, 32, use_smem, st);
      k_gj_update_mma<32><<<narrow, 256, 0, st>>>(gp, UT + 64, 128, k2, k3, k3 + 32, k2, k3);
      gp.UT = UT + 96;
      panel<32>(gp, n, k3, 32, use_smem, st);
      k_gj_update_mma<32><<<narrow, 256, 0, st>>>(gp, UT + 96, 128, k3, k2, k2 + 32, k3, k3 + 32);
      k_gj_update_mma<64><<<narrow, 256, 0, st>>>(gp, UT + 64, 128, k2, k0, k0 + 64, k2, k2 + 64);
      gp.UT = UT;
      k_gj_update_mma128<<<wide, 256, kUpd128Smem, st>>>(gp, UT, 128, k0, 0, ld, k0, k0 + 128);
      count_launch(7);
    }
  }
  gp.UT = UT;
  gp.utw = 64;
  for (int64_t k0 = kstart; k0 < n; k0 += 64) {
    const int kb1 = (int)((n - k0) < 32 ? (n - k0) : 32);
    const int64_t k1 = k0 + 32;
    const bool two = k1 < n;
    const int kb2 = two ? (int)((n - k1) < 32 ? (n - k1) : 32) : 0;
    if (reg_block) {
      if (n <= 256)
        k_gj_block64<1, 256><<<kNumPrimes, 256, 0, st>>>(gp, k0, kb1, kb2, 0, -1);
      else if (n <= 512)
        k_gj_block64<2, 256><<<kNumPrimes, 256, 0, st>>>(gp, k0, kb1, kb2, 0, -1);
      else
        k_gj_block64<4, 256><<<kNumPrimes, 256, 0, st>>>(gp, k0, kb1, kb2, 0, -1);
      count_launch();
    } else {
      gp.UT = UT;
      panel<32>(gp, n, k0, kb1, use_smem, st);
      if (two) {
        k_gj_update_mma<32><<<dim3(1, rtiles, kNumPrimes), 256, 0, st>>>(gp, UT, 64, k0, k1, k1 + 32, k0, k1);
        gp.UT = UT + 32;
        panel<32>(gp, n, k1, kb2, use_smem, st);
        k_gj_update_mma<32><<<dim3(1, rtiles, kNumPrimes), 256, 0, st>>>(gp, UT + 32, 64, k1, k0, k0 + 32, k1,
                                                                          k1 + 32);
        count_launch(2);
      }
      gp.UT = UT;
    }
    if (two)
      k_gj_update_mma<64><<<wide, 256, 0, st>>>(gp, UT, 64, k0, 0, ld, k0, k0 + 64);
    else
      k_gj_update_mma<32><<<wide, 256, 0, st>>>(gp, UT, 64, k0, 0, ld, k0, k0 + 32);
    count_launch();
  }
  gp.UT = UT;
  return cuda_status(cudaGetLastError(), "gauss-jordan blocks");
}

// ------------------------------------------------------------------ overlap
// Two SM partitions per device (green contexts, driver API looked up at run
// time): one of at least 53 SMs for the block kernels (one CTA per prime, a
// whole SM's registers each) and the rest for the updates, each with a
// stream.  While the panel partition brings block b + 1 up to date and
// factors it, the update of block b reaches every other column on the other:
//   update stream: [wait pb] stage b's pivot rows of the other columns -> (wn)
//                  -> update every column outside blocks b and b + 1
//   panel stream:  [wait wn] block b+1, which first applies block b's update
//                  to its own 64 columns -> (pb)
// The two kernels that run at the same time touch disjoint columns of W and
// disjoint rows of U^T.  Created once per device; es_release_workspace
// destroys them.
struct Partitions {
  bool tried = false, ok = false;
  CUgreenCtx gp = nullptr, gu = nullptr;
  cudaStream_t sp = nullptr, su = nullptr;
  cudaEvent_t fork = nullptr, pb = nullptr, wn[2] = {nullptr, nullptr}, join = nullptr;
};
std::mutex g_part_mu;
Partitions g_part[kMaxDevices];

template <class F>
bool driver_entry(const char* name, F* fn) {
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &ptr, CUDA_VERSION, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !ptr) {
    cudaGetLastError();
    return false;
  }
  *fn = reinterpret_cast<F>(ptr);
  return true;
}

using GreenDestroyFn = CUresult (*)(CUgreenCtx);

void drop_partitions(Partitions& P) {
  GreenDestroyFn destroy = nullptr;
  driver_entry("cuGreenCtxDestroy", &destroy);
  for (cudaStream_t* s : {&P.sp, &P.su})
    if (*s) cudaStreamDestroy(*s);
  for (cudaEvent_t* e : {&P.fork, &P.pb, &P.wn[0], &P.wn[1], &P.join})
    if (*e) cudaEventDestroy(*e);
  if (destroy) {
    if (P.gp) destroy(P.gp);
    if (P.gu) destroy(P.gu);
  }
  cudaGetLastError();
  P = Partitions{};
}

bool make_partitions(int dev, Partitions& P) {
  CUresult (*get_dev)(CUdevice*, int) = nullptr;
  CUresult (*get_res)(CUdevice, CUdevResource*, CUdevResourceType) = nullptr;
  CUresult (*split)(CUdevResource*, unsigned*, const CUdevResource*, CUdevResource*, unsigned, unsigned) = nullptr;
  CUresult (*gen_desc)(CUdevResourceDesc*, CUdevResource*, unsigned) = nullptr;
  CUresult (*create)(CUgreenCtx*, CUdevResourceDesc, CUdevice, unsigned) = nullptr;
  CUresult (*stream_create)(CUstream*, CUgreenCtx, unsigned, int) = nullptr;
  if (!driver_entry("cuDeviceGet", &get_dev) || !driver_entry("cuDeviceGetDevResource", &get_res) ||
      !driver_entry("cuDevSmResourceSplitByCount", &split) || !driver_entry("cuDevResourceGenerateDesc", &gen_desc) ||
      !driver_entry("cuGreenCtxCreate", &create) || !driver_entry("cuGreenCtxStreamCreate", &stream_create))
    return false;
  CUdevice d;
  CUdevResource all, grp[1], rest;
  unsigned ngroups = 1;
  if (get_dev(&d, dev) != CUDA_SUCCESS || get_res(d, &all, CU_DEV_RESOURCE_TYPE_SM) != CUDA_SUCCESS ||
      split(grp, &ngroups, &all, &rest, 0, kNumPrimes) != CUDA_SUCCESS || ngroups != 1 ||
      grp[0].sm.smCount < (unsigned)kNumPrimes || rest.sm.smCount < 32)
    return false;
  CUdevResourceDesc dp, du;
  CUstream sp = nullptr, su = nullptr;
  if (gen_desc(&dp, grp, 1) != CUDA_SUCCESS || gen_desc(&du, &rest, 1) != CUDA_SUCCESS ||
      create(&P.gp, dp, d, CU_GREEN_CTX_DEFAULT_STREAM) != CUDA_SUCCESS ||
      create(&P.gu, du, d, CU_GREEN_CTX_DEFAULT_STREAM) != CUDA_SUCCESS ||
      stream_create(&sp, P.gp, CU_STREAM_NON_BLOCKING, 0) != CUDA_SUCCESS ||
      stream_create(&su, P.gu, CU_STREAM_NON_BLOCKING, 0) != CUDA_SUCCESS) {
    P.sp = (cudaStream_t)sp;
    P.su = (cudaStream_t)su;
    drop_partitions(P);
    return false;
  }
  P.sp = (cudaStream_t)sp;
  P.su = (cudaStream_t)su;
  for (cudaEvent_t* e : {&P.fork, &P.pb, &P.wn[0], &P.wn[1], &P.join})
    if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) {
      drop_partitions(P);
      return false;
    }
  return true;
}

template <int R, int T>
void block64(GJParams& gp, int64_t k0, int kb1, int kb2, int own_only, int64_t prev, cudaStream_t st) {
  k_gj_block64<R, T><<<kNumPrimes, T, 0, st>>>(gp, k0, kb1, kb2, own_only, prev);
}

es_status run_blocks64_split(GJParams& gp, int64_t n, cudaStream_t st, Partitions& P) {
  const int64_t ld = gp.ld;
  const dim3 strips((unsigned)((ld + 63) / 64), kNumPrimes);
  gp.utw = 64;
  ES_CHECK(cuda_status(
      cudaFuncSetAttribute(k_gj_update_strip, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStripSmem),
      "update strip smem attribute"));
  ES_CHECK(cuda_status(cudaEventRecord(P.fork, st), "fork"));
  ES_CHECK(cuda_status(cudaStreamWaitEvent(P.sp, P.fork, 0), "fork panel"));
  ES_CHECK(cuda_status(cudaStreamWaitEvent(P.su, P.fork, 0), "fork update"));
  // Panel side: block k (after update k-2, which brings block k's columns
  // up to date through block k-2) first applies block k-1 to its own columns
  // with block k-1's pivot rows there, then factors.  Update side: block k's
  // update of all columns but blocks k and k+1, U read from its pivot rows.
  // The updates' completions alternate between two events.
  int64_t prev = -1;  // the previous block's first column
  int blk = 0;
  for (int64_t k0 = 0; k0 < n; k0 += 64, ++blk) {
    const int kb1 = (int)((n - k0) < 32 ? (n - k0) : 32);
    const int64_t k1 = k0 + 32, n0 = k0 + 64;
    const int kb2 = k1 < n ? (int)((n - k1) < 32 ? (n - k1) : 32) : 0;
    if (blk >= 2) ES_CHECK(cuda_status(cudaStreamWaitEvent(P.sp, P.wn[blk & 1], 0), "wait update"));
    if (n <= 256)
      block64<1, 256>(gp, k0, kb1, kb2, 1, prev, P.sp);
    else if (n <= 512)
      block64<2, 256>(gp, k0, kb1, kb2, 1, prev, P.sp);
    else
      block64<4, 256>(gp, k0, kb1, kb2, 1, prev, P.sp);
    ES_CHECK(cuda_status(cudaEventRecord(P.pb, P.sp), "record block"));
    ES_CHECK(cuda_status(cudaStreamWaitEvent(P.su, P.pb, 0), "wait block"));
    const int64_t xe = n0 < n ? n0 + 64 : n0;  // blocks k and k+1 stay with the panel side
    k_gj_update_strip<<<strips, 256, kStripSmem, P.su>>>(gp, k0, kb1, kb2, xe);
    ES_CHECK(cuda_status(cudaEventRecord(P.wn[blk & 1], P.su), "record update"));
    count_launch(2);
    prev = k0;
  }
  ES_CHECK(cuda_status(cudaEventRecord(P.join, P.su), "join"));
  ES_CHECK(cuda_status(cudaStreamWaitEvent(st, P.join, 0), "join wait"));
  return cuda_status(cudaGetLastError(), "gauss-jordan blocks (split)");
}
}  // namespace

size_t inverse_scratch_bytes(int64_t n) { return inverse_layout(n).total; }

void release_inverse_partitions(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return;
  std::lock_guard<std::mutex> lock(g_part_mu);
  drop_partitions(g_part[dev]);
}

es_status run_inverse(const int64_t* A_dev, int64_t n, int8_t* B_dev, uint8_t* good_dev, char* scratch,
                      void* stream, bool split, bool* used_split) {
  cudaStream_t st = (cudaStream_t)stream;
  InvLayout L = inverse_layout(n);
  bool use_smem;
  int nbp = choose_nbp(n, &use_smem);
  GJParams gp;
  gp.n = n;
  gp.ld = padded_ld(n);
  gp.W = reinterpret_cast<int8_t*>(scratch + L.W);
  gp.UT = reinterpret_cast<int8_t*>(scratch + L.UT);
  gp.utw = nbp;
  gp.piv = reinterpret_cast<int32_t*>(scratch + L.piv);
  gp.pinv = reinterpret_cast<int32_t*>(scratch + L.pinv);
  gp.used = reinterpret_cast<uint8_t*>(scratch + L.used);
  gp.bad = reinterpret_cast<int32_t*>(scratch + L.bad);
  gp.gpanel = use_smem ? nullptr : reinterpret_cast<int8_t*>(scratch + L.gpanel);
  ES_CHECK(cuda_status(cudaMemsetAsync(gp.used, 0, (size_t)kNumPrimes * n, st), "memset used"));
  ES_CHECK(cuda_status(cudaMemsetAsync(gp.bad, 0, (size_t)kNumPrimes * 4, st), "memset bad"));
  ES_CHECK(launch_residues_matrix(A_dev, n, gp.ld, gp.W, st));
  bool done = false;
  if (used_split) *used_split = false;
  if (nbp == 32 && n <= 1024 && split) {
    int dev = 0;
    ES_CHECK(cuda_status(cudaGetDevice(&dev), "get device"));
    if (dev >= 0 && dev < kMaxDevices) {
      std::lock_guard<std::mutex> lock(g_part_mu);
      Partitions& P = g_part[dev];
      if (!P.tried) {
        P.tried = true;
        P.ok = make_partitions(dev, P);
      }
      if (P.ok) {
        ES_CHECK(run_blocks64_split(gp, n, st, P));
        done = true;
        if (used_split) *used_split = true;
      }
    }
  }
  if (done) {
  } else if (nbp == 32) {
    ES_CHECK(run_blocks64(gp, n, use_smem, st));
  } else {
    ES_CHECK(run_blocks16(gp, n, use_smem, st));
  }
  k_gj_pinv<<<dim3((unsigned)((n + 255) / 256), kNumPrimes), 256, 0, st>>>(gp);
  count_launch(2);  // pinv + permute
  ES_CHECK(cuda_status(cudaGetLastError(), "k_gj_pinv"));
  if (n <= kPermuteMaxN) {
    const size_t psm = (size_t)(2 * n + 15) / 16 * 16 + 8 * (size_t)gp.ld;
    const dim3 grid((unsigned)((n + kPermuteRows - 1) / kPermuteRows), kNumPrimes);
    auto launch = [&](auto kern) -> es_status {
      if (psm > 48 * 1024)
        ES_CHECK(cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psm),
                             "permute smem attribute"));
      kern<<<grid, 256, psm, st>>>(gp, B_dev, good_dev);
      return cuda_status(cudaGetLastError(), "k_gj_permute_rows");
    };
    if (gp.ld <= 1024) return launch(k_gj_permute_rows<2>);
    if (gp.ld <= 4096) return launch(k_gj_permute_rows<8>);
    return launch(k_gj_permute_rows<kPermuteMaxN / 512>);
  }
  size_t rsm = (size_t)gp.ld;
  if (rsm > 48 * 1024)
    ES_CHECK(cuda_status(cudaFuncSetAttribute(k_gj_permute, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rsm),
                         "permute smem attribute"));
  k_gj_permute<<<dim3((unsigned)n, kNumPrimes), 256, rsm, st>>>(gp, B_dev, good_dev);
  return cuda_status(cudaGetLastError(), "k_gj_permute");
}

}  // namespace es

// Host self-check of the f32 residue arithmetic of the Gauss-Jordan kernels:
// for every odd prime q < 256 and every integer |x| < 2^20 (the domain the
// kernels use it on), fred(x) must be the balanced residue of x and fbyte of
// it that residue's two's complement low byte.  Returns the number of
// mismatches.
extern "C" int64_t es_selftest_gj_reduction(void) {
  using namespace es;
  const QInvTable qi = make_qinv_table();
  int64_t bad = 0;
  for (int j = 0; j < kNumPrimes; ++j) {
    const int32_t q = (int32_t)kPrimes[j], h = (q - 1) / 2;
    const ModF mf{(float)q, qi.v[j]};
    for (int32_t x = -(1 << 21) - 1024; x <= (1 << 21) + 1024; ++x) {
      int32_t r = x % q;
      if (r > h) r -= q;
      if (r < -h) r += q;
      const float f = fred((float)x, mf);
      if (f != (float)r || fbyte(f) != ((uint32_t)r & 0xFFu)) ++bad;
    }
  }
  return bad;
}
