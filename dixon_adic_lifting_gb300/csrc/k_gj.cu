// Batched modular inverse B_j = A^{-1} mod q_j for all 53 primes at once.
//
// exact-solve card, §Method: "a batched modular inverse (A^{-1} mod q_j for
// every prime by Gauss-Jordan over the augmented matrix, one grid per
// elimination step spanning all primes, Barrett reduction in place of
// hardware modulo)"; §Requirements: working memory scales with the prime
// count and n.
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
#include <cuda_runtime.h>

#include <climits>

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
  int8_t* UT;      // [53][ld][NBP] pivot rows' values, transposed, zero for a >= kb
  int8_t* gpanel;  // [53][n][NBP] panel in global memory when shared memory is too small
};

__device__ __forceinline__ int32_t sbyte(uint32_t w, int u) { return (int32_t)(w << (24 - 8 * u)) >> 24; }

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
  int8_t* UTj = p.UT + (int64_t)j * ld * NBP;
  for (int64_t idx = tid; idx < (int64_t)NBP * ld; idx += blockDim.x) {
    int a = (int)(idx / ld);
    int64_t col = idx - (int64_t)a * ld;
    int8_t v = 0;
    if (a < kb && (col < k0 || col >= k0 + kb)) {
      int64_t off = (int64_t)s_piv[a] * ld + col;
      v = Wj[off];
      Wj[off] = 0;
    }
    UTj[col * NBP + a] = v;
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
  const int8_t* UTj = p.UT + (int64_t)j * ld * NBP;
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
    if (col < ld) v = *reinterpret_cast<const int4*>(UTj + col * NBP + 16 * cch);
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

// ------------------------------------------------------------------ permute
__global__ void k_gj_pinv(GJParams p) {
  const int j = blockIdx.y;
  if (p.bad[j]) return;
  int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= p.n) return;
  p.pinv[(int64_t)j * p.n + p.piv[(int64_t)j * p.n + k]] = (int32_t)k;
}

// B[j][k][t] = W[j][piv[k]][pinv[t]] (t < n), zero for n <= t < ld.
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
  r.UT = L.add((size_t)kNumPrimes * ld * nbp);
  r.piv = L.add((size_t)kNumPrimes * n * 4);
  r.pinv = L.add((size_t)kNumPrimes * n * 4);
  r.used = L.add((size_t)kNumPrimes * n);
  r.bad = L.add((size_t)kNumPrimes * 4);
  r.gpanel = sm ? 0 : L.add((size_t)kNumPrimes * n * nbp);
  r.total = L.total;
  return r;
}

template <int NBP>
es_status run_blocks(GJParams& gp, int64_t n, bool use_smem, cudaStream_t st) {
  size_t smem = use_smem ? (size_t)n * NBP + (size_t)n : 0;
  ES_CHECK(cuda_status(cudaFuncSetAttribute(k_gj_panel<NBP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)kPanelSmemLimit + 1024),
                       "panel smem attribute"));
  dim3 ugrid((unsigned)((gp.ld + 127) / 128), (unsigned)((n + 63) / 64), kNumPrimes);
  for (int64_t k0 = 0; k0 < n; k0 += NBP) {
    int kb = (int)((n - k0) < NBP ? (n - k0) : NBP);
    k_gj_panel<NBP><<<kNumPrimes, 1024, smem, st>>>(gp, k0, kb, use_smem ? 1 : 0);
    k_gj_update<NBP><<<ugrid, 256, 0, st>>>(gp, k0, kb);
    count_launch(2);
  }
  return cuda_status(cudaGetLastError(), "gauss-jordan blocks");
}
}  // namespace

size_t inverse_scratch_bytes(int64_t n) { return inverse_layout(n).total; }

es_status run_inverse(const int64_t* A_dev, int64_t n, int8_t* B_dev, uint8_t* good_dev, char* scratch,
                      void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  InvLayout L = inverse_layout(n);
  bool use_smem;
  int nbp = choose_nbp(n, &use_smem);
  GJParams gp;
  gp.n = n;
  gp.ld = padded_ld(n);
  gp.W = reinterpret_cast<int8_t*>(scratch + L.W);
  gp.UT = reinterpret_cast<int8_t*>(scratch + L.UT);
  gp.piv = reinterpret_cast<int32_t*>(scratch + L.piv);
  gp.pinv = reinterpret_cast<int32_t*>(scratch + L.pinv);
  gp.used = reinterpret_cast<uint8_t*>(scratch + L.used);
  gp.bad = reinterpret_cast<int32_t*>(scratch + L.bad);
  gp.gpanel = use_smem ? nullptr : reinterpret_cast<int8_t*>(scratch + L.gpanel);
  ES_CHECK(cuda_status(cudaMemsetAsync(gp.used, 0, (size_t)kNumPrimes * n, st), "memset used"));
  ES_CHECK(cuda_status(cudaMemsetAsync(gp.bad, 0, (size_t)kNumPrimes * 4, st), "memset bad"));
  ES_CHECK(launch_residues_matrix(A_dev, n, gp.ld, gp.W, st));
  if (nbp == 32)
    ES_CHECK(run_blocks<32>(gp, n, use_smem, st));
  else
    ES_CHECK(run_blocks<16>(gp, n, use_smem, st));
  k_gj_pinv<<<dim3((unsigned)((n + 255) / 256), kNumPrimes), 256, 0, st>>>(gp);
  count_launch(2);  // pinv + permute
  ES_CHECK(cuda_status(cudaGetLastError(), "k_gj_pinv"));
  size_t rsm = (size_t)gp.ld;
  if (rsm > 48 * 1024)
    ES_CHECK(cuda_status(cudaFuncSetAttribute(k_gj_permute, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rsm),
                         "permute smem attribute"));
  k_gj_permute<<<dim3((unsigned)n, kNumPrimes), 256, rsm, st>>>(gp, B_dev, good_dev);
  return cuda_status(cudaGetLastError(), "k_gj_permute");
}

}  // namespace es
