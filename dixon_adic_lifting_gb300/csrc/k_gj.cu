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
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
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
  uint8_t inv[256];                  // inverses mod q
  __align__(16) int wmin[32];        // per-warp pivot candidates
  __align__(16) int32_t raw[32];     // pivot row, natural column order
  __align__(16) int32_t prow[32];    // scaled pivot row, rotated: entry t = column (a + t) mod NBP
  __align__(16) int32_t pupd[32];    // same with the pivot entry + 1
  int piv[32];                       // the panel's pivot rows
  __align__(16) uint32_t u[32][8];   // a narrow update's U: column c, pivot rows 4w .. 4w + 3 in word w
};

// The kb exchange steps of the panel at k0; writes the reduced panel back to
// W and the used flags, and leaves each of the thread's rows as 8 packed
// words in Fp.  False when the prime has no pivot (it is flagged bad).
template <int NBP, int R, int T>
__device__ __forceinline__ bool panel_factor(const GJParams& p, int j, const ModQ& m, int8_t* Wj, int64_t k0, int kb,
                                             PanelSmem& S, uint32_t (&Fp)[R][NBP / 4]) {
  const int n = (int)p.n, ld = (int)p.ld;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t v[R][NBP];
  bool used[R];
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
        for (int u = 0; u < 4; ++u) v[i][c4 * 16 + q4 * 4 + u] = sbyte(ww[q4], u);
    }
    used[i] = active ? p.used[(int64_t)j * n + row] != 0 : true;
  }
  __syncthreads();
#pragma unroll 1
  for (int a = 0; a < kb; ++a) {
    int32_t f[R];
    int cand = INT_MAX;
#pragma unroll
    for (int i = R - 1; i >= 0; --i) {  // rows grow with i: the smallest i wins
      f[i] = reduce_bal(v[i][0], m);
      if (!used[i] && f[i] != 0) cand = tid + T * i;
    }
    cand = __reduce_min_sync(0xffffffffu, cand);
    if (lane == 0) S.wmin[warp] = cand;
    __syncthreads();  // (1) candidates of every warp
    int pr = INT_MAX;
#pragma unroll
    for (int w4 = 0; w4 < T / 128; ++w4) {
      const int4 c = *reinterpret_cast<const int4*>(S.wmin + 4 * w4);
      pr = min(pr, min(min(c.x, c.y), min(c.z, c.w)));
    }
    if (pr == INT_MAX) {  // no pivot: q_j | det A
      if (tid == 0) p.bad[j] = 1;
      return false;
    }
#pragma unroll
    for (int i = 0; i < R; ++i)
      if (tid + T * i == pr) {
#pragma unroll
        for (int t = 0; t < NBP; ++t) S.raw[(a + t) & (NBP - 1)] = t == 0 ? f[i] : v[i][t];
        used[i] = true;
        S.piv[a] = pr;
        p.piv[(int64_t)j * n + k0 + a] = pr;
      }
    __syncthreads();  // (2) raw pivot row
    if (warp == 0) {
      const int32_t pf = S.raw[a];
      const uint32_t inv = S.inv[pf < 0 ? pf + (int32_t)m.q : pf];
      for (int t = lane; t < NBP; t += 32) {
        const int c = (a + t) & (NBP - 1);
        const int32_t pt =
            (t == 0) ? bal_from_unsigned(inv, m) : reduce_bal(reduce_bal(S.raw[c], m) * (int32_t)inv, m);
        S.prow[t] = pt;
        S.pupd[t] = (t == 0) ? pt + 1 : pt;
      }
    }
    __syncthreads();  // (3) scaled pivot row
    // v[t] <- (v[t + 1] - f u_{t + 1}), v[NBP - 1] <- (v[0] - f u_0); the pivot row takes p instead.
    // u_0 = p_a + 1 turns the pivot column into -f inv (mod q), as v[0] = f (mod q).
#pragma unroll
    for (int i = 0; i < R; ++i) {
      if (tid + T * i == pr) {
#pragma unroll
        for (int t4 = 0; t4 < NBP / 4; ++t4) {
          const int4 pp = *reinterpret_cast<const int4*>(S.prow + 4 * t4);
          const int32_t ps[4] = {pp.x, pp.y, pp.z, pp.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) v[i][(4 * t4 + u + NBP - 1) & (NBP - 1)] = ps[u];
        }
      } else {
        const int32_t fi = f[i], first = v[i][0] - fi * S.pupd[0];
#pragma unroll
        for (int t4 = 0; t4 < NBP / 4; ++t4) {
          const int4 uu = *reinterpret_cast<const int4*>(S.pupd + 4 * t4);
          const int32_t us[4] = {uu.x, uu.y, uu.z, uu.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int t = 4 * t4 + u;
            if (t > 0) v[i][t - 1] = v[i][t] - fi * us[u];
          }
        }
        v[i][NBP - 1] = first;
      }
    }
  }
  // rotate back by kb (entry t holds column (kb + t) mod NBP), log shifter
#pragma unroll
  for (int i = 0; i < R; ++i) {
#pragma unroll
    for (int sh = 1; sh < NBP; sh <<= 1) {
      if (kb & sh) {
        int32_t tmp[NBP];
#pragma unroll
        for (int t = 0; t < NBP; ++t) tmp[(t + sh) & (NBP - 1)] = v[i][t];
#pragma unroll
        for (int t = 0; t < NBP; ++t) v[i][t] = tmp[t];
      }
    }
  }
  // reduce and write the panel back (padding columns stay zero: their pivot-row entries are zero)
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int row = tid + T * i;
#pragma unroll
    for (int q = 0; q < NBP / 4; ++q) {
      uint32_t x = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) x |= ((uint32_t)(uint8_t)(int8_t)reduce_bal(v[i][4 * q + u], m)) << (8 * u);
      Fp[i][q] = x;
    }
    if (row >= n) continue;
#pragma unroll
    for (int c4 = 0; c4 < NBP / 16; ++c4)
      if (k0 + 16 * c4 < ld)
        *reinterpret_cast<int4*>(Wj + (int64_t)row * ld + k0 + 16 * c4) =
            make_int4(Fp[i][4 * c4], Fp[i][4 * c4 + 1], Fp[i][4 * c4 + 2], Fp[i][4 * c4 + 3]);
    p.used[(int64_t)j * n + row] = used[i] ? 1 : 0;
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

// W[r][c0 + c] += sum_a F[r][a] U[a][c] (mod q) for the 32 columns c0 .. c0+31
// and every row r of this thread (F = its packed panel rows, U = the staged
// pivot rows of those columns, UT[col][0..32) at row width utw): 8 dp4a per
// entry, exact (32 * 125^2 + 125 < 2^31).
template <int R, int T>
__device__ __forceinline__ void narrow_update(const GJParams& p, int8_t* Wj, const ModQ& m,
                                              const uint32_t (&Fp)[R][8], const int8_t* UTj, int utw, int64_t c0,
                                              PanelSmem& S) {
  const int n = (int)p.n;
  const int64_t ld = p.ld;
  const int tid = threadIdx.x;
  if (tid < 64) {
    const int c = tid >> 1, h = tid & 1;
    const int64_t col = c0 + c;
    const int4 x = col < ld ? *reinterpret_cast<const int4*>(UTj + col * utw + 16 * h) : make_int4(0, 0, 0, 0);
    *reinterpret_cast<int4*>(&S.u[c][4 * h]) = x;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int row = tid + T * i;
    if (row >= n) continue;
    int8_t* wr = Wj + (int64_t)row * ld + c0;
    const bool two = c0 + 16 < ld;
    const int4 o0 = *reinterpret_cast<const int4*>(wr), o1 = two ? *reinterpret_cast<const int4*>(wr + 16)
                                                                 : make_int4(0, 0, 0, 0);
    uint32_t w[8] = {(uint32_t)o0.x, (uint32_t)o0.y, (uint32_t)o0.z, (uint32_t)o0.w,
                     (uint32_t)o1.x, (uint32_t)o1.y, (uint32_t)o1.z, (uint32_t)o1.w};
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      uint32_t x = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = 4 * q + u;
        const int4 ua = *reinterpret_cast<const int4*>(&S.u[c][0]), ub = *reinterpret_cast<const int4*>(&S.u[c][4]);
        int32_t acc = 0;
        acc = __dp4a((int)Fp[i][0], ua.x, acc);
        acc = __dp4a((int)Fp[i][1], ua.y, acc);
        acc = __dp4a((int)Fp[i][2], ua.z, acc);
        acc = __dp4a((int)Fp[i][3], ua.w, acc);
        acc = __dp4a((int)Fp[i][4], ub.x, acc);
        acc = __dp4a((int)Fp[i][5], ub.y, acc);
        acc = __dp4a((int)Fp[i][6], ub.z, acc);
        acc = __dp4a((int)Fp[i][7], ub.w, acc);
        int32_t val = sbyte(w[q], u);
        if (c0 + c < n) val = reduce_bal(val + acc, m);
        x |= ((uint32_t)(uint8_t)(int8_t)val) << (8 * u);
      }
      w[q] = x;
    }
    *reinterpret_cast<int4*>(wr) = make_int4(w[0], w[1], w[2], w[3]);
    if (two) *reinterpret_cast<int4*>(wr + 16) = make_int4(w[4], w[5], w[6], w[7]);
  }
}

// One 64-column block (n <= 1024): panel k0 (kb1 columns), its U^T into
// UT[:, 0..32) with the pivot rows zeroed, the update of the block's other
// 32 columns, panel k0 + 32 (kb2 columns, 0 = none), its U^T into
// UT[:, 32..64), the update of the first 32 columns.  One CTA per prime.
// W[r][k0 + c] += sum_a F[r][a] U[a][c] (mod q) for the 64 columns of the
// block at k0 and every row r of this thread: the previous block's update of
// these columns, F = W[:, prev .. prev + 64) (its final columns), U = its
// staged pivot rows, UT[k0 + c][0 .. 64).  16 dp4a per entry, exact
// (64 * 125^2 + 125 < 2^31); U is broadcast from shared memory.
template <int R, int T>
__device__ __forceinline__ void catch_up(const GJParams& p, int8_t* Wj, const int8_t* UTj, const ModQ& m, int64_t prev,
                                         int64_t k0, uint32_t (*Us)[16]) {
  const int n = (int)p.n;
  const int64_t ld = p.ld;
  const int tid = threadIdx.x;
  for (int idx = tid; idx < 64 * 4; idx += T) {
    const int c = idx >> 2, h = idx & 3;
    const int64_t col = k0 + c;
    const int4 x = col < ld ? *reinterpret_cast<const int4*>(UTj + col * 64 + 16 * h) : make_int4(0, 0, 0, 0);
    *reinterpret_cast<int4*>(&Us[c][4 * h]) = x;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int row = tid + T * i;
    if (row >= n) continue;
    uint32_t f[16], w[16];
    const int4* fr = reinterpret_cast<const int4*>(Wj + (int64_t)row * ld + prev);
    int4* wr = reinterpret_cast<int4*>(Wj + (int64_t)row * ld + k0);
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int4 a = fr[h];
      const int4 b = (k0 + 16 * h < ld) ? wr[h] : make_int4(0, 0, 0, 0);
      f[4 * h] = a.x, f[4 * h + 1] = a.y, f[4 * h + 2] = a.z, f[4 * h + 3] = a.w;
      w[4 * h] = b.x, w[4 * h + 1] = b.y, w[4 * h + 2] = b.z, w[4 * h + 3] = b.w;
    }
#pragma unroll 4
    for (int q = 0; q < 16; ++q) {
      uint32_t x = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = 4 * q + u;
        int32_t acc = 0;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const uint4 uu = *reinterpret_cast<const uint4*>(&Us[c][4 * h]);
          acc = __dp4a((int)f[4 * h], (int)uu.x, acc);
          acc = __dp4a((int)f[4 * h + 1], (int)uu.y, acc);
          acc = __dp4a((int)f[4 * h + 2], (int)uu.z, acc);
          acc = __dp4a((int)f[4 * h + 3], (int)uu.w, acc);
        }
        int32_t val = sbyte(w[q], u);
        if (k0 + c < n) val = reduce_bal(val + acc, m);
        x |= ((uint32_t)(uint8_t)(int8_t)val) << (8 * u);
      }
      w[q] = x;
    }
#pragma unroll
    for (int h = 0; h < 4; ++h)
      if (k0 + 16 * h < ld) wr[h] = make_int4(w[4 * h], w[4 * h + 1], w[4 * h + 2], w[4 * h + 3]);
  }
  __syncthreads();
}

// own_only: stage only the block's own columns; the other columns' pivot
// rows are staged later by k_gj_stage64 (the schedule that overlaps this
// kernel with the previous block's update of those columns).  prev >= 0:
// first bring the block's columns up to date with the block at prev.
template <int R, int T>
__global__ void __launch_bounds__(T, 1) k_gj_block64(GJParams p, int64_t k0, int kb1, int kb2, int own_only,
                                                     int64_t prev) {
  const int j = blockIdx.x;
  if (p.bad[j]) return;
  const ModQ m = c_modq.v[j];
  int8_t* Wj = p.W + (int64_t)j * p.n * p.ld;
  int8_t* UTj = p.UT + (int64_t)j * p.ld * 64;
  __shared__ PanelSmem S;
  __shared__ __align__(16) uint32_t Us[64][16];
  for (int x = threadIdx.x; x < (int)m.q; x += T) S.inv[x] = x ? (uint8_t)inv_mod((uint32_t)x, m) : 0;
  if (prev >= 0) catch_up<R, T>(p, Wj, UTj, m, prev, k0, Us);
  uint32_t Fp[R][8];
  const int64_t cb = own_only ? k0 : 0, ce = own_only ? (k0 + 64 < p.ld ? k0 + 64 : p.ld) : p.ld;
  if (!panel_factor<32, R, T>(p, j, m, Wj, k0, kb1, S, Fp)) return;
  __syncthreads();
  panel_stage<32, T>(cb, ce, Wj, p.ld, k0, kb1, S, UTj, 64);
  if (kb2 == 0) return;
  const int64_t k1 = k0 + 32;
  __syncthreads();
  narrow_update<R, T>(p, Wj, m, Fp, UTj, 64, k1, S);
  __syncthreads();
  if (!panel_factor<32, R, T>(p, j, m, Wj, k1, kb2, S, Fp)) return;
  __syncthreads();
  panel_stage<32, T>(cb, ce, Wj, p.ld, k1, kb2, S, UTj + 32, 64);
  __syncthreads();
  narrow_update<R, T>(p, Wj, m, Fp, UTj + 32, 64, k0, S);
}

// The block's U^T for every column outside it: the pivot rows
// piv[k0 .. k0 + 64) (the first kb1 of the first panel, the second panel's at
// 32 .. 32 + kb2) go to UT[col][0 .. 64) (zero where there is no pivot) and
// are zeroed in W.  Thread per 4 consecutive columns and prime: one 4-byte
// load per pivot row (a warp reads whole 128-byte lines), all loads before
// any zeroing store, bytes transposed in registers.
__global__ void __launch_bounds__(128) k_gj_stage64(GJParams p, int64_t k0, int kb1, int kb2) {
  const int j = blockIdx.y;
  if (p.bad[j]) return;
  const int64_t n = p.n, ld = p.ld;
  const int64_t col = 4 * ((int64_t)blockIdx.x * blockDim.x + threadIdx.x);
  if (col >= ld || (col >= k0 && col < k0 + 64)) return;  // ld and k0 are multiples of 4
  int8_t* Wj = p.W + (int64_t)j * n * ld;
  const int32_t* pv = p.piv + (int64_t)j * n + k0;
  uint32_t x[64];
#pragma unroll
  for (int a = 0; a < 64; ++a) {
    const bool have = a < 32 ? a < kb1 : a - 32 < kb2;
    x[a] = have ? *reinterpret_cast<const uint32_t*>(Wj + (int64_t)pv[a] * ld + col) : 0u;
  }
#pragma unroll
  for (int a = 0; a < 64; ++a) {
    const bool have = a < 32 ? a < kb1 : a - 32 < kb2;
    if (have) *reinterpret_cast<uint32_t*>(Wj + (int64_t)pv[a] * ld + col) = 0u;
  }
  // column c of the four: bytes c of x[0 .. 64), packed four at a time
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    int4* dst = reinterpret_cast<int4*>(p.UT + ((int64_t)j * ld + col + c) * 64);
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int a0 = 16 * c4 + 4 * q;
        // gather byte c of x[a0 .. a0 + 4) into one word
        const uint32_t lo = __byte_perm(x[a0], x[a0 + 1], c | (c + 4) << 4);
        const uint32_t hi = __byte_perm(x[a0 + 2], x[a0 + 3], c | (c + 4) << 4);
        w[q] = __byte_perm(lo, hi, 0x5410);
      }
      dst[c4] = make_int4(w[0], w[1], w[2], w[3]);
    }
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
// F = W[:, k0 .. k0 + KW) and U^T (row width utw bytes, U^T[col][a] = pivot
// row a's entry of column col) are staged as int8 in shared memory with
// 16-byte loads (rows of 64 bytes, chunk c of row r at chunk c ^ ((r >> 1) & 3):
// conflict-free for the stores and for ldmatrix), read with ldmatrix as s8
// fragments of m16n8k32 shape and widened to f16 in registers.  A 32-bit s8
// fragment word holds four consecutive k; its low pair goes to the f16
// fragment register for k-slots 2t, 2t + 1 and its high pair to 2t + 8, 2t + 9,
// on both operands, so the products pair up the same k.
//
// The residue of v = old + (F U)[i][t] is taken in f32 as v - q rint(v / q~),
// q~ = fl(1/q): the quotient estimate errs by at most |v| / q * 2^-24 <
// 1/(16 q), while v / q is at least 1/(2 q) away from a half-integer (q odd),
// so the rounding is always the exact one and the result is the balanced
// residue.  CTA tile 64 rows x 128 columns, 8 warps of 32 x 32.  Columns
// updated: 32-column segments col0 with cbase <= col0 < cend outside
// [xb, xe) (which holds at least the panel).
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

// Four signed bytes -> f16x2 of bytes 0, 1 (lo) and of bytes 2, 3 (hi): with
// u = x + 128 (the top bit flipped), 0x64uu is the f16 1024 + u, and
// 1024 + u - 1152 = x exactly.
__device__ __forceinline__ void s8x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  lo = __byte_perm(u, 0x64646464u, 0x4140);
  hi = __byte_perm(u, 0x64646464u, 0x4342);
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(0x64806480u));
}

struct QInvTable {
  float v[kNumPrimes];
};
constexpr QInvTable make_qinv_table() {
  QInvTable t{};
  for (int i = 0; i < kNumPrimes; ++i) t.v[i] = 1.0f / (float)kPrimes[i];
  return t;
}
__constant__ QInvTable c_qinv = make_qinv_table();

__device__ __forceinline__ int rot3(int r) { return ((r << 1) | ((r >> 2) & 1)) & 7; }
__device__ __forceinline__ int swz64(int r, int c) { return r * 64 + 16 * (c ^ ((r >> 1) & 3)); }

template <int KW>
__global__ void __launch_bounds__(256) k_gj_update_mma(GJParams p, const int8_t* __restrict__ UT, int utw,
                                                       int64_t k0, int64_t cbase, int64_t cend, int64_t xb,
                                                       int64_t xe) {
  constexpr int KC = KW / 16;  // 16-byte chunks per operand row
  const int j = blockIdx.z;
  if (p.bad[j]) return;
  const int64_t n = p.n, ld = p.ld;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t rowc = (int64_t)blockIdx.y * 64, colc = cbase + (int64_t)blockIdx.x * 128;
  const int64_t row0 = rowc + (warp >> 2) * 32;
  const int64_t col0 = colc + (warp & 3) * 32;
  int8_t* Wj = p.W + (int64_t)j * n * ld;
  const int8_t* UTj = UT + (int64_t)j * ld * utw;
  __shared__ __align__(16) float Cs[8][32][32];
  __shared__ __align__(16) uint8_t As[64 * 64];
  __shared__ __align__(16) uint8_t Bs[128 * 64];
  // this thread's output row segment (row0 + lane, 32 columns), fetched early;
  // segments are 32-column aligned like the panel: one either lies in it or misses it
  const int64_t orow = row0 + lane;
  const bool rowok = orow < n && col0 < ld && col0 < cend && (col0 < xb || col0 >= xe);
  int4 old0 = make_int4(0, 0, 0, 0), old1 = old0;
  if (rowok) {
    old0 = *reinterpret_cast<const int4*>(Wj + orow * ld + col0);
    if (col0 + 16 < ld) old1 = *reinterpret_cast<const int4*>(Wj + orow * ld + col0 + 16);
  }
  for (int i = tid; i < 64 * KC; i += 256) {
    const int r = i / KC, c = i % KC;
    const int64_t row = rowc + r, col = k0 + 16 * c;
    int4 v = make_int4(0, 0, 0, 0);
    if (row < n && col < ld) v = *reinterpret_cast<const int4*>(Wj + row * ld + col);
    *reinterpret_cast<int4*>(As + swz64(r, c)) = v;
  }
  for (int i = tid; i < 128 * KC; i += 256) {
    const int r = i / KC, c = i % KC;
    const int64_t col = colc + r;
    int4 v = make_int4(0, 0, 0, 0);
    if (col < ld) v = *reinterpret_cast<const int4*>(UTj + col * utw + 16 * c);
    *reinterpret_cast<int4*>(Bs + swz64(r, c)) = v;
  }
  __syncthreads();
  const int mi8 = lane >> 3, rr = lane & 7;  // ldmatrix: matrix and row this lane addresses
  float acc[2][4][4];
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ni = 0; ni < 4; ++ni)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[mi][ni][r] = 0.f;
#pragma unroll
  for (int kk = 0; kk < KW / 32; ++kk) {
    // s8 fragments: A reg r = rows g + 8 (r & 1), k 4 t + 16 (r >> 1) + 0..3;
    // B reg r of column tile 2 np + (i >> 1) (i = 2 (ni & 1) + r) = column g, k 4 t + 16 r + 0..3
    uint32_t a8[2][4], b8[2][4];
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
      ldsm_x4(a8[mi], As + swz64((warp >> 2) * 32 + 16 * mi + rr + 8 * (mi8 & 1), 2 * kk + (mi8 >> 1)));
#pragma unroll
    for (int np = 0; np < 2; ++np)
      ldsm_x4(b8[np], Bs + swz64((warp & 3) * 32 + 8 * (2 * np + (mi8 >> 1)) + rr, 2 * kk + (mi8 & 1)));
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t af[2][4], bf[4][2];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        s8x4_to_f16(a8[mi][2 * h], af[mi][0], af[mi][2]);
        s8x4_to_f16(a8[mi][2 * h + 1], af[mi][1], af[mi][3]);
      }
#pragma unroll
      for (int ni = 0; ni < 4; ++ni) s8x4_to_f16(b8[ni >> 1][2 * (ni & 1) + h], bf[ni][0], bf[ni][1]);
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) mma_f16_16x8x16(acc[mi][ni], af[mi], bf[ni]);
    }
  }
  // C reg r = row g + 8 (r >> 1), column 2 t + (r & 1); within a row the
  // 16-byte chunk c sits at chunk c ^ rot(row) (rot = 3-bit left rotation of
  // row & 7): conflict-free for the 8-byte stores (per half-warp) and the
  // 16-byte row reads (per quarter-warp)
  {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int ni = 0; ni < 4; ++ni) {
        const int cw = 8 * ni + 2 * t, sw = (4 * ((cw >> 2) ^ rot3(g))) | (cw & 3);  // rows g, g + 8: same rot
        *reinterpret_cast<float2*>(&Cs[warp][16 * mi + g][sw]) = make_float2(acc[mi][ni][0], acc[mi][ni][1]);
        *reinterpret_cast<float2*>(&Cs[warp][16 * mi + g + 8][sw]) = make_float2(acc[mi][ni][2], acc[mi][ni][3]);
      }
  }
  __syncwarp();
  if (!rowok) return;
  const float qf = (float)c_modq.v[j].q, qinv = c_qinv.v[j];
  const float kM = 12582912.0f;  // 1.5 * 2^23: x + kM has ulp 1 for |x| < 2^22
  const uint32_t w[8] = {(uint32_t)old0.x, (uint32_t)old0.y, (uint32_t)old0.z, (uint32_t)old0.w,
                         (uint32_t)old1.x, (uint32_t)old1.y, (uint32_t)old1.z, (uint32_t)old1.w};
  uint32_t o[8];
  const int rl = rot3(lane);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float4 c4 = *reinterpret_cast<const float4*>(&Cs[warp][lane][4 * (q ^ rl)]);
    const float cv[4] = {c4.x, c4.y, c4.z, c4.w};
    const uint32_t wu = w[q] ^ 0x80808080u;  // bytes x + 128
    uint32_t rb[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      // 2^23 + x + 128 from the bits 0x4B0000uu
      const float fb = __int_as_float((int)__byte_perm(wu, 0x4B000000u, 0x7540 + u));
      const float v = __fadd_rn(__fadd_rn(cv[u], fb), -8388736.0f);
      const float k = __fadd_rn(__fmaf_rn(v, qinv, kM), -kM);
      rb[u] = (uint32_t)__float_as_int(__fadd_rn(__fmaf_rn(-k, qf, v), kM));  // low byte = residue
    }
    o[q] = __byte_perm(__byte_perm(rb[0], rb[1], 0x0040), __byte_perm(rb[2], rb[3], 0x0040), 0x5410);
  }
  if (col0 + 32 > n) {  // columns n .. ld - 1 keep their zero padding
#pragma unroll
    for (int q = 0; q < 8; ++q)
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (col0 + 4 * q + u >= n) o[q] = (o[q] & ~(0xFFu << (8 * u))) | (w[q] & (0xFFu << (8 * u)));
  }
  *reinterpret_cast<int4*>(Wj + orow * ld + col0) = make_int4(o[0], o[1], o[2], o[3]);
  if (col0 + 16 < ld) *reinterpret_cast<int4*>(Wj + orow * ld + col0 + 16) = make_int4(o[4], o[5], o[6], o[7]);
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
  r.UT = L.add((size_t)kNumPrimes * ld * (nbp == 32 ? 64 : nbp));  // NB = 32: two panels' U^T side by side
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
  k_gj_panel<NBP><<<kNumPrimes, 1024, use_smem ? (size_t)n * NBP + (size_t)n : 0, st>>>(gp, k0, kb,
                                                                                     use_smem ? 1 : 0);
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
es_status run_blocks64(GJParams& gp, int64_t n, bool use_smem, cudaStream_t st) {
  ES_CHECK(cuda_status(cudaFuncSetAttribute(k_gj_panel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)kPanelSmemLimit + 1024),
                       "panel smem attribute"));
  int8_t* const UT = gp.UT;
  const int64_t ld = gp.ld;
  const unsigned rtiles = (unsigned)((n + 63) / 64);
  const dim3 wide((unsigned)((ld + 127) / 128), rtiles, kNumPrimes);
  const bool reg_block = n <= 1024;  // the whole block in one launch, panel in registers
  gp.utw = 64;
  for (int64_t k0 = 0; k0 < n; k0 += 64) {
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
        k_gj_block64<2, 512><<<kNumPrimes, 512, 0, st>>>(gp, k0, kb1, kb2, 0, -1);
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
  cudaEvent_t fork = nullptr, pb = nullptr, wn = nullptr, join = nullptr;
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
  for (cudaEvent_t* e : {&P.fork, &P.pb, &P.wn, &P.join})
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
  for (cudaEvent_t* e : {&P.fork, &P.pb, &P.wn, &P.join})
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
  int8_t* const UT = gp.UT;
  const int64_t ld = gp.ld;
  const unsigned rtiles = (unsigned)((n + 63) / 64);
  const dim3 sgrid((unsigned)((ld / 4 + 127) / 128), kNumPrimes);
  const dim3 wide((unsigned)((ld + 127) / 128), rtiles, kNumPrimes);
  gp.utw = 64;
  ES_CHECK(cuda_status(cudaEventRecord(P.fork, st), "fork"));
  ES_CHECK(cuda_status(cudaStreamWaitEvent(P.sp, P.fork, 0), "fork panel"));
  ES_CHECK(cuda_status(cudaStreamWaitEvent(P.su, P.fork, 0), "fork update"));
  int64_t prev = -1;  // the previous block's first column
  for (int64_t k0 = 0; k0 < n; k0 += 64) {
    const int kb1 = (int)((n - k0) < 32 ? (n - k0) : 32);
    const int64_t k1 = k0 + 32, n0 = k0 + 64;
    const int kb2 = k1 < n ? (int)((n - k1) < 32 ? (n - k1) : 32) : 0;
    if (prev >= 0) ES_CHECK(cuda_status(cudaStreamWaitEvent(P.sp, P.wn, 0), "wait stage"));
    if (n <= 256)
      block64<1, 256>(gp, k0, kb1, kb2, 1, prev, P.sp);
    else if (n <= 512)
      block64<2, 256>(gp, k0, kb1, kb2, 1, prev, P.sp);
    else
      block64<2, 512>(gp, k0, kb1, kb2, 1, prev, P.sp);
    ES_CHECK(cuda_status(cudaEventRecord(P.pb, P.sp), "record block"));
    // stage this block's pivot rows of every other column (after the
    // previous block's update reached them), then update all but the next block
    ES_CHECK(cuda_status(cudaStreamWaitEvent(P.su, P.pb, 0), "wait block"));
    k_gj_stage64<<<sgrid, 128, 0, P.su>>>(gp, k0, kb1, kb2);
    ES_CHECK(cuda_status(cudaEventRecord(P.wn, P.su), "record stage"));
    const int64_t xe = n0 < n ? n0 + 64 : n0;  // keep off the next block (done on the panel side)
    if (kb2)
      k_gj_update_mma<64><<<wide, 256, 0, P.su>>>(gp, UT, 64, k0, 0, ld, k0, xe);
    else
      k_gj_update_mma<32><<<wide, 256, 0, P.su>>>(gp, UT, 64, k0, 0, ld, k0, xe);
    count_launch(3);
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
                      void* stream, bool split) {
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
  size_t rsm = (size_t)gp.ld;
  if (rsm > 48 * 1024)
    ES_CHECK(cuda_status(cudaFuncSetAttribute(k_gj_permute, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rsm),
                         "permute smem attribute"));
  k_gj_permute<<<dim3((unsigned)n, kNumPrimes), 256, rsm, st>>>(gp, B_dev, good_dev);
  return cuda_status(cudaGetLastError(), "k_gj_permute");
}

}  // namespace es
