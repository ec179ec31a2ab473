// Residue slicing and the statistics behind the range check and the
// Hadamard stop rule.
//
// exact-solve card, §Method: the per-prime products run on balanced
// residues of A and of the residual; the range is n * max|A_ij| < 2^63 and
// lifting stops once P^m exceeds twice the Hadamard bound on numerator and
// denominator.
#include <cuda_runtime.h>

#include <cmath>
#include <vector>

#include "es_common.cuh"
#include "es_internal.h"

namespace es {

// out[j*ostride + i] = bal(src[i] mod q_j) for all 53 primes.
__global__ void k_residues_vec(const int64_t* __restrict__ src, int64_t count, int8_t* __restrict__ out,
                               int64_t ostride) {
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= count) return;
  int64_t a = src[i];
#pragma unroll 4
  for (int j = 0; j < kNumPrimes; ++j) out[j * ostride + i] = (int8_t)reduce_i64_bal(a, c_modq.v[j]);
}

// A [n, n] int64 -> W [53][n][ld] int8 balanced; four columns per thread,
// padding columns (n <= k < ld) written as zero.
__global__ void k_residues_matrix(const int64_t* __restrict__ A, int64_t n, int64_t ld, int8_t* __restrict__ W) {
  int64_t words_per_row = ld / 4;
  int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n * words_per_row) return;
  int64_t row = t / words_per_row;
  int64_t k0 = (t - row * words_per_row) * 4;
  int64_t a[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) a[u] = (k0 + u < n) ? A[row * n + k0 + u] : 0;
  uint32_t* dst = reinterpret_cast<uint32_t*>(W) + row * words_per_row + (k0 / 4);
  int64_t plane = n * words_per_row;  // 32-bit words per prime
#pragma unroll 2
  for (int j = 0; j < kNumPrimes; ++j) {
    const ModQ& m = c_modq.v[j];
    uint32_t w = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) w |= ((uint32_t)(uint8_t)(int8_t)reduce_i64_bal(a[u], m)) << (8 * u);
    dst[j * plane] = w;
  }
}

es_status launch_residues(const int64_t* src, int64_t count, int8_t* out, int64_t ostride, void* stream) {
  if (count <= 0) return ES_OK;
  int threads = 256;
  int64_t blocks = (count + threads - 1) / threads;
  k_residues_vec<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(src, count, out, ostride);
  count_launch();
  return cuda_status(cudaGetLastError(), "k_residues_vec");
}

es_status launch_residues_matrix(const int64_t* A, int64_t n, int64_t ld, int8_t* W, void* stream) {
  int64_t total = n * (ld / 4);
  int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  k_residues_matrix<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(A, n, ld, W);
  count_launch();
  return cuda_status(cudaGetLastError(), "k_residues_matrix");
}

// ---------------------------------------------------------------- statistics
struct RowStat {
  double sumsq;     // ||a_i||^2 (rounded; relative error <= n 2^-53)
  double bmax2;     // max_k b_ik^2
  uint64_t maxabs;  // max_k |A_ik|
  uint64_t bmaxabs; // max_k |b_ik|
};

__device__ __forceinline__ uint64_t uabs64(int64_t v) {
  return v < 0 ? (uint64_t)(-(v + 1)) + 1u : (uint64_t)v;
}

// One warp per row.
__global__ void k_row_stats(const int64_t* __restrict__ A, const int64_t* __restrict__ b, int64_t n, int64_t c,
                            RowStat* __restrict__ out) {
  int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  int lane = threadIdx.x % 32;
  if (row >= n) return;
  double s = 0.0, bm = 0.0;
  uint64_t mx = 0, bmx = 0;
  for (int64_t k = lane; k < n; k += 32) {
    int64_t v = A[row * n + k];
    double d = (double)v;
    s = fma(d, d, s);
    uint64_t u = uabs64(v);
    mx = u > mx ? u : mx;
  }
  for (int64_t k = lane; k < c; k += 32) {
    int64_t v = b[row * c + k];
    double d = (double)v;
    bm = fmax(bm, d * d);
    uint64_t u = uabs64(v);
    bmx = u > bmx ? u : bmx;
  }
  for (int o = 16; o; o >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, o);
    bm = fmax(bm, __shfl_xor_sync(0xffffffffu, bm, o));
    uint64_t om = __shfl_xor_sync(0xffffffffu, mx, o);
    mx = om > mx ? om : mx;
    uint64_t ob = __shfl_xor_sync(0xffffffffu, bmx, o);
    bmx = ob > bmx ? ob : bmx;
  }
  if (lane == 0) out[row] = RowStat{s, bm, mx, bmx};
}

size_t stats_scratch_bytes(int64_t n) { return (size_t)n * sizeof(RowStat); }

bool in_range(int64_t n, uint64_t max_abs_a) {
  if (n < 1 || n > (int64_t(1) << 17)) return false;
  // n * max|A| < 2^63  <=>  max|A| <= (2^63 - 1) / n
  return max_abs_a <= (uint64_t)INT64_MAX / (uint64_t)n;
}

es_status compute_stats(const int64_t* A_dev, const int64_t* b_dev, int64_t n, int64_t c, char* scratch,
                        void* stream, Stats* out) {
  RowStat* rs = reinterpret_cast<RowStat*>(scratch);
  int warps = 8;
  int64_t blocks = (n + warps - 1) / warps;
  k_row_stats<<<(unsigned)blocks, warps * 32, 0, (cudaStream_t)stream>>>(A_dev, b_dev, n, c, rs);
  count_launch();
  ES_CHECK(cuda_status(cudaGetLastError(), "k_row_stats"));
  std::vector<RowStat> h((size_t)n);
  ES_CHECK(cuda_status(cudaMemcpyAsync(h.data(), rs, (size_t)n * sizeof(RowStat), cudaMemcpyDeviceToHost,
                                       (cudaStream_t)stream),
                       "stats D2H"));
  ES_CHECK(cuda_status(cudaStreamSynchronize((cudaStream_t)stream), "stats sync"));
  Stats s{0, 0, 0, 0.0, 0.0};
  for (int64_t i = 0; i < n; ++i) {
    const RowStat& r = h[(size_t)i];
    s.max_abs_a = r.maxabs > s.max_abs_a ? r.maxabs : s.max_abs_a;
    s.max_abs_b = r.bmaxabs > s.max_abs_b ? r.bmaxabs : s.max_abs_b;
    if (r.sumsq == 0.0) {
      s.zero_row = 1;
      continue;
    }
    s.log2_d += 0.5 * std::log2(r.sumsq);
    s.log2_n += 0.5 * std::log2(r.sumsq + r.bmax2);
  }
  *out = s;
  return ES_OK;
}

// Bit bounds with an upward margin covering the rounding of the double sums
// (relative error <= n 2^-53 per row sum, one rounding per log and per
// addition), then the least m with m log2 P' > num_bits + den_bits + 1.
void plan_from_stats(const Stats& s, const uint8_t* good, int64_t* num_bits, int64_t* den_bits, int32_t* m) {
  double n_rows_margin = 1e-9 * (std::fabs(s.log2_n) + std::fabs(s.log2_d)) + 1e-6;
  int64_t nb = (int64_t)std::ceil(s.log2_n + n_rows_margin);
  int64_t db = (int64_t)std::ceil(s.log2_d + n_rows_margin);
  if (nb < 0) nb = 0;
  if (db < 0) db = 0;
  double log2P = 0.0;
  for (int j = 0; j < kNumPrimes; ++j)
    if (good[j]) log2P += std::log2((double)kPrimes[j]);
  double need = (double)(nb + db + 1);
  int32_t mm = 1;
  if (log2P > 0) {
    mm = (int32_t)std::floor(need / log2P) + 1;
    if ((double)mm * log2P - need < 1e-6 * mm) ++mm;  // stay strictly above with margin
  }
  *num_bits = nb;
  *den_bits = db;
  *m = mm;
}

}  // namespace es

extern "C" es_status es_residues_device(const int64_t* A_dev, int64_t count, int8_t* out_dev, void* stream) {
  if (!A_dev || !out_dev || count < 0) return ES_ERR_ARG;
  void* s = es::resolve_stream(stream);
  ES_CHECK(es::launch_residues(A_dev, count, out_dev, count, s));
  return es::cuda_status(cudaStreamSynchronize((cudaStream_t)s), "es_residues_device");
}
