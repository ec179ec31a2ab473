// Dixon lift for one right-hand side (c == 1) as one persistent cooperative
// launch covering all m steps.
//
// exact-solve card, §Method: each step forms the per-prime products
// Y_j = B_j R_j (R_j = r_i mod q_j, balanced), the balanced CRT digit x_i of
// the E' residues, and the residual update r_{i+1} = (r_i - A x_i) P'^{-1}
// mod 2^64 read as a signed 64-bit integer.
//
// Work split.  The grid has one CTA per SM (G CTAs); CTA g owns the rows
// k = g, g + G, g + 2G, ... (at most one per consumer warp) for every good
// prime.  The products and the CRT digit of an owned row need only that row
// of every B_j and the full residue vectors, so they stay inside the CTA.
// Two grid barriers per step publish what is all-to-all:
//   barrier 1: x_i mod 2^64 of every row (each row of A x_i needs all of it)
//   barrier 2: the residues of r_{i+1} of every row (each product needs all)
// Because every CTA keeps reading the same rows of B, a die's L2 only ever
// sees the part of B that its SMs own.
//
// Warp roles (256 threads, so every thread may hold 255 registers):
//   warps 0..6  consumers: products from the shared-memory ring (slot s of a
//               step to warp s % 7) against the residues of the slot's primes,
//               held in registers, CRT digit of row t = warp, grid
//               barriers, residual update of that row (its row of A stays in
//               registers for the whole launch when A fits in int32).
//   warp 7      one thread: producer.  B never changes, so it streams the
//               CTA's rows of the streamed B_j with cp.async.bulk into a ring
//               of slots (up to 14 KB) and runs ahead into the next step while
//               the consumers sit in the grid barriers.
// Resident slots.  Most of the CTA's rows of B never leave the SM: the first
// two slots of every consumer warp (all four of warp 3, the only warp on its
// lane quarter) sit in tensor memory, written once at the start (each lane
// keeps the 16-byte chunks it multiplies, 56 words per slot and chunk column:
// two primes x seven rows), and each step reads them back with tcgen05.ld.
// Only the other slots (21 of 53 primes at E' = 53) are streamed, which takes
// about 60 % of the shared-memory traffic (bulk writes plus reads) and of the
// L2 reads off the product phase.
// Before the launch, k_lift_relayout copies B once into the order of
// ownership: CTA g's rows of all primes form one contiguous block, prime-major
// ([e][t][ld]), so every ring slot (all owned rows of two primes) is filled by
// a single bulk copy.
// Every wait is bounded by %globaltimer: on expiry the CTA records an error
// code, every consumer leaves at the same named barrier, the producer waits
// for the copies it has in flight, and the kernel returns.
#include <cuda_runtime.h>

#include <string>

#include "es_common.cuh"
#include "es_internal.h"
#include "lift_device.cuh"
#include "lift_internal.h"

namespace es {
namespace {

constexpr int kConsumerWarps = 7;
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr int kThreads = kConsumerThreads + 32;
constexpr int kPP = 2;                                               // primes per ring slot
constexpr int kSlotsPerWarp = ((kNumPrimes + kPP - 1) / kPP + 6) / 7;  // ring slots per consumer warp and step
constexpr int kChunksPerLane = (int)kFusedMaxLd / 16 / 32;           // 16-byte chunks of a row per lane
constexpr int kMaxLd = (int)kFusedMaxLd;   // A row in registers: 8 int4 chunks per lane
constexpr int kAChunks = kMaxLd / 4 / 32;  // int4 chunks of an int32 A row per lane
constexpr int kVStride = 64;               // Vs row stride (E' <= 53)
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr int kXBatch = 4;   // ulonglong2 loads per consumer thread for x_i mod 2^64
static_assert(kConsumerWarps == 7, "kSlotsPerWarp assumes seven consumer warps");
static_assert(kMaxLd / 2 <= kXBatch * kConsumerThreads, "one batch loads every x_i mod 2^64");
enum : int { kErrEmpty = 11, kErrFull = 12, kErrGrid = 13, kErrDrain = 14 };
constexpr int kErrDigit = kFusedErrDigit;

struct FusedArgs {
  const int8_t* Bf;     // [n][E'][ld] inverses in the order of ownership
  const int32_t* A32;   // [n][ld] A narrowed (zero padded), or null
  const int64_t* A64;   // [n][n] A (read when A32 is null)
  const int64_t* b;     // r_0
  const LiftConst* K;
  int8_t* R;            // [E'][ld] residues of r_i (zero padded), row owners write
  uint64_t* xl;         // [ld] x_i mod 2^64 (zero padded), row owners write
  uint64_t* D;          // [m][n][6] digits
  uint64_t* hs;         // digit stream into mapped host memory (null: none), see DigitStream
  int64_t hsrow[kStreamRows];
  unsigned* bar;        // grid barrier arrivals, zero at launch
  int* err;
  int n, ld, E, m, G, slots, slot_bytes;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t gtime() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
// Bounded wait for the phase of parity `parity`.  Gives up (false) when
// another CTA or thread has recorded an error (if watch_err) or after
// kTimeoutNs, recording `code`.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err, int code, bool watch_err) {
  uint64_t t0 = 0;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try(bar, parity)) return true;
    if ((it & 255) == 0) {
      if (watch_err && *(volatile int*)err) return false;
      const uint64_t now = gtime();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > kTimeoutNs) {
        atomicCAS(err, 0, code);
        return false;
      }
    }
  }
}
// One bulk copy global -> shared (size and both addresses multiples of 16),
// completing `bytes` of the mbarrier's transaction count, with an L2 policy.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// Tensor-memory residency of ring slot s (slot j = s / 7 of consumer warp
// w = s % 7): the first kResSlots slots of every warp, all slots of warp 3.
constexpr int kResSlots = 2;
constexpr int kTmCols = 512;        // allocated tensor-memory columns
constexpr int kTmSlotCols = 2 * 56;  // two chunk columns x (2 primes x 7 rows x 4 words)
__device__ __forceinline__ int res_slots(int w) { return w == 3 ? kSlotsPerWarp : kResSlots; }
__device__ __forceinline__ bool resident(int s) { return s / kConsumerWarps < res_slots(s % kConsumerWarps); }
// Streamed slots before slot s (the ring's fill order within a step).
__device__ __forceinline__ int stream_rank(int s) {
  int k = 0;
  for (int x = 0; x < s; ++x) k += resident(x) ? 0 : 1;
  return k;
}
// First tensor-memory column of warp w's resident slots (warps w and w + 4
// share a lane quarter: the second takes the upper columns).
__device__ __forceinline__ uint32_t tm_col0(int w) { return w >= 4 ? (uint32_t)(kResSlots * kTmSlotCols) : 0u; }
static_assert(2 * kResSlots * kTmSlotCols <= kTmCols && kSlotsPerWarp * kTmSlotCols <= kTmCols, "tensor memory");
// 56 consecutive 32-bit tensor-memory columns of this thread's lane (x32 + x16 + x8).
__device__ __forceinline__ void tm_ld56(uint32_t taddr, uint32_t (&r)[56]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr + 0));
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47])
               : "r"(taddr + 32));
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55])
               : "r"(taddr + 48));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tm_st56(uint32_t taddr, const uint32_t (&r)[56]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
               ::"r"(taddr + 0), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
               : "memory");
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
               ::"r"(taddr + 32), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47])
               : "memory");
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
               ::"r"(taddr + 48), "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55])
               : "memory");
}

// Named barrier 1 over the consumer warps only (the producer never joins).
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory"); }
// The same barrier, returning the OR of `v` over the consumer threads: every
// consumer sees the same answer, so all of them leave together on an error.
__device__ __forceinline__ bool csync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, 1, %2, q;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kConsumerThreads)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Grid barrier among the consumers of all G CTAs, in two halves.  Arrive:
// the CTA's writes are ordered before one release increment of the counter
// by the named barrier.  Wait: acquire loads until the counter reaches
// `target` (G x barriers so far); returns true when the CTA must stop.
__device__ __forceinline__ void grid_arrive(unsigned* bar) {
  csync();
  if (threadIdx.x == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(bar) : "memory");
}
__device__ __forceinline__ bool grid_wait(unsigned* bar, unsigned target, int* err) {
  uint32_t stop = 0;
  if (threadIdx.x == 0) {
    uint64_t t0 = 0;
    for (uint32_t it = 1; ld_acquire(bar) < target; ++it) {
      if ((it & 63) == 0) {
        if (*(volatile int*)err) {
          stop = 1;
          break;
        }
        const uint64_t now = gtime();
        if (t0 == 0) {
          t0 = now;
        } else if (now - t0 > kTimeoutNs) {
          atomicCAS(err, 0, kErrGrid);
          stop = 1;
          break;
        }
      }
    }
  }
  return csync_or(stop);
}
__device__ __forceinline__ bool grid_sync(unsigned* bar, unsigned target, int* err) {
  grid_arrive(bar);
  return grid_wait(bar, target, err);
}

// Sums of eight per-lane values over the warp in 9 shuffles (halving the
// values at each of the first three levels).  Lane l ends with the total of
// value t = bits 4, 3, 2 of l read as (b2 | b3 << 1 | b4 << 2).
__device__ __forceinline__ int32_t reduce_rows(int32_t (&a)[8], int lane) {
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
  for (int j = 0; j < 4; ++j) {  // keep values with bit 2 of t equal to b4
    const int32_t send = b4 ? a[j] : a[j + 4], keep = b4 ? a[j + 4] : a[j];
    a[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int32_t send = b3 ? a[j] : a[j + 2], keep = b3 ? a[j + 2] : a[j];
    a[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  {
    const int32_t send = b2 ? a[0] : a[1], keep = b2 ? a[1] : a[0];
    a[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  a[0] += __shfl_xor_sync(0xffffffffu, a[0], 2);
  a[0] += __shfl_xor_sync(0xffffffffu, a[0], 1);
  return a[0];
}

__device__ __forceinline__ uint64_t lo64(const uint32_t* w) { return (uint64_t)w[0] | ((uint64_t)w[1] << 32); }

// x mod 2^64 of the balanced CRT digit x from two 64-bit warp sums, lane l
// holding the residues of primes l and l + 32:
//   c_e = v_e w_e mod q_e,  x = sum_e c_e M_e - t P' (M_e = P'/q_e),
//   sum_e c_e / q_e = t + f, 0 <= f < 1; balanced x subtracts P' once more
//   exactly when f > 1/2.
// With F_e = floor(2^56 / q_e), T = sum_e c_e F_e satisfies
// 0 <= 2^56 sum_e c_e/q_e - T < sum_e c_e < 2^14 (E' <= 53, c_e <= 250), so
// with t' = T >> 56 and g = T mod 2^56:
//   g >= 2^55            f > 1/2 (or the sum just crossed an integer, where
//                        t' = t - 1 and subtracting P' once more is again exact)
//   g <  2^55 - 2^14     f < 1/2
// and x mod 2^64 = sum_e c_e (M_e mod 2^64) - t' P' - [g >= 2^55] P'.  The
// window in between returns false: the caller forms the full digit instead.
__device__ __forceinline__ bool fast_digit_lo(int32_t v0, int32_t v1, const ModQ& mq0, const ModQ& mq1, uint32_t w0,
                                              uint32_t w1, uint64_t f0, uint64_t f1, uint64_t m0, uint64_t m1,
                                              uint64_t P64, uint64_t* xlo) {
  const uint32_t c0 = barrett((uint32_t)(v0 < 0 ? v0 + (int32_t)mq0.q : v0) * w0, mq0);
  const uint32_t c1 = barrett((uint32_t)(v1 < 0 ? v1 + (int32_t)mq1.q : v1) * w1, mq1);
  uint64_t T = (uint64_t)c0 * f0 + (uint64_t)c1 * f1;   // f, m are 0 for lanes past E'
  uint64_t X = (uint64_t)c0 * m0 + (uint64_t)c1 * m1;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    T += __shfl_xor_sync(0xffffffffu, T, o);
    X += __shfl_xor_sync(0xffffffffu, X, o);
  }
  const uint64_t g = T & ((1ull << 56) - 1), half = 1ull << 55;
  if (g < half && g >= half - (1ull << 14)) return false;
  *xlo = X - (T >> 56) * P64 - (g >= half ? P64 : 0);
  return true;
}

// First row position of CTA g in the order of ownership.
__device__ __forceinline__ int64_t own_start(int g, int n, int G) {
  const int base = n / G, extra = n % G;
  return (int64_t)g * base + min(g, extra);
}

// Bf: CTA g's block (at own_start(g) E' ld) holds B_{pidx[e]}[k][:] for its
// rows k = g + t G at (e rows_g + t) ld.  One CTA per row k.
__global__ void __launch_bounds__(256) k_lift_relayout(const int8_t* __restrict__ B, const LiftConst* __restrict__ K,
                                                       int n, int ld, int G, int8_t* __restrict__ Bf) {
  const int k = blockIdx.x, g = k % G, t = k / G, E = K->E;
  const int rows = (n - 1 - g) / G + 1;
  const int cpr = ld / 16;  // int4 chunks per row
  int8_t* blk = Bf + own_start(g, n, G) * E * ld;
  for (int i = threadIdx.x; i < E * cpr; i += blockDim.x) {
    const int e = i / cpr, ch = i - e * cpr;
    reinterpret_cast<int4*>(blk + ((int64_t)e * rows + t) * ld)[ch] =
        __ldg(reinterpret_cast<const int4*>(B + ((int64_t)K->pidx[e] * n + k) * ld) + ch);
  }
}


template <bool kA32>
__global__ void __launch_bounds__(kThreads, 1) k_lift_fused(const FusedArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  uint64_t* xs = reinterpret_cast<uint64_t*>(ring + (size_t)a.slots * a.slot_bytes);
  int32_t* Vs = reinterpret_cast<int32_t*>(xs + a.ld);
  uint64_t* full = reinterpret_cast<uint64_t*>(Vs + kConsumerWarps * kVStride);
  uint64_t* empty = full + a.slots;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(empty + a.slots);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x, G = a.G, n = a.n, ld = a.ld, E = a.E;
  const unsigned slots = (unsigned)a.slots;
  const int rows = (n - 1 - g) / G + 1;  // owned rows, 1 ..  kConsumerWarps (G <= n)
  // A step's block is prime-major, [e][t][ld]; ring slot s of a step holds
  // all owned rows of primes 2s and 2s + 1.
  const int rowbytes = rows * ld;
  const int sps = (E + kPP - 1) / kPP;  // ring slots per step

  if (threadIdx.x == 0) {
    for (unsigned s = 0; s < slots; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);  // released by the one warp that consumed it
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(s_tmem)),
                 "r"(kTmCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    // Fill number q (all steps in order) goes to ring slot q % slots; its
    // (q / slots)-th use waits for the previous use to be released.
    if (lane != 0) return;
    const uint64_t pol = policy_evict_last();
    const int8_t* Bg = a.Bf + own_start(g, n, G) * E * ld;  // this CTA's rows, all primes
    unsigned q = 0, r = 0, use = 0;
    bool ok = true;
    for (int step = 0; step < a.m && ok; ++step) {
      for (int s = 0; s < sps; ++s) {
        if (resident(s)) continue;
        if (use > 0 && !mbar_wait(empty + r, (use - 1) & 1, a.err, kErrEmpty, true)) {
          ok = false;
          break;
        }
        const int e0 = kPP * s, np = min(kPP, E - e0);
        mbar_expect_tx(full + r, (uint32_t)(np * rowbytes));
        bulk_load(ring + (size_t)r * a.slot_bytes, Bg + (int64_t)e0 * rowbytes, (uint32_t)(np * rowbytes), full + r,
                  pol);
        ++q;
        if (++r == slots) {
          r = 0;
          ++use;
        }
      }
    }
    // Every copy issued lands before the CTA may exit (fills earlier than the
    // last `slots` were consumed, hence complete).
    for (unsigned f = q > slots ? q - slots : 0; f < q; ++f)
      if (!mbar_wait(full + f % slots, (f / slots) & 1, a.err, kErrDrain, false)) break;
    return;
  }

  // -------------------------------------------------------------- consumers
  const LiftConst* __restrict__ K = a.K;
  const bool own = warp < rows;
  const int64_t k = g + (int64_t)warp * G;  // this warp's row (when own)
  int64_t rk = own ? a.b[k] : 0;            // r_i of that row, identical in all lanes
  const int achunks = ld / 4;               // int4 chunks of an int32 A row
  int4 arow[kAChunks];
#pragma unroll
  for (int i = 0; i < kAChunks; ++i) {
    const int ch = lane + 32 * i;
    arow[i] = (kA32 && own && ch < achunks) ? __ldg(reinterpret_cast<const int4*>(a.A32 + k * ld) + ch)
                                            : make_int4(0, 0, 0, 0);
  }
  const int bchunks = ld / 16;
  // constants of this lane's primes e = lane and lane + 32, kept in registers
  const bool h0 = lane < E, h1 = lane + 32 < E;
  const int e0 = h0 ? lane : 0, e1 = h1 ? lane + 32 : 0;
  const ModQ mq0 = K->mq[e0], mq1 = K->mq[e1];
  const uint32_t w0 = K->w[e0], w1 = K->w[e1];
  const uint64_t f0 = h0 ? K->t56[e0] : 0, f1 = h1 ? K->t56[e1] : 0;
  const uint64_t m0 = h0 ? lo64(K->Mq[e0]) : 0, m1 = h1 ? lo64(K->Mq[e1]) : 0;
  const uint64_t P64 = lo64(K->P), Pinv = K->Pinv64;
  // this warp's resident slots into tensor memory: lane l keeps chunks l and
  // l + 32 of both primes' rows, 56 words per chunk column
  const int nres = res_slots(warp);
  const uint32_t tm_warp = *s_tmem + ((uint32_t)(32 * (warp & 3)) << 16) + tm_col0(warp);
  const int8_t* Bg = a.Bf + own_start(g, n, G) * E * ld;  // this CTA's rows, all primes, [e][t][ld]
  for (int j = 0; j < nres; ++j) {
    const int s = warp + kConsumerWarps * j;
#pragma unroll
    for (int cc = 0; cc < kChunksPerLane; ++cc) {
      const int ch = lane + 32 * cc;
      uint32_t w[56];
#pragma unroll
      for (int pe = 0; pe < kPP; ++pe)
#pragma unroll
        for (int t = 0; t < kConsumerWarps; ++t) {
          const int e = kPP * s + pe;
          int4 v = make_int4(0, 0, 0, 0);
          if (s < sps && e < E && t < rows && ch < bchunks)
            v = __ldg(reinterpret_cast<const int4*>(Bg + ((int64_t)e * rows + t) * ld) + ch);
          const int o = (pe * kConsumerWarps + t) * 4;
          w[o] = (uint32_t)v.x, w[o + 1] = (uint32_t)v.y, w[o + 2] = (uint32_t)v.z, w[o + 3] = (uint32_t)v.w;
        }
      tm_st56(tm_warp + (uint32_t)(j * kTmSlotCols + cc * 56), w);
    }
  }
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  int sstream = 0;  // streamed slots per step
  for (int s = 0; s < sps; ++s) sstream += resident(s) ? 0 : 1;
  unsigned target = 0;
  unsigned gs = 0;  // fills of all earlier steps
  // the steps; every way out (the end, or an error that all consumers leave
  // on together) comes back here to free tensor memory
  [&]() {
  // this warp's row in the digit stream (-1: none), and its pending words
  int si_stream = -1;
  if (a.hs && own) {
#pragma unroll
    for (int q = 0; q < kStreamRows; ++q)
      if (a.hsrow[q] == k) si_stream = q;
  }
  uint64_t hs_part = 0;
  int hs_step = -1;
  auto stream_out = [&]() {  // twelve 8-byte words: 32 bits of the digit, 32 of tag
    if (hs_step >= 0 && lane < 2 * kDigitLimbs) {
      const uint64_t w = ((lane & 1) ? hs_part >> 32 : hs_part & 0xffffffffull) | ((uint64_t)(hs_step + 1) << 32);
      asm volatile("st.relaxed.sys.global.u64 [%0], %1;" ::"l"(a.hs + ((int64_t)hs_step * kStreamRows + si_stream) *
                                                                           kStreamWords + lane),
                   "l"(w)
                   : "memory");
    }
    hs_step = -1;
  };
  for (int step = 0; step < a.m; ++step) {
    if (si_stream >= 0) stream_out();  // the previous step's digit
    // This warp's slots are s = warp + 7 j; their primes' residues of r_i go
    // straight to registers (chunks lane and lane + 32 of each row).
    int4 Rr[kSlotsPerWarp][kPP][kChunksPerLane];
#pragma unroll
    for (int j = 0; j < kSlotsPerWarp; ++j)
#pragma unroll
      for (int pe = 0; pe < kPP; ++pe) {
        const int e = kPP * (warp + kConsumerWarps * j) + pe;
#pragma unroll
        for (int cc = 0; cc < kChunksPerLane; ++cc) {
          const int ch = lane + 32 * cc;
          Rr[j][pe][cc] = (e < E && ch < bchunks) ? __ldcg(reinterpret_cast<const int4*>(a.R + (int64_t)e * ld) + ch)
                                                  : make_int4(0, 0, 0, 0);
        }
      }
    // products of the owned rows; raw sums (|sum| <= n 125^2) go to Vs and
    // are reduced in the CRT below
    bool fail = false;
#pragma unroll
    for (int j = 0; j < kSlotsPerWarp; ++j) {
      const int s = warp + kConsumerWarps * j;
      if (s >= sps) break;
      const bool res = j < nres;  // warp-uniform
      unsigned r = 0;
      if (!res) {
        const unsigned q = gs + (unsigned)stream_rank(s), use = q / slots;
        r = q % slots;
        if (!fail) fail = !mbar_wait(full + r, use & 1, a.err, kErrFull, true);
      }
      fail = __any_sync(0xffffffffu, fail);  // warp-uniform: the code below shuffles
      if (fail) break;
      const int eb = kPP * s, np = min(kPP, E - eb);
      const int4* src = reinterpret_cast<const int4*>(ring + (size_t)r * a.slot_bytes);
      int32_t acc[kPP][8];
#pragma unroll
      for (int pe = 0; pe < kPP; ++pe)
#pragma unroll
        for (int t = 0; t < 8; ++t) acc[pe][t] = 0;
#pragma unroll
      for (int cc = 0; cc < kChunksPerLane; ++cc) {
        const int ch = lane + 32 * cc;
        int4 x[kPP][kConsumerWarps];
        if (res) {  // every lane: tcgen05.ld is warp-wide
          uint32_t w[56];
          tm_ld56(tm_warp + (uint32_t)(j * kTmSlotCols + cc * 56), w);
#pragma unroll
          for (int pe = 0; pe < kPP; ++pe)
#pragma unroll
            for (int t = 0; t < kConsumerWarps; ++t) {
              const int o = (pe * kConsumerWarps + t) * 4;
              x[pe][t] = make_int4((int)w[o], (int)w[o + 1], (int)w[o + 2], (int)w[o + 3]);
            }
        }
        if (ch < bchunks) {
          if (!res) {
#pragma unroll
            for (int pe = 0; pe < kPP; ++pe)
#pragma unroll
              for (int t = 0; t < kConsumerWarps; ++t)
                x[pe][t] = (pe < np && t < rows) ? src[(pe * rows + t) * bchunks + ch] : make_int4(0, 0, 0, 0);
          }
#pragma unroll
          for (int pe = 0; pe < kPP; ++pe) {
            const int4 y = Rr[j][pe][cc];
#pragma unroll
            for (int t = 0; t < kConsumerWarps; ++t) {
              acc[pe][t] = __dp4a(x[pe][t].x, y.x, acc[pe][t]);
              acc[pe][t] = __dp4a(x[pe][t].y, y.y, acc[pe][t]);
              acc[pe][t] = __dp4a(x[pe][t].z, y.z, acc[pe][t]);
              acc[pe][t] = __dp4a(x[pe][t].w, y.w, acc[pe][t]);
            }
          }
        }
      }
      __syncwarp();
      if (!res && lane == 0) mbar_arrive(empty + r);  // the slot's bytes are in registers now
      const int t = (lane >> 2) & 7;           // the row whose total this lane ends with
#pragma unroll
      for (int pe = 0; pe < kPP; ++pe) {
        const int32_t v = reduce_rows(acc[pe], lane);
        if ((lane & 3) == 0 && t < rows && pe < np) Vs[t * kVStride + eb + pe] = v;
      }
    }
    gs += (unsigned)sstream;
    if (csync_or(fail)) return;
    // x_i mod 2^64 of this warp's row, on the short path (see fast_digit_lo),
    // published before the full digit is formed
    int32_t v0 = 0, v1 = 0;
    uint64_t xlo = 0;
    if (own) {
      v0 = h0 ? reduce_bal(Vs[warp * kVStride + lane], mq0) : 0;
      v1 = h1 ? reduce_bal(Vs[warp * kVStride + lane + 32], mq1) : 0;
      if (!fast_digit_lo(v0, v1, mq0, mq1, w0, w1, f0, f1, m0, m1, P64, &xlo)) {
        uint32_t S[kCrtWords];
        crt_warp(v0, v1, lane, K, S);
        xlo = (uint64_t)S[0] | ((uint64_t)S[1] << 32);
      }
      if (lane == 0) a.xl[k] = xlo;
    }
    const bool last = step + 1 == a.m;
    if (!last) grid_arrive(a.bar);
    // the full balanced digit (six limbs) while the barrier completes; its
    // low limb must equal the short path's
    if (own) {
      uint32_t S[kCrtWords];
      crt_warp(v0, v1, lane, K, S);
      uint64_t limb = 0;
#pragma unroll
      for (int l = 0; l < kDigitLimbs; ++l)
        if (lane == l) limb = (uint64_t)S[2 * l] | ((uint64_t)S[2 * l + 1] << 32);
      if (lane < kDigitLimbs) a.D[((int64_t)step * n + k) * kDigitLimbs + lane] = limb;
      if (lane == 0 && limb != xlo) atomicCAS(a.err, 0, kErrDigit);
      if (si_stream >= 0) {
        // a streamed row: its twelve self-tagged words go out at the start of
        // the next step's products (the last step's at once), so that the
        // stores to host memory do not hold up this step's second barrier
        hs_part = __shfl_sync(0xffffffffu, limb, (lane >> 1) % kDigitLimbs);
        hs_step = step;
        if (last) stream_out();
      }
    }
    if (last) break;
    target += G;
    if (grid_wait(a.bar, target, a.err)) return;
    // x_i mod 2^64 of every row: one batch of loads
    {
      const ulonglong2* src = reinterpret_cast<const ulonglong2*>(a.xl);
      ulonglong2* dst = reinterpret_cast<ulonglong2*>(xs);
      const int nx = ld / 2;
      ulonglong2 v[kXBatch];
#pragma unroll
      for (int q = 0; q < kXBatch; ++q) {
        const int i = threadIdx.x + q * kConsumerThreads;
        v[q] = i < nx ? __ldcg(src + i) : make_ulonglong2(0, 0);
      }
#pragma unroll
      for (int q = 0; q < kXBatch; ++q) {
        const int i = threadIdx.x + q * kConsumerThreads;
        if (i < nx) dst[i] = v[q];
      }
    }
    csync();
    // r_{i+1} of this warp's row and its residues
    if (own) {
      uint64_t sum = 0;
      if (kA32) {
#pragma unroll
        for (int i = 0; i < kAChunks; ++i) {
          const int ch = lane + 32 * i;
          if (ch < achunks) {
            const ulonglong2 x0 = reinterpret_cast<const ulonglong2*>(xs)[2 * ch];
            const ulonglong2 x1 = reinterpret_cast<const ulonglong2*>(xs)[2 * ch + 1];
            sum += (uint64_t)(int64_t)arow[i].x * x0.x + (uint64_t)(int64_t)arow[i].y * x0.y +
                   (uint64_t)(int64_t)arow[i].z * x1.x + (uint64_t)(int64_t)arow[i].w * x1.y;
          }
        }
      } else {
        const int64_t* Ak = a.A64 + k * n;
        for (int j = lane; j < n; j += 32) sum += (uint64_t)__ldg(Ak + j) * xs[j];
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      rk = (int64_t)(((uint64_t)rk - sum) * Pinv);
      if (h0) a.R[(int64_t)lane * ld + k] = (int8_t)reduce_i64_bal(rk, mq0);
      if (h1) a.R[(int64_t)(lane + 32) * ld + k] = (int8_t)reduce_i64_bal(rk, mq1);
    }
    target += G;
    if (grid_sync(a.bar, target, a.err)) return;
  }
  }();
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  csync();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(*s_tmem), "r"(kTmCols));
  }
}

size_t fused_smem_fixed(int64_t ld) { return 144 + (size_t)ld * 8 + (size_t)kConsumerWarps * kVStride * 4; }

}  // namespace

// Whether the fused lift can run this problem on `device`, and its shape.
bool fused_lift_plan(int64_t n, int64_t c, int E, int device, FusedPlan* p) {
  if (c != 1 || n < 1) return false;
  const int64_t ld = padded_ld(n);
  if (ld > kMaxLd) return false;
  int sms = 0, smem = 0, coop = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, device) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (!coop || sms < 1) return false;
  const int64_t G = n < sms ? n : sms;
  if ((n + G - 1) / G > kConsumerWarps) return false;
  const size_t fixed = fused_smem_fixed(ld);
  const int64_t rows_max = (n + G - 1) / G;
  const size_t slot_bytes = (size_t)((kPP * rows_max * ld + 127) / 128 * 128);
  const size_t per_slot = slot_bytes + 16;
  if ((size_t)smem < fixed + 2 * per_slot) return false;
  int slots = (int)(((size_t)smem - fixed) / per_slot);
  if (slots > 64) slots = 64;
  p->G = (int)G;
  p->slots = slots;
  p->slot_bytes = (int)slot_bytes;
  p->relayout_bytes = (size_t)E * n * ld;
  p->smem = fixed + (size_t)slots * per_slot;
  return true;
}

es_status fused_lift_relayout(const FusedPlan& p, const int8_t* B, const LiftConst* K, int8_t* Bf, int64_t n,
                              void* stream) {
  k_lift_relayout<<<(unsigned)n, 256, 0, (cudaStream_t)stream>>>(B, K, (int)n, (int)padded_ld(n), p.G, Bf);
  return cuda_status(cudaGetLastError(), "k_lift_relayout");
}

es_status fused_lift_launch(const FusedPlan& p, const int8_t* Bf, const int32_t* A32, const int64_t* A64,
                            const int64_t* b, const LiftConst* K, int8_t* R, uint64_t* xl, uint64_t* D,
                            unsigned* bar, int* err, int64_t n, int E, int32_t m, void* stream,
                            const DigitStream* ds) {
  FusedArgs a;
  a.Bf = Bf;
  a.A32 = A32;
  a.A64 = A64;
  a.b = b;
  a.K = K;
  a.R = R;
  a.xl = xl;
  a.D = D;
  a.hs = ds ? ds->dev : nullptr;
  for (int q = 0; q < kStreamRows; ++q) a.hsrow[q] = ds ? ds->rows[q] : -1;
  a.bar = bar;
  a.err = err;
  a.n = (int)n;
  a.ld = (int)padded_ld(n);
  a.E = E;
  a.m = m;
  a.G = p.G;
  a.slots = p.slots;
  a.slot_bytes = p.slot_bytes;
  const void* fn = A32 ? (const void*)k_lift_fused<true> : (const void*)k_lift_fused<false>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return cuda_status(e, "fused lift smem attribute");
  void* args[] = {&a};
  e = cudaLaunchCooperativeKernel(fn, dim3((unsigned)p.G), dim3(kThreads), args, p.smem, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return ES_ERR_RANGE;  // caller falls back to the per-step kernels
  }
  return ES_OK;
}

}  // namespace es
