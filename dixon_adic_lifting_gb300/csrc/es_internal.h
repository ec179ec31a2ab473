// Internal declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <memory>
#include <new>
#include <string>
#include <utility>
#include <vector>

#include "../../include/es.h"

namespace es {

constexpr int kMaxDevices = 64;

// ---------------------------------------------------------------- errors
void set_last_error(const std::string& s);
// Records the CUDA error (if any) and returns ES_ERR_CUDA / ES_OK.
es_status cuda_status(int cuda_err, const char* where);

#define ES_CHECK(expr)                     \
  do {                                     \
    es_status _st = (expr);                \
    if (_st != ES_OK) return _st;          \
  } while (0)

// ---------------------------------------------------------------- workspace
// Grow-only device workspace of the current device, carved into regions by
// a Layout.  Each region starts on a 256-byte boundary.
struct Layout {
  size_t total = 0;
  size_t add(size_t bytes) {
    size_t off = total;
    total += (bytes + 255) / 256 * 256;
    return off;
  }
};

// Ensures the current device's workspace holds at least `bytes`; returns its
// base in *base.  max_bytes != 0 caps the size (ES_ERR_NOMEM beyond it).
es_status workspace_get(size_t bytes, size_t max_bytes, bool inject_nomem, char** base);

// Stream to use for a caller-given handle (NULL -> the library's stream).
void* resolve_stream(void* user_stream);

// Current device's SM count (cached).
int sm_count();

// Row-stride of the int8 residue matrices: n rounded up to 16 bytes.
inline int64_t padded_ld(int64_t n) { return (n + 15) / 16 * 16; }

// ---------------------------------------------------------------- range
// Device statistics of A and b used by the range check and the bounds.
struct Stats {
  uint64_t max_abs_a;   // max |A_ij| (|-2^63| = 2^63 as uint64)
  uint64_t max_abs_b;   // max |b_ij|
  int zero_row;         // some row of A is zero
  double log2_d;        // sum_i 0.5 log2 ||a_i||^2
  double log2_n;        // sum_i 0.5 log2 (||a_i||^2 + max_k b_ik^2)
};
es_status compute_stats(const int64_t* A_dev, const int64_t* b_dev, int64_t n, int64_t c, char* scratch,
                        void* stream, Stats* out);
// scratch bytes compute_stats needs
size_t stats_scratch_bytes(int64_t n);
bool in_range(int64_t n, uint64_t max_abs_a);

// Bounds and step count from Stats and the good-prime flags.
void plan_from_stats(const Stats& s, const uint8_t* good, int64_t* num_bits, int64_t* den_bits, int32_t* m);

// ---------------------------------------------------------------- stages
// Residues of `count` int64 values for all 53 primes: out[j*ostride + i].
es_status launch_residues(const int64_t* src, int64_t count, int8_t* out, int64_t ostride, void* stream);
// Residues of A [n, n] into W [53][n][ld] (balanced, padding zero).
es_status launch_residues_matrix(const int64_t* A, int64_t n, int64_t ld, int8_t* W, void* stream);

// Batched modular inverse: A_dev -> B [53][n][ld], good [53] (device).
size_t inverse_scratch_bytes(int64_t n);
// split: run the blocks on two SM partitions (green contexts) when the
// device supports them (no extra streams otherwise); *used_split (if given)
// tells whether they ran that way.
es_status run_inverse(const int64_t* A_dev, int64_t n, int8_t* B_dev, uint8_t* good_dev, char* scratch,
                      void* stream, bool split = true, bool* used_split = nullptr);
// Destroys the SM partitions of device `dev` (es_release_workspace).
void release_inverse_partitions(int dev);

// Kernel accounting: every launch site adds to the launch counter; the lift
// optionally brackets each launch of its product kernel with CUDA events.
void count_launch(int64_t k = 1);
int64_t launch_count();
struct KernelTiming {
  bool events = false;       // bracket each launch of the dominant lift kernel with events
  bool fused = false;        // the lift ran as one fused launch (k_lift_fused)
  const char* name = "";     // that kernel's name
  int64_t launches = 0;      // its launches
  double ms = 0.0;           // their summed event time
  double bytes_per_launch = 0.0;
};

// Lift: m steps -> digits [m][n*c][6].
size_t lift_scratch_bytes(int64_t n, int64_t c, int E, bool a32);
// A lift in flight: run_lift_start enqueues every launch on the stream and
// returns without waiting; run_lift_finish waits for it, reads the kernels'
// error flag and fills the timing (the host is free in between).
struct LiftRun {
  void* stream = nullptr;
  std::vector<void*> ev;  // cudaEvent_t pairs around each launch of the dominant kernel
  int* err = nullptr;     // device error flag of the lift kernels
  bool fused = false, tc = false, a32 = false;
  int E = 0;
  int64_t n = 0, c = 0;
  int32_t m = 0;
  KernelTiming* kt = nullptr;
  LiftRun() = default;
  LiftRun(const LiftRun&) = delete;
  LiftRun& operator=(const LiftRun&) = delete;
  ~LiftRun();  // destroys the events
};
// Digits of a few components (c == 1) handed to the host while the fused lift
// forms them: `host` is a page-locked block mapped into the device's address
// space (dev, its device address), kStreamRows entries of kStreamWords words
// per step: entry (i, s) at (i kStreamRows + s) kStreamWords holds the digit
// of step i of component rows[s] as 12 words, word j = 32-bit part j of the
// digit's six limbs (little-endian) in its low half and the tag i + 1 in its
// high half.  Each 8-byte store is single-copy atomic, so a word whose tag
// reads i + 1 holds its part; no fence is needed (zero before the lift).
// Other lift paths leave the block untouched.
constexpr int kStreamRows = 4;
constexpr int kStreamWords = 16;
struct DigitStream {
  uint64_t* dev = nullptr;
  const volatile uint64_t* host = nullptr;
  int64_t rows[kStreamRows] = {-1, -1, -1, -1};
};
// stall_barrier: start the fused lift's grid-barrier counter 11 short of
// wrapping around, so that its first barrier never completes (fault injection
// of an expiring bounded wait).
es_status run_lift_start(const int64_t* A_dev, const int64_t* b_dev, int64_t n, int64_t c, const int8_t* B_dev,
                         const uint8_t* good_host, int32_t m, uint64_t* digits_dev, uint64_t max_abs_a,
                         char* scratch, void* stream, KernelTiming* kt, bool allow_fused, LiftRun* run,
                         bool stall_barrier = false, const DigitStream* stream_digits = nullptr);
es_status run_lift_finish(LiftRun* run);
es_status run_lift(const int64_t* A_dev, const int64_t* b_dev, int64_t n, int64_t c, const int8_t* B_dev,
                   const uint8_t* good_host, int32_t m, uint64_t* digits_dev, uint64_t max_abs_a, char* scratch,
                   void* stream, KernelTiming* kt = nullptr, bool allow_fused = true);

// ---------------------------------------------------------------- solution
// Host buffer of result limbs.  Blocks come from a small process-wide pool
// (host_pool.cpp): page-locked when a CUDA device is present (a device copy
// into them runs at full speed, with no page faults once warm), returned to
// the pool when the buffer dies.  resize() keeps no contents.
class LimbBuffer {
 public:
  LimbBuffer() = default;
  LimbBuffer(const LimbBuffer&) = delete;
  LimbBuffer& operator=(const LimbBuffer&) = delete;
  ~LimbBuffer() { release(); }
  void resize(size_t count);  // contents unspecified afterwards
  uint64_t* data() { return p_; }
  const uint64_t* data() const { return p_; }
  size_t size() const { return n_; }
  bool pinned() const { return pinned_; }

 private:
  void release();
  uint64_t* p_ = nullptr;
  size_t n_ = 0, cap_ = 0;
  bool pinned_ = false;
};

struct Solution {
  int64_t n = 0, c = 0, limbs = 0;
  LimbBuffer num;              // [n*c*limbs]
  std::vector<uint64_t> den;  // [limbs]
  double ms[ES_NUM_PHASES] = {0, 0, 0, 0, 0, 0};
  int32_t m = 0;
  int32_t primes_used = 0;
  int64_t launches = 0;
  bool inverse_split = false;  // the inverse ran on the two SM partitions
  KernelTiming top;
};

// Reconstruction with the numerator pass on the GPU (k_recon.cu): applicable
// when the low-digit certificate needs m' <= m digits.  digits on the device.
bool recon_device_applicable(int64_t n, int32_t m, const uint8_t* good, int64_t num_bits, int64_t den_bits,
                             const Stats& stats, int32_t* mp_out);
size_t recon_device_bytes(int64_t nc, int32_t mp, const uint8_t* good, int64_t num_bits, int64_t den_bits);
// Its digit-independent constants (P'^m, Q = P'^m', Q's reciprocal) are
// built first, on the host, while the lift runs.
struct ReconPlan;
void recon_plan_free(ReconPlan* p);
es_status recon_device_prepare(int64_t n, int64_t c, int32_t m, int32_t mp, const uint8_t* good, int64_t num_bits,
                               int64_t den_bits, const Stats& stats, ReconPlan** out);
// The components whose denominators seed the common denominator (the first
// round's sample), for `threads` host threads (0: all cores).
std::vector<int64_t> recon_samples(int64_t n, int64_t c, int threads);
// recon_device_prepare, and with a digit stream (ds, its first ns rows the
// samples) the samples' shifted sums formed from the low digit up as the
// digits arrive, both on the host pool while the lift runs.  lift_done: an
// event recorded after the lift's launches; a sample whose digits stop
// coming once it has completed leaves *pre empty (the reconstruction then
// reads the digits from the device as usual).
es_status recon_prepare_overlapped(int64_t n, int64_t c, int32_t m, int32_t mp, const uint8_t* good,
                                   int64_t num_bits, int64_t den_bits, const Stats& stats, int threads,
                                   const DigitStream* ds, int ns, void* lift_done, ReconPlan** out,
                                   std::vector<std::vector<uint64_t>>* pre);
// pre: the shifted sums (assemble_shifted) of the first round's sampled
// components, in the order sample_components gives, when they were formed
// already (from a DigitStream); null or empty: formed here from D_dev.
es_status reconstruct_device(ReconPlan* plan, const uint64_t* D_dev, int threads, char* scratch,
                             size_t scratch_bytes, void* stream, struct Solution* out,
                             const std::vector<std::vector<uint64_t>>* pre = nullptr);

// Host reconstruction (recon.cpp).  digits [m][n*c][6].
es_status reconstruct(const uint64_t* digits, int64_t n, int64_t c, int32_t m, const uint8_t* good,
                      int64_t num_bits, int64_t den_bits, int threads, bool inject_fault, Solution* out);

}  // namespace es

struct es_solution {
  es::Solution s;
};
