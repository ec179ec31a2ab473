// es_solve / es_solve_device and the stage entry points: argument checks,
// the device workspace, phase timing, and the sequence
//   statistics (range check, Hadamard terms) -> batched modular inverse ->
//   plan (prime set P', step count m) -> lift -> digits to host ->
//   rational reconstruction.
// exact-solve card, §API (solve returns None when A is singular over the
// rationals), §Method (stages, range), §Requirements and limits.
#include <cuda_runtime.h>

#include <atomic>
#include <chrono>
#include <cstring>
#include <memory>
#include <mutex>
#include <new>
#include <string>

#include "es_common.cuh"
#include "es_internal.h"

namespace es {

// ------------------------------------------------------------ errors
static thread_local std::string g_last_error;
void set_last_error(const std::string& s) { g_last_error = s; }
es_status cuda_status(int err, const char* where) {
  if (err == cudaSuccess) return ES_OK;
  g_last_error = std::string(where) + ": " + cudaGetErrorString((cudaError_t)err);
  cudaGetLastError();  // clear a non-sticky error
  return ES_ERR_CUDA;
}

// ------------------------------------------------------------ launch accounting
static std::atomic<int64_t> g_launches(0);
void count_launch(int64_t k) { g_launches.fetch_add(k, std::memory_order_relaxed); }
int64_t launch_count() { return g_launches.load(std::memory_order_relaxed); }

// ------------------------------------------------------------ per-device state
namespace {
struct DeviceState {
  std::mutex mu;
  char* ws = nullptr;
  size_t ws_size = 0;
  uint64_t* digits = nullptr;  // device digits buffer (grow-only)
  size_t digits_size = 0;
  uint64_t* hdigits = nullptr;  // pinned host copy (grow-only)
  size_t hdigits_size = 0;
  char* recon = nullptr;  // device reconstruction buffers (grow-only)
  size_t recon_size = 0;
  uint64_t* hstream = nullptr;  // page-locked, mapped: the fused lift's digit stream (grow-only)
  size_t hstream_words = 0;
  cudaEvent_t lift_done = nullptr;
  cudaStream_t stream = nullptr;
  int sms = 0;
};
DeviceState g_dev[kMaxDevices];

int current_device() {
  int d = 0;
  cudaGetDevice(&d);
  return d < kMaxDevices ? d : 0;
}

// The digit-stream block (page-locked, mapped into the device's address
// space) and the event that marks the lift's end; false when unavailable.
bool stream_buffer(DeviceState& dev, size_t words) {
  if (!dev.lift_done) {
    if (cudaEventCreateWithFlags(&dev.lift_done, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      dev.lift_done = nullptr;
      return false;
    }
  }
  if (words <= dev.hstream_words) return true;
  if (dev.hstream) cudaFreeHost(dev.hstream);
  dev.hstream = nullptr;
  dev.hstream_words = 0;
  if (cudaHostAlloc((void**)&dev.hstream, words * 8, cudaHostAllocMapped) != cudaSuccess) {
    cudaGetLastError();
    dev.hstream = nullptr;
    return false;
  }
  dev.hstream_words = words;
  return true;
}

es_status grow_device(void** p, size_t* have, size_t need, size_t cap_left, bool inject) {
  if (inject) return ES_ERR_NOMEM;
  if (cap_left && need > cap_left) return ES_ERR_NOMEM;  // the cap applies to what this call needs
  if (need <= *have) return ES_OK;
  if (*p) cudaFree(*p);
  *p = nullptr;
  *have = 0;
  cudaError_t e = cudaMalloc(p, need);
  if (e != cudaSuccess) {
    cudaGetLastError();
    *p = nullptr;
    set_last_error(std::string("cudaMalloc: ") + cudaGetErrorString(e));
    return ES_ERR_NOMEM;
  }
  *have = need;
  return ES_OK;
}
}  // namespace

es_status workspace_get(size_t bytes, size_t max_bytes, bool inject_nomem, char** base) {
  DeviceState& d = g_dev[current_device()];
  void* p = d.ws;
  ES_CHECK(grow_device(&p, &d.ws_size, bytes, max_bytes, inject_nomem));
  d.ws = (char*)p;
  *base = d.ws;
  return ES_OK;
}

void* resolve_stream(void* user_stream) {
  if (user_stream) return user_stream;
  DeviceState& d = g_dev[current_device()];
  if (!d.stream) cudaStreamCreateWithFlags(&d.stream, cudaStreamNonBlocking);
  return d.stream;
}

int sm_count() {
  DeviceState& d = g_dev[current_device()];
  if (!d.sms) {
    int dev = current_device();
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
  }
  return d.sms;
}

// ------------------------------------------------------------ the solve
namespace {

struct Options {
  void* stream = nullptr;
  size_t max_bytes = 0;
  int fault = 0;
  int threads = 0;
  bool timing = false;
  bool kernel_events = false;
  bool host_recon = false;
  bool step_lift = false;
  bool one_stream = false;
};
Options read_options(const es_options* o) {
  Options r;
  if (o) {
    r.stream = o->stream;
    r.max_bytes = o->max_device_bytes;
    r.fault = o->fault_stage;
    r.threads = o->threads;
    r.timing = o->timing != 0;
    r.kernel_events = o->timing >= 2;
    r.host_recon = (o->flags & ES_FLAG_HOST_RECON) != 0;
    r.step_lift = (o->flags & ES_FLAG_STEP_LIFT) != 0;
    r.one_stream = (o->flags & ES_FLAG_ONE_STREAM) != 0;
  }
  return r;
}

struct Timer {
  bool on;
  cudaStream_t st;
  cudaEvent_t ev[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
  Timer(bool on_, cudaStream_t s) : on(on_), st(s) {
    if (on)
      for (auto& e : ev) cudaEventCreate(&e);
  }
  ~Timer() {
    for (auto& e : ev)
      if (e) cudaEventDestroy(e);
  }
  void mark(int i) {
    if (on) cudaEventRecord(ev[i], st);
  }
  double between(int a, int b) {
    float ms = 0.f;
    if (on && cudaEventElapsedTime(&ms, ev[a], ev[b]) == cudaSuccess) return ms;
    return 0.0;
  }
};

struct SolveLayout {
  size_t A, b, B, good, stats, work, total;
};
SolveLayout solve_layout(int64_t n, int64_t c, bool stage_inputs) {
  Layout L;
  SolveLayout s;
  const int64_t ld = padded_ld(n);
  s.A = stage_inputs ? L.add((size_t)n * n * 8) : 0;
  s.b = stage_inputs ? L.add((size_t)n * c * 8) : 0;
  s.B = L.add((size_t)kNumPrimes * n * ld);
  s.good = L.add(kNumPrimes);
  s.stats = L.add(stats_scratch_bytes(n));
  size_t inv = inverse_scratch_bytes(n), lift = lift_scratch_bytes(n, c, kNumPrimes, true);
  s.work = L.add(inv > lift ? inv : lift);
  s.total = L.total;
  return s;
}

es_status check_args(int64_t n, int64_t c) {
  if (n < 1 || c < 1) return ES_ERR_ARG;
  if (n > (int64_t(1) << 17)) return ES_ERR_RANGE;
  if (c > (int64_t(1) << 24) || n * c > (int64_t(1) << 34)) return ES_ERR_ARG;
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) {
    cudaGetLastError();
    return ES_ERR_NODEVICE;
  }
  return ES_OK;
}

es_status solve_impl(const int64_t* A_in, const int64_t* b_in, bool host_inputs, int64_t n, int64_t c,
                     const es_options* opt, es_solution** out) {
  auto t_start = std::chrono::steady_clock::now();
  const int64_t launches0 = launch_count();
  if (!out || !A_in || !b_in) return ES_ERR_ARG;
  *out = nullptr;
  ES_CHECK(check_args(n, c));
  const Options o = read_options(opt);
  DeviceState& dev = g_dev[current_device()];
  std::lock_guard<std::mutex> lock(dev.mu);
  cudaStream_t st = (cudaStream_t)resolve_stream(o.stream);
  const int64_t ld = padded_ld(n), nc = n * c;
  (void)ld;

  SolveLayout SL = solve_layout(n, c, host_inputs);
  char* ws = nullptr;
  ES_CHECK(workspace_get(SL.total, o.max_bytes, o.fault == ES_FAULT_NOMEM, &ws));
  const int64_t* A = A_in;
  const int64_t* b = b_in;
  Timer tm(o.timing, st);
  tm.mark(0);
  if (host_inputs) {
    ES_CHECK(cuda_status(cudaMemcpyAsync(ws + SL.A, A_in, (size_t)n * n * 8, cudaMemcpyHostToDevice, st), "A H2D"));
    ES_CHECK(cuda_status(cudaMemcpyAsync(ws + SL.b, b_in, (size_t)nc * 8, cudaMemcpyHostToDevice, st), "b H2D"));
    A = reinterpret_cast<const int64_t*>(ws + SL.A);
    b = reinterpret_cast<const int64_t*>(ws + SL.b);
  }
  // range check and Hadamard terms
  Stats stats;
  ES_CHECK(compute_stats(A, b, n, c, ws + SL.stats, st, &stats));
  if (!in_range(n, stats.max_abs_a)) return ES_ERR_RANGE;
  if (o.fault == ES_FAULT_RESIDUES) {
    set_last_error("injected fault: residues");
    return ES_ERR_CUDA;
  }
  if (stats.zero_row) return ES_SINGULAR;  // det A = 0
  tm.mark(1);
  // batched modular inverse
  int8_t* B = reinterpret_cast<int8_t*>(ws + SL.B);
  uint8_t* good_dev = reinterpret_cast<uint8_t*>(ws + SL.good);
  bool inverse_split = false;
  ES_CHECK(run_inverse(A, n, B, good_dev, ws + SL.work, st, !o.one_stream, &inverse_split));
  uint8_t good[kNumPrimes];
  ES_CHECK(cuda_status(cudaMemcpyAsync(good, good_dev, kNumPrimes, cudaMemcpyDeviceToHost, st), "good D2H"));
  ES_CHECK(cuda_status(cudaStreamSynchronize(st), "inverse sync"));
  tm.mark(2);
  if (o.fault == ES_FAULT_INVERSE) {
    set_last_error("injected fault: inverse");
    return ES_ERR_CUDA;
  }
  int E = 0;
  for (int j = 0; j < kNumPrimes; ++j) E += good[j] ? 1 : 0;
  if (E == 0) return ES_SINGULAR;  // every prime divides det A (det A = 0 over Q)
  int64_t num_bits, den_bits;
  int32_t m;
  plan_from_stats(stats, good, &num_bits, &den_bits, &m);
  // lift
  const size_t dbytes = (size_t)m * (size_t)nc * kDigitLimbs * 8;
  {
    void* p = dev.digits;
    size_t cap_left = o.max_bytes ? (o.max_bytes > SL.total ? o.max_bytes - SL.total : 1) : 0;
    ES_CHECK(grow_device(&p, &dev.digits_size, dbytes, cap_left, false));
    dev.digits = (uint64_t*)p;
  }
  if (o.fault == ES_FAULT_LIFT) {
    set_last_error("injected fault: lift wait timed out");
    return ES_ERR_TIMEOUT;
  }
  KernelTiming kt;
  kt.events = o.kernel_events;
  int32_t mp = 0;
  const bool on_device = !o.host_recon && recon_device_applicable(n, m, good, num_bits, den_bits, stats, &mp);
  std::unique_ptr<ReconPlan, void (*)(ReconPlan*)> rplan(nullptr, recon_plan_free);
  // c == 1: the fused lift hands the sampled components' digits to the host
  // as it forms them, so that their sums are ready when it ends
  DigitStream ds;
  int ns = 0;
  std::vector<std::vector<uint64_t>> pre;
  if (on_device && c == 1 && !o.step_lift) {
    const std::vector<int64_t> sk = recon_samples(n, c, o.threads);
    const size_t words = (size_t)m * kStreamRows * kStreamWords;
    if (sk.size() <= (size_t)kStreamRows && stream_buffer(dev, words)) {
      std::memset(dev.hstream, 0, words * 8);
      ds.host = dev.hstream;
      void* dp = nullptr;
      if (cudaHostGetDevicePointer(&dp, dev.hstream, 0) == cudaSuccess) {
        ds.dev = static_cast<uint64_t*>(dp);
        ns = (int)sk.size();
        for (int q = 0; q < ns; ++q) ds.rows[q] = sk[(size_t)q];
      } else {
        cudaGetLastError();
        ds.host = nullptr;
      }
    }
  }
  {
    LiftRun lr;
    ES_CHECK(run_lift_start(A, b, n, c, B, good, m, dev.digits, stats.max_abs_a, ws + SL.work, st, &kt,
                            !o.step_lift, &lr, o.fault == ES_FAULT_LIFT_WAIT, ns ? &ds : nullptr));
    // while the GPU lifts: the reconstruction's digit-independent constants
    // and (fused lift) the streamed samples' sums
    es_status ps = ES_OK;
    if (on_device) {
      const bool streamed = ns && lr.fused &&
                            cudaEventRecord(dev.lift_done, st) == cudaSuccess;
      ReconPlan* rp = nullptr;
      ps = recon_prepare_overlapped(n, c, m, mp, good, num_bits, den_bits, stats, o.threads,
                                    streamed ? &ds : nullptr, ns, dev.lift_done, &rp, &pre);
      rplan.reset(rp);
    }
    ES_CHECK(run_lift_finish(&lr));
    ES_CHECK(ps);
  }
  tm.mark(3);
  if (o.fault == ES_FAULT_RECON) {
    set_last_error("injected fault: reconstruction");
    return ES_ERR_INTERNAL;
  }
  es_solution* sol = new (std::nothrow) es_solution;
  if (!sol) return ES_ERR_NOMEM;
  es_status rs = ES_OK;
  auto t_rec = std::chrono::steady_clock::now();
  if (on_device) {
    // numerators on the GPU from the low m' digits; sampled denominators on the host
    tm.mark(4);
    const size_t rbytes = recon_device_bytes(nc, mp, good, num_bits, den_bits);
    void* p = dev.recon;
    rs = grow_device(&p, &dev.recon_size, rbytes, 0, false);
    dev.recon = (char*)p;
    t_rec = std::chrono::steady_clock::now();
    if (rs == ES_OK)
      rs = reconstruct_device(rplan.get(), dev.digits, o.threads, dev.recon, dev.recon_size, st, &sol->s, &pre);
  } else {
    // all digits to the host, reconstruction on the host
    if (dbytes > dev.hdigits_size) {
      if (dev.hdigits) cudaFreeHost(dev.hdigits);
      dev.hdigits = nullptr;
      dev.hdigits_size = 0;
      if (cudaMallocHost((void**)&dev.hdigits, dbytes) != cudaSuccess) {
        cudaGetLastError();
        dev.hdigits = nullptr;
        delete sol;
        return ES_ERR_NOMEM;
      }
      dev.hdigits_size = dbytes;
    }
    rs = cuda_status(cudaMemcpyAsync(dev.hdigits, dev.digits, dbytes, cudaMemcpyDeviceToHost, st), "digits D2H");
    tm.mark(4);
    if (rs == ES_OK) rs = cuda_status(cudaStreamSynchronize(st), "digits sync");
    t_rec = std::chrono::steady_clock::now();
    if (rs == ES_OK) rs = reconstruct(dev.hdigits, n, c, m, good, num_bits, den_bits, o.threads, false, &sol->s);
  }
  if (rs != ES_OK) {
    delete sol;
    return rs;
  }
  auto t_end = std::chrono::steady_clock::now();
  Solution& S = sol->s;
  S.ms[0] = tm.between(0, 1);
  S.ms[1] = tm.between(1, 2);
  S.ms[2] = tm.between(2, 3);
  S.ms[3] = tm.between(3, 4);
  S.ms[4] = std::chrono::duration<double, std::milli>(t_end - t_rec).count();
  S.ms[5] = std::chrono::duration<double, std::milli>(t_end - t_start).count();
  S.m = m;
  S.primes_used = E;
  S.launches = launch_count() - launches0;
  S.inverse_split = inverse_split;
  S.top = kt;
  *out = sol;
  return ES_OK;
}

}  // namespace
// ------------------------------------------------------------ limb blocks
// Result limbs leave the device once per solve into a buffer the caller may
// keep.  A fresh pageable buffer costs page faults (and a staged copy); the
// blocks here are page-locked when a device is present, so the numerator
// kernel can write them directly, and recycled: a freed buffer's block waits
// in a short list for the next solve.  Blocks above kPinMax bytes are plain
// allocations, and the list holds at most kKeep blocks and kKeepBytes bytes.
namespace {
constexpr size_t kPinMax = size_t(8) << 30;
constexpr size_t kKeep = 4;
constexpr size_t kKeepBytes = size_t(8) << 30;
struct Block {
  uint64_t* p;
  size_t cap;
  bool pinned;
};
std::mutex g_blk_mu;
std::vector<Block> g_blocks;
size_t g_kept_bytes = 0;

Block block_new(size_t count) {
  Block b{nullptr, count, false};
  if (count * 8 <= kPinMax) {
    void* p = nullptr;
    if (cudaMallocHost(&p, count * 8) == cudaSuccess) {
      b.p = static_cast<uint64_t*>(p);
      b.pinned = true;
      return b;
    }
    cudaGetLastError();  // no device: fall back to a plain allocation
  }
  b.p = new (std::nothrow) uint64_t[count];
  return b;
}
void block_delete(const Block& b) {
  if (b.pinned)
    cudaFreeHost(b.p);
  else
    delete[] b.p;
}
}  // namespace

void LimbBuffer::resize(size_t count) {
  if (count <= cap_) {
    n_ = count;
    return;
  }
  release();
  Block b{nullptr, 0, false};
  {
    std::lock_guard<std::mutex> lk(g_blk_mu);
    size_t best = g_blocks.size();
    for (size_t i = 0; i < g_blocks.size(); ++i)
      if (g_blocks[i].cap >= count && (best == g_blocks.size() || g_blocks[i].cap < g_blocks[best].cap)) best = i;
    if (best < g_blocks.size()) {
      b = g_blocks[best];
      g_kept_bytes -= b.cap * 8;
      g_blocks.erase(g_blocks.begin() + (std::ptrdiff_t)best);
    }
  }
  if (!b.p) b = block_new(count);
  if (!b.p) throw std::bad_alloc();
  p_ = b.p;
  cap_ = b.cap;
  n_ = count;
  pinned_ = b.pinned;
}

void LimbBuffer::release() {
  if (!p_) return;
  Block b{p_, cap_, pinned_};
  p_ = nullptr;
  n_ = cap_ = 0;
  pinned_ = false;
  if (b.cap * 8 <= kPinMax) {
    // keep it, evicting smaller kept blocks while the list is full: a large
    // page-locked block costs far more to make again than a small one
    std::vector<Block> evict;
    bool kept = false;
    {
      std::lock_guard<std::mutex> lk(g_blk_mu);
      while (g_blocks.size() >= kKeep || g_kept_bytes + b.cap * 8 > kKeepBytes) {
        size_t small = 0;
        for (size_t i = 1; i < g_blocks.size(); ++i)
          if (g_blocks[i].cap < g_blocks[small].cap) small = i;
        if (g_blocks.empty() || g_blocks[small].cap >= b.cap) break;
        evict.push_back(g_blocks[small]);
        g_kept_bytes -= g_blocks[small].cap * 8;
        g_blocks.erase(g_blocks.begin() + (std::ptrdiff_t)small);
      }
      if (g_blocks.size() < kKeep && g_kept_bytes + b.cap * 8 <= kKeepBytes) {
        g_blocks.push_back(b);
        g_kept_bytes += b.cap * 8;
        kept = true;
      }
    }
    for (const Block& e : evict) block_delete(e);
    if (kept) return;
  }
  block_delete(b);
}

}  // namespace es

// ------------------------------------------------------------ C ABI
extern "C" {

es_status es_solve(const int64_t* A, const int64_t* b, int64_t n, int64_t c, const es_options* opt,
                   es_solution** out) {
  return es::solve_impl(A, b, true, n, c, opt, out);
}

es_status es_solve_device(const int64_t* A_dev, const int64_t* b_dev, int64_t n, int64_t c,
                          const es_options* opt, es_solution** out) {
  return es::solve_impl(A_dev, b_dev, false, n, c, opt, out);
}

es_status es_solution_shape(const es_solution* s, int64_t* n, int64_t* c, int64_t* limbs) {
  if (!s) return ES_ERR_ARG;
  if (n) *n = s->s.n;
  if (c) *c = s->s.c;
  if (limbs) *limbs = s->s.limbs;
  return ES_OK;
}

es_status es_solution_export(const es_solution* s, uint64_t* num, uint64_t* den) {
  if (!s) return ES_ERR_ARG;
  if (num) std::memcpy(num, s->s.num.data(), s->s.num.size() * 8);
  if (den) std::memcpy(den, s->s.den.data(), s->s.den.size() * 8);
  return ES_OK;
}

es_status es_solution_data(const es_solution* s, const uint64_t** num, const uint64_t** den) {
  if (!s) return ES_ERR_ARG;
  if (num) *num = s->s.num.data();
  if (den) *den = s->s.den.data();
  return ES_OK;
}

es_status es_solution_phase_ms(const es_solution* s, double* ms, int32_t* m, int32_t* primes_used) {
  if (!s) return ES_ERR_ARG;
  if (ms)
    for (int i = 0; i < ES_NUM_PHASES; ++i) ms[i] = s->s.ms[i];
  if (m) *m = s->s.m;
  if (primes_used) *primes_used = s->s.primes_used;
  return ES_OK;
}

es_status es_solution_kernels(const es_solution* s, int64_t* launches, int64_t* top_launches, double* top_ms,
                              double* top_bytes_per_launch) {
  if (!s) return ES_ERR_ARG;
  if (launches) *launches = s->s.launches;
  if (top_launches) *top_launches = s->s.top.launches;
  if (top_ms) *top_ms = s->s.top.ms;
  if (top_bytes_per_launch) *top_bytes_per_launch = s->s.top.bytes_per_launch;
  return ES_OK;
}

const char* es_solution_top_kernel(const es_solution* s) { return s && s->s.top.name ? s->s.top.name : ""; }

int32_t es_solution_inverse_split(const es_solution* s) { return s && s->s.inverse_split ? 1 : 0; }

void es_solution_free(es_solution* s) { delete s; }

const char* es_status_string(es_status st) {
  switch (st) {
    case ES_OK: return "ok";
    case ES_SINGULAR: return "singular: A is singular over the rationals";
    case ES_ERR_ARG: return "invalid argument";
    case ES_ERR_RANGE: return "out of range: need n <= 2^17 and n * max|A_ij| < 2^63";
    case ES_ERR_CUDA: return "CUDA error";
    case ES_ERR_NOMEM: return "out of memory";
    case ES_ERR_TIMEOUT: return "timed out";
    case ES_ERR_INTERNAL: return "internal self-check failed";
    case ES_ERR_NODEVICE: return "no CUDA device";
  }
  return "unknown status";
}

const char* es_last_error(void) { return es::g_last_error.c_str(); }

es_status es_release_workspace(void) {
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) {
    cudaGetLastError();
    return ES_ERR_NODEVICE;
  }
  es::DeviceState& d = es::g_dev[es::current_device()];
  std::lock_guard<std::mutex> lock(d.mu);
  if (d.ws) cudaFree(d.ws);
  if (d.digits) cudaFree(d.digits);
  if (d.hdigits) cudaFreeHost(d.hdigits);
  if (d.recon) cudaFree(d.recon);
  d.recon = nullptr;
  d.recon_size = 0;
  if (d.hstream) cudaFreeHost(d.hstream);
  d.hstream = nullptr;
  d.hstream_words = 0;
  d.ws = nullptr;
  d.digits = nullptr;
  d.hdigits = nullptr;
  d.ws_size = d.digits_size = d.hdigits_size = 0;
  es::release_inverse_partitions(es::current_device());
  return ES_OK;
}

int32_t es_version(void) { return 1; }

es_status es_inverse_mod_device(const int64_t* A_dev, int64_t n, int8_t* B_dev, uint8_t* good_dev,
                                void* stream) {
  if (!A_dev || !B_dev || !good_dev) return ES_ERR_ARG;
  ES_CHECK(es::check_args(n, 1));
  es::DeviceState& dev = es::g_dev[es::current_device()];
  std::lock_guard<std::mutex> lock(dev.mu);
  cudaStream_t st = (cudaStream_t)es::resolve_stream(stream);
  size_t need = es::stats_scratch_bytes(n) + 256 + es::inverse_scratch_bytes(n);
  char* ws = nullptr;
  ES_CHECK(es::workspace_get(need, 0, false, &ws));
  es::Stats stats;
  // range statistics of A alone (no columns of b)
  ES_CHECK(es::compute_stats(A_dev, A_dev, n, 0, ws, st, &stats));
  if (!es::in_range(n, stats.max_abs_a)) return ES_ERR_RANGE;
  size_t off = (es::stats_scratch_bytes(n) + 255) / 256 * 256;
  ES_CHECK(es::run_inverse(A_dev, n, B_dev, good_dev, ws + off, st));
  return es::cuda_status(cudaStreamSynchronize(st), "es_inverse_mod_device");
}

es_status es_plan_device(const int64_t* A_dev, const int64_t* b_dev, int64_t n, int64_t c, const uint8_t* good,
                         int64_t* num_bits, int64_t* den_bits, int32_t* m, void* stream) {
  if (!A_dev || !b_dev || !good || !num_bits || !den_bits || !m) return ES_ERR_ARG;
  ES_CHECK(es::check_args(n, c));
  es::DeviceState& dev = es::g_dev[es::current_device()];
  std::lock_guard<std::mutex> lock(dev.mu);
  cudaStream_t st = (cudaStream_t)es::resolve_stream(stream);
  char* ws = nullptr;
  ES_CHECK(es::workspace_get(es::stats_scratch_bytes(n), 0, false, &ws));
  es::Stats stats;
  ES_CHECK(es::compute_stats(A_dev, b_dev, n, c, ws, st, &stats));
  if (!es::in_range(n, stats.max_abs_a)) return ES_ERR_RANGE;
  int E = 0;
  for (int j = 0; j < es::kNumPrimes; ++j) E += good[j] ? 1 : 0;
  if (E == 0) return ES_ERR_ARG;
  es::plan_from_stats(stats, good, num_bits, den_bits, m);
  return ES_OK;
}

es_status es_lift_device(const int64_t* A_dev, const int64_t* b_dev, int64_t n, int64_t c, const int8_t* B_dev,
                         const uint8_t* good, int32_t m, uint64_t* digits_dev, void* stream) {
  if (!A_dev || !b_dev || !B_dev || !good || !digits_dev || m < 1) return ES_ERR_ARG;
  ES_CHECK(es::check_args(n, c));
  int E = 0;
  for (int j = 0; j < es::kNumPrimes; ++j) E += good[j] ? 1 : 0;
  if (E == 0) return ES_ERR_ARG;
  es::DeviceState& dev = es::g_dev[es::current_device()];
  std::lock_guard<std::mutex> lock(dev.mu);
  cudaStream_t st = (cudaStream_t)es::resolve_stream(stream);
  size_t soff = (es::stats_scratch_bytes(n) + 255) / 256 * 256;
  char* ws = nullptr;
  ES_CHECK(es::workspace_get(soff + es::lift_scratch_bytes(n, c, es::kNumPrimes, true), 0, false, &ws));
  es::Stats stats;
  ES_CHECK(es::compute_stats(A_dev, b_dev, n, c, ws, st, &stats));
  if (!es::in_range(n, stats.max_abs_a)) return ES_ERR_RANGE;
  return es::run_lift(A_dev, b_dev, n, c, B_dev, good, m, digits_dev, stats.max_abs_a, ws + soff, st);
}

}  // extern "C"
