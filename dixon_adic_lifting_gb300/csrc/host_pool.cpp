// Process-wide pool of host threads for the reconstruction stage.
//
// Starting and joining a thread costs tens of microseconds, which a
// reconstruction of a few milliseconds cannot afford for each of its
// parallel loops.  The workers are started once; after a job they poll for
// the next one for a short while and then sleep on a condition variable.
//
// A job hands out indices from one atomic word that also carries the job's
// number, and an index is taken by compare-and-swap only while the number
// matches.  A new job retags that word before it publishes its function and
// count, so a worker that arrives after its job has ended (or reads the next
// job's function) cannot take or skip an index of another job.  The
// caller takes indices too and returns once every index has completed.
// Calls from inside a job run inline on the calling thread.
#include <atomic>
#include <chrono>
#include <condition_variable>
#include <functional>
#include <mutex>
#include <thread>
#include <vector>

#include "recon_common.h"

namespace es {
namespace {

thread_local bool t_in_job = false;

class HostPool {
 public:
  explicit HostPool(int workers) {
    for (int i = 0; i < workers; ++i) threads_.emplace_back([this] { worker(); });
  }
  ~HostPool() {
    {
      std::lock_guard<std::mutex> lk(mu_);
      quit_.store(true, std::memory_order_release);
      gen_.fetch_add(1, std::memory_order_acq_rel);
    }
    cv_.notify_all();
    for (auto& t : threads_) t.join();
  }
  int workers() const { return (int)threads_.size(); }

  void run(int64_t count, int width, const std::function<void(int64_t)>& fn) {
    std::lock_guard<std::mutex> one(run_mu_);
    const uint64_t g = gen_.load(std::memory_order_relaxed) + 1;
    // the dispenser changes hands first: a worker that sees this job's
    // function or count (acquire) sees the new tag as well
    next_.store(tag(g), std::memory_order_relaxed);
    done_.store(0, std::memory_order_relaxed);
    count_.store(count, std::memory_order_release);
    fn_.store(&fn, std::memory_order_release);
    const int64_t helpers = (int64_t)width - 1 < count - 1 ? (int64_t)width - 1 : count - 1;
    slots_.store((int)helpers, std::memory_order_relaxed);
    {
      std::lock_guard<std::mutex> lk(mu_);
      gen_.store(g, std::memory_order_release);
    }
    cv_.notify_all();
    take(g, fn, count);
    int spins = 0;
    while (done_.load(std::memory_order_acquire) < count)
      if (++spins > 64) std::this_thread::yield();
  }

 private:
  static uint64_t tag(uint64_t g) { return (g & 0xFFFFFFull) << 40; }
  static constexpr uint64_t kIndexMask = (1ull << 40) - 1;

  // take and run indices of job g while it lasts
  void take(uint64_t g, const std::function<void(int64_t)>& fn, int64_t count) {
    const bool outer = t_in_job;
    t_in_job = true;
    for (;;) {
      uint64_t v = next_.load(std::memory_order_acquire);
      if ((v & ~kIndexMask) != tag(g)) break;
      const int64_t i = (int64_t)(v & kIndexMask);
      if (i >= count) break;
      if (!next_.compare_exchange_weak(v, v + 1, std::memory_order_acq_rel)) continue;
      fn(i);
      done_.fetch_add(1, std::memory_order_acq_rel);
    }
    t_in_job = outer;
  }

  void worker() {
    uint64_t seen = 0;
    for (;;) {
      uint64_t g;
      const auto t0 = std::chrono::steady_clock::now();
      int spins = 0;
      while ((g = gen_.load(std::memory_order_acquire)) == seen) {
        if (++spins < 1024) continue;
        spins = 0;
        if (std::chrono::steady_clock::now() - t0 < std::chrono::milliseconds(2)) {
          std::this_thread::yield();
          continue;
        }
        std::unique_lock<std::mutex> lk(mu_);
        cv_.wait(lk, [&] { return gen_.load(std::memory_order_acquire) != seen; });
      }
      seen = g;
      if (quit_.load(std::memory_order_acquire)) return;
      if (slots_.fetch_sub(1, std::memory_order_acq_rel) <= 0) continue;
      const std::function<void(int64_t)>* fn = fn_.load(std::memory_order_acquire);
      const int64_t count = count_.load(std::memory_order_acquire);
      take(g, *fn, count);  // stops at once if the job is no longer g
    }
  }

  std::vector<std::thread> threads_;
  std::mutex run_mu_;  // one job at a time
  std::mutex mu_;
  std::condition_variable cv_;
  std::atomic<bool> quit_{false};
  std::atomic<uint64_t> gen_{0};
  std::atomic<uint64_t> next_{0};
  std::atomic<int64_t> done_{0};
  std::atomic<int> slots_{0};
  std::atomic<const std::function<void(int64_t)>*> fn_{nullptr};
  std::atomic<int64_t> count_{0};
};

HostPool& pool() {
  static HostPool p(std::max(0, (int)std::thread::hardware_concurrency() - 1));
  return p;
}

}  // namespace

void host_parallel_for(int64_t count, int threads, const std::function<void(int64_t)>& fn) {
  if (count <= 0) return;
  int width = threads > 0 ? threads : (int)std::thread::hardware_concurrency();
  if (width > count) width = (int)count;
  if (width <= 1 || t_in_job) {
    for (int64_t i = 0; i < count; ++i) fn(i);
    return;
  }
  HostPool& p = pool();
  if (p.workers() == 0) {
    for (int64_t i = 0; i < count; ++i) fn(i);
    return;
  }
  p.run(count, width, fn);
}

}  // namespace es
