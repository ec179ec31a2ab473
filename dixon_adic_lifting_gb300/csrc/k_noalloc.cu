// Batched modular inverse that allocates nothing.
//
// Some callers cannot call cudaMalloc: code embedded in a framework whose
// caching allocator has already reserved (nearly) all device memory, where a
// foreign cudaMalloc fails; and latency-bound serving loops that must not
// stall, since cudaFree synchronizes the whole device and cudaMalloc may.
// For them, es_inverse_mod_device_noalloc runs the same kernels as
// es_inverse_mod_device with its working memory (the [53][n][ld] residue
// matrices, pivot bookkeeping and panel staging) taken from the fixed array
// below instead of the library's grown workspace.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its kNoAllocScratchBytes until the process exits.  Host code
// cannot use the array's name as a device address (on the host it names a
// shadow variable), so the address is fetched with cudaGetSymbolAddress once
// per device, with that device current, the first time the entry point runs
// on it.  That first call should therefore come before any stream capture.
// Every call synchronises the stream it was given before returning.  The
// address is kept for the life of the process, so a caller that resets a
// device (cudaDeviceReset, which may reload the module elsewhere) must not
// call the entry point on that device again.
#include <cuda_runtime.h>

#include <mutex>

#include "es_common.cuh"
#include "es_internal.h"

namespace es {

// Working memory for n <= kNoAllocMaxN: inverse_scratch_bytes(256) is
// 4,464,128 bytes (W 3.47 MB, U^T of two panels 0.87 MB, pivots 0.11 MB,
// flags).
constexpr int64_t kNoAllocMaxN = 256;
constexpr size_t kNoAllocScratchBytes = size_t(4608) << 10;  // 4.5 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kMaxDev = 64;
std::mutex g_noalloc_mu;                 // one call at a time: all calls share the array
void* g_noalloc_ptr[kMaxDev] = {nullptr};  // device address of the array, per device
}  // namespace

}  // namespace es

extern "C" es_status es_inverse_mod_device_noalloc(const int64_t* A_dev, int64_t n, int8_t* B_dev,
                                                   uint8_t* good_dev, void* stream) {
  if (!A_dev || !B_dev || !good_dev || n < 1) return ES_ERR_ARG;
  if (n > es::kNoAllocMaxN || es::inverse_scratch_bytes(n) > es::kNoAllocScratchBytes) {
    es::set_last_error("es_inverse_mod_device_noalloc: n exceeds the no-allocation maximum of 256");
    return ES_ERR_RANGE;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= es::kMaxDev) {
    cudaGetLastError();
    return ES_ERR_NODEVICE;
  }
  std::lock_guard<std::mutex> lock(es::g_noalloc_mu);
  if (!es::g_noalloc_ptr[dev]) {
    void* p = nullptr;
    ES_CHECK(es::cuda_status(cudaGetSymbolAddress(&p, es::g_noalloc_scratch), "cudaGetSymbolAddress"));
    es::g_noalloc_ptr[dev] = p;
  }
  cudaStream_t st = (cudaStream_t)stream;  // NULL: the legacy default stream (no stream is created)
  // one stream, no SM partitions: this entry point creates nothing
  ES_CHECK(es::run_inverse(A_dev, n, B_dev, good_dev, static_cast<char*>(es::g_noalloc_ptr[dev]), st, false));
  return es::cuda_status(cudaStreamSynchronize(st), "es_inverse_mod_device_noalloc");
}
