// apr_qgemm_noalloc: the tensor-core GEMM entry point without any device
// allocation, for callers that cannot allocate device memory.
//
// apr_qgemm takes its fp16 copy of the activations from a memory pool that the
// library creates and grows on demand. Some callers cannot allow that: a
// serving process that reserves nearly all of HBM up front (weights and a
// preallocated KV-cache arena) and treats any later device allocation as a
// fault, a runtime whose allocation happens once at start-up under its own
// allocator, or a real-time path that must not stall on, or fail in, an
// allocator after initialisation. For them, this file holds the scratch as a
// fixed module-scope device array: it is created when the library's module is
// loaded on a device and lives until the process exits, and no call here
// allocates or frees device memory.

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include <cuda_runtime.h>

#include "apr_qgemm.h"
#include "apr_internal.h"

namespace apr {
namespace {

// Capacity of the fixed scratch, in fp16 values of the activation copy: T * k
// must not exceed it (16 MiB of device memory per GPU that loads the library).
constexpr size_t kNoAllocScratchElems = size_t(APR_NOALLOC_MAX_TK);

__device__ __align__(256) uint16_t g_noalloc_x16[kNoAllocScratchElems];

struct NoAllocDevice {
  std::atomic<bool> ready{false};
  uint16_t* scratch = nullptr;  // device address of g_noalloc_x16
  unsigned* status = nullptr;   // device address of the library's status word
};
NoAllocDevice g_na[64];
std::mutex g_na_mu;

// Per device, with that device current: check it, then look up the device
// addresses of the scratch array and of the status word. In host code the
// array's name only stands in for the symbol; the kernels need the address
// cudaGetSymbolAddress returns. Only a successful lookup is kept: a failed
// one (for instance made during a stream capture, which the header warns
// against) is tried again on the next call.
int setup(NoAllocDevice** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return set_error(APR_E_DEVICE, "no usable CUDA device");
  }
  NoAllocDevice& st = g_na[dev];
  if (!st.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_na_mu);
    if (!st.ready.load(std::memory_order_relaxed)) {
      cudaDeviceProp prop;
      if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess || prop.major != 10 || prop.minor != 3) {
        cudaGetLastError();
        return set_error(APR_E_DEVICE, "device is not a compute capability 10.3 GPU (GB300)");
      }
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_x16);
      if (e != cudaSuccess) {
        cudaGetLastError();
        return set_error(APR_E_DEVICE, "looking up the fixed scratch failed (retried on the next call)");
      }
      unsigned* status = status_word_address();
      if (!status) return set_error(APR_E_DEVICE, "looking up the status word failed (retried on the next call)");
      st.scratch = static_cast<uint16_t*>(p);
      st.status = status;
      st.ready.store(true, std::memory_order_release);
    }
  }
  *out = &st;
  return APR_OK;
}

}  // namespace
}  // namespace apr

extern "C" int apr_qgemm_noalloc(int qtype, const void* W, int n, int k, const float* X, int T, float* Y,
                                 const float* residual, apr_stream_t stream) {
  using namespace apr;
  int rc = check_gemm_args(qtype, W, n, k, X, T, Y, residual);
  if (rc == 1) return APR_OK;
  if (rc != APR_OK) return rc;
  if (k % 256 != 0) return set_error(APR_E_INVAL, "apr_qgemm_noalloc needs k % 256 == 0");
  if ((size_t)T * (size_t)k > kNoAllocScratchElems) {
    char msg[160];
    snprintf(msg, sizeof msg, "apr_qgemm_noalloc: T*k = %zu exceeds its fixed scratch of %zu fp16 values",
             (size_t)T * (size_t)k, kNoAllocScratchElems);
    return set_error(APR_E_INVAL, msg);
  }
  NoAllocDevice* st = nullptr;
  rc = setup(&st);
  if (rc != APR_OK) return rc;
  const cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = launch_x_to_f16(X, st->scratch, (size_t)T * (size_t)k, s);
  if (e != cudaSuccess) return set_error(APR_E_LAUNCH, cudaGetErrorString(e));
  char msg[256] = "";
  const GemmPlan plan = plan_gemm_tc(n, k, T, false);
  // the fixed array also covers kMinXRows rows of X when they fit
  const int xr = (size_t)padded_x_rows(T) * (size_t)k <= kNoAllocScratchElems ? padded_x_rows(T) : T;
  if (launch_gemm_tc(plan, qtype, W, nullptr, n, k, st->scratch, T, Y, n, residual, st->status, s, msg, sizeof msg,
                     kEarlyWR, xr) != 0)
    return set_error(APR_E_LAUNCH, msg);
  return APR_OK;
}
