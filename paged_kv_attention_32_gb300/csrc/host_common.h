// Host-side helpers shared by the C-ABI translation units: status codes,
// the thread-local last-error message and CUDA error mapping.
#pragma once

#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <string>

#include <cuda_runtime.h>

#include "pka.h"

namespace pka {

// Records `fmt` as the calling thread's last error and returns `code`.
int fail(int code, const char* fmt, ...);

// Clears the calling thread's last error.
void clear_error();

// Maps a CUDA runtime error to PKA_ERR_CUDA with a message naming `what`.
// Raises a kernel's dynamic shared memory limit once per device: `done` is the
// calling launcher's own bit set (devices 0-63; a higher device sets it on
// every launch).  The attribute stays set for the life of the process.
template <typename Kernel>
inline cudaError_t set_smem_once(Kernel kern, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

inline int cuda_fail(cudaError_t e, const char* what) {
  return fail(PKA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace pka

#define PKA_CHECK_ARG(cond, ...)                          \
  do {                                                    \
    if (!(cond)) return ::pka::fail(PKA_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)

#define PKA_CUDA_TRY(expr, what)                          \
  do {                                                    \
    cudaError_t _e = (expr);                              \
    if (_e != cudaSuccess) return ::pka::cuda_fail(_e, what); \
  } while (0)
