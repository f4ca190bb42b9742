// Host-side helpers shared by the C-ABI translation units: status codes,
// the thread-local last-error message and CUDA error mapping.
#pragma once

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
