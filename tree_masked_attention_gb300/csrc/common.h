// Internal helpers shared by the library's translation units (host side).
#pragma once
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <string>

#include "tree_attn.h"

namespace tree {

// Records a failure for tree_last_error() on this host thread and returns `status`.
int fail(int status, const char* fmt, ...);
void clear_error();

// Device address of this device's error word (one int per device, in status.cu).
// Kernels OR a TREE_ERR_* code into it; tree_check_device_status() reads and clears it.
int* device_error_word();

// Counts one kernel launch (reported by tree_launch_count()).
void count_launch();

// CUDA-event brackets around a call's main kernel, when tree_kernel_timing(1) is on:
// 0 = attention forward, 1 = attention backward, 2 = conv1d forward, 3 = conv1d backward
// (its kernel and the dw / dbias reduction); tree_kernel_last_ms reads them.
constexpr int kTimedKernels = 4;
void timing_begin(int which, void* stream);
void timing_end(int which, void* stream);

// Opts `func` in to `bytes` of dynamic shared memory on the current device. The attribute
// is per device, so the first call on each device sets it; later calls only look it up.
int smem_opt_in(const void* func, int bytes);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace tree

// Return TREE_ERR_CUDA from the enclosing function if a CUDA call failed.
#define TREE_CUDA_TRY(expr)                                                              \
  do {                                                                                   \
    cudaError_t e_ = (expr);                                                             \
    if (e_ != cudaSuccess)                                                               \
      return ::tree::fail(TREE_ERR_CUDA, "%s failed: %s (%s:%d)", #expr,                \
                          cudaGetErrorString(e_), __FILE__, __LINE__);                   \
  } while (0)

// After a kernel launch: report a launch-configuration error.
#define TREE_LAUNCH_CHECK(name)                                                          \
  do {                                                                                   \
    ::tree::count_launch();                                                              \
    cudaError_t e_ = cudaGetLastError();                                                 \
    if (e_ != cudaSuccess)                                                               \
      return ::tree::fail(TREE_ERR_CUDA, "launch of %s failed: %s", name,               \
                          cudaGetErrorString(e_));                                       \
  } while (0)
