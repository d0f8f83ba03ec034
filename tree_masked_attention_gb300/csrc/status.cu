// Error reporting: the thread-local host message and the per-device error word.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <tuple>
#include <vector>

#include "common.h"
#include "sm100.cuh"

namespace tree {

static thread_local std::string g_msg;

int fail(int status, const char* fmt, ...) {
  char buf[1024];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_msg = buf;
  return status;
}

void clear_error() { g_msg.clear(); }

static std::atomic<uint64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// One error word per device; a kernel ORs a TREE_ERR_* code into it.
static __device__ int g_device_error;

static int* g_err_ptr[128];
static std::mutex g_err_mu;

int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lock(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  return g_err_ptr[dev];
}

// (device, kernel) pairs whose dynamic shared-memory limit was raised, with the bytes set.
static std::mutex g_attr_mu;
static std::vector<std::tuple<int, const void*, int>> g_attr_done;

int smem_opt_in(const void* func, int bytes) {
  int dev = 0;
  TREE_CUDA_TRY(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lock(g_attr_mu);
  for (const auto& e : g_attr_done)
    if (std::get<0>(e) == dev && std::get<1>(e) == func && std::get<2>(e) >= bytes) return TREE_OK;
  TREE_CUDA_TRY(cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
  g_attr_done.emplace_back(dev, func, bytes);
  return TREE_OK;
}

}  // namespace tree

extern "C" int tree_check_device_status(tree_stream_t stream) {
  tree::clear_error();
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  TREE_CUDA_TRY(cudaStreamSynchronize(s));
  int* w = tree::device_error_word();
  if (!w) return tree::fail(TREE_ERR_CUDA, "cannot resolve the device error word");
  int v = 0;
  TREE_CUDA_TRY(cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost));
  if (v != 0) {
    int zero = 0;
    TREE_CUDA_TRY(cudaMemcpy(w, &zero, sizeof(int), cudaMemcpyHostToDevice));
    if (v & (1 << TREE_ERR_TIMEOUT))
      return tree::fail(TREE_ERR_TIMEOUT, "a bounded device-side wait gave up (flags 0x%x)", v);
    return tree::fail(TREE_ERR_DEVICE_CHECK, "a device-side range check failed (flags 0x%x)", v);
  }
  return TREE_OK;
}

extern "C" const char* tree_last_error(void) { return tree::g_msg.c_str(); }

extern "C" uint64_t tree_launch_count(void) { return tree::g_launches.load(); }

namespace tree {
static std::atomic<int> g_timing{0};
static cudaEvent_t g_tev[128][kTimedKernels][2];
static bool g_trecorded[128][kTimedKernels];

static void timing_record(int which, void* stream, int edge) {
  if (!g_timing.load(std::memory_order_relaxed) || which < 0 || which >= kTimedKernels) return;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return;
  std::lock_guard<std::mutex> lock(g_err_mu);
  cudaEvent_t& e = g_tev[dev][which][edge];
  if (!e && cudaEventCreate(&e) != cudaSuccess) {
    e = nullptr;
    return;
  }
  if (cudaEventRecord(e, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess && edge == 1)
    g_trecorded[dev][which] = true;
}
void timing_begin(int which, void* stream) { timing_record(which, stream, 0); }
void timing_end(int which, void* stream) { timing_record(which, stream, 1); }
}  // namespace tree

extern "C" int tree_kernel_timing(int enable) {
  tree::g_timing.store(enable ? 1 : 0);
  return TREE_OK;
}

extern "C" float tree_kernel_last_ms(int which) {
  int dev = 0;
  if (which < 0 || which >= tree::kTimedKernels || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128)
    return -1.f;
  cudaEvent_t b, e;
  {
    std::lock_guard<std::mutex> lock(tree::g_err_mu);
    if (!tree::g_trecorded[dev][which]) return -1.f;
    b = tree::g_tev[dev][which][0];
    e = tree::g_tev[dev][which][1];
  }
  float ms = -1.f;
  if (cudaEventSynchronize(e) != cudaSuccess || cudaEventElapsedTime(&ms, b, e) != cudaSuccess) return -1.f;
  return ms;
}

namespace tree {
__global__ void selftest_exp2_kernel(const float* __restrict__ x, float* __restrict__ y, int64_t n) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (2 * t + 1 < n) {
    const float2 r = sm100::exp2_fma2(make_float2(x[2 * t], x[2 * t + 1]));
    y[2 * t] = r.x;
    y[2 * t + 1] = r.y;
  } else if (2 * t < n) {
    y[2 * t] = sm100::exp2_fma2(make_float2(x[2 * t], 0.f)).x;
  }
}
}  // namespace tree

extern "C" int tree_selftest_exp2(const float* x, float* y, int64_t n, tree_stream_t stream) {
  tree::clear_error();
  if (n < 0 || (n > 0 && (!x || !y))) return tree::fail(TREE_ERR_INVALID_ARG, "tree_selftest_exp2: bad arguments");
  if (n == 0) return TREE_OK;
  const int64_t pairs = (n + 1) / 2;
  tree::selftest_exp2_kernel<<<static_cast<unsigned>((pairs + 255) / 256), 256, 0,
                               reinterpret_cast<cudaStream_t>(stream)>>>(x, y, n);
  TREE_LAUNCH_CHECK("selftest_exp2_kernel");
  return TREE_OK;
}

extern "C" const char* tree_version(void) { return "tree_masked_attention_gb300 0.1 (sm_103a)"; }
