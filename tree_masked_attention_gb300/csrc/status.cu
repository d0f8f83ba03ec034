// Error reporting: the thread-local host message and the per-device error word.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "common.h"

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

extern "C" const char* tree_version(void) { return "tree_masked_attention_gb300 0.1 (sm_103a)"; }
