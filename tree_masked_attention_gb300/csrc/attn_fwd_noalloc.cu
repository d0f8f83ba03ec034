// tree_attn_fwd_noalloc: the tree-attention forward without a caller workspace.
//
// tree_attn_fwd needs a small scratch area for its per-tile metadata, and takes it
// from a workspace the caller allocates. Some callers cannot do that: a host
// framework whose memory pool already owns all of the device memory it may use,
// a serving loop whose policy forbids cudaMalloc after start-up (an allocation can
// synchronise the device and stall every stream), or a plugin interface that has
// no slot through which a workspace could be passed. For them this entry point
// keeps the scratch in a fixed array in device memory that is part of the loaded
// library (every GPU that loads the library holds it until the process exits).
//
// The array serves trees of up to kNoAllocMaxRows packed rows; larger trees are
// rejected. All calls share it: two calls whose kernels overlap on the GPU (for
// example on two streams) race on it, so issue them in order on one stream. Each
// call rewrites every entry it reads before reading it, so nothing has to start
// at zero and leftovers of an earlier call do no harm.
//
// The first call on a device looks up the array's device address with
// cudaGetSymbolAddress (with that device current) and caches it; make that first
// call before any stream capture. No call allocates or frees device memory.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "attn_internal.h"
#include "common.h"

namespace tree {
namespace {

constexpr int64_t kNoAllocMaxRows = 65536;
constexpr size_t kTiles32 = kNoAllocMaxRows / 32, kTiles128 = kNoAllocMaxRows / 128;
// kmax32, kmin32, kmax128, kmin128, padded subtree_end; each region 256-byte aligned.
constexpr size_t kOff32a = 0;
constexpr size_t kOff32b = kOff32a + kTiles32 * 4;
constexpr size_t kOff128a = kOff32b + kTiles32 * 4;
constexpr size_t kOff128b = kOff128a + kTiles128 * 4;
constexpr size_t kOffPad = kOff128b + kTiles128 * 4;
constexpr size_t kScratchBytes = kOffPad + kNoAllocMaxRows * 4;
static_assert(kOff32b % 256 == 0 && kOff128a % 256 == 0 && kOff128b % 256 == 0 && kOffPad % 256 == 0,
              "scratch regions must stay 256-byte aligned");

// The forward's metadata scratch (about 276 KB).
static __device__ __align__(256) unsigned char g_fwd_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch[128];

// Device address of g_fwd_scratch on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = 0;
  TREE_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 128) return fail(TREE_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_fwd_scratch);
    if (e != cudaSuccess || !p)
      return fail(TREE_ERR_CUDA, "cudaGetSymbolAddress of the forward scratch failed: %s",
                  cudaGetErrorString(e));
    g_scratch[dev] = p;
  }
  *out = g_scratch[dev];
  return TREE_OK;
}

}  // namespace
}  // namespace tree

using namespace tree;

extern "C" int tree_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                                     const int32_t* subtree_end, int64_t T, int Hq, int Hkv, int d, int dtype,
                                     float softmax_scale, tree_stream_t stream) {
  clear_error();
  if (dtype != TREE_DTYPE_F32 && dtype != TREE_DTYPE_BF16)
    return fail(TREE_ERR_DTYPE, "tree_attn_fwd_noalloc: dtype %d is not TREE_DTYPE_F32/BF16", dtype);
  if (T < 1) return fail(TREE_ERR_SHAPE, "tree_attn_fwd_noalloc: T = %lld < 1", static_cast<long long>(T));
  if (T > kNoAllocMaxRows)
    return fail(TREE_ERR_SHAPE,
                "tree_attn_fwd_noalloc: T = %lld exceeds the %lld rows its fixed scratch serves; "
                "use tree_attn_fwd with a workspace",
                static_cast<long long>(T), static_cast<long long>(kNoAllocMaxRows));
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Hq > 65535)
    return fail(TREE_ERR_SHAPE, "tree_attn_fwd_noalloc: Hq = %d, Hkv = %d", Hq, Hkv);
  if (d != 64 && d != 128) return fail(TREE_ERR_SHAPE, "tree_attn_fwd_noalloc: head size %d", d);
  if (!q || !k || !v || !o || !lse || !subtree_end)
    return fail(TREE_ERR_INVALID_ARG, "tree_attn_fwd_noalloc: null tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(TREE_ERR_ALIGNMENT, "tree_attn_fwd_noalloc: q/k/v/o not 16-byte aligned");
  void* base = nullptr;
  int rc = scratch_address(&base);
  if (rc) return rc;
  char* b = static_cast<char*>(base);
  AttnArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse; a.end = subtree_end;
  a.T = T; a.Hq = Hq; a.Hkv = Hkv; a.d = d; a.dtype = dtype;
  a.scale = softmax_scale > 0.f ? softmax_scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  a.ws.kmax32 = reinterpret_cast<int32_t*>(b + kOff32a);
  a.ws.kmin32 = reinterpret_cast<int32_t*>(b + kOff32b);
  a.ws.kmax128 = reinterpret_cast<int32_t*>(b + kOff128a);
  a.ws.kmin128 = reinterpret_cast<int32_t*>(b + kOff128b);
  a.ws.end_pad = reinterpret_cast<int32_t*>(b + kOffPad);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (attn_fwd_tc_supported(dtype, d, Hq, Hkv)) return attn_fwd_tc(a, st);
  if (attn_tc32_supported(dtype, d)) return attn_fwd_tc32(a, st);
  return attn_fwd_simt(a, st);
}
