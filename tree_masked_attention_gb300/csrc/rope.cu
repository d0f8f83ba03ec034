// tree_rope: rotary position embedding on depth positions, in place on Q and K.
//
// Tree Training (arXiv 2511.00413) §3.2 "Position Embedding", eq. 9, and Trie
// packing "Step 1 - Store each node once": each packed row is rotated by its
// depth, the position it has in its own per-path sequence. Rotate-half pairing
// (x[k], x[k + d/2]) with angle pos * base^(-2k/d).
//
// Memory-bound: every element of Q and K is read and written once. One thread owns
// one row, 8 consecutive frequencies and 4 heads (of Q, then K): it forms the 8
// (cos, sin) pairs once and applies them to those 4 heads, so sincosf runs a quarter
// as often as per element while the grid still has T * (d/16) * (Hq+Hkv)/4 threads
// to keep every SM's memory pipe busy. Consecutive threads cover consecutive
// 16-byte pieces of a head's row, so warp accesses are fully used 128-byte lines.
#include <cmath>

#include "common.h"
#include "device_common.cuh"

namespace tree {

template <typename T>
__global__ void rope_kernel(T* __restrict__ q, T* __restrict__ k, const int32_t* __restrict__ pos,
                            int64_t n_rows, int Hq, int Hkv, int d, float neg2_log2base_over_d,
                            float sign, int* err) {
  constexpr int kHeadsPerThread = 4;
  const int groups = d / 16;  // groups of 8 frequencies per row
  const int n_heads = Hq + Hkv, chunks = (n_heads + kHeadsPerThread - 1) / kHeadsPerThread;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int g = static_cast<int>(tid % groups);
  const int64_t rest = tid / groups;
  const int chunk = static_cast<int>(rest % chunks);
  const int64_t row = rest / chunks;
  if (row >= n_rows) return;
  const int p0 = pos[row];
  if (p0 < 0) { raise_error(err, TREE_ERR_DEVICE_CHECK); return; }
  float c[8], s[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int kf = g * 8 + i;
    const float inv_freq = exp2f(static_cast<float>(kf) * neg2_log2base_over_d);
    sincosf(static_cast<float>(p0) * inv_freq, &s[i], &c[i]);
    s[i] *= sign;
  }
  const int half = d / 2;
  for (int hh = chunk * kHeadsPerThread; hh < min(n_heads, (chunk + 1) * kHeadsPerThread); ++hh) {
    T* base = hh < Hq ? q : k;
    if (!base) continue;
    const int H = hh < Hq ? Hq : Hkv, h = hh < Hq ? hh : hh - Hq;
    T* r = base + (row * static_cast<int64_t>(H) + h) * d + g * 8;
    float x1[8], x2[8], y1[8], y2[8];
    load8(r, x1);
    load8(r + half, x2);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      y1[i] = x1[i] * c[i] - x2[i] * s[i];
      y2[i] = x2[i] * c[i] + x1[i] * s[i];
    }
    store8(r, y1);
    store8(r + half, y2);
  }
}

// Scalar path for head sizes that are not a multiple of 16.
template <typename T>
__global__ void rope_scalar_kernel(T* __restrict__ x, const int32_t* __restrict__ pos, int64_t n_rows,
                                   int H, int d, float neg2_log2base_over_d, float sign, int* err) {
  const int half = d / 2;
  const int64_t n = n_rows * H * half;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < n;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int kf = static_cast<int>(t % half);
    const int64_t rh = t / half;
    const int64_t row = rh / H;
    const int p = pos[row];
    if (p < 0) { raise_error(err, TREE_ERR_DEVICE_CHECK); continue; }
    float sn, cs;
    sincosf(static_cast<float>(p) * exp2f(static_cast<float>(kf) * neg2_log2base_over_d), &sn, &cs);
    sn *= sign;
    T* r = x + rh * d;
    const float x1 = to_f32(r[kf]), x2 = to_f32(r[kf + half]);
    r[kf] = from_f32<T>(x1 * cs - x2 * sn);
    r[kf + half] = from_f32<T>(x2 * cs + x1 * sn);
  }
}

template <typename T>
static int launch_rope(void* q, void* k, const int32_t* pos, int64_t n_rows, int Hq, int Hkv, int d,
                       float theta_base, int inverse, cudaStream_t st) {
  const float e = static_cast<float>(-2.0 * std::log2(static_cast<double>(theta_base)) / d);
  const float sign = inverse ? -1.f : 1.f;
  int* err = device_error_word();
  if (d % 16 == 0) {
    const int64_t threads = n_rows * (d / 16) * ((Hq + Hkv + 3) / 4);
    const int bs = 256;
    const int64_t grid = (threads + bs - 1) / bs;
    rope_kernel<T><<<static_cast<unsigned>(grid), bs, 0, st>>>(static_cast<T*>(q), static_cast<T*>(k), pos,
                                                               n_rows, Hq, Hkv, d, e, sign, err);
    TREE_LAUNCH_CHECK("rope_kernel");
  } else {
    if (q) {
      rope_scalar_kernel<T><<<1024, 256, 0, st>>>(static_cast<T*>(q), pos, n_rows, Hq, d, e, sign, err);
      TREE_LAUNCH_CHECK("rope_scalar_kernel");
    }
    if (k) {
      rope_scalar_kernel<T><<<1024, 256, 0, st>>>(static_cast<T*>(k), pos, n_rows, Hkv, d, e, sign, err);
      TREE_LAUNCH_CHECK("rope_scalar_kernel");
    }
  }
  return TREE_OK;
}

int rope_launch(void* q, void* k, const int32_t* pos, int64_t T, int Hq, int Hkv, int d, float theta_base,
                int dtype, int inverse, cudaStream_t st) {
  if (dtype == TREE_DTYPE_BF16)
    return launch_rope<__nv_bfloat16>(q, k, pos, T, Hq, Hkv, d, theta_base, inverse, st);
  return launch_rope<float>(q, k, pos, T, Hq, Hkv, d, theta_base, inverse, st);
}

}  // namespace tree
