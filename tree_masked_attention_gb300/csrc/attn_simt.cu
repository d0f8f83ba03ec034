// Tree attention on the CUDA cores, for the one shape the tensor-core kernels leave out:
// fp32 storage with head size 128. (The tf32-split kernels hold each fp32 operand as two
// tf32 tiles; at head size 128 the dQ pass would need Q and dO resident as 4 x 64 KB, more
// than a CTA's shared memory.) Forward, backward preprocess (Delta), dQ and dK/dV. The
// per-tile metadata kernel here also serves the tf32-split kernels.
//
// Visibility (Tree Training, arXiv 2511.00413, §3.2 "Attention Mask"; Trie
// packing "Step 2 - Allow only ancestors and self"): key j is visible to query i
// iff j <= i <= subtree_end[j]. A key tile is skipped for a query tile when no
// key in it is visible to any of the queries: max(subtree_end over the tile) is
// below the first query, or its first key is past the last query. Since every
// row between a key tile's first key and that maximum lies in some key's
// subtree, the queries a key tile serves are exactly that contiguous range
// (used by the dK/dV kernel to bound its query loop).
//
// Scores are handled in the base-2 domain: s2 = q.k * scale * log2(e), so that
// p = exp2(s2 - m2) and LSE = ln(2) * (m2 + log2 l).
//
// Layout: 4 threads share one row (query, or key for dK/dV); thread `part` owns
// the dimensions t*4 + part, t < D/4, so the 4 threads of a row read 4
// consecutive floats of a shared-memory row (no bank conflicts) and the 8 rows
// of a warp broadcast the same addresses.
#include <cmath>

#include "attn_internal.h"
#include "common.h"
#include "device_common.cuh"

namespace tree {

constexpr int kSimtTile = 32;     // query rows and keys per tile
constexpr int kSimtThreads = 128; // 32 rows x 4 threads

// Per key tile: max and min subtree_end; range-checks every entry.
__global__ void tile_meta_kernel(const int32_t* __restrict__ end, int64_t n, int tile,
                                 int32_t* __restrict__ kmax, int32_t* __restrict__ kmin, int* err) {
  const int64_t kt = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  const int64_t n_tiles = (n + tile - 1) / tile;
  if (kt >= n_tiles) return;
  int mx = -1, mn = INT32_MAX;
  bool bad = false;
  for (int64_t j = kt * tile + lane; j < min(n, (kt + 1) * tile); j += 32) {
    const int e = end[j];
    bad |= (e < j) || (e >= n);
    mx = max(mx, e);
    mn = min(mn, e);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) raise_error(err, TREE_ERR_DEVICE_CHECK);
  if (lane == 0) {
    kmax[kt] = mx;
    kmin[kt] = mn;
  }
}

int tile_meta_launch(const int32_t* end, int64_t n, int tile, int32_t* kmax, int32_t* kmin,
                     cudaStream_t st) {
  const int64_t n_tiles = (n + tile - 1) / tile;
  const int64_t blocks = (n_tiles * 32 + 255) / 256;
  tile_meta_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(end, n, tile, kmax, kmin,
                                                                   device_error_word());
  TREE_LAUNCH_CHECK("tile_meta_kernel");
  return TREE_OK;
}

__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}

template <typename T, int D>
__global__ void __launch_bounds__(kSimtThreads)
attn_fwd_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     T* __restrict__ o, float* __restrict__ lse, const int32_t* __restrict__ end,
                     const int32_t* __restrict__ kmax, int64_t n, int Hq, int Hkv, float scale_log2) {
  constexpr int B = kSimtTile, DPT = D / 4;
  __shared__ float Ks[B][D], Vs[B][D];
  __shared__ int Es[B];
  const int h = blockIdx.y, kvh = h / (Hq / Hkv);
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * B;
  const int r = threadIdx.x / 4, part = threadIdx.x % 4;
  const int64_t i = i0 + r;
  const bool valid = i < n;
  float qr[DPT], acc[DPT];
#pragma unroll
  for (int t = 0; t < DPT; ++t) {
    qr[t] = valid ? to_f32(q[(i * Hq + h) * D + t * 4 + part]) * scale_log2 : 0.f;
    acc[t] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int64_t last = min(n - 1, i0 + B - 1);
  for (int64_t kt = 0; kt * B <= last; ++kt) {
    if (kmax[kt] < i0) continue;  // no key of this tile sees any query of the tile
    const int64_t j0 = kt * B;
    __syncthreads();
    for (int e = threadIdx.x; e < B * D; e += kSimtThreads) {
      const int jj = e / D, dd = e % D;
      const int64_t j = j0 + jj;
      Ks[jj][dd] = j < n ? to_f32(k[(j * Hkv + kvh) * D + dd]) : 0.f;
      Vs[jj][dd] = j < n ? to_f32(v[(j * Hkv + kvh) * D + dd]) : 0.f;
    }
    if (threadIdx.x < B) Es[threadIdx.x] = j0 + threadIdx.x < n ? end[j0 + threadIdx.x] : -1;
    __syncthreads();
    float s[B];
    float mt = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < B; ++jj) {
      float dot = 0.f;
#pragma unroll
      for (int t = 0; t < DPT; ++t) dot += qr[t] * Ks[jj][t * 4 + part];
      dot = quad_sum(dot);
      const int64_t j = j0 + jj;
      const bool vis = valid && j <= i && i <= Es[jj];
      s[jj] = vis ? dot : -INFINITY;
      mt = fmaxf(mt, s[jj]);
    }
    if (mt == -INFINITY) continue;
    const float mn = fmaxf(m, mt);
    const float corr = exp2f(m - mn);
    m = mn;
    l *= corr;
#pragma unroll
    for (int t = 0; t < DPT; ++t) acc[t] *= corr;
#pragma unroll
    for (int jj = 0; jj < B; ++jj) {
      const float p = exp2f(s[jj] - m);
      l += p;
#pragma unroll
      for (int t = 0; t < DPT; ++t) acc[t] += p * Vs[jj][t * 4 + part];
    }
  }
  if (!valid) return;
  const float inv = 1.f / l;
#pragma unroll
  for (int t = 0; t < DPT; ++t) o[(i * Hq + h) * D + t * 4 + part] = from_f32<T>(acc[t] * inv);
  if (part == 0) lse[static_cast<int64_t>(h) * n + i] = (m + log2f(l)) * 0.6931471805599453f;
}

// Delta_i = dO_i . O_i per query head: one warp per (row, head).
template <typename T>
__global__ void attn_delta_kernel(const T* __restrict__ o, const T* __restrict__ dout,
                                  float* __restrict__ delta, int64_t n, int Hq, int d) {
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (w >= n * Hq) return;
  const int64_t i = w / Hq;
  const int h = static_cast<int>(w % Hq);
  float s = 0.f;
  for (int dd = lane; dd < d; dd += 32) s += to_f32(o[w * d + dd]) * to_f32(dout[w * d + dd]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) delta[static_cast<int64_t>(h) * n + i] = s;
}

// dQ_i = scale * sum_j P_ij (dO_i . v_j - Delta_i) k_j, query-stationary.
template <typename T, int D>
__global__ void __launch_bounds__(kSimtThreads)
attn_dq_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                    const T* __restrict__ dout, const float* __restrict__ lse,
                    const float* __restrict__ delta, T* __restrict__ dq, const int32_t* __restrict__ end,
                    const int32_t* __restrict__ kmax, int64_t n, int Hq, int Hkv, float scale_log2,
                    float scale) {
  constexpr int B = kSimtTile, DPT = D / 4;
  __shared__ float Ks[B][D], Vs[B][D];
  __shared__ int Es[B];
  const int h = blockIdx.y, kvh = h / (Hq / Hkv);
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * B;
  const int r = threadIdx.x / 4, part = threadIdx.x % 4;
  const int64_t i = i0 + r;
  const bool valid = i < n;
  float qr[DPT], dor[DPT], acc[DPT];
#pragma unroll
  for (int t = 0; t < DPT; ++t) {
    const int64_t idx = (i * Hq + h) * D + t * 4 + part;
    qr[t] = valid ? to_f32(q[idx]) * scale_log2 : 0.f;
    dor[t] = valid ? to_f32(dout[idx]) : 0.f;
    acc[t] = 0.f;
  }
  const float lse2 = valid ? lse[static_cast<int64_t>(h) * n + i] * 1.4426950408889634f : 0.f;
  const float dl = valid ? delta[static_cast<int64_t>(h) * n + i] : 0.f;
  const int64_t last = min(n - 1, i0 + B - 1);
  for (int64_t kt = 0; kt * B <= last; ++kt) {
    if (kmax[kt] < i0) continue;
    const int64_t j0 = kt * B;
    __syncthreads();
    for (int e = threadIdx.x; e < B * D; e += kSimtThreads) {
      const int jj = e / D, dd = e % D;
      const int64_t j = j0 + jj;
      Ks[jj][dd] = j < n ? to_f32(k[(j * Hkv + kvh) * D + dd]) : 0.f;
      Vs[jj][dd] = j < n ? to_f32(v[(j * Hkv + kvh) * D + dd]) : 0.f;
    }
    if (threadIdx.x < B) Es[threadIdx.x] = j0 + threadIdx.x < n ? end[j0 + threadIdx.x] : -1;
    __syncthreads();
#pragma unroll 4
    for (int jj = 0; jj < B; ++jj) {
      float sd = 0.f, pd = 0.f;
#pragma unroll
      for (int t = 0; t < DPT; ++t) {
        sd += qr[t] * Ks[jj][t * 4 + part];
        pd += dor[t] * Vs[jj][t * 4 + part];
      }
      sd = quad_sum(sd);
      pd = quad_sum(pd);
      const int64_t j = j0 + jj;
      const bool vis = valid && j <= i && i <= Es[jj];
      const float p = vis ? exp2f(sd - lse2) : 0.f;
      const float ds = p * (pd - dl);
#pragma unroll
      for (int t = 0; t < DPT; ++t) acc[t] += ds * Ks[jj][t * 4 + part];
    }
  }
  if (!valid) return;
#pragma unroll
  for (int t = 0; t < DPT; ++t) dq[(i * Hq + h) * D + t * 4 + part] = from_f32<T>(acc[t] * scale);
}

// dK_j, dV_j: key-stationary; queries j0 .. kmax[tile] of every query head of the group.
template <typename T, int D>
__global__ void __launch_bounds__(kSimtThreads)
attn_dkdv_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                      const T* __restrict__ dout, const float* __restrict__ lse,
                      const float* __restrict__ delta, T* __restrict__ dk, T* __restrict__ dv,
                      const int32_t* __restrict__ end, const int32_t* __restrict__ kmax, int64_t n,
                      int Hq, int Hkv, float scale_log2, float scale) {
  constexpr int B = kSimtTile, DPT = D / 4;
  __shared__ float Qs[B][D], Ds[B][D];
  __shared__ float Ls[B], Dl[B];
  const int kvh = blockIdx.y, group = Hq / Hkv;
  const int64_t kt = blockIdx.x, j0 = kt * B;
  const int r = threadIdx.x / 4, part = threadIdx.x % 4;
  const int64_t j = j0 + r;
  const bool valid = j < n;
  const int ej = valid ? end[j] : -1;
  float kr[DPT], vr[DPT], dka[DPT], dva[DPT];
#pragma unroll
  for (int t = 0; t < DPT; ++t) {
    const int64_t idx = (j * Hkv + kvh) * D + t * 4 + part;
    kr[t] = valid ? to_f32(k[idx]) * scale_log2 : 0.f;
    vr[t] = valid ? to_f32(v[idx]) : 0.f;
    dka[t] = 0.f;
    dva[t] = 0.f;
  }
  const int64_t qlast = min(static_cast<int64_t>(kmax[kt]), n - 1);
  for (int hh = 0; hh < group; ++hh) {
    const int h = kvh * group + hh;
    for (int64_t i0 = (j0 / B) * B; i0 <= qlast; i0 += B) {
      __syncthreads();
      for (int e = threadIdx.x; e < B * D; e += kSimtThreads) {
        const int ii = e / D, dd = e % D;
        const int64_t i = i0 + ii;
        Qs[ii][dd] = i < n ? to_f32(q[(i * Hq + h) * D + dd]) : 0.f;
        Ds[ii][dd] = i < n ? to_f32(dout[(i * Hq + h) * D + dd]) : 0.f;
      }
      if (threadIdx.x < B) {
        const int64_t i = i0 + threadIdx.x;
        Ls[threadIdx.x] = i < n ? lse[static_cast<int64_t>(h) * n + i] * 1.4426950408889634f : 0.f;
        Dl[threadIdx.x] = i < n ? delta[static_cast<int64_t>(h) * n + i] : 0.f;
      }
      __syncthreads();
#pragma unroll 4
      for (int ii = 0; ii < B; ++ii) {
        float sd = 0.f, pd = 0.f;
#pragma unroll
        for (int t = 0; t < DPT; ++t) {
          sd += kr[t] * Qs[ii][t * 4 + part];
          pd += vr[t] * Ds[ii][t * 4 + part];
        }
        sd = quad_sum(sd);
        pd = quad_sum(pd);
        const int64_t i = i0 + ii;
        const bool vis = valid && i < n && j <= i && i <= ej;
        const float p = vis ? exp2f(sd - Ls[ii]) : 0.f;
        const float ds = p * (pd - Dl[ii]);
#pragma unroll
        for (int t = 0; t < DPT; ++t) {
          dva[t] += p * Ds[ii][t * 4 + part];
          dka[t] += ds * Qs[ii][t * 4 + part];
        }
      }
    }
  }
  if (!valid) return;
#pragma unroll
  for (int t = 0; t < DPT; ++t) {
    const int64_t idx = (j * Hkv + kvh) * D + t * 4 + part;
    dk[idx] = from_f32<T>(dka[t] * scale);
    dv[idx] = from_f32<T>(dva[t]);
  }
}

template <typename T, int D>
static int fwd_simt(const AttnArgs& a, cudaStream_t st) {
  int32_t* kmax = a.ws.kmax32;
  int32_t* kmin = a.ws.kmin32;
  int rc = tile_meta_launch(a.end, a.T, kSimtTile, kmax, kmin, st);
  if (rc) return rc;
  dim3 grid(static_cast<unsigned>((a.T + kSimtTile - 1) / kSimtTile), a.Hq);
  attn_fwd_simt_kernel<T, D><<<grid, kSimtThreads, 0, st>>>(
      static_cast<const T*>(a.q), static_cast<const T*>(a.k), static_cast<const T*>(a.v),
      static_cast<T*>(a.o), a.lse, a.end, kmax, a.T, a.Hq, a.Hkv, a.scale * 1.4426950408889634f);
  TREE_LAUNCH_CHECK("attn_fwd_simt_kernel");
  return TREE_OK;
}

template <typename T, int D>
static int bwd_simt(const AttnArgs& a, cudaStream_t st) {
  int32_t* kmax = a.ws.kmax32;
  int32_t* kmin = a.ws.kmin32;
  int rc = tile_meta_launch(a.end, a.T, kSimtTile, kmax, kmin, st);
  if (rc) return rc;
  const int64_t warps = a.T * a.Hq;
  attn_delta_kernel<T><<<static_cast<unsigned>((warps * 32 + 255) / 256), 256, 0, st>>>(
      static_cast<const T*>(a.o), static_cast<const T*>(a.dout), a.ws.delta, a.T, a.Hq, D);
  TREE_LAUNCH_CHECK("attn_delta_kernel");
  const float sl2 = a.scale * 1.4426950408889634f;
  dim3 gq(static_cast<unsigned>((a.T + kSimtTile - 1) / kSimtTile), a.Hq);
  attn_dq_simt_kernel<T, D><<<gq, kSimtThreads, 0, st>>>(
      static_cast<const T*>(a.q), static_cast<const T*>(a.k), static_cast<const T*>(a.v),
      static_cast<const T*>(a.dout), a.lse, a.ws.delta, static_cast<T*>(a.dq), a.end, kmax, a.T,
      a.Hq, a.Hkv, sl2, a.scale);
  TREE_LAUNCH_CHECK("attn_dq_simt_kernel");
  dim3 gk(static_cast<unsigned>((a.T + kSimtTile - 1) / kSimtTile), a.Hkv);
  attn_dkdv_simt_kernel<T, D><<<gk, kSimtThreads, 0, st>>>(
      static_cast<const T*>(a.q), static_cast<const T*>(a.k), static_cast<const T*>(a.v),
      static_cast<const T*>(a.dout), a.lse, a.ws.delta, static_cast<T*>(a.dk), static_cast<T*>(a.dv),
      a.end, kmax, a.T, a.Hq, a.Hkv, sl2, a.scale);
  TREE_LAUNCH_CHECK("attn_dkdv_simt_kernel");
  return TREE_OK;
}

int attn_fwd_simt(const AttnArgs& a, cudaStream_t st) {
  if (a.dtype != TREE_DTYPE_F32 || a.d != 128)
    return fail(TREE_ERR_SHAPE, "CUDA-core attention serves fp32 with head size 128 only");
  return fwd_simt<float, 128>(a, st);
}

int attn_bwd_simt(const AttnArgs& a, cudaStream_t st) {
  if (a.dtype != TREE_DTYPE_F32 || a.d != 128)
    return fail(TREE_ERR_SHAPE, "CUDA-core attention serves fp32 with head size 128 only");
  return bwd_simt<float, 128>(a, st);
}

}  // namespace tree
