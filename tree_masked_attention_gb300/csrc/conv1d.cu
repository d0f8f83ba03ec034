// tree_conv1d_fwd / tree_conv1d_bwd: tree-correct causal depthwise conv1d (the short
// convolution of SSM / linear-attention layers) over a packed prefix tree.
//
// Tree Training (arXiv 2511.00413) §3.2 "(ii) Causal convolution", eq. 11 and Fig. 4: a
// causal conv of kernel size K reads the K-1 tokens before a token; in the preorder
// serialisation the rows just before a child chunk belong to a sibling, so the left
// context of a row is taken from its ancestors instead, which reproduces what the row
// sees in an independent per-branch pass. Row i's m-th ancestor a_m(i) (a_0 = i,
// a_{m+1} = parent_row[a_m], none above a root) gets tap K-1-m:
//   y[i, c] = bias[c] + sum_{m<K} w[c, K-1-m] x[a_m(i), c]          (zero past the root)
// Backward, with D_m[j] = sum of dy[i] over the rows i whose m-th ancestor is j:
//   dx[j, c] = sum_{m<K} w[c, K-1-m] D_m[j, c]
//   dw[c, K-1-m] = sum_j x[j, c] D_m[j, c],     dbias[c] = sum_i dy[i, c].
//
// Both directions are HBM-bound (read x / write y; read x, dy / write dx) and use no
// atomics. A CTA of 256 threads owns 1024 channels (4 per thread, so a warp touches 256
// contiguous bytes of a bf16 row) and a group of consecutive rows; the grid is one wave
// on GB300 (3 forward / 2 backward CTAs per SM). Thread 0 stages the group's rows in
// chunks of 8 through a ring of shared-memory buffers filled by bulk asynchronous copies
// (one cp.async.bulk per row segment, completion on an mbarrier), so each SM keeps
// >100 KB of loads in flight without spending registers on them. Every thread of a CTA
// walks the same rows: the tree logic is uniform, only the channel data differ.
//  - Forward, rows in increasing order: a register window holds x at the current row's
//    K ancestors. A chunk whose rows all continue the previous row (parent_row[i] ==
//    i-1, the common case inside a chunk of the tree) takes a fast path whose window
//    indices are compile-time constants (the chunk's own rows plus the window carried
//    from the row before it). Otherwise each row either shifts the window by one or, at
//    a later sibling or the group's first row, refills it by walking parent links.
//  - Backward, rows in decreasing order: a window holds D_0..D_{K-1} of the current
//    row. A chunk in which every row's only child is the next row takes the fast path
//    (D_m of row q is dy of row q+m, or the carried window of the row after the chunk).
//    Otherwise a row whose only child is j+1 (subtree_end[j+1] == subtree_end[j])
//    shifts the window, a leaf has D_m = 0 for m > 0, and a fork (or the group's last
//    row) enumerates its descendants within depth K-1 in preorder from subtree_end and
//    the depth positions. dw and dbias are summed per group in fp32, then a second
//    kernel adds the groups in a fixed order in fp64.
#include <algorithm>

#include "common.h"
#include "device_common.cuh"
#include "sm100.cuh"

namespace tree {
namespace {

using namespace sm100;

constexpr int kConvThreads = 256;
constexpr int kConvVec = 4;                             // channels per thread
constexpr int kConvChan = kConvThreads * kConvVec;      // channels per CTA (one row segment)
constexpr int kStageRows = 8;                           // rows per pipeline stage
constexpr int kFwdStages = 4;                           // x:      4 x 8 rows x 2 KB (bf16) = 64 KB
constexpr int kBwdStages = 3;                           // x, dy:  3 x 8 rows x 4 KB (bf16) = 96 KB
// One wave of CTAs on GB300's 152 SMs: 3 forward / 2 backward CTAs fit per SM by shared memory.
constexpr int kFwdTargetCtas = 152 * 3;
constexpr int kBwdTargetCtas = 152 * 2;
constexpr int kConvMaxK = 8;                            // largest kernel size
static_assert(kStageRows >= kConvMaxK, "the chain fast paths take a window of K rows from one stage");

template <typename T> constexpr size_t fwd_smem() { return sizeof(T) * kFwdStages * kStageRows * kConvChan; }
template <typename T> constexpr size_t bwd_smem() { return sizeof(T) * kBwdStages * 2 * kStageRows * kConvChan; }

// Rows are split into groups of whole stages; grid = (groups, channel tiles).
struct ConvGrid {
  int64_t rows_per_group, groups;
  int ctiles;
};
ConvGrid conv_grid(int64_t n_rows, int C, int target_ctas) {
  ConvGrid g;
  g.ctiles = (C + kConvChan - 1) / kConvChan;
  const int64_t chunks = std::max<int64_t>((n_rows + kStageRows - 1) / kStageRows, 1);
  int64_t groups = std::max<int64_t>(1, std::min<int64_t>(chunks, (target_ctas + g.ctiles - 1) / g.ctiles));
  const int64_t per = (chunks + groups - 1) / groups;
  g.rows_per_group = per * kStageRows;
  g.groups = (chunks + per - 1) / per;
  return g;
}

// 4 consecutive elements <-> 4 floats (8-byte access for bf16, 16-byte for fp32).
__device__ __forceinline__ void ld4(const __nv_bfloat16* p, float* f) {
  uint2 u = *reinterpret_cast<const uint2*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
  float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}
__device__ __forceinline__ void ld4(const float* p, float* f) {
  float4 a = *reinterpret_cast<const float4*>(p);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
}
__device__ __forceinline__ void st4(__nv_bfloat16* p, const float* f) {
  uint2 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
  h[0] = __floats2bfloat162_rn(f[0], f[1]);
  h[1] = __floats2bfloat162_rn(f[2], f[3]);
  *reinterpret_cast<uint2*>(p) = u;
}
__device__ __forceinline__ void st4(float* p, const float* f) {
  *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
}

// Taps of this thread's channels: wt[k][v] = w[c0 + v, k]; bias in b (0 if none).
template <typename T, int K>
__device__ __forceinline__ void load_taps(const T* __restrict__ w, const T* __restrict__ bias, int c0,
                                          bool active, float (&wt)[K][kConvVec], float* b) {
#pragma unroll
  for (int v = 0; v < kConvVec; ++v) {
    b[v] = (active && bias) ? to_f32(bias[c0 + v]) : 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) wt[k][v] = active ? to_f32(w[static_cast<int64_t>(c0 + v) * K + k]) : 0.f;
  }
}

// Thread 0: one bulk copy per row of `rows` rows starting at `r`, each `row_bytes` long
// (the CTA's channel slice), into `dst` (rows kConvChan elements apart), completing on `bar`.
template <typename T>
__device__ __forceinline__ void stage_rows(T* dst, const T* src, int64_t r, int rows, int C, int ct0,
                                           uint32_t row_bytes, uint64_t* bar) {
  for (int q = 0; q < rows; ++q)
    bulk_load(dst + q * kConvChan, src + (r + q) * C + ct0, row_bytes, bar);
}

// After a timed-out wait: thread 0 waits (bounded) for the stages still being filled, so
// no copy lands in shared memory after the CTA has left.
__device__ __forceinline__ void drain_stages(uint64_t* full, int n_stages, int first, int last_issued,
                                             int* err) {
  for (int c = first; c <= last_issued; ++c) mbar_wait(&full[c % n_stages], (c / n_stages) & 1, err);
}

template <typename T, int K>
__global__ void __launch_bounds__(kConvThreads, K <= 4 ? 3 : 2) conv1d_fwd_kernel(
    const T* __restrict__ x, const T* __restrict__ w, const T* __restrict__ bias, T* __restrict__ y,
    const int32_t* __restrict__ parent, int64_t n_rows, int C, int64_t rows_per_group, int* err) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ uint64_t full[kFwdStages];
  T* stage = reinterpret_cast<T*>(smem_raw);  // [kFwdStages][kStageRows][kConvChan]
  const int64_t g0 = static_cast<int64_t>(blockIdx.x) * rows_per_group;
  const int64_t g1 = min(g0 + rows_per_group, n_rows);
  const int ct0 = blockIdx.y * kConvChan;
  const uint32_t row_bytes = static_cast<uint32_t>(min(kConvChan, C - ct0) * sizeof(T));
  const int c0 = ct0 + threadIdx.x * kConvVec;
  const bool active = c0 < C;
  const int n_chunks = static_cast<int>((g1 - g0 + kStageRows - 1) / kStageRows);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kFwdStages; ++s) mbar_init(&full[s], 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  int issued = -1;  // last chunk whose copies thread 0 has issued
  auto issue = [&](int c) {
    const int s = c % kFwdStages;
    const int64_t r = g0 + static_cast<int64_t>(c) * kStageRows;
    const int rows = static_cast<int>(min(static_cast<int64_t>(kStageRows), g1 - r));
    mbar_arrive_expect_tx(&full[s], rows * row_bytes);
    stage_rows(stage + s * kStageRows * kConvChan, x, r, rows, C, ct0, row_bytes, &full[s]);
    issued = c;
  };
  if (threadIdx.x == 0)
    for (int c = 0; c < min(kFwdStages - 1, n_chunks); ++c) issue(c);

  float wt[K][kConvVec], b[kConvVec];
  load_taps<T, K>(w, bias, c0, active, wt, b);
  float win[K][kConvVec];  // win[m] = x at the m-th ancestor of the current row
#pragma unroll
  for (int m = 0; m < K; ++m)
#pragma unroll
    for (int v = 0; v < kConvVec; ++v) win[m][v] = 0.f;

  for (int c = 0; c < n_chunks; ++c) {
    // the stage of chunk c + kFwdStages - 1 was read in iteration c - 1 (barrier below)
    if (threadIdx.x == 0 && c + kFwdStages - 1 < n_chunks) issue(c + kFwdStages - 1);
    const bool ok = mbar_wait(&full[c % kFwdStages], (c / kFwdStages) & 1, err);
    if (ok) {
      const T* sx = stage + (c % kFwdStages) * kStageRows * kConvChan + threadIdx.x * kConvVec;
      const int64_t r = g0 + static_cast<int64_t>(c) * kStageRows;
      const int rows = static_cast<int>(min(static_cast<int64_t>(kStageRows), g1 - r));
      int pb[kStageRows];  // the chunk's parent links, loaded together
#pragma unroll
      for (int q = 0; q < kStageRows; ++q) pb[q] = q < rows ? parent[r + q] : -1;
      bool chain = rows == kStageRows && r > g0;
#pragma unroll
      for (int q = 0; q < kStageRows; ++q) chain = chain && pb[q] == r + q - 1;
      if (chain) {
        // Every row of the chunk continues the previous one: row q's m-th ancestor is
        // row q - m of the chunk, or (q < m) the (m - q - 1)-th ancestor of the row
        // before the chunk, which win holds. All indices are fixed at compile time.
        float xr[kStageRows][kConvVec];
#pragma unroll
        for (int q = 0; q < kStageRows; ++q) {
          if (active) {
            ld4(sx + q * kConvChan, xr[q]);
          } else {
#pragma unroll
            for (int v = 0; v < kConvVec; ++v) xr[q][v] = 0.f;
          }
        }
#pragma unroll
        for (int q = 0; q < kStageRows; ++q) {
          float out[kConvVec];
#pragma unroll
          for (int v = 0; v < kConvVec; ++v) {
            float acc = b[v];
#pragma unroll
            for (int m = 0; m < K; ++m) acc = fmaf(wt[K - 1 - m][v], q >= m ? xr[q - m][v] : win[m - q - 1][v], acc);
            out[v] = acc;
          }
          if (active) st4(y + (r + q) * C + c0, out);
        }
#pragma unroll
        for (int m = 0; m < K; ++m)
#pragma unroll
          for (int v = 0; v < kConvVec; ++v) win[m][v] = xr[kStageRows - 1 - m][v];
      } else {
#pragma unroll
      for (int q = 0; q < kStageRows; ++q) {
        const int64_t i = r + q;
        if (q >= rows) break;
        int p = pb[q];
        if (p < -1 || p >= i) {  // a parent must be an earlier row (or -1 for a root)
          raise_error(err, TREE_ERR_DEVICE_CHECK);
          p = -1;
        }
        if (i > g0 && p == i - 1) {
#pragma unroll
          for (int m = K - 1; m > 0; --m)
#pragma unroll
            for (int v = 0; v < kConvVec; ++v) win[m][v] = win[m - 1][v];
        } else {
          int64_t a = p;
#pragma unroll
          for (int m = 1; m < K; ++m) {
            if (a >= 0) {
              if (active) ld4(x + a * C + c0, win[m]);
              int64_t pa = parent[a];
              if (pa < -1 || pa >= a) {
                raise_error(err, TREE_ERR_DEVICE_CHECK);
                pa = -1;
              }
              a = pa;
            } else {
#pragma unroll
              for (int v = 0; v < kConvVec; ++v) win[m][v] = 0.f;
            }
          }
        }
        if (active) ld4(sx + q * kConvChan, win[0]);
        float out[kConvVec];
#pragma unroll
        for (int v = 0; v < kConvVec; ++v) {
          float acc = b[v];
#pragma unroll
          for (int m = 0; m < K; ++m) acc = fmaf(wt[K - 1 - m][v], win[m][v], acc);
          out[v] = acc;
        }
        if (active) st4(y + i * C + c0, out);
      }
      }
    }
    if (!__syncthreads_and(ok)) {
      if (threadIdx.x == 0) drain_stages(full, kFwdStages, c + 1, issued, err);
      return;
    }
  }
}

template <typename T, int K>
__global__ void __launch_bounds__(kConvThreads, K <= 4 ? 2 : 1) conv1d_bwd_kernel(
    const T* __restrict__ x, const T* __restrict__ w, const T* __restrict__ dy, T* __restrict__ dx,
    const int32_t* __restrict__ end, const int32_t* __restrict__ pos, int64_t n_rows, int C,
    int64_t rows_per_group, float* __restrict__ part, int* err) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ uint64_t full[kBwdStages];
  T* stage = reinterpret_cast<T*>(smem_raw);  // [kBwdStages][x, dy][kStageRows][kConvChan]
  const int64_t g0 = static_cast<int64_t>(blockIdx.x) * rows_per_group;
  const int64_t g1 = min(g0 + rows_per_group, n_rows);
  const int ct0 = blockIdx.y * kConvChan;
  const uint32_t row_bytes = static_cast<uint32_t>(min(kConvChan, C - ct0) * sizeof(T));
  const int c0 = ct0 + threadIdx.x * kConvVec;
  const bool active = c0 < C;
  const int n_chunks = static_cast<int>((g1 - g0 + kStageRows - 1) / kStageRows);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kBwdStages; ++s) mbar_init(&full[s], 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  // chunks are consumed last row first: consumption step c reads chunk n_chunks - 1 - c
  int issued = -1;
  auto issue = [&](int c) {
    const int s = c % kBwdStages;
    const int64_t r = g0 + static_cast<int64_t>(n_chunks - 1 - c) * kStageRows;
    const int rows = static_cast<int>(min(static_cast<int64_t>(kStageRows), g1 - r));
    T* dst = stage + s * 2 * kStageRows * kConvChan;
    mbar_arrive_expect_tx(&full[s], 2 * rows * row_bytes);
    stage_rows(dst, x, r, rows, C, ct0, row_bytes, &full[s]);
    stage_rows(dst + kStageRows * kConvChan, dy, r, rows, C, ct0, row_bytes, &full[s]);
    issued = c;
  };
  if (threadIdx.x == 0)
    for (int c = 0; c < min(kBwdStages - 1, n_chunks); ++c) issue(c);

  float wt[K][kConvVec], unused_b[kConvVec];
  load_taps<T, K>(w, static_cast<const T*>(nullptr), c0, active, wt, unused_b);
  float D[K][kConvVec];  // D[m] = sum of dy over the current row's depth-m descendants
  float dwacc[K][kConvVec], dbacc[kConvVec];
#pragma unroll
  for (int v = 0; v < kConvVec; ++v) {
    dbacc[v] = 0.f;
#pragma unroll
    for (int m = 0; m < K; ++m) D[m][v] = dwacc[m][v] = 0.f;
  }
  int64_t end_next = -1;  // subtree_end of the row processed just before (j + 1)

  for (int c = 0; c < n_chunks; ++c) {
    if (threadIdx.x == 0 && c + kBwdStages - 1 < n_chunks) issue(c + kBwdStages - 1);
    const bool ok = mbar_wait(&full[c % kBwdStages], (c / kBwdStages) & 1, err);
    if (ok) {
      const T* sx = stage + (c % kBwdStages) * 2 * kStageRows * kConvChan + threadIdx.x * kConvVec;
      const T* sg = sx + kStageRows * kConvChan;
      const int64_t r = g0 + static_cast<int64_t>(n_chunks - 1 - c) * kStageRows;
      const int rows = static_cast<int>(min(static_cast<int64_t>(kStageRows), g1 - r));
      int eb[kStageRows];  // the chunk's subtree ends, loaded together
#pragma unroll
      for (int q = 0; q < kStageRows; ++q) eb[q] = q < rows ? end[r + q] : 0;
      bool chain = rows == kStageRows && r + kStageRows < g1;
#pragma unroll
      for (int q = 0; q < kStageRows; ++q)
        chain = chain && eb[q] > r + q && eb[q] == (q + 1 < kStageRows ? static_cast<int64_t>(eb[q + 1]) : end_next);
      if (chain) {
        // Every row's only child is the next row: row q's depth-m descendant is row q + m
        // of the chunk, or (q + m >= kStageRows) D[q + m - kStageRows] of the row after the
        // chunk, which D holds. All indices are fixed at compile time.
        float gr[kStageRows][kConvVec];
#pragma unroll
        for (int q = 0; q < kStageRows; ++q) {
          if (active) {
            ld4(sg + q * kConvChan, gr[q]);
          } else {
#pragma unroll
            for (int v = 0; v < kConvVec; ++v) gr[q][v] = 0.f;
          }
        }
#pragma unroll
        for (int q = kStageRows - 1; q >= 0; --q) {
          float xv[kConvVec], out[kConvVec];
          if (active) {
            ld4(sx + q * kConvChan, xv);
          } else {
#pragma unroll
            for (int v = 0; v < kConvVec; ++v) xv[v] = 0.f;
          }
#pragma unroll
          for (int v = 0; v < kConvVec; ++v) {
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < K; ++m) {
              const float d = q + m < kStageRows ? gr[q + m][v] : D[q + m - kStageRows][v];
              acc = fmaf(wt[K - 1 - m][v], d, acc);
              dwacc[K - 1 - m][v] = fmaf(xv[v], d, dwacc[K - 1 - m][v]);
            }
            out[v] = acc;
            dbacc[v] += gr[q][v];
          }
          if (active) st4(dx + (r + q) * C + c0, out);
        }
#pragma unroll
        for (int m = 0; m < K; ++m)
#pragma unroll
          for (int v = 0; v < kConvVec; ++v) D[m][v] = gr[m][v];
        end_next = eb[0];
      } else {
#pragma unroll
      for (int q = kStageRows - 1; q >= 0; --q) {
        const int64_t j = r + q;
        if (q >= rows) continue;
        int64_t e = eb[q];
        if (e < j || e >= n_rows) {  // a subtree holds its root and ends inside the tree
          raise_error(err, TREE_ERR_DEVICE_CHECK);
          e = j;
        }
        if (j + 1 < g1 && j + 1 <= e && end_next == e) {
          // j's only child is j + 1, processed just before: its window, one level down
#pragma unroll
          for (int m = K - 1; m > 0; --m)
#pragma unroll
            for (int v = 0; v < kConvVec; ++v) D[m][v] = D[m - 1][v];
        } else {
#pragma unroll
          for (int m = 1; m < K; ++m)
#pragma unroll
            for (int v = 0; v < kConvVec; ++v) D[m][v] = 0.f;
          if (K > 1 && e > j) {
            // descendants of j within depth K-1, in preorder: a row at depth K-1 below j
            // is added and its subtree skipped; a shallower row steps to the next row
            const int pj = pos[j];
            int64_t rr = j + 1;
            while (rr <= e) {
              const int dr = pos[rr] - pj;
              int64_t er = end[rr];
              if (er < rr) {
                raise_error(err, TREE_ERR_DEVICE_CHECK);
                er = rr;
              }
              if (dr < 1 || dr >= K) {  // depths inconsistent with the subtree intervals
                raise_error(err, TREE_ERR_DEVICE_CHECK);
                rr = er + 1;
                continue;
              }
              if (active) {
                float g[kConvVec];
                ld4(dy + rr * C + c0, g);
#pragma unroll
                for (int m = 1; m < K; ++m)
                  if (dr == m) {
#pragma unroll
                    for (int v = 0; v < kConvVec; ++v) D[m][v] += g[v];
                  }
              }
              rr = dr == K - 1 ? er + 1 : rr + 1;
            }
          }
        }
        end_next = e;
        float xv[kConvVec];
        if (active) {
          ld4(sg + q * kConvChan, D[0]);
          ld4(sx + q * kConvChan, xv);
        } else {
#pragma unroll
          for (int v = 0; v < kConvVec; ++v) D[0][v] = xv[v] = 0.f;
        }
        float out[kConvVec];
#pragma unroll
        for (int v = 0; v < kConvVec; ++v) {
          float acc = 0.f;
#pragma unroll
          for (int m = 0; m < K; ++m) {
            acc = fmaf(wt[K - 1 - m][v], D[m][v], acc);
            dwacc[K - 1 - m][v] = fmaf(xv[v], D[m][v], dwacc[K - 1 - m][v]);
          }
          out[v] = acc;
          dbacc[v] += D[0][v];
        }
        if (active) st4(dx + j * C + c0, out);
      }
      }
    }
    if (!__syncthreads_and(ok)) {
      if (threadIdx.x == 0) drain_stages(full, kBwdStages, c + 1, issued, err);
      return;
    }
  }
  if (active) {
    float* pt = part + static_cast<int64_t>(blockIdx.x) * (K + 1) * C + c0;
#pragma unroll
    for (int k = 0; k < K; ++k) st4(pt + static_cast<int64_t>(k) * C, dwacc[k]);
    st4(pt + static_cast<int64_t>(K) * C, dbacc);
  }
}

// dw[c, k] (k < K) and dbias[c] (k == K) from the per-group partials part[group][k][c]:
// a CTA covers 32 channels with 8 threads per channel, each adding every 8th group in
// fp64; the 8 sums are then added in a fixed order (the result does not depend on
// scheduling).
constexpr int kRedC = 32, kRedG = 8;
__global__ void __launch_bounds__(kRedC * kRedG) conv1d_reduce_kernel(const float* __restrict__ part,
                                                                    int64_t n_groups, int C, int K,
                                                                    float* __restrict__ dw,
                                                                    float* __restrict__ dbias) {
  __shared__ double acc[kRedG][kRedC];
  const int c = blockIdx.x * kRedC + threadIdx.x;
  const int k = blockIdx.y;
  double s = 0.0;
  if (c < C) {
#pragma unroll 4
    for (int64_t g = threadIdx.y; g < n_groups; g += kRedG) s += part[(g * (K + 1) + k) * C + c];
  }
  acc[threadIdx.y][threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.y == 0 && c < C) {
    double tot = 0.0;
#pragma unroll
    for (int q = 0; q < kRedG; ++q) tot += acc[q][threadIdx.x];
    if (k < K) {
      if (dw) dw[static_cast<int64_t>(c) * K + k] = static_cast<float>(tot);
    } else if (dbias) {
      dbias[c] = static_cast<float>(tot);
    }
  }
}

template <typename T, int K>
int launch_fwd(const void* x, const void* w, const void* bias, void* y, const int32_t* parent, int64_t T_,
               int C, cudaStream_t st) {
  if (int rc_ = smem_opt_in(reinterpret_cast<const void*>(conv1d_fwd_kernel<T, K>), static_cast<int>(fwd_smem<T>()))) return rc_;
  const ConvGrid g = conv_grid(T_, C, kFwdTargetCtas);
  dim3 grid(static_cast<unsigned>(g.groups), static_cast<unsigned>(g.ctiles));
  timing_begin(2, st);
  conv1d_fwd_kernel<T, K><<<grid, kConvThreads, fwd_smem<T>(), st>>>(
      static_cast<const T*>(x), static_cast<const T*>(w), static_cast<const T*>(bias), static_cast<T*>(y), parent,
      T_, C, g.rows_per_group, device_error_word());
  TREE_LAUNCH_CHECK("conv1d_fwd_kernel");
  timing_end(2, st);
  return TREE_OK;
}

template <typename T, int K>
int launch_bwd(const void* x, const void* w, const void* dy, void* dx, float* dw, float* dbias,
               const int32_t* end, const int32_t* pos, int64_t T_, int C, float* part, cudaStream_t st) {
  if (int rc_ = smem_opt_in(reinterpret_cast<const void*>(conv1d_bwd_kernel<T, K>), static_cast<int>(bwd_smem<T>()))) return rc_;
  const ConvGrid g = conv_grid(T_, C, kBwdTargetCtas);
  dim3 grid(static_cast<unsigned>(g.groups), static_cast<unsigned>(g.ctiles));
  int* err = device_error_word();
  timing_begin(3, st);
  conv1d_bwd_kernel<T, K><<<grid, kConvThreads, bwd_smem<T>(), st>>>(
      static_cast<const T*>(x), static_cast<const T*>(w), static_cast<const T*>(dy), static_cast<T*>(dx), end, pos,
      T_, C, g.rows_per_group, part, err);
  TREE_LAUNCH_CHECK("conv1d_bwd_kernel");
  if (dw || dbias) {
    dim3 rgrid(static_cast<unsigned>((C + kRedC - 1) / kRedC), static_cast<unsigned>(K + 1));
    conv1d_reduce_kernel<<<rgrid, dim3(kRedC, kRedG), 0, st>>>(part, g.groups, C, K, dw, dbias);
    TREE_LAUNCH_CHECK("conv1d_reduce_kernel");
  }
  timing_end(3, st);
  return TREE_OK;
}

template <typename T>
int dispatch_fwd(int K, const void* x, const void* w, const void* bias, void* y, const int32_t* parent,
                 int64_t T_, int C, cudaStream_t st) {
  switch (K) {
    case 1: return launch_fwd<T, 1>(x, w, bias, y, parent, T_, C, st);
    case 2: return launch_fwd<T, 2>(x, w, bias, y, parent, T_, C, st);
    case 3: return launch_fwd<T, 3>(x, w, bias, y, parent, T_, C, st);
    case 4: return launch_fwd<T, 4>(x, w, bias, y, parent, T_, C, st);
    case 5: return launch_fwd<T, 5>(x, w, bias, y, parent, T_, C, st);
    case 6: return launch_fwd<T, 6>(x, w, bias, y, parent, T_, C, st);
    case 7: return launch_fwd<T, 7>(x, w, bias, y, parent, T_, C, st);
    default: return launch_fwd<T, 8>(x, w, bias, y, parent, T_, C, st);
  }
}

template <typename T>
int dispatch_bwd(int K, const void* x, const void* w, const void* dy, void* dx, float* dw, float* dbias,
                 const int32_t* end, const int32_t* pos, int64_t T_, int C, float* part, cudaStream_t st) {
  switch (K) {
    case 1: return launch_bwd<T, 1>(x, w, dy, dx, dw, dbias, end, pos, T_, C, part, st);
    case 2: return launch_bwd<T, 2>(x, w, dy, dx, dw, dbias, end, pos, T_, C, part, st);
    case 3: return launch_bwd<T, 3>(x, w, dy, dx, dw, dbias, end, pos, T_, C, part, st);
    case 4: return launch_bwd<T, 4>(x, w, dy, dx, dw, dbias, end, pos, T_, C, part, st);
    case 5: return launch_bwd<T, 5>(x, w, dy, dx, dw, dbias, end, pos, T_, C, part, st);
    case 6: return launch_bwd<T, 6>(x, w, dy, dx, dw, dbias, end, pos, T_, C, part, st);
    case 7: return launch_bwd<T, 7>(x, w, dy, dx, dw, dbias, end, pos, T_, C, part, st);
    default: return launch_bwd<T, 8>(x, w, dy, dx, dw, dbias, end, pos, T_, C, part, st);
  }
}

int check_conv_args(int64_t T_, int C, int K, int dtype, const char* who) {
  if (dtype != TREE_DTYPE_F32 && dtype != TREE_DTYPE_BF16) return fail(TREE_ERR_DTYPE, "%s: bad dtype %d", who, dtype);
  if (T_ < 0 || T_ > INT32_MAX) return fail(TREE_ERR_SHAPE, "%s: T = %lld outside [0, 2^31)", who, (long long)T_);
  if (C < 8 || C % 8 != 0 || C > (1 << 24))
    return fail(TREE_ERR_SHAPE, "%s: channels C = %d must be a positive multiple of 8 (<= 2^24)", who, C);
  if (K < 1 || K > kConvMaxK) return fail(TREE_ERR_SHAPE, "%s: kernel size K = %d outside [1, %d]", who, K, kConvMaxK);
  return TREE_OK;
}

}  // namespace

size_t conv1d_ws_bytes(int64_t T_, int C, int K) {
  const ConvGrid g = conv_grid(T_, C, kBwdTargetCtas);
  return round_up(static_cast<size_t>(g.groups) * (K + 1) * C * sizeof(float), 256);
}

}  // namespace tree

using namespace tree;

extern "C" size_t tree_conv1d_workspace_size(int64_t T, int C, int K) {
  if (T < 0 || C < 1 || K < 1 || K > kConvMaxK) return 0;
  return conv1d_ws_bytes(T, C, K);
}

extern "C" int tree_conv1d_fwd(const void* x, const void* w, const void* bias, void* y, const int32_t* parent_row,
                               int64_t T, int C, int K, int dtype, tree_stream_t stream) {
  clear_error();
  int rc = check_conv_args(T, C, K, dtype, "tree_conv1d_fwd");
  if (rc) return rc;
  if (T == 0) return TREE_OK;
  if (!x || !w || !y || !parent_row) return fail(TREE_ERR_INVALID_ARG, "tree_conv1d_fwd: null pointer");
  if (!aligned16(x) || !aligned16(y)) return fail(TREE_ERR_ALIGNMENT, "tree_conv1d_fwd: x / y not 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == TREE_DTYPE_BF16) return dispatch_fwd<__nv_bfloat16>(K, x, w, bias, y, parent_row, T, C, st);
  return dispatch_fwd<float>(K, x, w, bias, y, parent_row, T, C, st);
}

extern "C" int tree_conv1d_bwd(const void* x, const void* w, const void* dy, void* dx, float* dw, float* dbias,
                               const int32_t* subtree_end, const int32_t* position_ids, int64_t T, int C, int K,
                               int dtype, void* workspace, size_t workspace_bytes, tree_stream_t stream) {
  clear_error();
  int rc = check_conv_args(T, C, K, dtype, "tree_conv1d_bwd");
  if (rc) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) {  // no rows: the weight and bias gradients are zero
    if (dw) TREE_CUDA_TRY(cudaMemsetAsync(dw, 0, sizeof(float) * C * K, st));
    if (dbias) TREE_CUDA_TRY(cudaMemsetAsync(dbias, 0, sizeof(float) * C, st));
    return TREE_OK;
  }
  if (!x || !w || !dy || !dx || !subtree_end || !position_ids)
    return fail(TREE_ERR_INVALID_ARG, "tree_conv1d_bwd: null pointer");
  if (!aligned16(x) || !aligned16(dy) || !aligned16(dx))
    return fail(TREE_ERR_ALIGNMENT, "tree_conv1d_bwd: x / dy / dx not 16-byte aligned");
  const size_t need = conv1d_ws_bytes(T, C, K);
  if (workspace_bytes < need)
    return fail(TREE_ERR_WORKSPACE, "tree_conv1d_bwd: workspace of %zu bytes, %zu needed", workspace_bytes, need);
  if (!workspace) return fail(TREE_ERR_INVALID_ARG, "tree_conv1d_bwd: workspace is null");
  if (!aligned256(workspace)) return fail(TREE_ERR_ALIGNMENT, "tree_conv1d_bwd: workspace not 256-byte aligned");
  float* part = static_cast<float*>(workspace);
  if (dtype == TREE_DTYPE_BF16)
    return dispatch_bwd<__nv_bfloat16>(K, x, w, dy, dx, dw, dbias, subtree_end, position_ids, T, C, part, st);
  return dispatch_bwd<float>(K, x, w, dy, dx, dw, dbias, subtree_end, position_ids, T, C, part, st);
}
