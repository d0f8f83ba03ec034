// Shared-logit log-probs, SIMT fp32 kernels (the fp32 path).
//
// Trie packing (agillm.io), "Share logits, preserve every prediction" and "The
// training-loop change is small": one logits row z_r = h_r W per packed row,
// log-softmax, and the log-prob of every occurrence's target; "Same chain rule,
// shared computation graph", Step 1: G_z = p - e_y per target, contributions of
// several targets at one row add. With g_o = dL/dlogp_o:
//   G_z[r] = sum_{o at r} g_o e_{y_o} - c_r softmax(z_r),  c_r = sum_{o at r} g_o.
//
// Forward: a tiled GEMM whose epilogue keeps, per row and vocabulary tile, the
// tile max and sum of exp (never storing the logits) and writes the target logit
// of every occurrence whose target falls in the tile into logp[o]; a per-row
// combine kernel forms LSE and subtracts it from the row's target logits.
// Backward: the same GEMM recomputes z and writes G_z (fp32) to the workspace,
// then two GEMMs give dH = G_z W^T and dW = H^T G_z.
#include <cmath>

#include "attn_internal.h"
#include "common.h"
#include "device_common.cuh"

namespace tree {

constexpr int GB = 64;   // output tile rows and columns
constexpr int GK = 16;   // depth of a K step
constexpr int GT = 256;  // threads: 16 x 16, each 4 x 4 outputs

enum { EPI_STORE = 0, EPI_LSE = 1, EPI_GZ = 2 };

struct GemmEpi {
  // EPI_STORE
  void* c;
  int64_t ldc;
  int out_bf16;
  // EPI_LSE / EPI_GZ
  int64_t T, V;
  const int32_t* row_ptr;
  const int32_t* perm;
  const int32_t* targets;
  int64_t n_occ;
  float* part_max;
  float* part_sum;
  float* logp;        // EPI_LSE: receives target logits
  const float* lse;   // EPI_GZ
  const float* crow;  // EPI_GZ
  const float* grad;  // EPI_GZ
  float* gz;          // EPI_GZ: [T, V]
  int* err;
};

// C[m, n] = sum_k A(m, k) B(k, n); A(m, k) = A[m*sam + k*sak], B(k, n) = B[k*sbk + n*sbn].
template <typename TA, typename TB, int EPI>
__global__ void __launch_bounds__(GT)
simt_gemm_kernel(const TA* __restrict__ A, int64_t sam, int64_t sak, const TB* __restrict__ B,
                 int64_t sbk, int64_t sbn, int64_t M, int64_t N, int64_t K, GemmEpi ep) {
  __shared__ float As[GK][GB + 4], Bs[GK][GB + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * GB, n0 = static_cast<int64_t>(blockIdx.x) * GB;
  float acc[4][4] = {};
  for (int64_t k0 = 0; k0 < K; k0 += GK) {
    __syncthreads();
    for (int e = threadIdx.x; e < GB * GK; e += GT) {
      // A: k fastest when A is k-contiguous, else m fastest
      int mm, kk;
      if (sak == 1) { mm = e / GK; kk = e % GK; } else { kk = e / GB; mm = e % GB; }
      const int64_t m = m0 + mm, k = k0 + kk;
      As[kk][mm] = (m < M && k < K) ? to_f32(A[m * sam + k * sak]) : 0.f;
      int nn, kb;
      if (sbn == 1) { kb = e / GB; nn = e % GB; } else { nn = e / GK; kb = e % GK; }
      const int64_t n = n0 + nn, kq = k0 + kb;
      Bs[kb][nn] = (n < N && kq < K) ? to_f32(B[kq * sbk + n * sbn]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < GK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        a[t] = As[kk][ty * 4 + t];
        b[t] = Bs[kk][tx * 4 + t];
      }
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] += a[x] * b[y];
    }
  }
  if constexpr (EPI == EPI_STORE) {
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int64_t m = m0 + ty * 4 + x;
      if (m >= M) continue;
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const int64_t n = n0 + tx * 4 + y;
        if (n >= N) continue;
        if (ep.out_bf16)
          static_cast<__nv_bfloat16*>(ep.c)[m * ep.ldc + n] = __float2bfloat16_rn(acc[x][y]);
        else
          static_cast<float*>(ep.c)[m * ep.ldc + n] = acc[x][y];
      }
    }
  } else {
    const int64_t c_lo = n0 + tx * 4;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int64_t m = m0 + ty * 4 + x;
      const bool row_ok = m < M;
      int64_t o_begin = 0, o_end = 0;
      if (row_ok) {
        o_begin = ep.row_ptr[m];
        o_end = ep.row_ptr[m + 1];
        if (o_begin < 0 || o_end < o_begin || o_end > ep.n_occ) {
          raise_error(ep.err, TREE_ERR_DEVICE_CHECK);
          o_end = o_begin = 0;
        }
      }
      if constexpr (EPI == EPI_LSE) {
        float mx = -INFINITY;
#pragma unroll
        for (int y = 0; y < 4; ++y)
          if (c_lo + y < N) mx = fmaxf(mx, acc[x][y]);
#pragma unroll
        for (int off = 1; off < 16; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        float sm = 0.f;
#pragma unroll
        for (int y = 0; y < 4; ++y)
          if (c_lo + y < N) sm += expf(acc[x][y] - mx);
#pragma unroll
        for (int off = 1; off < 16; off <<= 1) sm += __shfl_xor_sync(0xffffffffu, sm, off);
        if (row_ok && tx == 0) {
          ep.part_max[static_cast<int64_t>(blockIdx.x) * ep.T + m] = mx;
          ep.part_sum[static_cast<int64_t>(blockIdx.x) * ep.T + m] = sm;
        }
        for (int64_t q = o_begin; q < o_end; ++q) {
          const int o = ep.perm[q];
          if (o < 0 || o >= ep.n_occ) { raise_error(ep.err, TREE_ERR_DEVICE_CHECK); continue; }
          const int64_t y = ep.targets[o];
          if (y < 0 || y >= ep.V) { raise_error(ep.err, TREE_ERR_DEVICE_CHECK); continue; }
          if (y >= c_lo && y < c_lo + 4) {
#pragma unroll
            for (int t = 0; t < 4; ++t)
              if (y == c_lo + t) ep.logp[o] = acc[x][t];
          }
        }
      } else {  // EPI_GZ
        if (!row_ok) continue;
        const float l = ep.lse[m], c = ep.crow[m];
        float g[4];
#pragma unroll
        for (int y = 0; y < 4; ++y) g[y] = -c * expf(acc[x][y] - l);
        for (int64_t q = o_begin; q < o_end; ++q) {
          const int o = ep.perm[q];
          if (o < 0 || o >= ep.n_occ) { raise_error(ep.err, TREE_ERR_DEVICE_CHECK); continue; }
          const int64_t y = ep.targets[o];
          if (y < 0 || y >= ep.V) { raise_error(ep.err, TREE_ERR_DEVICE_CHECK); continue; }
#pragma unroll
          for (int t = 0; t < 4; ++t)
            if (y == c_lo + t) g[t] += ep.grad[o];
        }
#pragma unroll
        for (int y = 0; y < 4; ++y)
          if (c_lo + y < N) ep.gz[m * ep.V + c_lo + y] = g[y];
      }
    }
  }
}

// Per row: LSE from the tile partials, then logp[o] = z_target - LSE for the row's occurrences.
__global__ void lse_combine_kernel(const float* __restrict__ part_max, const float* __restrict__ part_sum,
                                   int n_tiles, int64_t T, const int32_t* __restrict__ row_ptr,
                                   const int32_t* __restrict__ perm, int64_t n_occ,
                                   float* __restrict__ lse, float* __restrict__ logp) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= T) return;
  float mx = -INFINITY;
  for (int t = 0; t < n_tiles; ++t) mx = fmaxf(mx, part_max[t * T + r]);
  float s = 0.f;
  for (int t = 0; t < n_tiles; ++t) s += part_sum[t * T + r] * expf(part_max[t * T + r] - mx);
  const float L = mx + logf(s);
  lse[r] = L;
  const int64_t b = row_ptr[r], e = row_ptr[r + 1];
  if (b < 0 || e < b || e > n_occ) return;  // reported by the GEMM epilogue
  for (int64_t q = b; q < e; ++q) {
    const int o = perm[q];
    if (o >= 0 && o < n_occ) logp[o] -= L;
  }
}

// c_r = sum of grad_logp over row r's occurrences.
__global__ void row_grad_sum_kernel(const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ perm,
                                    const float* __restrict__ grad, int64_t T, int64_t n_occ,
                                    float* __restrict__ crow) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= T) return;
  const int64_t b = row_ptr[r], e = row_ptr[r + 1];
  float c = 0.f;
  if (b >= 0 && e >= b && e <= n_occ)
    for (int64_t q = b; q < e; ++q) {
      const int o = perm[q];
      if (o >= 0 && o < n_occ) c += grad[o];
    }
  crow[r] = c;
}

template <typename T>
static int fwd_impl(const LogprobArgs& a, cudaStream_t st) {
  GemmEpi ep{};
  ep.T = a.T; ep.V = a.V; ep.row_ptr = a.row_ptr; ep.perm = a.perm; ep.targets = a.targets;
  ep.n_occ = a.n_occ; ep.part_max = a.ws.part_max; ep.part_sum = a.ws.part_sum; ep.logp = a.logp;
  ep.err = device_error_word();
  const int n_vt = static_cast<int>((a.V + GB - 1) / GB);
  dim3 grid(n_vt, static_cast<unsigned>((a.T + GB - 1) / GB));
  const T* H = static_cast<const T*>(a.h);
  const T* W = static_cast<const T*>(a.w);
  simt_gemm_kernel<T, T, EPI_LSE><<<grid, GT, 0, st>>>(H, a.K, 1, W, a.V, 1, a.T, a.V, a.K, ep);
  TREE_LAUNCH_CHECK("simt_gemm_kernel<lse>");
  lse_combine_kernel<<<static_cast<unsigned>((a.T + 255) / 256), 256, 0, st>>>(
      a.ws.part_max, a.ws.part_sum, n_vt, a.T, a.row_ptr, a.perm, a.n_occ, a.lse, a.logp);
  TREE_LAUNCH_CHECK("lse_combine_kernel");
  return TREE_OK;
}

template <typename T>
static int bwd_impl(const LogprobArgs& a, cudaStream_t st) {
  row_grad_sum_kernel<<<static_cast<unsigned>((a.T + 255) / 256), 256, 0, st>>>(
      a.row_ptr, a.perm, a.grad, a.T, a.n_occ, a.ws.crow);
  TREE_LAUNCH_CHECK("row_grad_sum_kernel");
  GemmEpi ep{};
  ep.T = a.T; ep.V = a.V; ep.row_ptr = a.row_ptr; ep.perm = a.perm; ep.targets = a.targets;
  ep.n_occ = a.n_occ; ep.lse = a.lse; ep.crow = a.ws.crow; ep.grad = a.grad;
  ep.gz = static_cast<float*>(a.ws.gz); ep.err = device_error_word();
  const T* H = static_cast<const T*>(a.h);
  const T* W = static_cast<const T*>(a.w);
  const float* G = static_cast<const float*>(a.ws.gz);
  dim3 g1(static_cast<unsigned>((a.V + GB - 1) / GB), static_cast<unsigned>((a.T + GB - 1) / GB));
  simt_gemm_kernel<T, T, EPI_GZ><<<g1, GT, 0, st>>>(H, a.K, 1, W, a.V, 1, a.T, a.V, a.K, ep);
  TREE_LAUNCH_CHECK("simt_gemm_kernel<gz>");
  GemmEpi e2{};
  e2.out_bf16 = a.dtype == TREE_DTYPE_BF16;
  // dH[T, K] = G[T, V] . W^T : A(m, k) = G[m*V + k], B(k, n) = W[n*V + k]
  e2.c = a.dh; e2.ldc = a.K;
  dim3 g2(static_cast<unsigned>((a.K + GB - 1) / GB), static_cast<unsigned>((a.T + GB - 1) / GB));
  simt_gemm_kernel<float, T, EPI_STORE><<<g2, GT, 0, st>>>(G, a.V, 1, W, 1, a.V, a.T, a.K, a.V, e2);
  TREE_LAUNCH_CHECK("simt_gemm_kernel<dh>");
  // dW[K, V] = H^T . G : A(m, k) = H[k*K + m], B(k, n) = G[k*V + n]
  e2.c = a.dw; e2.ldc = a.V;
  dim3 g3(static_cast<unsigned>((a.V + GB - 1) / GB), static_cast<unsigned>((a.K + GB - 1) / GB));
  simt_gemm_kernel<T, float, EPI_STORE><<<g3, GT, 0, st>>>(H, 1, a.K, G, a.V, 1, a.K, a.V, a.T, e2);
  TREE_LAUNCH_CHECK("simt_gemm_kernel<dw>");
  return TREE_OK;
}

int lse_combine_launch(const float* part_max, const float* part_sum, int n_tiles, int64_t T, const int32_t* row_ptr,
                       const int32_t* perm, int64_t n_occ, float* lse, float* logp, cudaStream_t st) {
  lse_combine_kernel<<<static_cast<unsigned>((T + 255) / 256), 256, 0, st>>>(part_max, part_sum, n_tiles, T, row_ptr,
                                                                           perm, n_occ, lse, logp);
  TREE_LAUNCH_CHECK("lse_combine_kernel");
  return TREE_OK;
}

int row_grad_sum_launch(const int32_t* row_ptr, const int32_t* perm, const float* grad, int64_t T, int64_t n_occ,
                        float* crow, cudaStream_t st) {
  row_grad_sum_kernel<<<static_cast<unsigned>((T + 255) / 256), 256, 0, st>>>(row_ptr, perm, grad, T, n_occ, crow);
  TREE_LAUNCH_CHECK("row_grad_sum_kernel");
  return TREE_OK;
}

int logprob_fwd_simt(const LogprobArgs& a, cudaStream_t st) {
  return a.dtype == TREE_DTYPE_BF16 ? fwd_impl<__nv_bfloat16>(a, st) : fwd_impl<float>(a, st);
}

int logprob_bwd_simt(const LogprobArgs& a, cudaStream_t st) {
  return a.dtype == TREE_DTYPE_BF16 ? bwd_impl<__nv_bfloat16>(a, st) : bwd_impl<float>(a, st);
}

}  // namespace tree
