// Shared-logit log-probs in fp32: the GEMMs on the tcgen05 tensor cores (kind::tf32 with the
// two-term split of tc32.cuh), the softmax statistics and G_z in their epilogues.
//
// Trie packing (agillm.io), "Share logits, preserve every prediction" and "The training-loop
// change is small": one logits row z_r = h_r W per packed row, log-softmax, and the log-prob
// of every occurrence's target; "Same chain rule, shared computation graph", Step 1:
// G_z = p - e_y per target, contributions of several targets at one row add. With
// g_o = dL/dlogp_o:
//   G_z[r] = sum_{o at r} g_o e_{y_o} - c_r softmax(z_r),  c_r = sum_{o at r} g_o.
//
// Forward: z tiles of 128 rows x 128 vocabulary columns; the epilogue keeps per row and tile
// the max and the sum of exp (the logits are never stored) and writes the target logit of
// every occurrence whose target falls in the tile into logp[o]; a per-row combine forms LSE
// and subtracts it. Backward: the same GEMM recomputes z and writes G_z (fp32) to the
// workspace, then dH = G_z W^T and dW = H^T G_z.
//
// GEMM kernel: 128 threads, one 128 x 128 output tile per CTA, K in steps of 32 (one 128-byte
// swizzle row of fp32), operand tiles double-buffered in shared memory: while the MMAs of
// step k run, the threads load, split and store step k + 1; every kGroup steps the products
// are added into a running fp32 sum in TMEM. Thread t then owns accumulator row t (TMEM
// lane t) for the epilogue.
#include <cmath>
#include <type_traits>

#include "attn_internal.h"
#include "common.h"
#include "device_common.cuh"
#include "tc32.cuh"

namespace tree {
namespace ltc32 {

using namespace sm100;
using namespace tc32;

constexpr int TM = 128, TN = 128, TK = 32;
constexpr int kThreads = 128;
constexpr int kOpB = TM * TK * 4;                 // one operand tile, hi or lo (16 KB)
constexpr int kStageB = 4 * kOpB;                 // A hi/lo + B hi/lo
constexpr int kSmem = 2 * kStageB + 1024 + 256;   // two stages

enum { EPI_STORE = 0, EPI_LSE = 1, EPI_GZ = 2 };

struct Epi {
  void* c;            // EPI_STORE: [M, ldc] fp32 or bf16
  int64_t ldc;
  int out_bf16;
  int64_t T, V;       // EPI_LSE / EPI_GZ
  const int32_t* row_ptr;
  const int32_t* perm;
  const int32_t* targets;
  int64_t n_occ;
  float* part_max;    // [n_tiles, T]
  float* part_sum;
  float* logp;        // EPI_LSE: receives target logits
  const float* lse;   // EPI_GZ
  const float* crow;
  const float* grad;
  float* gz;          // EPI_GZ: [T, V]
  int* err;
};

// One K step of a 128-row operand tile: element (r, k) = X[(r0 + r) * s_r + (k0 + k) * s_k],
// zero outside [0, rows) x [0, K). One of s_r, s_k is 1; 4 consecutive elements along it
// are loaded at once (rows and K are multiples of 4 there).
template <typename TX>
__device__ __forceinline__ void stage_op(const TX* X, int64_t s_r, int64_t s_k, int64_t r0, int64_t rows,
                                         int64_t k0, int64_t K, uint8_t* hi, uint8_t* lo) {
  if (s_k == 1) {
    for (int idx = threadIdx.x; idx < TM * TK / 4; idx += kThreads) {
      const int r = idx / (TK / 4), c = (idx % (TK / 4)) * 4;
      const int64_t g = r0 + r, kk = k0 + c;
      const float4 x = (g < rows && kk < K) ? load4(X + g * s_r + kk) : make_float4(0.f, 0.f, 0.f, 0.f);
      put4<TM>(hi, lo, r, c, x);
    }
  } else {
    for (int idx = threadIdx.x; idx < TM * TK / 4; idx += kThreads) {
      const int r = (idx % (TM / 4)) * 4, c = idx / (TM / 4);
      const int64_t g = r0 + r, kk = k0 + c;
      const float4 x = (g < rows && kk < K) ? load4(X + g + kk * s_k) : make_float4(0.f, 0.f, 0.f, 0.f);
      put1<TM>(hi, lo, r + 0, c, x.x);
      put1<TM>(hi, lo, r + 1, c, x.y);
      put1<TM>(hi, lo, r + 2, c, x.z);
      put1<TM>(hi, lo, r + 3, c, x.w);
    }
  }
}

// The tensor cores' fp32 accumulation does not round to nearest and its error grows with
// the number of MMAs adding into one accumulator; over a long K (dW sums over every row)
// that would leave fp32 results short of fp32 accuracy. So the MMAs of kGroup K steps go
// to a fresh TMEM block, which is then added into a running sum with IEEE fp32 adds.
constexpr int kGroup = 4;

__device__ __forceinline__ void tmem_accumulate128(uint32_t run, uint32_t step, bool first) {
#pragma unroll 1
  for (int c0 = 0; c0 < TN; c0 += 32) {
    uint32_t x[32], y[32];
    tmem_ld32(step + c0, x);
    if (!first) tmem_ld32(run + c0, y);
    tmem_ld_wait();
    if (!first) {
#pragma unroll
      for (int c = 0; c < 32; ++c) x[c] = __float_as_uint(__uint_as_float(x[c]) + __uint_as_float(y[c]));
    }
    tmem_st32(run + c0, x);
  }
  tmem_st_wait();
}

// C[m, n] = sum_k A(m, k) B(k, n); A(m, k) = A[m*sam + k*sak], B(k, n) = B[k*sbk + n*sbn].
template <typename TA, typename TB, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
lm_gemm_tc32_kernel(const TA* __restrict__ A, int64_t sam, int64_t sak, const TB* __restrict__ B, int64_t sbk,
                    int64_t sbn, int64_t M, int64_t N, int64_t K, Epi ep) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(base + 2 * kStageB);  // [2] one per stage
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 2);
  const int t = threadIdx.x, warp = t / 32;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * TM, n0 = static_cast<int64_t>(blockIdx.x) * TN;
  if (t == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbarrier_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 2 * TN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tstep = *tmem_slot, tmem = tstep + TN;  // a group's products; the running sum
  const uint32_t lanes = static_cast<uint32_t>(warp * 32) << 16;
  constexpr bool a_exact = !std::is_same<TA, float>::value, b_exact = !std::is_same<TB, float>::value;

  const int64_t n_k = (K + TK - 1) / TK;
  uint32_t used[2] = {0, 0};  // commits issued per stage
  bool ok = true;
  for (int64_t kb = 0; kb < n_k; ++kb) {
    const int s = static_cast<int>(kb & 1);
    uint8_t* st = base + s * kStageB;
    if (used[s] > 0) {  // the MMAs that last read this stage are done
      ok = mbar_wait(&bar[s], (used[s] - 1) & 1, ep.err);
      if (!(ok = __syncthreads_and(ok) != 0)) break;
    }
    stage_op(A, sam, sak, m0, M, kb * TK, K, st, st + kOpB);
    stage_op(B, sbn, sbk, n0, N, kb * TK, K, st + 2 * kOpB, st + 3 * kOpB);
    fence_proxy_async_smem();
    __syncthreads();
    if (t == 0) {
      tc_fence_after();
      mma3<TM, TN, TK>(tstep, smem_u32(st), smem_u32(st + kOpB), smem_u32(st + 2 * kOpB),
                       smem_u32(st + 3 * kOpB), kb % kGroup ? 1u : 0u, a_exact, b_exact);
      mma_commit(&bar[s]);
    }
    ++used[s];
    if (kb % kGroup == kGroup - 1 || kb == n_k - 1) {  // the group's MMAs done: add it to the sum
      ok = mbar_wait(&bar[s], (used[s] - 1) & 1, ep.err);
      if (!(ok = __syncthreads_and(ok) != 0)) break;
      tc_fence_after();
      tmem_accumulate128(tmem + lanes, tstep + lanes, kb < kGroup);
      tc_fence_before();  // the next group's MMAs overwrite the step block
    }
  }
  // the last commit covers every MMA issued before it
  if (ok && n_k > 0) {
    const int s = static_cast<int>((n_k - 1) & 1);
    ok = mbar_wait(&bar[s], (used[s] - 1) & 1, ep.err);
  }
  ok = __syncthreads_and(ok) != 0;
  tc_fence_after();

  if (ok) {
    const int64_t m = m0 + t;
    const bool row_ok = m < M;
    int64_t o_begin = 0, o_end = 0;
    if constexpr (EPI != EPI_STORE) {
      if (row_ok) {
        o_begin = ep.row_ptr[m];
        o_end = ep.row_ptr[m + 1];
        if (o_begin < 0 || o_end < o_begin || o_end > ep.n_occ) {
          raise_error(ep.err, TREE_ERR_DEVICE_CHECK);
          o_end = o_begin = 0;
        }
      }
    }
    float mx = -INFINITY, sm = 0.f, l = 0.f, c = 0.f;
    if constexpr (EPI == EPI_GZ) {
      if (row_ok) {
        l = ep.lse[m];
        c = ep.crow[m];
      }
    }
#pragma unroll 1
    for (int c0 = 0; c0 < TN; c0 += 32) {
      uint32_t u[32];
      tmem_ld32(tmem + lanes + c0, u);
      tmem_ld_wait();
      float z[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) z[e] = __uint_as_float(u[e]);
      const int64_t nb = n0 + c0;
      if constexpr (EPI == EPI_STORE) {
        if (row_ok) {
          if (ep.out_bf16) {
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(ep.c) + m * ep.ldc;
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (nb + e < N) out[nb + e] = __float2bfloat16_rn(z[e]);
          } else {
            float* out = static_cast<float*>(ep.c) + m * ep.ldc;
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (nb + e < N) out[nb + e] = z[e];
          }
        }
      } else if constexpr (EPI == EPI_LSE) {
        float cm = -INFINITY;
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (nb + e < N) cm = fmaxf(cm, z[e]);
        if (cm > -INFINITY) {
          const float nm = fmaxf(mx, cm);
          float s2 = 0.f;
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (nb + e < N) s2 += expf(z[e] - nm);
          sm = sm * expf(mx - nm) + s2;
          mx = nm;
        }
        for (int64_t qq = o_begin; qq < o_end; ++qq) {
          const int o = ep.perm[qq];
          if (o < 0 || o >= ep.n_occ) { raise_error(ep.err, TREE_ERR_DEVICE_CHECK); continue; }
          const int64_t y = ep.targets[o];
          if (y < 0 || y >= ep.V) { raise_error(ep.err, TREE_ERR_DEVICE_CHECK); continue; }
          if (y >= nb && y < nb + 32) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (y == nb + e) ep.logp[o] = z[e];
          }
        }
      } else {  // EPI_GZ
        if (row_ok) {
#pragma unroll
          for (int e = 0; e < 32; ++e) z[e] = -c * expf(z[e] - l);
          for (int64_t qq = o_begin; qq < o_end; ++qq) {
            const int o = ep.perm[qq];
            if (o < 0 || o >= ep.n_occ) { raise_error(ep.err, TREE_ERR_DEVICE_CHECK); continue; }
            const int64_t y = ep.targets[o];
            if (y < 0 || y >= ep.V) { raise_error(ep.err, TREE_ERR_DEVICE_CHECK); continue; }
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (y == nb + e) z[e] += ep.grad[o];
          }
          float* out = ep.gz + m * ep.V;
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (nb + e < N) out[nb + e] = z[e];
        }
      }
    }
    if constexpr (EPI == EPI_LSE) {
      if (row_ok) {
        ep.part_max[static_cast<int64_t>(blockIdx.x) * ep.T + m] = mx;
        ep.part_sum[static_cast<int64_t>(blockIdx.x) * ep.T + m] = sm;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tstep, 2 * TN);
  }
}

template <typename TA, typename TB, int EPI>
int gemm(const TA* A, int64_t sam, int64_t sak, const TB* B, int64_t sbk, int64_t sbn, int64_t M, int64_t N,
         int64_t K, const Epi& ep, cudaStream_t st, const char* name) {
  auto* kern = lm_gemm_tc32_kernel<TA, TB, EPI>;
  int rc = smem_opt_in(reinterpret_cast<const void*>(kern), kSmem);
  if (rc) return rc;
  dim3 grid(static_cast<unsigned>((N + TN - 1) / TN), static_cast<unsigned>((M + TM - 1) / TM));
  kern<<<grid, kThreads, kSmem, st>>>(A, sam, sak, B, sbk, sbn, M, N, K, ep);
  TREE_LAUNCH_CHECK(name);
  return TREE_OK;
}

// Per row: LSE from the tile partials, then logp[o] = z_target - LSE for the row's occurrences.
__global__ void lse_combine_kernel(const float* __restrict__ part_max, const float* __restrict__ part_sum,
                                   int n_tiles, int64_t T, const int32_t* __restrict__ row_ptr,
                                   const int32_t* __restrict__ perm, int64_t n_occ, float* __restrict__ lse,
                                   float* __restrict__ logp) {
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

}  // namespace ltc32

int lse_combine_launch(const float* part_max, const float* part_sum, int n_tiles, int64_t T, const int32_t* row_ptr,
                       const int32_t* perm, int64_t n_occ, float* lse, float* logp, cudaStream_t st) {
  ltc32::lse_combine_kernel<<<static_cast<unsigned>((T + 255) / 256), 256, 0, st>>>(part_max, part_sum, n_tiles, T,
                                                                                  row_ptr, perm, n_occ, lse, logp);
  TREE_LAUNCH_CHECK("lse_combine_kernel");
  return TREE_OK;
}

int row_grad_sum_launch(const int32_t* row_ptr, const int32_t* perm, const float* grad, int64_t T, int64_t n_occ,
                        float* crow, cudaStream_t st) {
  ltc32::row_grad_sum_kernel<<<static_cast<unsigned>((T + 255) / 256), 256, 0, st>>>(row_ptr, perm, grad, T, n_occ,
                                                                                   crow);
  TREE_LAUNCH_CHECK("row_grad_sum_kernel");
  return TREE_OK;
}

int logprob_fwd_tc32(const LogprobArgs& a, cudaStream_t st) {
  using namespace ltc32;
  Epi ep{};
  ep.T = a.T; ep.V = a.V; ep.row_ptr = a.row_ptr; ep.perm = a.perm; ep.targets = a.targets;
  ep.n_occ = a.n_occ; ep.part_max = a.ws.part_max; ep.part_sum = a.ws.part_sum; ep.logp = a.logp;
  ep.err = device_error_word();
  const float* H = static_cast<const float*>(a.h);
  const float* W = static_cast<const float*>(a.w);
  int rc = gemm<float, float, EPI_LSE>(H, a.K, 1, W, a.V, 1, a.T, a.V, a.K, ep, st, "lm_gemm_tc32_kernel<lse>");
  if (rc) return rc;
  const int n_vt = static_cast<int>((a.V + TN - 1) / TN);
  return lse_combine_launch(a.ws.part_max, a.ws.part_sum, n_vt, a.T, a.row_ptr, a.perm, a.n_occ, a.lse, a.logp, st);
}

int logprob_bwd_tc32(const LogprobArgs& a, cudaStream_t st) {
  using namespace ltc32;
  int rc = row_grad_sum_launch(a.row_ptr, a.perm, a.grad, a.T, a.n_occ, a.ws.crow, st);
  if (rc) return rc;
  Epi ep{};
  ep.T = a.T; ep.V = a.V; ep.row_ptr = a.row_ptr; ep.perm = a.perm; ep.targets = a.targets;
  ep.n_occ = a.n_occ; ep.lse = a.lse; ep.crow = a.ws.crow; ep.grad = a.grad;
  ep.gz = static_cast<float*>(a.ws.gz); ep.err = device_error_word();
  const float* H = static_cast<const float*>(a.h);
  const float* W = static_cast<const float*>(a.w);
  const float* G = static_cast<const float*>(a.ws.gz);
  if ((rc = gemm<float, float, EPI_GZ>(H, a.K, 1, W, a.V, 1, a.T, a.V, a.K, ep, st, "lm_gemm_tc32_kernel<gz>")))
    return rc;
  Epi e2{};
  e2.err = ep.err;
  // dH[T, K] = G[T, V] . W^T : A(m, k) = G[m*V + k], B(k, n) = W[n*V + k]
  e2.c = a.dh; e2.ldc = a.K; e2.out_bf16 = 0;
  if ((rc = gemm<float, float, EPI_STORE>(G, a.V, 1, W, 1, a.V, a.T, a.K, a.V, e2, st, "lm_gemm_tc32_kernel<dh>")))
    return rc;
  // dW[K, V] = H^T . G : A(m, k) = H[k*K + m], B(k, n) = G[k*V + n]
  e2.c = a.dw; e2.ldc = a.V; e2.out_bf16 = 0;
  return gemm<float, float, EPI_STORE>(H, 1, a.K, G, a.V, 1, a.K, a.V, a.T, e2, st, "lm_gemm_tc32_kernel<dw>");
}

}  // namespace tree
