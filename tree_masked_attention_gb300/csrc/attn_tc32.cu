// Tree attention on the tcgen05 tensor cores for head size 64, fp32 or bf16 storage: every
// contraction (S = Q K^T, O = P V, dP = dO V^T, dV = P^T dO, dK = dS^T Q, dQ = dS K) is a
// kind::tf32 MMA with the two-term split of tc32.cuh, so fp32 inputs keep fp32 accuracy
// (the split's error is about 2^-21 per product) and bf16 inputs, exact in tf32, take one
// pass per contraction of P or dS and none of the lo-terms of their own operands.
//
// Visibility (Tree Training, arXiv 2511.00413, §3.2 "Attention Mask"; Trie packing "Step 2
// - Allow only ancestors and self"): key j is visible to query i iff j <= i <= subtree_end[j].
// A key tile with max(subtree_end) below a query tile's first row is skipped; the queries a
// key tile serves are the contiguous rows from its first key to that maximum.
//
// Kernels (128 threads; thread t owns TMEM lane t, i.e. one query row or one key row):
//   forward   one CTA per (128 query rows, query head); 64-key tiles; online softmax in
//             registers (base 2), O accumulated in registers from a fresh P V per tile.
//   dK / dV   one CTA per (128 keys, KV head); every query head of the group and every 32-row
//             query tile the key tile serves, in a fixed order; each step's dV and dK come
//             out of the MMAs into a fresh TMEM block and are added into running sums in fp32.
//   dQ        one CTA per (128 query rows, query head); 32-key tiles in key order, each
//             tile's dQ added into a running sum likewise.
// The backward takes no atomics: both gradients come out in one fixed order, so repeated
// calls are bitwise equal whatever `deterministic` asks.
#include <cmath>
#include <type_traits>

#include "attn_internal.h"
#include "common.h"
#include "device_common.cuh"
#include "tc32.cuh"

namespace tree {
namespace atc32 {

using namespace sm100;
using namespace tc32;

constexpr int kThreads = 128;
constexpr int BM = 128;  // query rows (forward, dQ) or keys (dK/dV) per CTA = TMEM lanes
constexpr int D = 64;
constexpr int BNF = 64;  // keys per forward step
constexpr int BQ = 32;   // query rows per dK/dV step
constexpr int BNQ = 32;  // keys per dQ step
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct Params {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  const void* dout;
  const float* delta;
  void* dq;
  void* dk;
  void* dv;
  const int32_t* end;
  const int32_t* kmax32;
  int64_t T;
  int Hq, Hkv;
  float scale, scale_log2;
  int* err;
};

template <typename T>
constexpr bool kExact = std::is_same<T, __nv_bfloat16>::value;

__device__ __forceinline__ void store4(float* p, float4 x) { *reinterpret_cast<float4*>(p) = x; }
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 x) {
  uint2 u;
  u.x = pack_bf16(x.x, x.y);
  u.y = pack_bf16(x.z, x.w);
  *reinterpret_cast<uint2*>(p) = u;
}

// Rows [r0, r0 + R) of a [T, H, D] tensor at head h -> a K-major tile (rows, D) and, when
// `tr` is set, its transpose (D rows, R columns); rows past T are zero.
template <int R, typename T>
__device__ __forceinline__ void stage_rows(const T* src, int64_t r0, int64_t n, int H, int h, uint8_t* hi,
                                           uint8_t* lo, uint8_t* thi, uint8_t* tlo) {
  for (int idx = threadIdx.x; idx < R * (D / 4); idx += kThreads) {
    const int r = idx / (D / 4), c = (idx % (D / 4)) * 4;
    const int64_t g = r0 + r;
    const float4 x = g < n ? load4(src + (g * H + h) * D + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    if (hi) put4<R>(hi, lo, r, c, x);
    if (thi) {
      put1<D>(thi, tlo, c + 0, r, x.x);
      put1<D>(thi, tlo, c + 1, r, x.y);
      put1<D>(thi, tlo, c + 2, r, x.z);
      put1<D>(thi, tlo, c + 3, r, x.w);
    }
  }
}

__device__ __forceinline__ void ld_row32(uint32_t taddr, float (&x)[32]) {
  uint32_t r[32];
  tmem_ld32(taddr, r);
  tmem_ld_wait();
#pragma unroll
  for (int c = 0; c < 32; ++c) x[c] = __uint_as_float(r[c]);
}

// The tensor cores' fp32 accumulation does not round to nearest, and its error grows with
// the number of MMAs that add into one accumulator (a thousand-row chain put dV 2e-5
// relative off). So each step's products go to a fresh TMEM block (a dozen MMAs), and the
// running sum is kept in a second block, added to with IEEE fp32 adds: `run` (+)= `step`
// over D columns of this warp's lanes; `first` copies instead of adding.
__device__ __forceinline__ void tmem_accumulate(uint32_t run, uint32_t step, bool first) {
#pragma unroll
  for (int c0 = 0; c0 < D; c0 += 32) {
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

// Waits for the next MMA commit on `bar`; every thread of the CTA takes part and gets the
// same answer.
__device__ __forceinline__ bool wait_mma(uint64_t* bar, uint32_t& phase, int* err) {
  const bool ok = mbar_wait(bar, phase, err);
  phase ^= 1;
  const bool all = __syncthreads_and(ok) != 0;
  tc_fence_after();
  return all;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// ------------------------------------------------------------------------ forward
constexpr int kQB = BM * D * 4, kKB = BNF * D * 4, kPB = BM * BNF * 4;
constexpr int kFwdSmem = 2 * (kQB + 2 * kKB + kPB) + 1024 + 512;

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_tc32_kernel(Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint8_t *Qh = base, *Ql = Qh + kQB, *Kh = Ql + kQB, *Kl = Kh + kKB, *Vh = Kl + kKB, *Vl = Vh + kKB,
          *Ph = Vl + kKB, *Pl = Ph + kPB;
  int32_t* ends = reinterpret_cast<int32_t*>(Pl + kPB);
  uint64_t* bar = reinterpret_cast<uint64_t*>(ends + BNF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);

  const int t = threadIdx.x, warp = t / 32, h = blockIdx.y, kvh = h / (p.Hq / p.Hkv);
  const int64_t q0 = static_cast<int64_t>(blockIdx.x) * BM, i = q0 + t;
  const bool valid = i < p.T;
  const int64_t q_last = min(p.T - 1, q0 + BM - 1);
  const T* q = static_cast<const T*>(p.q);
  const T* k = static_cast<const T*>(p.k);
  const T* v = static_cast<const T*>(p.v);

  if (t == 0) {
    mbar_init(bar, 1);
    fence_mbarrier_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 128);
  stage_rows<BM>(q, q0, p.T, p.Hq, h, Qh, Ql, nullptr, nullptr);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot, tS = tmem, tO = tmem + BNF;
  const uint32_t lanes = static_cast<uint32_t>(warp * 32) << 16;

  float o[D];
#pragma unroll
  for (int c = 0; c < D; ++c) o[c] = 0.f;
  float m = -INFINITY, l = 0.f;
  uint32_t phase = 0;
  bool ok = true;
  for (int64_t kt = 0; kt * BNF <= q_last && ok; ++kt) {
    int km = p.kmax32[2 * kt];
    if ((2 * kt + 1) * 32 < p.T) km = max(km, p.kmax32[2 * kt + 1]);
    if (km < q0) continue;
    const int64_t j0 = kt * BNF;
    __syncthreads();
    stage_rows<BNF>(k, j0, p.T, p.Hkv, kvh, Kh, Kl, nullptr, nullptr);
    stage_rows<BNF>(v, j0, p.T, p.Hkv, kvh, nullptr, nullptr, Vh, Vl);
    if (t < BNF) ends[t] = j0 + t < p.T ? p.end[j0 + t] : -1;
    fence_proxy_async_smem();
    __syncthreads();
    if (t == 0) {
      tc_fence_after();
      mma3<BM, BNF, D>(tS, smem_u32(Qh), smem_u32(Ql), smem_u32(Kh), smem_u32(Kl), 0, kExact<T>, kExact<T>);
      mma_commit(bar);
    }
    if (!(ok = wait_mma(bar, phase, p.err))) break;

    float s[BNF];
    {
      float x[32];
#pragma unroll
      for (int c0 = 0; c0 < BNF; c0 += 32) {
        ld_row32(tS + lanes + c0, x);
#pragma unroll
        for (int c = 0; c < 32; ++c) s[c0 + c] = x[c];
      }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < BNF; ++c) {
      const int64_t j = j0 + c;
      const bool vis = valid && j <= i && i <= ends[c];
      s[c] = vis ? s[c] * p.scale_log2 : -INFINITY;
      mx = fmaxf(mx, s[c]);
    }
    const float mn = fmaxf(m, mx);
    const float corr = mn == -INFINITY ? 1.f : exp2f(m - mn);
    float sum = 0.f;
#pragma unroll
    for (int c = 0; c < BNF; ++c) {
      s[c] = mn == -INFINITY ? 0.f : exp2f(s[c] - mn);
      sum += s[c];
    }
    m = mn;
    l = l * corr + sum;
#pragma unroll
    for (int c = 0; c < D; ++c) o[c] *= corr;
#pragma unroll
    for (int c = 0; c < BNF; c += 4) put4<BM>(Ph, Pl, t, c, make_float4(s[c], s[c + 1], s[c + 2], s[c + 3]));
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (t == 0) {
      tc_fence_after();
      mma3<BM, D, BNF>(tO, smem_u32(Ph), smem_u32(Pl), smem_u32(Vh), smem_u32(Vl), 0, false, kExact<T>);
      mma_commit(bar);
    }
    if (!(ok = wait_mma(bar, phase, p.err))) break;
    {
      float x[32];
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        ld_row32(tO + lanes + c0, x);
#pragma unroll
        for (int c = 0; c < 32; ++c) o[c0 + c] += x[c];
      }
    }
  }
  if (ok && valid) {
    const float inv = 1.f / l;
    T* out = static_cast<T*>(p.o) + (i * p.Hq + h) * D;
#pragma unroll
    for (int c = 0; c < D; c += 4)
      store4(out + c, make_float4(o[c] * inv, o[c + 1] * inv, o[c + 2] * inv, o[c + 3] * inv));
    p.lse[static_cast<int64_t>(h) * p.T + i] = (m + log2f(l)) * kLn2;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// ------------------------------------------------------------------------ backward
// Delta_i = dO_i . O_i per query head: one warp per (row, head).
template <typename T>
__global__ void attn_delta_tc32_kernel(const T* __restrict__ o, const T* __restrict__ dout, float* __restrict__ delta,
                                       int64_t n, int Hq) {
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (w >= n * Hq) return;
  const int64_t i = w / Hq;
  const int h = static_cast<int>(w % Hq);
  float s = 0.f;
  for (int c = lane * 2; c < D; c += 64) {
    s += to_f32(o[w * D + c]) * to_f32(dout[w * D + c]);
    s += to_f32(o[w * D + c + 1]) * to_f32(dout[w * D + c + 1]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) delta[static_cast<int64_t>(h) * n + i] = s;
}

constexpr int kKVB = BM * D * 4, kQtB = BQ * D * 4, kXB = BM * BQ * 4;
constexpr int kDkvSmem = 2 * (2 * kKVB + 4 * kQtB + kXB) + 2 * BQ * 4 + 1024 + 512;

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) attn_dkdv_tc32_kernel(Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint8_t *Kh = base, *Kl = Kh + kKVB, *Vh = Kl + kKVB, *Vl = Vh + kKVB;
  uint8_t *Qh = Vl + kKVB, *Ql = Qh + kQtB, *QTh = Ql + kQtB, *QTl = QTh + kQtB;
  uint8_t *Oh = QTl + kQtB, *Ol = Oh + kQtB, *OTh = Ol + kQtB, *OTl = OTh + kQtB;
  uint8_t *Xh = OTl + kQtB, *Xl = Xh + kXB;
  float* lse2 = reinterpret_cast<float*>(Xl + kXB);
  float* dl = lse2 + BQ;
  uint64_t* bar = reinterpret_cast<uint64_t*>(dl + BQ);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  __shared__ int qmax_s;

  const int t = threadIdx.x, warp = t / 32, kvh = blockIdx.y, group = p.Hq / p.Hkv;
  const int64_t k0 = static_cast<int64_t>(blockIdx.x) * BM, j = k0 + t;
  const bool jvalid = j < p.T;
  const int ej = jvalid ? p.end[j] : -1;
  const T* q = static_cast<const T*>(p.q);
  const T* dout = static_cast<const T*>(p.dout);

  if (t == 0) {
    qmax_s = -1;
    mbar_init(bar, 1);
    fence_mbarrier_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 512);
  __syncthreads();
  atomicMax(&qmax_s, ej);
  stage_rows<BM>(static_cast<const T*>(p.k), k0, p.T, p.Hkv, kvh, Kh, Kl, nullptr, nullptr);
  stage_rows<BM>(static_cast<const T*>(p.v), k0, p.T, p.Hkv, kvh, Vh, Vl, nullptr, nullptr);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // S^T, dP^T, this step's dV and dK, their running sums
  const uint32_t tmem = *tmem_slot, tST = tmem, tdPT = tmem + 32, tdV = tmem + 64, tdK = tmem + 64 + D,
                 tV = tmem + 64 + 2 * D, tK = tmem + 64 + 3 * D;
  const uint32_t lanes = static_cast<uint32_t>(warp * 32) << 16;
  const int64_t q_last = min(static_cast<int64_t>(qmax_s), p.T - 1);

  uint32_t phase = 0;
  bool ok = true, first = true;
  for (int hh = 0; hh < group && ok; ++hh) {
    const int h = kvh * group + hh;
    for (int64_t i0 = k0; i0 <= q_last; i0 += BQ) {
      __syncthreads();
      stage_rows<BQ>(q, i0, p.T, p.Hq, h, Qh, Ql, QTh, QTl);
      stage_rows<BQ>(dout, i0, p.T, p.Hq, h, Oh, Ol, OTh, OTl);
      if (t < BQ) {
        const int64_t i = i0 + t;
        lse2[t] = i < p.T ? p.lse[static_cast<int64_t>(h) * p.T + i] * kLog2e : 0.f;
        dl[t] = i < p.T ? p.delta[static_cast<int64_t>(h) * p.T + i] : 0.f;
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (t == 0) {
        tc_fence_after();
        mma3<BM, BQ, D>(tST, smem_u32(Kh), smem_u32(Kl), smem_u32(Qh), smem_u32(Ql), 0, kExact<T>, kExact<T>);
        mma3<BM, BQ, D>(tdPT, smem_u32(Vh), smem_u32(Vl), smem_u32(Oh), smem_u32(Ol), 0, kExact<T>, kExact<T>);
        mma_commit(bar);
      }
      if (!(ok = wait_mma(bar, phase, p.err))) break;
      float s[32], dp[32];
      ld_row32(tST + lanes, s);
      ld_row32(tdPT + lanes, dp);
#pragma unroll
      for (int c = 0; c < BQ; ++c) {
        const int64_t i = i0 + c;
        const bool vis = jvalid && i < p.T && j <= i && i <= ej;
        s[c] = vis ? exp2f(s[c] * p.scale_log2 - lse2[c]) : 0.f;  // P^T
        dp[c] = s[c] * (dp[c] - dl[c]);                              // dS^T
      }
#pragma unroll
      for (int c = 0; c < BQ; c += 4) put4<BM>(Xh, Xl, t, c, make_float4(s[c], s[c + 1], s[c + 2], s[c + 3]));
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      if (t == 0) {
        tc_fence_after();
        mma3<BM, D, BQ>(tdV, smem_u32(Xh), smem_u32(Xl), smem_u32(OTh), smem_u32(OTl), 0, false, kExact<T>);
        mma_commit(bar);
      }
      if (!(ok = wait_mma(bar, phase, p.err))) break;
#pragma unroll
      for (int c = 0; c < BQ; c += 4)
        put4<BM>(Xh, Xl, t, c, make_float4(dp[c], dp[c + 1], dp[c + 2], dp[c + 3]));
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      if (t == 0) {
        tc_fence_after();
        mma3<BM, D, BQ>(tdK, smem_u32(Xh), smem_u32(Xl), smem_u32(QTh), smem_u32(QTl), 0, false, kExact<T>);
        mma_commit(bar);
      }
      if (!(ok = wait_mma(bar, phase, p.err))) break;
      tmem_accumulate(tV + lanes, tdV + lanes, first);
      tmem_accumulate(tK + lanes, tdK + lanes, first);
      tc_fence_before();  // the next step's MMAs overwrite the step blocks
      first = false;
    }
  }
  if (ok) {  // the TMEM loads are warp-collective: every lane takes them, valid rows store
    T* dk = static_cast<T*>(p.dk) + (j * p.Hkv + kvh) * D;
    T* dv = static_cast<T*>(p.dv) + (j * p.Hkv + kvh) * D;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      float a[32], b[32];
      if (first) {
#pragma unroll
        for (int c = 0; c < 32; ++c) a[c] = b[c] = 0.f;
      } else {
        ld_row32(tK + lanes + c0, a);
        ld_row32(tV + lanes + c0, b);
      }
      if (!jvalid) continue;
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        store4(dk + c0 + c, make_float4(a[c] * p.scale, a[c + 1] * p.scale, a[c + 2] * p.scale, a[c + 3] * p.scale));
        store4(dv + c0 + c, make_float4(b[c], b[c + 1], b[c + 2], b[c + 3]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

constexpr int kQqB = BM * D * 4, kKqB = BNQ * D * 4, kXqB = BM * BNQ * 4;
constexpr int kDqSmem = 2 * (2 * kQqB + 3 * kKqB + kXqB) + 1024 + 512;

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) attn_dq_tc32_kernel(Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint8_t *Qh = base, *Ql = Qh + kQqB, *Oh = Ql + kQqB, *Ol = Oh + kQqB;
  uint8_t *Kh = Ol + kQqB, *Kl = Kh + kKqB, *Vh = Kl + kKqB, *Vl = Vh + kKqB, *KTh = Vl + kKqB, *KTl = KTh + kKqB;
  uint8_t *Xh = KTl + kKqB, *Xl = Xh + kXqB;
  int32_t* ends = reinterpret_cast<int32_t*>(Xl + kXqB);
  uint64_t* bar = reinterpret_cast<uint64_t*>(ends + BNQ);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);

  const int t = threadIdx.x, warp = t / 32, h = blockIdx.y, kvh = h / (p.Hq / p.Hkv);
  const int64_t q0 = static_cast<int64_t>(blockIdx.x) * BM, i = q0 + t;
  const bool valid = i < p.T;
  const int64_t q_last = min(p.T - 1, q0 + BM - 1);
  const T* k = static_cast<const T*>(p.k);
  const T* v = static_cast<const T*>(p.v);

  if (t == 0) {
    mbar_init(bar, 1);
    fence_mbarrier_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 256);
  stage_rows<BM>(static_cast<const T*>(p.q), q0, p.T, p.Hq, h, Qh, Ql, nullptr, nullptr);
  stage_rows<BM>(static_cast<const T*>(p.dout), q0, p.T, p.Hq, h, Oh, Ol, nullptr, nullptr);
  const float lse2 = valid ? p.lse[static_cast<int64_t>(h) * p.T + i] * kLog2e : 0.f;
  const float dl = valid ? p.delta[static_cast<int64_t>(h) * p.T + i] : 0.f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // S, dP, this key tile's dQ, the running sum
  const uint32_t tmem = *tmem_slot, tS = tmem, tdP = tmem + 32, tdQ = tmem + 64, tQ = tmem + 64 + D;
  const uint32_t lanes = static_cast<uint32_t>(warp * 32) << 16;

  uint32_t phase = 0;
  bool ok = true, first = true;
  for (int64_t kt = 0; kt * BNQ <= q_last; ++kt) {
    if (p.kmax32[kt] < q0) continue;
    const int64_t j0 = kt * BNQ;
    __syncthreads();
    stage_rows<BNQ>(k, j0, p.T, p.Hkv, kvh, Kh, Kl, KTh, KTl);
    stage_rows<BNQ>(v, j0, p.T, p.Hkv, kvh, Vh, Vl, nullptr, nullptr);
    if (t < BNQ) ends[t] = j0 + t < p.T ? p.end[j0 + t] : -1;
    fence_proxy_async_smem();
    __syncthreads();
    if (t == 0) {
      tc_fence_after();
      mma3<BM, BNQ, D>(tS, smem_u32(Qh), smem_u32(Ql), smem_u32(Kh), smem_u32(Kl), 0, kExact<T>, kExact<T>);
      mma3<BM, BNQ, D>(tdP, smem_u32(Oh), smem_u32(Ol), smem_u32(Vh), smem_u32(Vl), 0, kExact<T>, kExact<T>);
      mma_commit(bar);
    }
    if (!(ok = wait_mma(bar, phase, p.err))) break;
    float s[32], dp[32];
    ld_row32(tS + lanes, s);
    ld_row32(tdP + lanes, dp);
#pragma unroll
    for (int c = 0; c < BNQ; ++c) {
      const int64_t j = j0 + c;
      const bool vis = valid && j <= i && i <= ends[c];
      const float pr = vis ? exp2f(s[c] * p.scale_log2 - lse2) : 0.f;
      dp[c] = pr * (dp[c] - dl);
    }
#pragma unroll
    for (int c = 0; c < BNQ; c += 4) put4<BM>(Xh, Xl, t, c, make_float4(dp[c], dp[c + 1], dp[c + 2], dp[c + 3]));
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (t == 0) {
      tc_fence_after();
      mma3<BM, D, BNQ>(tdQ, smem_u32(Xh), smem_u32(Xl), smem_u32(KTh), smem_u32(KTl), 0, false, kExact<T>);
      mma_commit(bar);
    }
    if (!(ok = wait_mma(bar, phase, p.err))) break;
    tmem_accumulate(tQ + lanes, tdQ + lanes, first);
    tc_fence_before();
    first = false;
  }
  if (ok) {  // warp-collective TMEM loads by every lane, stores by valid rows
    T* dq = static_cast<T*>(p.dq) + (i * p.Hq + h) * D;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      float a[32];
      if (first) {
#pragma unroll
        for (int c = 0; c < 32; ++c) a[c] = 0.f;
      } else {
        ld_row32(tQ + lanes + c0, a);
      }
      if (!valid) continue;
#pragma unroll
      for (int c = 0; c < 32; c += 4)
        store4(dq + c0 + c, make_float4(a[c] * p.scale, a[c + 1] * p.scale, a[c + 2] * p.scale, a[c + 3] * p.scale));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

static_assert(kFwdSmem <= 232448 && kDkvSmem <= 232448 && kDqSmem <= 232448, "shared memory per CTA");

Params make_params(const AttnArgs& a) {
  Params p{};
  p.q = a.q; p.k = a.k; p.v = a.v; p.o = a.o; p.lse = a.lse; p.dout = a.dout; p.delta = a.ws.delta;
  p.dq = a.dq; p.dk = a.dk; p.dv = a.dv; p.end = a.end; p.kmax32 = a.ws.kmax32;
  p.T = a.T; p.Hq = a.Hq; p.Hkv = a.Hkv; p.scale = a.scale; p.scale_log2 = a.scale * kLog2e;
  p.err = device_error_word();
  return p;
}

template <typename T>
int fwd(const AttnArgs& a, cudaStream_t st) {
  int rc = tile_meta_launch(a.end, a.T, 32, a.ws.kmax32, a.ws.kmin32, st);
  if (rc) return rc;
  auto* kern = attn_fwd_tc32_kernel<T>;
  if ((rc = smem_opt_in(reinterpret_cast<const void*>(kern), kFwdSmem))) return rc;
  dim3 grid(static_cast<unsigned>((a.T + BM - 1) / BM), a.Hq);
  kern<<<grid, kThreads, kFwdSmem, st>>>(make_params(a));
  TREE_LAUNCH_CHECK("attn_fwd_tc32_kernel");
  return TREE_OK;
}

template <typename T>
int bwd(const AttnArgs& a, cudaStream_t st) {
  int rc = tile_meta_launch(a.end, a.T, 32, a.ws.kmax32, a.ws.kmin32, st);
  if (rc) return rc;
  const int64_t warps = a.T * a.Hq;
  attn_delta_tc32_kernel<T><<<static_cast<unsigned>((warps * 32 + 255) / 256), 256, 0, st>>>(
      static_cast<const T*>(a.o), static_cast<const T*>(a.dout), a.ws.delta, a.T, a.Hq);
  TREE_LAUNCH_CHECK("attn_delta_tc32_kernel");
  const Params p = make_params(a);
  auto* kdq = attn_dq_tc32_kernel<T>;
  auto* kkv = attn_dkdv_tc32_kernel<T>;
  if ((rc = smem_opt_in(reinterpret_cast<const void*>(kdq), kDqSmem))) return rc;
  if ((rc = smem_opt_in(reinterpret_cast<const void*>(kkv), kDkvSmem))) return rc;
  const unsigned tiles = static_cast<unsigned>((a.T + BM - 1) / BM);
  kdq<<<dim3(tiles, a.Hq), kThreads, kDqSmem, st>>>(p);
  TREE_LAUNCH_CHECK("attn_dq_tc32_kernel");
  kkv<<<dim3(tiles, a.Hkv), kThreads, kDkvSmem, st>>>(p);
  TREE_LAUNCH_CHECK("attn_dkdv_tc32_kernel");
  return TREE_OK;
}

}  // namespace atc32

bool attn_tc32_supported(int dtype, int d) {
  return d == atc32::D && (dtype == TREE_DTYPE_F32 || dtype == TREE_DTYPE_BF16);
}

int attn_fwd_tc32(const AttnArgs& a, cudaStream_t st) {
  return a.dtype == TREE_DTYPE_BF16 ? atc32::fwd<__nv_bfloat16>(a, st) : atc32::fwd<float>(a, st);
}

int attn_bwd_tc32(const AttnArgs& a, cudaStream_t st) {
  return a.dtype == TREE_DTYPE_BF16 ? atc32::bwd<__nv_bfloat16>(a, st) : atc32::bwd<float>(a, st);
}

}  // namespace tree
