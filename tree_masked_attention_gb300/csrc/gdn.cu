// tree_gdn_fwd: Gated DeltaNet forward over a packed prefix tree, the recurrent state
// routed along the tree.
//
// Tree Training (arXiv 2511.00413) §3.2 "SSM Layers (GDN)", eq. 10 and Appendix A.2:
// each chunk (tree node) starts from the end state of its parent chunk, a root chunk from
// zero, instead of from the chunk before it in preorder (a sibling branch). Per head the
// state S [Dv, Dk] follows the gated delta rule
//   S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t.
//
// Work item = (a sub-chunk of at most 64 rows of one node, a head). Inside a sub-chunk
// of rows 0..L-1 starting from state h0 = S^T [Dk, Dv], with lg_t the running sum of g:
//   A[t][s] = beta_t exp(lg_t - lg_s) (k_t . k_s)  (s < t),  P[t][s] = exp(lg_t - lg_s) (q_t . k_s)  (s <= t)
//   u solves (I + A) u = beta o (V - exp(lg) o (K h0))          (forward substitution)
//   O = exp(lg) o (Q h0) + P u,   h_end = exp(lg_{L-1}) h0 + sum_s exp(lg_{L-1} - lg_s) k_s u_s^T
// which is the recurrence solved for the whole sub-chunk at once (the delta-rule
// corrections u depend on each other only through the lower-triangular A).
// The sub-chunk's h0 is the end state of its predecessor: the previous sub-chunk of the
// same node, or the parent node's last sub-chunk (eq. 10). Items are handed out from a
// counter in order of chain depth (a sub-chunk's depth is its predecessor's plus one), so
// all sub-chunks of one depth -- siblings and other branches -- run together, and a
// predecessor always comes earlier: it was taken by a CTA that is running or done, and
// the bounded wait for its published end state terminates.
//
// One CTA (256 threads) per SM holds the sub-chunk's K, Q, V rows, the state, A and P in
// ~197 KB of shared memory; arithmetic is fp32 on the CUDA cores (a first version: the
// chunk products are small GEMMs that a tensor-core version would take over).
#include <algorithm>
#include <cmath>

#include "common.h"
#include "device_common.cuh"
#include "sm100.cuh"

namespace tree {
namespace {

constexpr int kGdnThreads = 256;
constexpr int kMaxGdnCtas = 1024;  // upper bound of the persistent grid (one CTA per SM)
constexpr int kChunk = 64;       // rows per sub-chunk
constexpr int kMaxD = 128;       // largest Dk, Dv
constexpr int kPad = kMaxD + 1;  // row stride of K, Q (bank-conflict-free column walks)

constexpr size_t kGdnSmemFloats = 2 * kChunk * kPad     // K, Q
                                  + kChunk * kMaxD      // V, then R, then u
                                  + kMaxD * kMaxD       // state h = S^T [Dk, Dv]
                                  + 2 * kChunk * kChunk // A, P
                                  + 3 * kChunk;         // lg, beta, end-decay weights
constexpr size_t kGdnSmemBytes = kGdnSmemFloats * sizeof(float);
static_assert(kGdnSmemBytes <= 227 * 1024, "GDN shared memory exceeds the per-block limit");

struct GdnParams {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  void* o;
  int T, H, Dk, Dv;
  const int4* chunks;  // {first row, rows, predecessor sub-chunk or -1, chain depth}
  const int* order;    // sub-chunks by increasing chain depth
  const int* n_chunks;
  int* counter;
  int* flags;          // [max_chunks * H] 1 once the end state is published
  int* abort;
  float* states;       // [max_chunks, H, Dk, Dv] end states
  int* err;
};

__device__ __forceinline__ float ldf(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p, int64_t i) { return __bfloat162float(p[i]); }

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Sub-chunk table from the node arrays (one thread walks the nodes in preorder, checking
// that they tile [0, T) with earlier parents), then the schedule: sub-chunks by
// increasing chain depth (a counting sort, stable in preorder); all threads clear the
// flags and counter.
__global__ void __launch_bounds__(1024) gdn_setup_kernel(const int32_t* __restrict__ node_start,
                                                         const int32_t* __restrict__ node_end,
                                                         const int32_t* __restrict__ node_parent, int n_nodes,
                                                         int T, int H, int max_chunks, int4* chunks,
                                                         int* node_last, int* order, int* depth_count,
                                                         int* n_chunks, int* counter, int* flags, int* abort,
                                                         int* err) {
  for (int64_t i = threadIdx.x; i < static_cast<int64_t>(max_chunks) * H; i += blockDim.x) flags[i] = 0;
  if (threadIdx.x != 0) return;
  *counter = 0;
  *abort = 0;
  int m = 0, next = 0;
  bool ok = true;
  for (int n = 0; n < n_nodes && ok; ++n) {
    const int s = node_start[n], e = node_end[n] + 1, par = node_parent[n];
    if (s != next || e <= s || e > T || par >= n || par < -1) {
      ok = false;
      break;
    }
    next = e;
    int pred = par >= 0 ? node_last[par] : -1;
    for (int c0 = s; c0 < e; c0 += kChunk) {
      if (m >= max_chunks) { ok = false; break; }
      const int depth = pred >= 0 ? chunks[pred].w + 1 : 0;
      chunks[m] = make_int4(c0, min(kChunk, e - c0), pred, depth);
      pred = m++;
    }
    node_last[n] = pred;
  }
  if (!ok || next != T) {
    raise_error(err, TREE_ERR_DEVICE_CHECK);
    m = 0;
  }
  // counting sort by chain depth (depths are < m)
  for (int d = 0; d <= m; ++d) depth_count[d] = 0;
  for (int c = 0; c < m; ++c) ++depth_count[chunks[c].w + 1];
  for (int d = 1; d <= m; ++d) depth_count[d] += depth_count[d - 1];
  for (int c = 0; c < m; ++c) order[depth_count[chunks[c].w]++] = c;
  *n_chunks = m;
}

template <typename Tin>
__global__ void __launch_bounds__(kGdnThreads, 1) gdn_fwd_kernel(const GdnParams p) {
  extern __shared__ float sm[];
  float* Ks = sm;                       // [64][kPad]
  float* Qs = Ks + kChunk * kPad;       // [64][kPad]
  float* Vs = Qs + kChunk * kPad;       // [64][kMaxD]  V -> R -> u
  float* Hs = Vs + kChunk * kMaxD;      // [kMaxD][kMaxD] h[i][j], i < Dk, j < Dv
  float* Am = Hs + kMaxD * kMaxD;       // [64][64]
  float* Pm = Am + kChunk * kChunk;     // [64][64]
  float* lg = Pm + kChunk * kChunk;     // [64]
  float* bs = lg + kChunk;              // [64]
  float* wd = bs + kChunk;              // [64] exp(lg_{L-1} - lg_s)
  __shared__ int s_item;
  __shared__ int s_ok;
  const int tid = threadIdx.x;
  const Tin* q = static_cast<const Tin*>(p.q);
  const Tin* k = static_cast<const Tin*>(p.k);
  const Tin* v = static_cast<const Tin*>(p.v);
  Tin* o = static_cast<Tin*>(p.o);
  const int H = p.H, Dk = p.Dk, Dv = p.Dv;
  const int items = *p.n_chunks * H;
  const int j = tid % kMaxD;          // the state / value column this thread owns
  const int half = tid / kMaxD;       // rows 32 * half .. 32 * half + 31 of the sub-chunk
  while (true) {
    if (tid == 0) s_item = *reinterpret_cast<volatile int*>(p.abort) ? items : atomicAdd(p.counter, 1);
    __syncthreads();
    const int item = s_item;
    if (item >= items) break;
    const int c = p.order[item / H], h = item % H;
    const int4 ck = p.chunks[c];
    const int r0 = ck.x, L = ck.y, pred = ck.z;
    // wait until the predecessor's end state is published (bounded)
    if (tid == 0) {
      int ok = 1;
      if (pred >= 0) {
        const int* f = p.flags + static_cast<int64_t>(pred) * H + h;
        if (!ld_acquire(f)) {
          const unsigned long long t0 = sm100::globaltimer();
          while (!ld_acquire(f)) {
            if (sm100::globaltimer() - t0 > sm100::kWaitNs) {
              ok = 0;
              raise_error(p.err, TREE_ERR_TIMEOUT);
              atomicExch(p.abort, 1);
              break;
            }
            __nanosleep(64);
          }
        }
      }
      s_ok = ok;
    }
    __syncthreads();
    if (!s_ok) break;
    // K, Q, V rows (zero past L), per-row decay sums and beta, the starting state
    for (int idx = tid; idx < kChunk * kMaxD; idx += kGdnThreads) {
      const int t = idx / kMaxD, i = idx % kMaxD;
      const bool in = t < L;
      const int64_t row = static_cast<int64_t>(r0 + t) * H + h;
      Ks[t * kPad + i] = (in && i < Dk) ? ldf(k, row * Dk + i) : 0.f;
      Qs[t * kPad + i] = (in && i < Dk) ? ldf(q, row * Dk + i) : 0.f;
      Vs[t * kMaxD + i] = (in && i < Dv) ? ldf(v, row * Dv + i) : 0.f;
    }
    const float* h0 = pred >= 0 ? p.states + (static_cast<int64_t>(pred) * H + h) * Dk * Dv : nullptr;
    for (int idx = tid; idx < kMaxD * kMaxD; idx += kGdnThreads) {
      const int i = idx / kMaxD, jj = idx % kMaxD;
      Hs[idx] = (h0 && i < Dk && jj < Dv) ? __ldcg(h0 + i * Dv + jj) : 0.f;
    }
    if (tid == 0) {
      float run = 0.f;
      for (int t = 0; t < kChunk; ++t) {
        const bool in = t < L;
        const int64_t row = static_cast<int64_t>(r0 + t) * H + h;
        run += in ? p.g[row] : 0.f;
        lg[t] = run;
        bs[t] = in ? p.beta[row] : 0.f;
      }
    }
    __syncthreads();
    if (tid < kChunk) wd[tid] = tid < L ? expf(lg[L - 1] - lg[tid]) : 0.f;
    // A and P: 64 x 64 dot products of length Dk
    for (int idx = tid; idx < kChunk * kChunk; idx += kGdnThreads) {
      const int t = idx / kChunk, s = idx % kChunk;
      float a = 0.f, b = 0.f;
      if (t < L && s <= t) {
        const float* kt = Ks + t * kPad;
        const float* qt = Qs + t * kPad;
        const float* ks = Ks + s * kPad;
        for (int i = 0; i < Dk; ++i) {
          a = fmaf(kt[i], ks[i], a);
          b = fmaf(qt[i], ks[i], b);
        }
        const float r = expf(lg[t] - lg[s]);
        a = s < t ? bs[t] * r * a : 0.f;
        b = r * b;
      }
      Am[idx] = a;
      Pm[idx] = b;
    }
    // K h0 and Q h0 for this thread's 32 rows and column j; R = beta (V - exp(lg) K h0)
    float qh[32];
    {
      float kh[32];
#pragma unroll
      for (int u = 0; u < 32; ++u) kh[u] = qh[u] = 0.f;
      if (j < Dv) {
        for (int i = 0; i < Dk; ++i) {
          const float hij = Hs[i * kMaxD + j];
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const int t = 32 * half + u;
            kh[u] = fmaf(Ks[t * kPad + i], hij, kh[u]);
            qh[u] = fmaf(Qs[t * kPad + i], hij, qh[u]);
          }
        }
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int t = 32 * half + u;
          Vs[t * kMaxD + j] = bs[t] * (Vs[t * kMaxD + j] - expf(lg[t]) * kh[u]);
        }
      }
    }
    __syncthreads();
    // forward substitution per column: u_t = R_t - sum_{s<t} A[t][s] u_s (in place)
    if (half == 0 && j < Dv) {
      for (int t = 1; t < L; ++t) {
        float acc = Vs[t * kMaxD + j];
        for (int s = 0; s < t; ++s) acc = fmaf(-Am[t * kChunk + s], Vs[s * kMaxD + j], acc);
        Vs[t * kMaxD + j] = acc;
      }
    }
    __syncthreads();
    // outputs: O = exp(lg) Q h0 + P u, this thread's 32 rows of column j
    if (j < Dv) {
#pragma unroll
      for (int u = 0; u < 32; ++u) {
        const int t = 32 * half + u;
        if (t < L) {
          float acc = expf(lg[t]) * qh[u];
          for (int s = 0; s <= t; ++s) acc = fmaf(Pm[t * kChunk + s], Vs[s * kMaxD + j], acc);
          const int64_t off = (static_cast<int64_t>(r0 + t) * H + h) * Dv + j;
          o[off] = from_f32<Tin>(acc);
        }
      }
    }
    // end state: h = exp(lg_{L-1}) h0 + sum_s wd_s k_s u_s^T (rows i of this thread's half)
    if (j < Dv) {
      const float gl = expf(lg[L - 1]);
      for (int i = half; i < Dk; i += 2) {
        float acc = gl * Hs[i * kMaxD + j];
        for (int s = 0; s < L; ++s) acc = fmaf(wd[s] * Ks[s * kPad + i], Vs[s * kMaxD + j], acc);
        Hs[i * kMaxD + j] = acc;
      }
    }
    __syncthreads();
    float* hout = p.states + (static_cast<int64_t>(c) * H + h) * Dk * Dv;
    for (int idx = tid; idx < Dk * Dv; idx += kGdnThreads) {
      const int i = idx / Dv, jj = idx % Dv;
      __stcg(hout + idx, Hs[i * kMaxD + jj]);
    }
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      st_release(p.flags + static_cast<int64_t>(c) * H + h, 1);
    }
  }
}

int64_t gdn_max_chunks(int64_t T, int64_t n_nodes) { return n_nodes + T / kChunk + 1; }

struct GdnWs {
  int4* chunks;
  int* node_last;
  int* order;
  int* depth_count;
  int* n_chunks;
  int* counter;
  int* abort;
  int* flags;
  float* states;
};

size_t gdn_ws_layout(int64_t T, int64_t n_nodes, int H, int Dk, int Dv, void* base, GdnWs* w) {
  const int64_t mc = gdn_max_chunks(T, n_nodes);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    off = round_up(off, 256);
    void* ptr = base ? static_cast<char*>(base) + off : nullptr;
    off += bytes;
    return ptr;
  };
  GdnWs x{};
  x.chunks = static_cast<int4*>(take(sizeof(int4) * mc));
  x.node_last = static_cast<int*>(take(sizeof(int) * std::max<int64_t>(n_nodes, 1)));
  x.order = static_cast<int*>(take(sizeof(int) * mc));
  x.depth_count = static_cast<int*>(take(sizeof(int) * (mc + 1)));
  x.n_chunks = static_cast<int*>(take(sizeof(int)));
  x.counter = static_cast<int*>(take(sizeof(int)));
  x.abort = static_cast<int*>(take(sizeof(int)));
  x.flags = static_cast<int*>(take(sizeof(int) * mc * H));
  x.states = static_cast<float*>(take(sizeof(float) * mc * H * Dk * Dv));
  if (w) *w = x;
  return round_up(off, 256);
}

int sm_count_gdn(int* n) {
  int dev = 0;
  TREE_CUDA_TRY(cudaGetDevice(&dev));
  TREE_CUDA_TRY(cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev));
  return TREE_OK;
}

template <typename Tin>
int launch_gdn(const GdnParams& p, cudaStream_t st) {
  if (int rc_ = smem_opt_in(reinterpret_cast<const void*>(gdn_fwd_kernel<Tin>), static_cast<int>(kGdnSmemBytes))) return rc_;
  int n_sm = 0;
  int rc = sm_count_gdn(&n_sm);
  if (rc) return rc;
  gdn_fwd_kernel<Tin><<<std::min(n_sm, kMaxGdnCtas), kGdnThreads, kGdnSmemBytes, st>>>(p);
  TREE_LAUNCH_CHECK("gdn_fwd_kernel");
  return TREE_OK;
}

}  // namespace
}  // namespace tree

using namespace tree;

extern "C" size_t tree_gdn_workspace_size(int64_t T, int64_t n_nodes, int H, int Dk, int Dv) {
  if (T < 1 || n_nodes < 1 || H < 1 || Dk < 1 || Dv < 1) return 0;
  return gdn_ws_layout(T, n_nodes, H, Dk, Dv, nullptr, nullptr);
}

extern "C" int tree_gdn_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta, void* o,
                            const int32_t* node_start, const int32_t* node_end, const int32_t* node_parent,
                            int64_t T, int64_t n_nodes, int H, int Dk, int Dv, int dtype, void* workspace,
                            size_t workspace_bytes, tree_stream_t stream) {
  clear_error();
  if (dtype != TREE_DTYPE_F32 && dtype != TREE_DTYPE_BF16) return fail(TREE_ERR_DTYPE, "tree_gdn_fwd: bad dtype %d", dtype);
  if (T < 0 || n_nodes < 0 || T > (1 << 30) || n_nodes > T)
    return fail(TREE_ERR_SHAPE, "tree_gdn_fwd: T = %lld, n_nodes = %lld", (long long)T, (long long)n_nodes);
  if (H < 1 || Dk < 1 || Dv < 1 || Dk > kMaxD || Dv > kMaxD)
    return fail(TREE_ERR_SHAPE, "tree_gdn_fwd: H = %d, Dk = %d, Dv = %d (need Dk, Dv <= %d)", H, Dk, Dv, kMaxD);
  if (T == 0) return TREE_OK;
  if (n_nodes < 1) return fail(TREE_ERR_SHAPE, "tree_gdn_fwd: no nodes for %lld rows", (long long)T);
  // work items are counted in 32 bits, and every CTA draws once past the last item
  if (gdn_max_chunks(T, n_nodes) * H + kMaxGdnCtas > INT32_MAX)
    return fail(TREE_ERR_SHAPE, "tree_gdn_fwd: %lld sub-chunks x %d heads exceed the 32-bit work counter",
                (long long)gdn_max_chunks(T, n_nodes), H);
  if (!q || !k || !v || !g || !beta || !o || !node_start || !node_end || !node_parent)
    return fail(TREE_ERR_INVALID_ARG, "tree_gdn_fwd: null pointer");
  const size_t need = gdn_ws_layout(T, n_nodes, H, Dk, Dv, nullptr, nullptr);
  if (workspace_bytes < need)
    return fail(TREE_ERR_WORKSPACE, "tree_gdn_fwd: workspace of %zu bytes, %zu needed", workspace_bytes, need);
  if (!workspace || !aligned256(workspace))
    return fail(TREE_ERR_ALIGNMENT, "tree_gdn_fwd: workspace null or not 256-byte aligned");
  GdnWs w{};
  gdn_ws_layout(T, n_nodes, H, Dk, Dv, workspace, &w);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t mc = gdn_max_chunks(T, n_nodes);
  gdn_setup_kernel<<<1, 1024, 0, st>>>(node_start, node_end, node_parent, static_cast<int>(n_nodes),
                                       static_cast<int>(T), H, static_cast<int>(mc), w.chunks, w.node_last,
                                       w.order, w.depth_count, w.n_chunks, w.counter, w.flags, w.abort,
                                       device_error_word());
  TREE_LAUNCH_CHECK("gdn_setup_kernel");
  GdnParams p{};
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.o = o;
  p.T = static_cast<int>(T); p.H = H; p.Dk = Dk; p.Dv = Dv;
  p.chunks = w.chunks; p.order = w.order; p.n_chunks = w.n_chunks; p.counter = w.counter; p.flags = w.flags; p.abort = w.abort;
  p.states = w.states; p.err = device_error_word();
  if (dtype == TREE_DTYPE_BF16) return launch_gdn<__nv_bfloat16>(p, st);
  return launch_gdn<float>(p, st);
}
