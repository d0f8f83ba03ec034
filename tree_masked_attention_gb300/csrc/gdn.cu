// tree_gdn_fwd / tree_gdn_bwd: Gated DeltaNet over a packed prefix tree, the recurrent
// state routed along the tree.
//
// Tree Training (arXiv 2511.00413) §3.2 "SSM Layers (GDN)", eq. 10 and Appendix A.2:
// each chunk (tree node) starts from the end state of its parent chunk, a root chunk from
// zero, instead of from the chunk before it in preorder (a sibling branch). Per head the
// state S [Dv, Dk] follows the gated delta rule
//   S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t.
//
// Every node is cut into sub-chunks of at most 64 rows. Inside a sub-chunk of rows
// 0..L-1 starting from state h0 = S^T [Dk, Dv], with lg_t the running sum of g from the
// sub-chunk's first row, E_t = exp(lg_t), f_ts = exp(lg_t - lg_s), w_s = exp(lg_{L-1} - lg_s):
//   A = strictly-lower(beta_t f_ts k_t.k_s),   P = lower(f_ts q_t.k_s),   X = (I + A)^-1
//   W = X (beta E o K),   U0 = X (beta o V)                 (no dependence on h0)
//   u = U0 - W h0,   O = E o (Q h0) + P u,   h_end = E_{L-1} h0 + sum_s w_s k_s u_s^T
// which is the recurrence solved for the whole sub-chunk at once (the delta-rule
// corrections u depend on each other only through the lower-triangular A).
//
// Forward, four launches:
//   setup  sub-chunk table, schedule by chain depth, successor lists, flags cleared;
//   prep   per (sub-chunk, head), all in parallel: A, P, X, W, U0;
//   chain  per (sub-chunk, head, 32-column slice of the state), handed out by increasing
//          chain depth: h0 is the predecessor's published end state (the previous
//          sub-chunk of the node, or the parent node's last one: eq. 10); u and h_end,
//          then h_end is published. Columns of the state never mix in the recurrence, so
//          the slices are independent chains;
//   out    per (sub-chunk, head), in parallel: O = E o (Q h0) + P u.
// Backward (gradients of sum(dO . O)): setup, prep and chain again (they give every h0
// and u), then
//   bchain per (sub-chunk, head, slice) by decreasing chain depth: the end-state gradient
//          dh_end is the sum, in a fixed order, of the successors' start-state gradients;
//          du = w o (K dh_end) + P^T dO, dr = X^T du, dv = beta o dr,
//          dh0 = E_{L-1} dh_end + Q^T (E o dO) - K^T (beta E o dr), published;
//   grads  per (sub-chunk, head), in parallel: dP = lower(dO u^T), dA = -strict(dr u^T),
//          dQ = (dP o f) K + (E o dO) h0^T,
//          dK = (dP o f)^T Q + (dA o beta f) K + (dA o beta f)^T K + w o (u dh_end^T)
//               - (beta E o dr) h0^T,
//          and dg, dbeta from the per-row sums of the reverse mode (dg is the reverse
//          running sum of d lg over the sub-chunk).
// Chain items are handed out from a counter in dependency order, so every item a CTA
// waits for was taken earlier by a CTA that is running or done; every wait is bounded.
// Arithmetic is fp32 on the CUDA cores.
#include <algorithm>
#include <atomic>
#include <cmath>

#include "common.h"
#include "device_common.cuh"
#include "sm100.cuh"

namespace tree {
namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 64;        // rows per sub-chunk
constexpr int kMaxD = 128;        // largest Dk, Dv
constexpr int kSlice = 32;        // state columns per chain item
constexpr int kMaxCtas = 1024;    // upper bound of a persistent grid
constexpr int kRow = kMaxD + 4;   // row stride (floats) of [64][D] tiles: 16-byte rows, float4 reads conflict-free
constexpr int kSq = kChunk + 4;   // row stride of [64][64] matrices (16-byte rows)
constexpr int kSl = kSlice + 4;   // row stride of [*][32] slices read along their rows (16-byte rows)
constexpr int kSt = 17;           // row stride of [128][16] stagings read down their columns

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

// Asynchronous global -> shared copies (no registers, many in flight), waited for together.
__device__ __forceinline__ void cp16(void* s, const void* g) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sm100::smem_u32(s)), "l"(g) : "memory");
}
__device__ __forceinline__ void cp4(void* s, const void* g) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(sm100::smem_u32(s)), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// A row-major [rows][cols] fp32 block (cols a multiple of 4) into shared memory rows of
// stride sstride floats (a multiple of 4), 16 bytes per copy.
__device__ __forceinline__ void cp_block(float* s, int sstride, const float* g, int rows, int cols) {
  const int per = cols / 4, n = rows * per;
  for (int p = threadIdx.x; p < n; p += kThreads) cp16(s + (p / per) * sstride + (p % per) * 4, g + 4 * static_cast<int64_t>(p));
}

struct GdnWs {
  int4* chunks;     // [mc] {first row, rows, predecessor sub-chunk or -1, chain depth}
  int* node_last;   // [n_nodes] last sub-chunk of each node
  int* order;       // [mc] sub-chunks by increasing chain depth
  int* depth_count; // [mc + 1]
  int* succ_ptr;    // [mc + 1] successors (sub-chunks whose predecessor is c), CSR
  int* succ;        // [mc]
  int* ctl;         // [4] n_chunks, forward counter, backward counter, abort
  int* flags_f;     // [mc, H, slices] end state published
  float* Pm;        // [mc, H, 64, 64]
  float* Xm;        // [mc, H, 64, 64]  (I + A)^-1
  float* W;         // [mc, H, 64, DkP]  (DkP = Dk rounded up to 4; zero past Dk and past the rows)
  float* U0;        // [mc, H, slices, 64, 32]
  float* u;         // [mc, H, slices, 64, 32]
  float* states;    // [mc, H, slices, Dk, 32] end states (columns past Dv zero)
  // backward only
  int* flags_b;     // [mc, H, slices] start-state gradient published
  float* dstart;    // [mc, H, slices, Dk, 32] start-state gradients
  float* dend;      // [mc, H, slices, Dk, 32] end-state gradients
  float* dr;        // [mc, H, slices, 64, 32]
  float* part;      // [slices, 2, T, H] per-row partial sums (dw, dr . v)
  float* part_he;   // [slices, mc, H] partial sums of dh_end . h0
  int* scratch;     // set-up working arrays when they do not fit in shared memory
};

int64_t gdn_max_chunks(int64_t T, int64_t n_nodes) { return n_nodes + T / kChunk + 1; }
int gdn_slices(int Dv) { return (Dv + kSlice - 1) / kSlice; }

// Block of one (sub-chunk, head, slice) in the [mc, H, slices, rows, 32] layouts.
__device__ __forceinline__ float* slice_block(float* base, int c, int h, int sl, int H, int ns, int rows) {
  return base + ((static_cast<int64_t>(c) * H + h) * ns + sl) * rows * kSlice;
}

size_t gdn_ws_layout(int64_t T, int64_t n_nodes, int H, int Dk, int Dv, bool bwd, void* base, GdnWs* w) {
  const int64_t mc = gdn_max_chunks(T, n_nodes);
  const int64_t ns = gdn_slices(Dv);
  const int64_t DkP = (Dk + 3) / 4 * 4;
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
  x.succ_ptr = static_cast<int*>(take(sizeof(int) * (mc + 1)));
  x.succ = static_cast<int*>(take(sizeof(int) * mc));
  x.ctl = static_cast<int*>(take(sizeof(int) * 4));
  x.scratch = static_cast<int*>(take(sizeof(int) * (4 * std::max<int64_t>(n_nodes, 1) + 4 * mc + 2)));
  x.flags_f = static_cast<int*>(take(sizeof(int) * mc * H * ns));
  x.Pm = static_cast<float*>(take(sizeof(float) * mc * H * kChunk * kChunk));
  x.Xm = static_cast<float*>(take(sizeof(float) * mc * H * kChunk * kChunk));
  x.W = static_cast<float*>(take(sizeof(float) * mc * H * kChunk * DkP));
  x.U0 = static_cast<float*>(take(sizeof(float) * mc * H * ns * kChunk * kSlice));
  x.u = static_cast<float*>(take(sizeof(float) * mc * H * ns * kChunk * kSlice));
  x.states = static_cast<float*>(take(sizeof(float) * mc * H * ns * Dk * kSlice));
  if (bwd) {
    x.flags_b = static_cast<int*>(take(sizeof(int) * mc * H * ns));
    x.dstart = static_cast<float*>(take(sizeof(float) * mc * H * ns * Dk * kSlice));
    x.dend = static_cast<float*>(take(sizeof(float) * mc * H * ns * Dk * kSlice));
    x.dr = static_cast<float*>(take(sizeof(float) * mc * H * ns * kChunk * kSlice));
    x.part = static_cast<float*>(take(sizeof(float) * ns * 2 * T * H));
    x.part_he = static_cast<float*>(take(sizeof(float) * ns * mc * H));
  }
  if (w) *w = x;
  return round_up(off, 256);
}

// ------------------------------------------------------------------------------ setup
// Sub-chunk table from the node arrays (one thread walks the nodes in preorder, checking
// that they tile [0, T) with earlier parents), the schedule (sub-chunks by increasing
// chain depth: a counting sort, stable in preorder) and the successor lists; all threads
// clear the flags. On a malformed table nothing is scheduled (n_chunks = 0). The walk's
// working arrays (copies of the node arrays, each node's last sub-chunk, each sub-chunk's
// depth and predecessor, the sort's counters) live in shared memory when they fit
// (`fits`), else in the workspace.
constexpr int kSetupThreads = 1024;

__host__ __device__ constexpr int64_t setup_ints(int64_t n_nodes, int64_t max_chunks) {
  return 4 * n_nodes + 4 * max_chunks + 2;  // node arrays, nlast; depth, pred, two counters of mc + 1
}

__global__ void __launch_bounds__(kSetupThreads) gdn_setup_kernel(const int32_t* __restrict__ node_start,
                                                                  const int32_t* __restrict__ node_end,
                                                                  const int32_t* __restrict__ node_parent,
                                                                  int n_nodes, int T, int64_t n_flags, GdnWs w,
                                                                  int max_chunks, int fits, int* err) {
  extern __shared__ int ssm[];
  for (int64_t i = threadIdx.x; i < n_flags; i += blockDim.x) {
    w.flags_f[i] = 0;
    if (w.flags_b) w.flags_b[i] = 0;
  }
  int* nst = fits ? ssm : w.scratch;
  int* nen = nst + n_nodes;
  int* npa = nen + n_nodes;
  int* nlast = npa + n_nodes;
  int* cdepth = nlast + n_nodes;
  int* cpred = cdepth + max_chunks;
  int* dc = cpred + max_chunks;   // [max_chunks + 1]
  int* sp = dc + max_chunks + 1;  // [max_chunks + 1]
  for (int i = threadIdx.x; i < n_nodes; i += blockDim.x) {
    nst[i] = node_start[i];
    nen[i] = node_end[i];
    npa[i] = node_parent[i];
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  w.ctl[1] = 0;
  w.ctl[2] = 0;
  w.ctl[3] = 0;
  int m = 0, next = 0;
  bool ok = true;
  for (int n = 0; n < n_nodes && ok; ++n) {
    const int s = nst[n], e = nen[n] + 1, par = npa[n];
    if (s != next || e <= s || e > T || par >= n || par < -1) {
      ok = false;
      break;
    }
    next = e;
    int pred = par >= 0 ? nlast[par] : -1;
    int depth = pred >= 0 ? cdepth[pred] + 1 : 0;
    for (int c0 = s; c0 < e; c0 += kChunk, ++depth) {
      if (m >= max_chunks) { ok = false; break; }
      cpred[m] = pred;
      cdepth[m] = depth;
      w.chunks[m] = make_int4(c0, min(kChunk, e - c0), pred, depth);
      pred = m++;
    }
    nlast[n] = pred;
  }
  if (!ok || next != T) {
    raise_error(err, TREE_ERR_DEVICE_CHECK);
    m = 0;
  }
  for (int d = 0; d <= m; ++d) dc[d] = 0;
  for (int c = 0; c < m; ++c) ++dc[cdepth[c] + 1];
  for (int d = 1; d <= m; ++d) dc[d] += dc[d - 1];
  for (int c = 0; c < m; ++c) w.order[dc[cdepth[c]]++] = c;
  // successor lists: the successors of c in increasing sub-chunk index
  for (int c = 0; c <= m; ++c) sp[c] = 0;
  for (int c = 0; c < m; ++c)
    if (cpred[c] >= 0) ++sp[cpred[c] + 1];
  for (int c = 1; c <= m; ++c) sp[c] += sp[c - 1];
  for (int c = 0; c <= m; ++c) {
    w.succ_ptr[c] = sp[c];
    dc[c] = sp[c];  // fill cursors
  }
  for (int c = 0; c < m; ++c)
    if (cpred[c] >= 0) w.succ[dc[cpred[c]]++] = c;
  w.ctl[0] = m;
}

// Running log-decay of a sub-chunk and the factors built from it: the first two warps load
// g and beta of one row each and form the running sum with a warp scan (the same order in
// every kernel, so every kernel sees the same lg). Ends with a block barrier.
__device__ __forceinline__ void decay_factors(const float* __restrict__ g, const float* __restrict__ beta, int r0,
                                              int L, int H, int h, float* lg, float* E, float* wv, float* bs) {
  __shared__ float s_carry;
  const int t = threadIdx.x;
  float x = 0.f;
  if (t < kChunk) {
    const bool in = t < L;
    const int64_t row = static_cast<int64_t>(r0 + t) * H + h;
    x = in ? g[row] : 0.f;
    bs[t] = in ? beta[row] : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if ((t & 31) >= o) x += y;
    }
    if (t == 31) s_carry = x;
  }
  __syncthreads();
  if (t < kChunk) {
    if (t >= 32) x += s_carry;
    lg[t] = x;
    E[t] = t < L ? expf(x) : 0.f;
  }
  __syncthreads();
  if (t < kChunk) wv[t] = t < L ? expf(lg[L - 1] - lg[t]) : 0.f;
  __syncthreads();
}

// 8 bf16 or 4 fp32 values of one 16-byte vector, widened to fp32.
__device__ __forceinline__ void widen(const uint4& v, float* f, const __nv_bfloat16*) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x = __bfloat1622float2(b[i]);
    f[2 * i] = x.x;
    f[2 * i + 1] = x.y;
  }
}
__device__ __forceinline__ void widen(const uint4& v, float* f, const float*) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}

// Columns [col0, col0 + ncols) of rows [r0, r0 + 64) of a [T, H, D] tensor (head h) into
// an fp32 shared tile (row stride `stride`), zero past L rows and past D columns (up to
// ncols, a multiple of 4). Every thread issues all of its 16-byte loads before using any,
// so their latencies overlap; rows whose width is not a whole number of vectors take a
// scalar path. The input pointer is 16-byte aligned (checked on the host).
template <typename Tin>
__device__ __forceinline__ void load_tile(float* dst, int stride, const Tin* __restrict__ src, int r0, int L, int H,
                                          int h, int D, int col0, int ncols) {
  constexpr int kVec = 16 / sizeof(Tin);                       // 8 bf16 or 4 fp32
  constexpr int kPer = kChunk * kMaxD / kVec / kThreads;        // most vectors a thread loads
  const int nv = ncols / kVec, total = kChunk * nv;
  if (D % kVec == 0 && ncols % kVec == 0) {
    uint4 buf[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int idx = threadIdx.x + u * kThreads;
      const int t = idx / max(nv, 1), cv = col0 + (idx % max(nv, 1)) * kVec;
      buf[u] = make_uint4(0u, 0u, 0u, 0u);
      if (idx < total && t < L && cv < D)
        buf[u] = __ldg(reinterpret_cast<const uint4*>(src + (static_cast<int64_t>(r0 + t) * H + h) * D + cv));
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int idx = threadIdx.x + u * kThreads;
      if (idx < total) {
        const int t = idx / nv, cl = (idx % nv) * kVec;
        float f[kVec];
        widen(buf[u], f, src);
#pragma unroll
        for (int e = 0; e < kVec; e += 4)
          *reinterpret_cast<float4*>(dst + t * stride + cl + e) = make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
      }
    }
  } else {
#pragma unroll 8
    for (int idx = threadIdx.x; idx < kChunk * ncols; idx += kThreads) {
      const int t = idx / ncols, cl = idx % ncols, cv = col0 + cl;
      dst[t * stride + cl] = (t < L && cv < D) ? ldf(src, (static_cast<int64_t>(r0 + t) * H + h) * D + cv) : 0.f;
    }
  }
}

__device__ __forceinline__ float dot4(const float* a, const float* b, int n4) {
  float acc = 0.f;
  for (int i = 0; i < n4; i += 4) {
    const float4 x = *reinterpret_cast<const float4*>(a + i);
    const float4 y = *reinterpret_cast<const float4*>(b + i);
    acc = fmaf(x.x, y.x, acc);
    acc = fmaf(x.y, y.y, acc);
    acc = fmaf(x.z, y.z, acc);
    acc = fmaf(x.w, y.w, acc);
  }
  return acc;
}

struct GdnArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  void* o;
  const void* dout;
  void* dq;
  void* dk;
  void* dv;
  float* dg;
  float* dbeta;
  int T, H, Dk, Dv, ns, DkP;
  int withhold;                 // test hook: this sub-chunk's publications are withheld (-1: none)
  unsigned long long wait_ns;   // limit of every wait on a publication
  GdnWs w;
  int* err;
};

// ------------------------------------------------------------------------------ prep
// Per (sub-chunk, head): P and X = (I + A)^-1 to the workspace, W = X (beta E o K) and
// U0 = X (beta o V), all 64 rows (zero past L) and every padding column written.
constexpr size_t kPrepSmem = (2 * kChunk * kRow + 2 * kChunk * kSq + 4 * kChunk) * sizeof(float);

template <typename Tin>
__global__ void __launch_bounds__(kThreads) gdn_prep_kernel(const GdnArgs a) {
  extern __shared__ __align__(16) float sm[];
  float* Ks = sm;                        // [64][kRow]
  float* QV = Ks + kChunk * kRow;        // [64][kRow]: Q, then V
  float* Am = QV + kChunk * kRow;        // [64][kSq]
  float* Xm = Am + kChunk * kSq;         // [64][kSq]
  float* lg = Xm + kChunk * kSq;
  float* E = lg + kChunk;
  float* wv = E + kChunk;
  float* bs = wv + kChunk;
  const int c = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  if (c >= a.w.ctl[0]) return;
  const int4 ck = a.w.chunks[c];
  const int r0 = ck.x, L = ck.y, H = a.H, Dk = a.Dk, Dv = a.Dv, DkP = a.DkP, ns = a.ns;
  const int Dk4 = (Dk + 3) & ~3, Dv4 = (Dv + 3) & ~3;
  load_tile(Ks, kRow, static_cast<const Tin*>(a.k), r0, L, H, h, Dk, 0, Dk4);
  load_tile(QV, kRow, static_cast<const Tin*>(a.q), r0, L, H, h, Dk, 0, Dk4);
  decay_factors(a.g, a.beta, r0, L, H, h, lg, E, wv, bs);  // ends with a barrier
  float* Pg = a.w.Pm + (static_cast<int64_t>(c) * H + h) * kChunk * kChunk;
  float* Xg = a.w.Xm + (static_cast<int64_t>(c) * H + h) * kChunk * kChunk;
  for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) {
    const int t = idx / kChunk, s = idx % kChunk;
    float av = 0.f, pv = 0.f;
    if (t < L && s <= t) {
      const float f = expf(lg[t] - lg[s]);
      pv = f * dot4(QV + t * kRow, Ks + s * kRow, Dk4);
      if (s < t) av = bs[t] * f * dot4(Ks + t * kRow, Ks + s * kRow, Dk4);
    }
    Am[t * kSq + s] = av;
    Pg[idx] = pv;
  }
  __syncthreads();
  // V over Q (Q is done); X by forward substitution, one column per thread
  load_tile(QV, kRow, static_cast<const Tin*>(a.v), r0, L, H, h, Dv, 0, Dv4);
  if (tid < kChunk) {
    const int cc = tid;
    for (int t = 0; t < kChunk; ++t) Xm[t * kSq + cc] = t == cc ? 1.f : 0.f;
    for (int t = cc + 1; t < L; ++t) {
      float acc = 0.f;
      for (int s = cc; s < t; ++s) acc = fmaf(-Am[t * kSq + s], Xm[s * kSq + cc], acc);
      Xm[t * kSq + cc] = acc;
    }
  }
  __syncthreads();
  for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) Xg[idx] = Xm[(idx / kChunk) * kSq + idx % kChunk];
  // W = X (beta E o K), U0 = X (beta o V): column `col` per thread, 32 rows each
  const int col = tid % kMaxD, half = tid / kMaxD;
  float* Wg = a.w.W + (static_cast<int64_t>(c) * H + h) * kChunk * DkP;
  for (int m = 0; m < 32; ++m) {
    const int t = 32 * half + m;
    float wa = 0.f, ua = 0.f;
    if (t < L) {
      for (int s = 0; s <= t; ++s) {
        const float x = Xm[t * kSq + s] * bs[s];
        wa = fmaf(x * E[s], Ks[s * kRow + col], wa);
        ua = fmaf(x, QV[s * kRow + col], ua);
      }
    }
    if (col < DkP) Wg[t * DkP + col] = col < Dk ? wa : 0.f;
    if (col < ns * kSlice)
      slice_block(a.w.U0, c, h, col / kSlice, H, ns, kChunk)[t * kSlice + col % kSlice] = col < Dv ? ua : 0.f;
  }
}

// ------------------------------------------------------------------------------ waits
// Bounded wait for a publication flag: gives up after wait_ns, or at once when another
// CTA has already given up (the abort word), raising TREE_ERR_TIMEOUT.
__device__ bool wait_flag(const int* f, const GdnArgs& a, int* abort) {
  if (ld_acquire(f)) return true;
  const unsigned long long t0 = sm100::globaltimer();
  while (!ld_acquire(f)) {
    if (*reinterpret_cast<volatile int*>(abort) || sm100::globaltimer() - t0 > a.wait_ns) {
      raise_error(a.err, TREE_ERR_TIMEOUT);
      atomicExch(abort, 1);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

// Next chain item of this CTA (thread 0 draws it; every thread calls).
__device__ __forceinline__ int next_item(int* counter, int* abort, int items, int* s_item) {
  __syncthreads();
  if (threadIdx.x == 0) *s_item = *reinterpret_cast<volatile int*>(abort) ? items : atomicAdd(counter, 1);
  __syncthreads();
  return *s_item;
}

// ------------------------------------------------------------------------------ chain
// Per (sub-chunk, head, slice of 32 state columns), by increasing chain depth:
//   u = U0 - W h0,   h_end = E_{L-1} h0 + sum_t w_t k_t u_t^T.
// The item's loads are issued together right after its predecessor's flag is seen.
constexpr size_t kChainSmem = (2 * kChunk * kRow + kMaxD * kSl + kChunk * kSl + 4 * kChunk) * sizeof(float);

template <typename Tin>
__global__ void __launch_bounds__(kThreads) gdn_chain_kernel(const GdnArgs a) {
  extern __shared__ __align__(16) float sm[];
  float* Ws = sm;                       // [64][kRow]
  float* Ks = Ws + kChunk * kRow;       // [64][kRow]
  float* Hs = Ks + kChunk * kRow;       // [128][kSl] h0 slice
  float* Us = Hs + kMaxD * kSl;         // [64][kSl] U0, then u
  float* lg = Us + kChunk * kSl;
  float* E = lg + kChunk;
  float* wv = E + kChunk;
  float* bs = wv + kChunk;
  __shared__ int s_item, s_ok;
  const GdnWs& w = a.w;
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int H = a.H, Dk = a.Dk, ns = a.ns, DkP = a.DkP;
  const int Dk4 = (Dk + 3) & ~3;
  const int items = w.ctl[0] * H * ns;
  while (true) {
    const int item = next_item(&w.ctl[1], &w.ctl[3], items, &s_item);
    if (item >= items) break;
    const int c = w.order[item / (H * ns)], rem = item % (H * ns), h = rem / ns, sl = rem % ns;
    const int4 ck = w.chunks[c];
    const int r0 = ck.x, L = ck.y, pred = ck.z;
    // loads that do not depend on the predecessor first
    cp_block(Ws, kRow, w.W + (static_cast<int64_t>(c) * H + h) * kChunk * DkP, kChunk, DkP);
    cp_block(Us, kSl, slice_block(w.U0, c, h, sl, H, ns, kChunk), kChunk, kSlice);
    load_tile(Ks, kRow, static_cast<const Tin*>(a.k), r0, L, H, h, Dk, 0, Dk4);
    if (tid == 0)
      s_ok = pred < 0 || wait_flag(w.flags_f + (static_cast<int64_t>(pred) * H + h) * ns + sl, a, &w.ctl[3]);
    __syncthreads();
    if (!s_ok) {
      cp_wait();
      break;
    }
    if (pred >= 0) {
      cp_block(Hs, kSl, slice_block(w.states, pred, h, sl, H, ns, Dk), Dk, kSlice);
    } else {
      for (int idx = tid; idx < Dk * kSlice; idx += kThreads) Hs[(idx / kSlice) * kSl + idx % kSlice] = 0.f;
    }
    cp_wait();
    decay_factors(a.g, a.beta, r0, L, H, h, lg, E, wv, bs);  // ends with a barrier
    // u = U0 - W h0: rows t = warp + 8 m of column `lane` (zero past L)
    float* ug = slice_block(w.u, c, h, sl, H, ns, kChunk);
    for (int t = warp; t < kChunk; t += 8) {
      float acc = 0.f;
      if (t < L) {
        acc = Us[t * kSl + lane];
        for (int i = 0; i < Dk; ++i) acc = fmaf(-Ws[t * kRow + i], Hs[i * kSl + lane], acc);
      }
      Us[t * kSl + lane] = acc;
      ug[t * kSlice + lane] = acc;
    }
    __syncthreads();
    // h_end = E_{L-1} h0 + sum_t w_t k_t u_t^T: rows i = warp + 8 m of column `lane`
    float* hend = slice_block(w.states, c, h, sl, H, ns, Dk);
    const float gl = E[L - 1];
    for (int i = warp; i < Dk; i += 8) {
      float acc = gl * Hs[i * kSl + lane];
      for (int t = 0; t < L; ++t) acc = fmaf(wv[t] * Ks[t * kRow + i], Us[t * kSl + lane], acc);
      __stcg(hend + i * kSlice + lane, acc);
    }
    __syncthreads();
    if (tid == 0 && c != a.withhold) {
      __threadfence();
      st_release(w.flags_f + (static_cast<int64_t>(c) * H + h) * ns + sl, 1);
    }
  }
}

// ------------------------------------------------------------------------------ out
// Per (sub-chunk, head): O = E o (Q h0) + P u.
constexpr size_t kOutSmem = (2 * kChunk * kRow + kMaxD * kRow + kChunk * kSq + 4 * kChunk) * sizeof(float);

template <typename Tin>
__global__ void __launch_bounds__(kThreads) gdn_out_kernel(const GdnArgs a) {
  extern __shared__ __align__(16) float sm[];
  float* Qs = sm;                      // [64][kRow]
  float* Us = Qs + kChunk * kRow;      // [64][kRow] u
  float* Hs = Us + kChunk * kRow;      // [128][kRow] h0
  float* Ps = Hs + kMaxD * kRow;       // [64][kSq]
  float* lg = Ps + kChunk * kSq;
  float* E = lg + kChunk;
  float* wv = E + kChunk;
  float* bs = wv + kChunk;
  const int c = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const GdnWs& w = a.w;
  if (c >= w.ctl[0]) return;
  if (*reinterpret_cast<volatile int*>(&w.ctl[3])) return;  // the chain gave up: outputs unspecified
  const int4 ck = w.chunks[c];
  const int r0 = ck.x, L = ck.y, pred = ck.z, H = a.H, Dk = a.Dk, Dv = a.Dv, ns = a.ns;
  const int Dk4 = (Dk + 3) & ~3;
  for (int sl = 0; sl < ns; ++sl) {
    cp_block(Us + sl * kSlice, kRow, slice_block(w.u, c, h, sl, H, ns, kChunk), kChunk, kSlice);
    if (pred >= 0) cp_block(Hs + sl * kSlice, kRow, slice_block(w.states, pred, h, sl, H, ns, Dk), Dk, kSlice);
  }
  cp_block(Ps, kSq, w.Pm + (static_cast<int64_t>(c) * H + h) * kChunk * kChunk, kChunk, kChunk);
  load_tile(Qs, kRow, static_cast<const Tin*>(a.q), r0, L, H, h, Dk, 0, Dk4);
  cp_wait();
  decay_factors(a.g, a.beta, r0, L, H, h, lg, E, wv, bs);  // ends with a barrier
  const int j = tid % kMaxD, half = tid / kMaxD;
  if (j >= Dv) return;
  Tin* o = static_cast<Tin*>(a.o);
  float acc[32];
#pragma unroll
  for (int m = 0; m < 32; ++m) acc[m] = 0.f;
  if (pred >= 0) {
    for (int i = 0; i < Dk; ++i) {
      const float hij = Hs[i * kRow + j];
#pragma unroll
      for (int m = 0; m < 32; ++m) acc[m] = fmaf(Qs[(32 * half + m) * kRow + i], hij, acc[m]);
    }
  }
#pragma unroll
  for (int m = 0; m < 32; ++m) {
    const int t = 32 * half + m;
    if (t < L) {
      float x = E[t] * acc[m];
      for (int s = 0; s <= t; ++s) x = fmaf(Ps[t * kSq + s], Us[s * kRow + j], x);
      o[(static_cast<int64_t>(r0 + t) * H + h) * Dv + j] = from_f32<Tin>(x);
    }
  }
}

// ------------------------------------------------------------------------------ bchain
// Per (sub-chunk, head, slice), by decreasing chain depth: dh_end (the sum of the
// successors' start-state gradients), du, dr, dv, dh0; per-row partial sums for dg, dbeta.
constexpr size_t kBchainSmem =
    (2 * kChunk * kRow + 2 * kChunk * kSq + 2 * kMaxD * kSl + 4 * kChunk * kSl + 4 * kChunk) * sizeof(float);

template <typename Tin>
__global__ void __launch_bounds__(kThreads) gdn_bchain_kernel(const GdnArgs a) {
  extern __shared__ __align__(16) float sm[];
  float* Ks = sm;                        // [64][kRow]
  float* Qs = Ks + kChunk * kRow;        // [64][kRow]
  float* Ps = Qs + kChunk * kRow;        // [64][kSq]
  float* Xs = Ps + kChunk * kSq;         // [64][kSq]
  float* Ds = Xs + kChunk * kSq;         // [128][kSl] dh_end slice
  float* Hs = Ds + kMaxD * kSl;          // [128][kSl] h0 slice
  float* Os = Hs + kMaxD * kSl;          // [64][kSl] dO slice
  float* Us = Os + kChunk * kSl;         // [64][kSl] u slice
  float* Vs = Us + kChunk * kSl;         // [64][kSl] v slice
  float* Rs = Vs + kChunk * kSl;         // [64][kSl] du, then dr
  float* lg = Rs + kChunk * kSl;
  float* E = lg + kChunk;
  float* wv = E + kChunk;
  float* bs = wv + kChunk;
  __shared__ int s_item, s_ok;
  __shared__ float s_red[kThreads / 32];
  const GdnWs& w = a.w;
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int H = a.H, Dk = a.Dk, Dv = a.Dv, ns = a.ns, T = a.T;
  const int Dk4 = (Dk + 3) & ~3;
  const int n_chunks = w.ctl[0];
  const int items = n_chunks * H * ns;
  const Tin* tdo = static_cast<const Tin*>(a.dout);
  Tin* tdv = static_cast<Tin*>(a.dv);
  while (true) {
    const int item = next_item(&w.ctl[2], &w.ctl[3], items, &s_item);
    if (item >= items) break;
    const int c = w.order[n_chunks - 1 - item / (H * ns)], rem = item % (H * ns), h = rem / ns, sl = rem % ns;
    const int4 ck = w.chunks[c];
    const int r0 = ck.x, L = ck.y, pred = ck.z;
    const int j = sl * kSlice + lane;
    const int sb = w.succ_ptr[c], se = w.succ_ptr[c + 1];
    // loads that do not depend on the successors first
    const int64_t mo = (static_cast<int64_t>(c) * H + h) * kChunk * kChunk;
    cp_block(Ps, kSq, w.Pm + mo, kChunk, kChunk);
    cp_block(Xs, kSq, w.Xm + mo, kChunk, kChunk);
    cp_block(Us, kSl, slice_block(w.u, c, h, sl, H, ns, kChunk), kChunk, kSlice);
    if (pred >= 0) cp_block(Hs, kSl, slice_block(w.states, pred, h, sl, H, ns, Dk), Dk, kSlice);
    load_tile(Ks, kRow, static_cast<const Tin*>(a.k), r0, L, H, h, Dk, 0, Dk4);
    load_tile(Qs, kRow, static_cast<const Tin*>(a.q), r0, L, H, h, Dk, 0, Dk4);
    load_tile(Os, kSl, tdo, r0, L, H, h, Dv, sl * kSlice, kSlice);
    load_tile(Vs, kSl, static_cast<const Tin*>(a.v), r0, L, H, h, Dv, sl * kSlice, kSlice);
    if (pred < 0)
      for (int idx = tid; idx < Dk * kSlice; idx += kThreads) Hs[(idx / kSlice) * kSl + idx % kSlice] = 0.f;
    if (tid == 0) {
      bool ok = true;
      for (int s = sb; ok && s < se; ++s)
        ok = wait_flag(w.flags_b + (static_cast<int64_t>(w.succ[s]) * H + h) * ns + sl, a, &w.ctl[3]);
      s_ok = ok;
    }
    __syncthreads();
    if (!s_ok) {
      cp_wait();
      break;
    }
    // dh_end slice = the sum of the successors' dh0 (fixed order), kept for the grads kernel
    {
      constexpr int kPer = kMaxD * kSlice / 4 / kThreads;  // float4 per thread
      float4 acc[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s = sb; s < se; ++s) {
        const float4* src = reinterpret_cast<const float4*>(slice_block(w.dstart, w.succ[s], h, sl, H, ns, Dk));
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int p = tid + u * kThreads;
          if (p < Dk * kSlice / 4) {
            const float4 x = __ldcg(src + p);
            acc[u].x += x.x; acc[u].y += x.y; acc[u].z += x.z; acc[u].w += x.w;
          }
        }
      }
      float4* dend = reinterpret_cast<float4*>(slice_block(w.dend, c, h, sl, H, ns, Dk));
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int p = tid + u * kThreads;
        if (p < Dk * kSlice / 4) {
          __stcg(dend + p, acc[u]);
          *reinterpret_cast<float4*>(Ds + (p / (kSlice / 4)) * kSl + (p % (kSlice / 4)) * 4) = acc[u];
        }
      }
    }
    cp_wait();
    __syncthreads();
    float he = 0.f;  // partial sum of dh_end . h0
    for (int idx = tid; idx < Dk * kSlice; idx += kThreads) {
      const int i = idx / kSlice, jj = idx % kSlice;
      he = fmaf(Ds[i * kSl + jj], Hs[i * kSl + jj], he);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) he += __shfl_xor_sync(0xffffffffu, he, o);
    if (lane == 0) s_red[warp] = he;
    decay_factors(a.g, a.beta, r0, L, H, h, lg, E, wv, bs);  // ends with a barrier
    if (tid == 0) {
      float x = 0.f;
      for (int u = 0; u < kThreads / 32; ++u) x += s_red[u];
      w.part_he[(static_cast<int64_t>(sl) * n_chunks + c) * H + h] = x;
    }
    // du = w o (K dh_end) + P^T dO; partial dw_t = w_t sum_j (K dh_end)_tj u_tj
    for (int t = warp; t < L; t += 8) {
      float kd = 0.f;
      for (int i = 0; i < Dk; ++i) kd = fmaf(Ks[t * kRow + i], Ds[i * kSl + lane], kd);
      float du = wv[t] * kd;
      for (int t2 = t; t2 < L; ++t2) du = fmaf(Ps[t2 * kSq + t], Os[t2 * kSl + lane], du);
      Rs[t * kSl + lane] = du;
      float dw = wv[t] * kd * Us[t * kSl + lane];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dw += __shfl_xor_sync(0xffffffffu, dw, o);
      if (lane == 0) w.part[((static_cast<int64_t>(sl) * 2 + 0) * T + r0 + t) * H + h] = dw;
    }
    __syncthreads();
    // dr = X^T du (in registers first: every row reads the whole column of du), dv = beta o dr
    float drr[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int t = warp + 8 * m;
      float x = 0.f;
      if (t < L)
        for (int t2 = t; t2 < L; ++t2) x = fmaf(Xs[t2 * kSq + t], Rs[t2 * kSl + lane], x);
      drr[m] = x;
    }
    __syncthreads();
    float* drg = slice_block(w.dr, c, h, sl, H, ns, kChunk);
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int t = warp + 8 * m;
      Rs[t * kSl + lane] = drr[m];
      drg[t * kSlice + lane] = drr[m];
      if (t < L) {
        if (j < Dv) tdv[(static_cast<int64_t>(r0 + t) * H + h) * Dv + j] = from_f32<Tin>(bs[t] * drr[m]);
        float rv = drr[m] * Vs[t * kSl + lane];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) rv += __shfl_xor_sync(0xffffffffu, rv, o);
        if (lane == 0) w.part[((static_cast<int64_t>(sl) * 2 + 1) * T + r0 + t) * H + h] = rv;
      }
    }
    __syncthreads();
    // dh0 = E_{L-1} dh_end + Q^T (E o dO) - K^T (beta E o dr)
    float* dst = slice_block(w.dstart, c, h, sl, H, ns, Dk);
    const float gl = E[L - 1];
    for (int i = warp; i < Dk; i += 8) {
      float acc = gl * Ds[i * kSl + lane];
      for (int t = 0; t < L; ++t)
        acc = fmaf(E[t], fmaf(Qs[t * kRow + i], Os[t * kSl + lane], -bs[t] * Ks[t * kRow + i] * Rs[t * kSl + lane]),
                   acc);
      __stcg(dst + i * kSlice + lane, acc);
    }
    __syncthreads();
    if (tid == 0 && c != a.withhold) {
      __threadfence();
      st_release(w.flags_b + (static_cast<int64_t>(c) * H + h) * ns + sl, 1);
    }
  }
}

// ------------------------------------------------------------------------------ grads
// Per (sub-chunk, head): dQ, dK (dtype), dg, dbeta (fp32).
constexpr size_t kGradsSmem = (5 * kChunk * kRow + 3 * kChunk * kSq + 6 * kChunk) * sizeof(float);
static_assert(kGradsSmem <= 227 * 1024, "GDN grads shared memory exceeds the per-block limit");
static_assert(kBchainSmem <= 227 * 1024 && kPrepSmem <= 227 * 1024 && kChainSmem <= 227 * 1024 &&
                  kOutSmem <= 227 * 1024,
              "GDN shared memory exceeds the per-block limit");
static_assert(2 * kMaxD * kSt <= kChunk * kSq, "h0 / dh_end staging must fit in the M1 buffer");

template <typename Tin>
__global__ void __launch_bounds__(kThreads, 1) gdn_grads_kernel(const GdnArgs a) {
  extern __shared__ __align__(16) float sm[];
  float* Ks = sm;                       // [64][kRow]
  float* Qs = Ks + kChunk * kRow;       // [64][kRow]
  float* Us = Qs + kChunk * kRow;       // [64][kRow] u
  float* Os = Us + kChunk * kRow;       // [64][kRow] dO
  float* Rs = Os + kChunk * kRow;       // [64][kRow] dr
  float* Fp = Rs + kChunk * kRow;       // [64][kSq] dP o f
  float* Fa = Fp + kChunk * kSq;        // [64][kSq] dA o beta f
  float* M1 = Fa + kChunk * kSq;        // [64][kSq] dP o P + dA o A; later staging and reductions
  float* lg = M1 + kChunk * kSq;
  float* E = lg + kChunk;
  float* wv = E + kChunk;
  float* bs = wv + kChunk;
  float* dlg = bs + kChunk;             // d lg per row
  float* dbt = dlg + kChunk;            // dbeta per row
  __shared__ float s_part[4];
  const int c = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const GdnWs& w = a.w;
  const int n_chunks = w.ctl[0];
  if (c >= n_chunks) return;
  if (*reinterpret_cast<volatile int*>(&w.ctl[3])) return;  // a chain gave up: outputs unspecified
  const int4 ck = w.chunks[c];
  const int r0 = ck.x, L = ck.y, pred = ck.z, H = a.H, Dk = a.Dk, Dv = a.Dv, T = a.T, ns = a.ns;
  const int Dk4 = (Dk + 3) & ~3, Dv4 = (Dv + 3) & ~3;
  for (int sl = 0; sl < ns; ++sl) {
    cp_block(Us + sl * kSlice, kRow, slice_block(w.u, c, h, sl, H, ns, kChunk), kChunk, kSlice);
    cp_block(Rs + sl * kSlice, kRow, slice_block(w.dr, c, h, sl, H, ns, kChunk), kChunk, kSlice);
  }
  load_tile(Ks, kRow, static_cast<const Tin*>(a.k), r0, L, H, h, Dk, 0, Dk4);
  load_tile(Qs, kRow, static_cast<const Tin*>(a.q), r0, L, H, h, Dk, 0, Dk4);
  load_tile(Os, kRow, static_cast<const Tin*>(a.dout), r0, L, H, h, Dv, 0, Dv4);
  cp_wait();
  decay_factors(a.g, a.beta, r0, L, H, h, lg, E, wv, bs);  // ends with a barrier
  // pairs (t, s), s <= t: four threads per row t, s = sub + 4 m
  {
    const int t = tid / 4, sub = tid % 4;
    float rowsum = 0.f, rowb = 0.f;
    for (int s = sub; s < kChunk; s += 4) {
      float fp = 0.f, fa = 0.f, m1 = 0.f;
      if (t < L && s <= t) {
        const float f = expf(lg[t] - lg[s]);
        const float qk = dot4(Qs + t * kRow, Ks + s * kRow, Dk4);
        const float dp = dot4(Os + t * kRow, Us + s * kRow, Dv4);
        fp = dp * f;
        m1 = fp * qk;  // dP o P
        if (s < t) {
          const float kk = dot4(Ks + t * kRow, Ks + s * kRow, Dk4);
          const float da = -dot4(Rs + t * kRow, Us + s * kRow, Dv4);
          fa = da * bs[t] * f;
          m1 = fmaf(fa, kk, m1);           // dA o A
          rowb = fmaf(da * f, kk, rowb);   // dA o f o KK (dbeta)
        }
      }
      Fp[t * kSq + s] = fp;
      Fa[t * kSq + s] = fa;
      M1[t * kSq + s] = m1;
      rowsum += m1;
    }
    rowsum += __shfl_xor_sync(0xffffffffu, rowsum, 1);
    rowsum += __shfl_xor_sync(0xffffffffu, rowsum, 2);
    rowb += __shfl_xor_sync(0xffffffffu, rowb, 1);
    rowb += __shfl_xor_sync(0xffffffffu, rowb, 2);
    if (sub == 0) {
      dlg[t] = rowsum;
      dbt[t] = rowb;
    }
  }
  __syncthreads();
  if (tid < kChunk) {  // column sums of M1, in row order
    float x = 0.f;
    for (int t = 0; t < kChunk; ++t) x += M1[t * kSq + tid];
    dlg[tid] -= x;
  }
  // dQ, dK: column i per thread, 16 rows per pass, two passes per half
  const int i = tid % kMaxD, half = tid / kMaxD;
  float* hst = M1;                      // [128][kSt] 16 columns of h0, staged
  float* dst = M1 + kMaxD * kSt;        // [128][kSt] the same columns of dh_end
  Tin* dq = static_cast<Tin*>(a.dq);
  Tin* dk = static_cast<Tin*>(a.dk);
  for (int pass = 0; pass < 2; ++pass) {
    const int t0 = 32 * half + 16 * pass;
    float qa[16], ka[16], z1[16], z2[16], z3[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) qa[m] = ka[m] = z1[m] = z2[m] = z3[m] = 0.f;
    for (int s = 0; s < kChunk; ++s) {
      const float kv = Ks[s * kRow + i], qv = Qs[s * kRow + i];
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const int t = t0 + m;
        qa[m] = fmaf(Fp[t * kSq + s], kv, qa[m]);                       // (dP o f) K
        ka[m] = fmaf(Fp[s * kSq + t], qv, ka[m]);                       // (dP o f)^T Q
        ka[m] = fmaf(Fa[t * kSq + s] + Fa[s * kSq + t], kv, ka[m]);     // (dA o b f) K + its transpose
      }
    }
    for (int j0 = 0; j0 < ns * kSlice; j0 += 16) {
      const int sl = j0 / kSlice, off = j0 % kSlice;
      __syncthreads();
      const float* hg = pred >= 0 ? slice_block(w.states, pred, h, sl, H, ns, Dk) : nullptr;
      const float* dg = slice_block(w.dend, c, h, sl, H, ns, Dk);
      for (int idx = tid; idx < Dk * 16; idx += kThreads) {
        const int ii = idx / 16, jj = idx % 16;
        if (hg) cp4(hst + ii * kSt + jj, hg + ii * kSlice + off + jj);
        else hst[ii * kSt + jj] = 0.f;
        cp4(dst + ii * kSt + jj, dg + ii * kSlice + off + jj);
      }
      cp_wait();
      __syncthreads();
      const int jn = min(16, Dv - j0);
      if (i < Dk) {
        for (int jj = 0; jj < jn; ++jj) {
          const float hv = hst[i * kSt + jj], dv = dst[i * kSt + jj];
#pragma unroll
          for (int m = 0; m < 16; ++m) {
            const int t = t0 + m;
            z1[m] = fmaf(Os[t * kRow + j0 + jj], hv, z1[m]);   // (dO h0^T)_ti
            z2[m] = fmaf(Rs[t * kRow + j0 + jj], hv, z2[m]);   // (dr h0^T)_ti
            z3[m] = fmaf(Us[t * kRow + j0 + jj], dv, z3[m]);   // (u dh_end^T)_ti
          }
        }
      }
    }
    __syncthreads();
    // the d lg terms E_t q_t . (dO h0^T)_t and -beta_t E_t k_t . (dr h0^T)_t and the dbeta
    // term -E_t k_t . (dr h0^T)_t: dot products over i, reduced over the 128 threads of a half
    float* red = M1;  // [2 halves][16 rows][8]
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const int t = t0 + m;
      float cq = i < Dk ? Qs[t * kRow + i] * z1[m] : 0.f;   // columns past Dk hold no data
      float ck2 = i < Dk ? Ks[t * kRow + i] * z2[m] : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        cq += __shfl_xor_sync(0xffffffffu, cq, o);
        ck2 += __shfl_xor_sync(0xffffffffu, ck2, o);
      }
      if (lane == 0) {
        red[(half * 16 + m) * 8 + (warp % 4)] = cq;
        red[(half * 16 + m) * 8 + 4 + (warp % 4)] = ck2;
      }
      if (t < L && i < Dk) {
        const int64_t off = (static_cast<int64_t>(r0 + t) * H + h) * Dk + i;
        dq[off] = from_f32<Tin>(qa[m] + E[t] * z1[m]);
        dk[off] = from_f32<Tin>(ka[m] + wv[t] * z3[m] - bs[t] * E[t] * z2[m]);
      }
    }
    __syncthreads();
    if (tid < 32) {  // lane (half, m) finishes row 32 half + 16 pass + m
      const int hh = tid / 16, m = tid % 16, t = 32 * hh + 16 * pass + m;
      const float* rr = red + (hh * 16 + m) * 8;
      const float cq = (rr[0] + rr[1]) + (rr[2] + rr[3]);
      const float ck2 = (rr[4] + rr[5]) + (rr[6] + rr[7]);
      dlg[t] += E[t] * cq - bs[t] * E[t] * ck2;
      dbt[t] -= E[t] * ck2;
    }
  }
  __syncthreads();
  // the chain's per-row sums (over the slices, in order), then dg as the reverse running
  // sum of d lg over the sub-chunk: the first two warps own one row each
  float dw = 0.f;
  if (tid < kChunk && tid < L) {
    float rv = 0.f;
    for (int sl = 0; sl < ns; ++sl) {
      dw += w.part[((static_cast<int64_t>(sl) * 2 + 0) * T + r0 + tid) * H + h];
      rv += w.part[((static_cast<int64_t>(sl) * 2 + 1) * T + r0 + tid) * H + h];
    }
    dlg[tid] -= dw;
    dbt[tid] += rv;
  }
  if (tid < kChunk) {
    float x = dw;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) s_part[warp] = x;
  }
  if (tid == 64) {
    float he = 0.f;
    for (int sl = 0; sl < ns; ++sl) he += w.part_he[(static_cast<int64_t>(sl) * n_chunks + c) * H + h];
    s_part[2] = he;
  }
  __syncthreads();
  if (tid == 0) dlg[L - 1] += (s_part[0] + s_part[1]) + E[L - 1] * s_part[2];
  __syncthreads();
  if (tid < kChunk) {
    float x = tid < L ? dlg[L - 1 - tid] : 0.f;   // reversed rows, then an inclusive scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (tid == 31) s_part[3] = x;
    M1[tid] = x;
  }
  __syncthreads();
  if (tid < L) {
    const float x = M1[tid] + (tid >= 32 ? s_part[3] : 0.f);
    a.dg[static_cast<int64_t>(r0 + L - 1 - tid) * H + h] = x;
    a.dbeta[static_cast<int64_t>(r0 + tid) * H + h] = dbt[tid];
  }
}

int sm_count(int* n) {
  int dev = 0;
  TREE_CUDA_TRY(cudaGetDevice(&dev));
  TREE_CUDA_TRY(cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev));
  return TREE_OK;
}

// Test hook: the next GDN call withholds the publications of one sub-chunk and waits at
// most this long for any publication.
std::atomic<long long> g_withhold{-1};
std::atomic<unsigned long long> g_wait_ns{0};

template <typename Tin>
int run_forward_chain(GdnArgs& a, int64_t mc, int n_sm, cudaStream_t st) {
  int rc;
  if ((rc = smem_opt_in(reinterpret_cast<const void*>(gdn_prep_kernel<Tin>), static_cast<int>(kPrepSmem))) ||
      (rc = smem_opt_in(reinterpret_cast<const void*>(gdn_chain_kernel<Tin>), static_cast<int>(kChainSmem))))
    return rc;
  dim3 grid(static_cast<unsigned>(mc), static_cast<unsigned>(a.H));
  gdn_prep_kernel<Tin><<<grid, kThreads, kPrepSmem, st>>>(a);
  TREE_LAUNCH_CHECK("gdn_prep_kernel");
  gdn_chain_kernel<Tin><<<std::min(2 * n_sm, kMaxCtas), kThreads, kChainSmem, st>>>(a);
  TREE_LAUNCH_CHECK("gdn_chain_kernel");
  return TREE_OK;
}

// Shared argument checks and set-up of both calls; fills `a` and enqueues the setup
// kernel. Returns TREE_OK with *empty = true when there is nothing to compute.
int gdn_begin(GdnArgs& a, const void* q, const void* k, const void* v, const float* g, const float* beta,
              const int32_t* node_start, const int32_t* node_end, const int32_t* node_parent, int64_t T,
              int64_t n_nodes, int H, int Dk, int Dv, int dtype, void* workspace, size_t workspace_bytes,
              bool bwd, bool outs_ok, const char* name, cudaStream_t st, int64_t* mc_out, bool* empty) {
  *empty = false;
  if (dtype != TREE_DTYPE_F32 && dtype != TREE_DTYPE_BF16) return fail(TREE_ERR_DTYPE, "%s: bad dtype %d", name, dtype);
  if (T < 0 || n_nodes < 0 || T > (1 << 30) || n_nodes > T)
    return fail(TREE_ERR_SHAPE, "%s: T = %lld, n_nodes = %lld", name, (long long)T, (long long)n_nodes);
  if (H < 1 || Dk < 1 || Dv < 1 || Dk > kMaxD || Dv > kMaxD)
    return fail(TREE_ERR_SHAPE, "%s: H = %d, Dk = %d, Dv = %d (need Dk, Dv <= %d)", name, H, Dk, Dv, kMaxD);
  if (H > 65535) return fail(TREE_ERR_SHAPE, "%s: H = %d exceeds 65535", name, H);
  if (T == 0) {
    *empty = true;
    return TREE_OK;
  }
  if (n_nodes < 1) return fail(TREE_ERR_SHAPE, "%s: no nodes for %lld rows", name, (long long)T);
  const int64_t mc = gdn_max_chunks(T, n_nodes);
  // chain items are counted in 32 bits, and every CTA draws once past the last item
  if (mc * H * gdn_slices(Dv) + kMaxCtas > INT32_MAX || mc > INT32_MAX / 2)
    return fail(TREE_ERR_SHAPE, "%s: %lld sub-chunks x %d heads exceed the 32-bit work counter", name,
                (long long)mc, H);
  if (!q || !k || !v || !g || !beta || !node_start || !node_end || !node_parent || !outs_ok)
    return fail(TREE_ERR_INVALID_ARG, "%s: null pointer", name);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v))
    return fail(TREE_ERR_ALIGNMENT, "%s: q, k or v not 16-byte aligned", name);
  const size_t need = gdn_ws_layout(T, n_nodes, H, Dk, Dv, bwd, nullptr, nullptr);
  if (workspace_bytes < need)
    return fail(TREE_ERR_WORKSPACE, "%s: workspace of %zu bytes, %zu needed", name, workspace_bytes, need);
  if (!workspace || !aligned256(workspace))
    return fail(TREE_ERR_ALIGNMENT, "%s: workspace null or not 256-byte aligned", name);
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
  a.T = static_cast<int>(T); a.H = H; a.Dk = Dk; a.Dv = Dv; a.ns = gdn_slices(Dv); a.DkP = (Dk + 3) / 4 * 4;
  a.withhold = static_cast<int>(g_withhold.exchange(-1));
  const unsigned long long wns = g_wait_ns.exchange(0);
  a.wait_ns = wns ? wns : sm100::kWaitNs;
  a.err = device_error_word();
  gdn_ws_layout(T, n_nodes, H, Dk, Dv, bwd, workspace, &a.w);
  const int64_t n_flags = mc * H * a.ns;
  const size_t setup_bytes = sizeof(int) * setup_ints(n_nodes, mc);
  const int fits = setup_bytes <= 200 * 1024;
  if (fits) {
    int rc = smem_opt_in(reinterpret_cast<const void*>(gdn_setup_kernel), static_cast<int>(setup_bytes));
    if (rc) return rc;
  }
  gdn_setup_kernel<<<1, kSetupThreads, fits ? setup_bytes : 0, st>>>(
      node_start, node_end, node_parent, static_cast<int>(n_nodes), static_cast<int>(T), n_flags, a.w,
      static_cast<int>(mc), fits, a.err);
  TREE_LAUNCH_CHECK("gdn_setup_kernel");
  *mc_out = mc;
  return TREE_OK;
}

template <typename Tin>
int gdn_forward(GdnArgs& a, int64_t mc, cudaStream_t st) {
  int n_sm = 0, rc;
  if ((rc = sm_count(&n_sm)) || (rc = run_forward_chain<Tin>(a, mc, n_sm, st))) return rc;
  if ((rc = smem_opt_in(reinterpret_cast<const void*>(gdn_out_kernel<Tin>), static_cast<int>(kOutSmem)))) return rc;
  gdn_out_kernel<Tin><<<dim3(static_cast<unsigned>(mc), static_cast<unsigned>(a.H)), kThreads, kOutSmem, st>>>(a);
  TREE_LAUNCH_CHECK("gdn_out_kernel");
  return TREE_OK;
}

template <typename Tin>
int gdn_backward(GdnArgs& a, int64_t mc, cudaStream_t st) {
  int n_sm = 0, rc;
  if ((rc = sm_count(&n_sm)) || (rc = run_forward_chain<Tin>(a, mc, n_sm, st))) return rc;
  if ((rc = smem_opt_in(reinterpret_cast<const void*>(gdn_bchain_kernel<Tin>), static_cast<int>(kBchainSmem))) ||
      (rc = smem_opt_in(reinterpret_cast<const void*>(gdn_grads_kernel<Tin>), static_cast<int>(kGradsSmem))))
    return rc;
  gdn_bchain_kernel<Tin><<<std::min(n_sm, kMaxCtas), kThreads, kBchainSmem, st>>>(a);
  TREE_LAUNCH_CHECK("gdn_bchain_kernel");
  gdn_grads_kernel<Tin><<<dim3(static_cast<unsigned>(mc), static_cast<unsigned>(a.H)), kThreads, kGradsSmem, st>>>(a);
  TREE_LAUNCH_CHECK("gdn_grads_kernel");
  return TREE_OK;
}

}  // namespace
}  // namespace tree

using namespace tree;

extern "C" size_t tree_gdn_workspace_size(int64_t T, int64_t n_nodes, int H, int Dk, int Dv) {
  if (T < 1 || n_nodes < 1 || H < 1 || Dk < 1 || Dv < 1) return 0;
  return gdn_ws_layout(T, n_nodes, H, Dk, Dv, false, nullptr, nullptr);
}

extern "C" size_t tree_gdn_bwd_workspace_size(int64_t T, int64_t n_nodes, int H, int Dk, int Dv) {
  if (T < 1 || n_nodes < 1 || H < 1 || Dk < 1 || Dv < 1) return 0;
  return gdn_ws_layout(T, n_nodes, H, Dk, Dv, true, nullptr, nullptr);
}

extern "C" int tree_gdn_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta, void* o,
                            const int32_t* node_start, const int32_t* node_end, const int32_t* node_parent,
                            int64_t T, int64_t n_nodes, int H, int Dk, int Dv, int dtype, void* workspace,
                            size_t workspace_bytes, tree_stream_t stream) {
  clear_error();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  GdnArgs a{};
  int64_t mc = 0;
  bool empty = false;
  int rc = gdn_begin(a, q, k, v, g, beta, node_start, node_end, node_parent, T, n_nodes, H, Dk, Dv, dtype,
                     workspace, workspace_bytes, false, o != nullptr, "tree_gdn_fwd", st, &mc, &empty);
  if (rc || empty) return rc;
  a.o = o;
  return dtype == TREE_DTYPE_BF16 ? gdn_forward<__nv_bfloat16>(a, mc, st) : gdn_forward<float>(a, mc, st);
}

extern "C" int tree_gdn_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                            const void* dout, void* dq, void* dk, void* dv, float* dg, float* dbeta,
                            const int32_t* node_start, const int32_t* node_end, const int32_t* node_parent,
                            int64_t T, int64_t n_nodes, int H, int Dk, int Dv, int dtype, void* workspace,
                            size_t workspace_bytes, tree_stream_t stream) {
  clear_error();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  GdnArgs a{};
  int64_t mc = 0;
  bool empty = false;
  int rc = gdn_begin(a, q, k, v, g, beta, node_start, node_end, node_parent, T, n_nodes, H, Dk, Dv, dtype,
                     workspace, workspace_bytes, true, dout && dq && dk && dv && dg && dbeta, "tree_gdn_bwd", st,
                     &mc, &empty);
  if (rc || empty) return rc;
  if (!aligned16(dout)) return fail(TREE_ERR_ALIGNMENT, "tree_gdn_bwd: dout not 16-byte aligned");
  a.dout = dout; a.dq = dq; a.dk = dk; a.dv = dv; a.dg = dg; a.dbeta = dbeta;
  return dtype == TREE_DTYPE_BF16 ? gdn_backward<__nv_bfloat16>(a, mc, st) : gdn_backward<float>(a, mc, st);
}

extern "C" int tree_gdn_test_withhold(int64_t sub_chunk, double wait_seconds) {
  clear_error();
  if (sub_chunk < -1 || sub_chunk > INT32_MAX || !(wait_seconds > 0.0) || wait_seconds > 2.0)
    return fail(TREE_ERR_INVALID_ARG, "tree_gdn_test_withhold: sub_chunk %lld, wait %g s", (long long)sub_chunk,
                wait_seconds);
  g_wait_ns.store(static_cast<unsigned long long>(wait_seconds * 1e9));
  g_withhold.store(sub_chunk);
  return TREE_OK;
}
