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
// and u; the saved form takes them from the forward's workspace), then
//   bprep  per (sub-chunk, head), in parallel: the chain-independent products
//          du0 = P^T dO and c0 = Q^T (E o dO);
//   bchain per (sub-chunk, head, slice) by decreasing chain depth: the end-state gradient
//          dh_end is the sum, in a fixed order, of the successors' start-state gradients;
//          du = w o (K dh_end) + du0, dr = X^T du, dv = beta o dr,
//          dh0 = E_{L-1} dh_end + c0 - K^T (beta E o dr), published;
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
template <int NT = kThreads>
__device__ __forceinline__ void cp_block(float* s, int sstride, const float* g, int rows, int cols) {
  const int per = cols / 4, n = rows * per;
  for (int p = threadIdx.x; p < n; p += NT) cp16(s + (p / per) * sstride + (p % per) * 4, g + 4 * static_cast<int64_t>(p));
}

struct GdnWs {
  int4* chunks;     // [mc] {first row, rows, predecessor sub-chunk or -1, chain depth}
  int* node_last;   // [n_nodes] last sub-chunk of each node
  int* order;       // [mc] sub-chunks by increasing chain depth
  int* depth_count; // [mc + 1]
  int* succ_ptr;    // [mc + 1] successors (sub-chunks whose predecessor is c), CSR
  int* succ;        // [mc]
  int* ctl;         // [8] n_chunks, forward counter, backward counter, abort, stamp (below)
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
  float* du0;       // [mc, H, slices, 64, 32] P^T dO
  float* c0;        // [mc, H, slices, Dk, 32] Q^T (E o dO)
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
  x.ctl = static_cast<int*>(take(sizeof(int) * 8));
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
    x.du0 = static_cast<float*>(take(sizeof(float) * mc * H * ns * kChunk * kSlice));
    x.c0 = static_cast<float*>(take(sizeof(float) * mc * H * ns * Dk * kSlice));
  }
  if (w) *w = x;
  return round_up(off, 256);
}

// ------------------------------------------------------------------------------ setup
// Sub-chunk table from the node arrays (one thread walks the nodes in preorder, checking
// that they tile [0, T) with earlier parents), the schedule (sub-chunks by increasing
// chain depth: a counting sort, stable in preorder) and the successor lists; all threads
// clear the flags. On a malformed table nothing is scheduled (n_chunks = 0). ctl[4] holds
// the stamp of the inputs whose forward results (factors, corrections, end states) the
// workspace holds: written by the calls that compute them (kStampWrite), checked and then
// cleared by a backward that takes them from the workspace (kStampUse), which schedules
// nothing on a mismatch. The walk's
// working arrays (copies of the node arrays, each node's last sub-chunk, each sub-chunk's
// depth and predecessor, the sort's counters) live in shared memory when they fit
// (`fits`), else in the workspace.
constexpr int kSetupThreads = 1024;
constexpr int kStampWrite = 0, kStampUse = 1;

__host__ __device__ constexpr int64_t setup_ints(int64_t n_nodes, int64_t max_chunks) {
  return 4 * n_nodes + 4 * max_chunks + 2;  // node arrays, nlast; depth, pred, two counters of mc + 1
}

__global__ void __launch_bounds__(kSetupThreads) gdn_setup_kernel(const int32_t* __restrict__ node_start,
                                                                  const int32_t* __restrict__ node_end,
                                                                  const int32_t* __restrict__ node_parent,
                                                                  int n_nodes, int T, int64_t n_flags, GdnWs w,
                                                                  int max_chunks, int fits, int stamp,
                                                                  int stamp_mode, int* err) {
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
  if (stamp_mode == kStampUse) {
    ok = w.ctl[4] == stamp;  // the forward of exactly these inputs ran on this workspace
    w.ctl[4] = 0;            // and its results serve one backward
  } else {
    w.ctl[4] = stamp;
  }
  for (int n = 0; ok && n < n_nodes; ++n) {
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
template <typename Tin, int NT = kThreads>
__device__ __forceinline__ void load_tile(float* dst, int stride, const Tin* __restrict__ src, int r0, int L, int H,
                                          int h, int D, int col0, int ncols) {
  constexpr int kVec = 16 / sizeof(Tin);                       // 8 bf16 or 4 fp32
  constexpr int kPer = (kChunk * kMaxD / kVec + NT - 1) / NT;   // most vectors a thread loads
  const int nv = ncols / kVec, total = kChunk * nv;
  if (D % kVec == 0 && ncols % kVec == 0) {
    uint4 buf[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int idx = threadIdx.x + u * NT;
      const int t = idx / max(nv, 1), cv = col0 + (idx % max(nv, 1)) * kVec;
      buf[u] = make_uint4(0u, 0u, 0u, 0u);
      if (idx < total && t < L && cv < D)
        buf[u] = __ldg(reinterpret_cast<const uint4*>(src + (static_cast<int64_t>(r0 + t) * H + h) * D + cv));
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int idx = threadIdx.x + u * NT;
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
    for (int idx = threadIdx.x; idx < kChunk * ncols; idx += NT) {
      const int t = idx / ncols, cl = idx % ncols, cv = col0 + cl;
      dst[t * stride + cl] = (t < L && cv < D) ? ldf(src, (static_cast<int64_t>(r0 + t) * H + h) * D + cv) : 0.f;
    }
  }
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
  const int lane = tid % 32, warp = tid / 32;
  {
    // A and P: each thread a 4 x 4 block of pairs, rows t0 + 16a, columns s0 + 16b (the
    // eight lanes of a quarter-warp read eight consecutive K rows: no bank conflicts)
    const int s0 = lane & 15, t0 = (lane >> 4) + 2 * warp;
    float qk[4][4], kk[4][4];
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 4; ++y) qk[x][y] = kk[x][y] = 0.f;
    for (int i = 0; i < Dk4; i += 4) {
      float4 qv[4], kt[4], ks[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        qv[x] = *reinterpret_cast<const float4*>(QV + (t0 + 16 * x) * kRow + i);
        kt[x] = *reinterpret_cast<const float4*>(Ks + (t0 + 16 * x) * kRow + i);
        ks[x] = *reinterpret_cast<const float4*>(Ks + (s0 + 16 * x) * kRow + i);
      }
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          qk[x][y] = fmaf(qv[x].x, ks[y].x, fmaf(qv[x].y, ks[y].y, fmaf(qv[x].z, ks[y].z, fmaf(qv[x].w, ks[y].w, qk[x][y]))));
          kk[x][y] = fmaf(kt[x].x, ks[y].x, fmaf(kt[x].y, ks[y].y, fmaf(kt[x].z, ks[y].z, fmaf(kt[x].w, ks[y].w, kk[x][y]))));
        }
    }
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const int t = t0 + 16 * x, ss = s0 + 16 * y;
        float av = 0.f, pv = 0.f;
        if (t < L && ss <= t) {
          const float f = expf(lg[t] - lg[ss]);
          pv = f * qk[x][y];
          if (ss < t) av = bs[t] * f * kk[x][y];
        }
        Am[t * kSq + ss] = av;
        Pg[t * kChunk + ss] = pv;
      }
  }
  __syncthreads();
  // V over Q (Q is done); X by forward substitution, one column per thread
  load_tile(QV, kRow, static_cast<const Tin*>(a.v), r0, L, H, h, Dv, 0, Dv4);
  // X = (I + A)^-1 in 16 x 16 blocks (A strictly lower-triangular, so X is unit lower-
  // triangular): first the four diagonal blocks, each column by forward substitution
  // (64 threads), then the blocks below the diagonal by their distance d = k - l:
  //   X_kl = -X_kk sum_{l <= m < k} A_km X_ml,
  // all blocks of one distance at once, every thread a few elements of the sums.
  for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) Xm[(idx / kChunk) * kSq + idx % kChunk] = 0.f;
  __syncthreads();
  if (tid < kChunk) {
    const int cc = tid, b0 = cc & ~15;  // column cc of the diagonal block starting at b0
    Xm[cc * kSq + cc] = 1.f;
    for (int t = cc + 1; t < b0 + 16; ++t) {
      float acc = 0.f;
      for (int q = cc; q < t; ++q) acc = fmaf(Am[t * kSq + q], Xm[q * kSq + cc], acc);
      Xm[t * kSq + cc] = -acc;
    }
  }
  __syncthreads();
  float* Ym = Am;  // A's blocks on and above the diagonal are not read: Y blocks go there
  for (int d = 1; d < 4; ++d) {
    const int nb = 4 - d;  // blocks (k, l) = (l + d, l), l < nb
    // Y_kl = sum_{l <= m < k} A_km X_ml  -> stored in A's upper block (l, k)
    for (int e = tid; e < nb * 256; e += kThreads) {
      const int l = e / 256, k = l + d, r = (e % 256) / 16, cl = e % 16;
      float acc = 0.f;
      for (int m = l; m < k; ++m)
        for (int q = 0; q < 16; ++q) acc = fmaf(Am[(16 * k + r) * kSq + 16 * m + q], Xm[(16 * m + q) * kSq + 16 * l + cl], acc);
      Ym[(16 * l + r) * kSq + 16 * k + cl] = acc;
    }
    __syncthreads();
    // X_kl = -X_kk Y_kl
    for (int e = tid; e < nb * 256; e += kThreads) {
      const int l = e / 256, k = l + d, r = (e % 256) / 16, cl = e % 16;
      float acc = 0.f;
      for (int q = 0; q <= r; ++q)
        acc = fmaf(Xm[(16 * k + r) * kSq + 16 * k + q], Ym[(16 * l + q) * kSq + 16 * k + cl], acc);
      Xm[(16 * k + r) * kSq + 16 * l + cl] = -acc;
    }
    __syncthreads();
  }
  // beta E o K and beta o V in place (K is not needed otherwise any more)
  for (int idx = tid; idx < kChunk * Dk4; idx += kThreads) {
    const int t = idx / Dk4, i = idx % Dk4;
    Ks[t * kRow + i] *= bs[t] * E[t];
  }
  for (int idx = tid; idx < kChunk * Dv4; idx += kThreads) {
    const int t = idx / Dv4, j = idx % Dv4;
    QV[t * kRow + j] *= bs[t];
  }
  __syncthreads();
  for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) Xg[idx] = Xm[(idx / kChunk) * kSq + idx % kChunk];
  // W = X (beta E o K), U0 = X (beta o V): four consecutive columns and rows warp + 8 m per
  // thread; X is lower-triangular (identity rows past L)
  {
    const int c4 = lane * 4;
    float4 wacc[8], uacc[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) wacc[m] = uacc[m] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q = 0; q < L; ++q) {
      const float4 k4 = *reinterpret_cast<const float4*>(Ks + q * kRow + c4);
      const float4 v4 = *reinterpret_cast<const float4*>(QV + q * kRow + c4);
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const float x = Xm[(warp + 8 * m) * kSq + q];
        wacc[m].x = fmaf(x, k4.x, wacc[m].x); wacc[m].y = fmaf(x, k4.y, wacc[m].y);
        wacc[m].z = fmaf(x, k4.z, wacc[m].z); wacc[m].w = fmaf(x, k4.w, wacc[m].w);
        uacc[m].x = fmaf(x, v4.x, uacc[m].x); uacc[m].y = fmaf(x, v4.y, uacc[m].y);
        uacc[m].z = fmaf(x, v4.z, uacc[m].z); uacc[m].w = fmaf(x, v4.w, uacc[m].w);
      }
    }
    float* Wg = a.w.W + (static_cast<int64_t>(c) * H + h) * kChunk * DkP;
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int t = warp + 8 * m;
      if (c4 < DkP) *reinterpret_cast<float4*>(Wg + t * DkP + c4) = c4 < Dk4 ? wacc[m] : z4;
      if (c4 < ns * kSlice)
        *reinterpret_cast<float4*>(slice_block(a.w.U0, c, h, c4 / kSlice, H, ns, kChunk) + t * kSlice + c4 % kSlice) =
            c4 < Dv4 ? uacc[m] : z4;
    }
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
__global__ void __launch_bounds__(kThreads, 2) gdn_chain_kernel(const GdnArgs a) {
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
      for (int idx = Dk * kSlice + tid; idx < kMaxD * kSlice; idx += kThreads)  // rows past Dk
        Hs[(idx / kSlice) * kSl + idx % kSlice] = 0.f;
    } else {
      for (int idx = tid; idx < kMaxD * kSlice; idx += kThreads) Hs[(idx / kSlice) * kSl + idx % kSlice] = 0.f;
    }
    cp_wait();
    decay_factors(a.g, a.beta, r0, L, H, h, lg, E, wv, bs);  // ends with a barrier
    // u = U0 - W h0: each thread rows t and t + 32 (t = lane / 8 + 4 warp) by four
    // consecutive columns j0 = 4 (lane % 8): two float4 of W and four of h0 per four steps
    // of i feed 32 FMAs. W rows past L are zero.
    float* ug = slice_block(w.u, c, h, sl, H, ns, kChunk);
    const int cg = (lane & 7) * 4;
    {
      const int t = (lane >> 3) + 4 * warp;
      float4 acc0 = *reinterpret_cast<const float4*>(Us + t * kSl + cg);
      float4 acc1 = *reinterpret_cast<const float4*>(Us + (t + 32) * kSl + cg);
      for (int i = 0; i < Dk4; i += 4) {
        const float4 w0 = *reinterpret_cast<const float4*>(Ws + t * kRow + i);
        const float4 w1 = *reinterpret_cast<const float4*>(Ws + (t + 32) * kRow + i);
        const float wa[4] = {w0.x, w0.y, w0.z, w0.w}, wb[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float4 h4 = *reinterpret_cast<const float4*>(Hs + (i + e) * kSl + cg);
          acc0.x = fmaf(-wa[e], h4.x, acc0.x); acc0.y = fmaf(-wa[e], h4.y, acc0.y);
          acc0.z = fmaf(-wa[e], h4.z, acc0.z); acc0.w = fmaf(-wa[e], h4.w, acc0.w);
          acc1.x = fmaf(-wb[e], h4.x, acc1.x); acc1.y = fmaf(-wb[e], h4.y, acc1.y);
          acc1.z = fmaf(-wb[e], h4.z, acc1.z); acc1.w = fmaf(-wb[e], h4.w, acc1.w);
        }
      }
      __syncthreads();  // every thread has read U0
      *reinterpret_cast<float4*>(Us + t * kSl + cg) = acc0;
      *reinterpret_cast<float4*>(Us + (t + 32) * kSl + cg) = acc1;
      *reinterpret_cast<float4*>(ug + t * kSlice + cg) = acc0;
      *reinterpret_cast<float4*>(ug + (t + 32) * kSlice + cg) = acc1;
    }
    __syncthreads();
    // h_end = E_{L-1} h0 + sum_t w_t k_t u_t^T: each thread rows 4 rq .. 4 rq + 3
    // (rq = lane / 8 + 4 warp) by columns j0 .. j0 + 3: one float4 of K and one of u per t
    // feed 16 FMAs
    {
      float* hend = slice_block(w.states, c, h, sl, H, ns, Dk);
      const float gl = E[L - 1];
      const int i0 = 4 * ((lane >> 3) + 4 * warp);
      float4 acc[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float4 h4 = *reinterpret_cast<const float4*>(Hs + (i0 + m) * kSl + cg);
        acc[m] = make_float4(gl * h4.x, gl * h4.y, gl * h4.z, gl * h4.w);
      }
      for (int t = 0; t < L; ++t) {
        const float wt = wv[t];
        const float4 u4 = *reinterpret_cast<const float4*>(Us + t * kSl + cg);
        const float4 k4 = *reinterpret_cast<const float4*>(Ks + t * kRow + i0);
        const float ka[4] = {k4.x * wt, k4.y * wt, k4.z * wt, k4.w * wt};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          acc[m].x = fmaf(ka[m], u4.x, acc[m].x); acc[m].y = fmaf(ka[m], u4.y, acc[m].y);
          acc[m].z = fmaf(ka[m], u4.z, acc[m].z); acc[m].w = fmaf(ka[m], u4.w, acc[m].w);
        }
      }
#pragma unroll
      for (int m = 0; m < 4; ++m)
        if (i0 + m < Dk) __stcg(reinterpret_cast<float4*>(hend + (i0 + m) * kSlice + cg), acc[m]);
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
  // four consecutive columns and rows warp + 8 m per thread
  const int lane = tid % 32, warp = tid / 32, c4 = lane * 4;
  if (c4 >= Dv) return;
  Tin* o = static_cast<Tin*>(a.o);
  float4 acc[8];
#pragma unroll
  for (int m = 0; m < 8; ++m) acc[m] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (pred >= 0) {
    for (int i = 0; i < Dk; ++i) {
      const float4 h4 = *reinterpret_cast<const float4*>(Hs + i * kRow + c4);
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const float q = Qs[(warp + 8 * m) * kRow + i];
        acc[m].x = fmaf(q, h4.x, acc[m].x); acc[m].y = fmaf(q, h4.y, acc[m].y);
        acc[m].z = fmaf(q, h4.z, acc[m].z); acc[m].w = fmaf(q, h4.w, acc[m].w);
      }
    }
  }
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const float e = E[warp + 8 * m];
    acc[m].x *= e; acc[m].y *= e; acc[m].z *= e; acc[m].w *= e;
  }
  for (int q = 0; q < L; ++q) {  // P is lower-triangular
    const float4 u4 = *reinterpret_cast<const float4*>(Us + q * kRow + c4);
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const float pv = Ps[(warp + 8 * m) * kSq + q];
      acc[m].x = fmaf(pv, u4.x, acc[m].x); acc[m].y = fmaf(pv, u4.y, acc[m].y);
      acc[m].z = fmaf(pv, u4.z, acc[m].z); acc[m].w = fmaf(pv, u4.w, acc[m].w);
    }
  }
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int t = warp + 8 * m;
    if (t < L) {
      const float v4[4] = {acc[m].x, acc[m].y, acc[m].z, acc[m].w};
      Tin* dst = o + (static_cast<int64_t>(r0 + t) * H + h) * Dv + c4;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (c4 + e < Dv) dst[e] = from_f32<Tin>(v4[e]);
    }
  }
}

// ------------------------------------------------------------------------------ bprep
// Per (sub-chunk, head), in parallel: the two products of the state-gradient chain that do
// not depend on it, du0 = P^T dO ([64, Dv]) and c0 = Q^T (E o dO) ([Dk, Dv]), into the
// [mc, H, slices, rows, 32] layout the chain reads. Each thread owns four consecutive
// columns c4 of rows warp + 8 m.
constexpr size_t kBprepSmem = (kChunk * kSq + 2 * kChunk * kRow + 4 * kChunk) * sizeof(float);

template <typename Tin>
__global__ void __launch_bounds__(kThreads, 2) gdn_bprep_kernel(const GdnArgs a) {
  extern __shared__ __align__(16) float sm[];
  float* Ps = sm;                 // [64][kSq]
  float* Qs = Ps + kChunk * kSq;  // [64][kRow]
  float* Os = Qs + kChunk * kRow; // [64][kRow] dO, then E o dO
  float* lg = Os + kChunk * kRow;
  float* E = lg + kChunk;
  float* wv = E + kChunk;
  float* bs = wv + kChunk;
  const int c = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const GdnWs& w = a.w;
  if (c >= w.ctl[0]) return;
  if (*reinterpret_cast<volatile int*>(&w.ctl[3])) return;  // a chain gave up: outputs unspecified
  const int4 ck = w.chunks[c];
  const int r0 = ck.x, L = ck.y, H = a.H, Dk = a.Dk, Dv = a.Dv, ns = a.ns;
  const int Dk4 = (Dk + 3) & ~3, nc = ns * kSlice;  // dO columns past Dv up to the slices' end are zero
  cp_block(Ps, kSq, w.Pm + (static_cast<int64_t>(c) * H + h) * kChunk * kChunk, kChunk, kChunk);
  load_tile(Qs, kRow, static_cast<const Tin*>(a.q), r0, L, H, h, Dk, 0, Dk4);
  load_tile(Os, kRow, static_cast<const Tin*>(a.dout), r0, L, H, h, Dv, 0, nc);
  cp_wait();
  decay_factors(a.g, a.beta, r0, L, H, h, lg, E, wv, bs);  // ends with a barrier
  const int c4 = lane * 4;
  const bool col_ok = c4 < nc;
  {  // du0 = P^T dO (P lower-triangular, zero past L): rows warp + 8 m, m < 8
    float4 acc[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) acc[m] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int t2 = 0; t2 < L; ++t2) {
      const float4 o4 = *reinterpret_cast<const float4*>(Os + t2 * kRow + c4);
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const float pv = Ps[t2 * kSq + warp + 8 * m];
        acc[m].x = fmaf(pv, o4.x, acc[m].x); acc[m].y = fmaf(pv, o4.y, acc[m].y);
        acc[m].z = fmaf(pv, o4.z, acc[m].z); acc[m].w = fmaf(pv, o4.w, acc[m].w);
      }
    }
    if (col_ok) {
      float* dst = slice_block(w.du0, c, h, c4 / kSlice, H, ns, kChunk) + c4 % kSlice;
#pragma unroll
      for (int m = 0; m < 8; ++m) *reinterpret_cast<float4*>(dst + (warp + 8 * m) * kSlice) = acc[m];
    }
  }
  __syncthreads();
  for (int idx = tid; idx < L * (nc / 4); idx += kThreads) {  // E o dO
    const int t = idx / (nc / 4), j = (idx % (nc / 4)) * 4;
    float4* o = reinterpret_cast<float4*>(Os + t * kRow + j);
    const float e = E[t];
    float4 x = *o;
    x.x *= e; x.y *= e; x.z *= e; x.w *= e;
    *o = x;
  }
  __syncthreads();
  {  // c0 = Q^T (E o dO): rows i = warp + 8 m, m < 16
    float4 acc[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) acc[m] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int t = 0; t < L; ++t) {
      const float4 o4 = *reinterpret_cast<const float4*>(Os + t * kRow + c4);
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float qv = Qs[t * kRow + warp + 8 * m];
        acc[m].x = fmaf(qv, o4.x, acc[m].x); acc[m].y = fmaf(qv, o4.y, acc[m].y);
        acc[m].z = fmaf(qv, o4.z, acc[m].z); acc[m].w = fmaf(qv, o4.w, acc[m].w);
      }
    }
    if (col_ok) {
      float* dst = slice_block(w.c0, c, h, c4 / kSlice, H, ns, Dk) + c4 % kSlice;
#pragma unroll
      for (int m = 0; m < 16; ++m)
        if (warp + 8 * m < Dk) *reinterpret_cast<float4*>(dst + (warp + 8 * m) * kSlice) = acc[m];
    }
  }
}

// ------------------------------------------------------------------------------ bchain
// Per (sub-chunk, head, slice), by decreasing chain depth: dh_end (the sum of the
// successors' start-state gradients), du, dr, dv, dh0; per-row partial sums for dg, dbeta.
// The chain-independent du0 and c0 come from gdn_bprep_kernel, staged in the Os and Qs
// buffers.
constexpr int kBThreads = 512;                  // 16 warps: latency of one chain item is the critical path
constexpr int kBRows = kChunk / (kBThreads / 32);  // rows of du / dr per warp (4); dh0 rows per warp 2 kBRows
static_assert(kBRows == 4 && 2 * kBRows * (kBThreads / 32) == kMaxD, "bchain row mapping");
constexpr size_t kBchainSmem =
    (2 * kChunk * kRow + 2 * kChunk * kSq + 2 * kMaxD * kSl + 4 * kChunk * kSl + 4 * kChunk) * sizeof(float);

template <typename Tin>
__global__ void __launch_bounds__(kBThreads, 1) gdn_bchain_kernel(const GdnArgs a) {
  extern __shared__ __align__(16) float sm[];
  float* Ks = sm;                        // [64][kRow]
  float* Qs = Ks + kChunk * kRow;        // [128][kSl] c0 slice (the region of a [64][kRow] tile)
  float* Ps = Qs + kChunk * kRow;        // [64][kSq] (unused)
  float* Xs = Ps + kChunk * kSq;         // [64][kSq]
  float* Ds = Xs + kChunk * kSq;         // [128][kSl] dh_end slice
  float* Hs = Ds + kMaxD * kSl;          // [128][kSl] h0 slice
  float* Os = Hs + kMaxD * kSl;          // [64][kSl] du0 slice
  float* Us = Os + kChunk * kSl;         // [64][kSl] u slice
  float* Vs = Us + kChunk * kSl;         // [64][kSl] v slice
  float* Rs = Vs + kChunk * kSl;         // [64][kSl] du, then dr
  float* lg = Rs + kChunk * kSl;
  float* E = lg + kChunk;
  float* wv = E + kChunk;
  float* bs = wv + kChunk;
  __shared__ int s_item, s_ok;
  __shared__ float s_red[kBThreads / 32];
  const GdnWs& w = a.w;
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int H = a.H, Dk = a.Dk, Dv = a.Dv, ns = a.ns, T = a.T;
  const int Dk4 = (Dk + 3) & ~3;
  const int n_chunks = w.ctl[0];
  const int items = n_chunks * H * ns;
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
    cp_block<kBThreads>(Xs, kSq, w.Xm + mo, kChunk, kChunk);
    cp_block<kBThreads>(Os, kSl, slice_block(w.du0, c, h, sl, H, ns, kChunk), kChunk, kSlice);
    cp_block<kBThreads>(Qs, kSl, slice_block(w.c0, c, h, sl, H, ns, Dk), Dk, kSlice);
    cp_block<kBThreads>(Us, kSl, slice_block(w.u, c, h, sl, H, ns, kChunk), kChunk, kSlice);
    if (pred >= 0) cp_block<kBThreads>(Hs, kSl, slice_block(w.states, pred, h, sl, H, ns, Dk), Dk, kSlice);
    load_tile<Tin, kBThreads>(Ks, kRow, static_cast<const Tin*>(a.k), r0, L, H, h, Dk, 0, Dk4);
    load_tile<Tin, kBThreads>(Vs, kSl, static_cast<const Tin*>(a.v), r0, L, H, h, Dv, sl * kSlice, kSlice);
    if (pred < 0)
      for (int idx = tid; idx < Dk * kSlice; idx += kBThreads) Hs[(idx / kSlice) * kSl + idx % kSlice] = 0.f;
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
      constexpr int kPer = kMaxD * kSlice / 4 / kBThreads;  // float4 per thread
      float4 acc[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s = sb; s < se; ++s) {
        const float4* src = reinterpret_cast<const float4*>(slice_block(w.dstart, w.succ[s], h, sl, H, ns, Dk));
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int p = tid + u * kBThreads;
          if (p < Dk * kSlice / 4) {
            const float4 x = __ldcg(src + p);
            acc[u].x += x.x; acc[u].y += x.y; acc[u].z += x.z; acc[u].w += x.w;
          }
        }
      }
      float4* dend = reinterpret_cast<float4*>(slice_block(w.dend, c, h, sl, H, ns, Dk));
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int p = tid + u * kBThreads;
        if (p < Dk * kSlice / 4) {
          __stcg(dend + p, acc[u]);
          *reinterpret_cast<float4*>(Ds + (p / (kSlice / 4)) * kSl + (p % (kSlice / 4)) * 4) = acc[u];
        }
      }
      for (int idx = Dk * kSlice + tid; idx < kMaxD * kSlice; idx += kBThreads)  // rows past Dk
        Ds[(idx / kSlice) * kSl + idx % kSlice] = 0.f;
    }
    cp_wait();
    __syncthreads();
    float he = 0.f;  // partial sum of dh_end . h0
    for (int idx = tid; idx < Dk * kSlice; idx += kBThreads) {
      const int i = idx / kSlice, jj = idx % kSlice;
      he = fmaf(Ds[i * kSl + jj], Hs[i * kSl + jj], he);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) he += __shfl_xor_sync(0xffffffffu, he, o);
    if (lane == 0) s_red[warp] = he;
    decay_factors(a.g, a.beta, r0, L, H, h, lg, E, wv, bs);  // ends with a barrier
    if (tid == 0) {
      float x = 0.f;
      for (int u = 0; u < kBThreads / 32; ++u) x += s_red[u];
      w.part_he[(static_cast<int64_t>(sl) * n_chunks + c) * H + h] = x;
    }
    // du = w o (K dh_end) + du0 for rows t = 4 warp + m of column `lane` (K and du0 rows
    // past L are zero, so every row is computed); partial dw_t = w_t sum_j (K dh_end)_tj u_tj
    {
      float kd[kBRows];
#pragma unroll
      for (int m = 0; m < kBRows; ++m) kd[m] = 0.f;
      for (int i = 0; i < Dk4; i += 4) {
        const float d0 = Ds[i * kSl + lane], d1 = Ds[(i + 1) * kSl + lane], d2 = Ds[(i + 2) * kSl + lane],
                    d3 = Ds[(i + 3) * kSl + lane];
#pragma unroll
        for (int m = 0; m < kBRows; ++m) {
          const float4 k4 = *reinterpret_cast<const float4*>(Ks + (kBRows * warp + m) * kRow + i);
          kd[m] = fmaf(k4.x, d0, fmaf(k4.y, d1, fmaf(k4.z, d2, fmaf(k4.w, d3, kd[m]))));
        }
      }
      float du[kBRows];
#pragma unroll
      for (int m = 0; m < kBRows; ++m)
        du[m] = fmaf(wv[kBRows * warp + m], kd[m], Os[(kBRows * warp + m) * kSl + lane]);
#pragma unroll
      for (int m = 0; m < kBRows; ++m) {
        const int t = kBRows * warp + m;
        Rs[t * kSl + lane] = du[m];
        if (t < L) {
          float dw = wv[t] * kd[m] * Us[t * kSl + lane];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) dw += __shfl_xor_sync(0xffffffffu, dw, o);
          if (lane == 0) w.part[((static_cast<int64_t>(sl) * 2 + 0) * T + r0 + t) * H + h] = dw;
        }
      }
    }
    __syncthreads();
    // dr = X^T du (X lower-triangular), dv = beta o dr
    float drr[kBRows];
#pragma unroll
    for (int m = 0; m < kBRows; ++m) drr[m] = 0.f;
    for (int t2 = 0; t2 < L; ++t2) {
      const float rr = Rs[t2 * kSl + lane];
      const float4 x0 = *reinterpret_cast<const float4*>(Xs + t2 * kSq + kBRows * warp);
      drr[0] = fmaf(x0.x, rr, drr[0]); drr[1] = fmaf(x0.y, rr, drr[1]); drr[2] = fmaf(x0.z, rr, drr[2]);
      drr[3] = fmaf(x0.w, rr, drr[3]);
    }
    __syncthreads();
    float* drg = slice_block(w.dr, c, h, sl, H, ns, kChunk);
#pragma unroll
    for (int m = 0; m < kBRows; ++m) {
      const int t = kBRows * warp + m;
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
    // dh0 = E_{L-1} dh_end + c0 - K^T (beta E o dr): rows i = 8 warp + m (c0 rows past Dk
    // are never read: those rows are not stored)
    {
      float* dst = slice_block(w.dstart, c, h, sl, H, ns, Dk);
      const float gl = E[L - 1];
      const int i0 = 2 * kBRows * warp;
      float acc[2 * kBRows];
#pragma unroll
      for (int m = 0; m < 2 * kBRows; ++m)
        acc[m] = i0 + m < Dk ? fmaf(gl, Ds[(i0 + m) * kSl + lane], Qs[(i0 + m) * kSl + lane]) : 0.f;
      for (int t = 0; t < L; ++t) {
        const float br = -bs[t] * E[t] * Rs[t * kSl + lane];
        const float4* kr = reinterpret_cast<const float4*>(Ks + t * kRow + i0);
#pragma unroll
        for (int q = 0; q < 2 * kBRows / 4; ++q) {
          const float4 k4 = kr[q];
          acc[4 * q] = fmaf(k4.x, br, acc[4 * q]);
          acc[4 * q + 1] = fmaf(k4.y, br, acc[4 * q + 1]);
          acc[4 * q + 2] = fmaf(k4.z, br, acc[4 * q + 2]);
          acc[4 * q + 3] = fmaf(k4.w, br, acc[4 * q + 3]);
        }
      }
#pragma unroll
      for (int m = 0; m < 2 * kBRows; ++m)
        if (i0 + m < Dk) __stcg(dst + (i0 + m) * kSlice + lane, acc[m]);
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
                  2 * kBprepSmem <= 227 * 1024 && kMaxD * kSl <= kChunk * kRow &&
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
  // pairs (t, s): each thread a 4 x 4 block, rows t0 + 16 x, columns s0 + 16 y (the eight
  // lanes of a quarter-warp read eight consecutive rows of the column operand)
  {
    const int s0 = lane & 15, t0 = (lane >> 4) + 2 * warp;
    float qk[4][4], kk[4][4], dp[4][4], da[4][4];
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 4; ++y) qk[x][y] = kk[x][y] = dp[x][y] = da[x][y] = 0.f;
    for (int i = 0; i < Dk4; i += 4) {
      float4 qv[4], kt[4], ks[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        qv[x] = *reinterpret_cast<const float4*>(Qs + (t0 + 16 * x) * kRow + i);
        kt[x] = *reinterpret_cast<const float4*>(Ks + (t0 + 16 * x) * kRow + i);
        ks[x] = *reinterpret_cast<const float4*>(Ks + (s0 + 16 * x) * kRow + i);
      }
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          qk[x][y] = fmaf(qv[x].x, ks[y].x, fmaf(qv[x].y, ks[y].y, fmaf(qv[x].z, ks[y].z, fmaf(qv[x].w, ks[y].w, qk[x][y]))));
          kk[x][y] = fmaf(kt[x].x, ks[y].x, fmaf(kt[x].y, ks[y].y, fmaf(kt[x].z, ks[y].z, fmaf(kt[x].w, ks[y].w, kk[x][y]))));
        }
    }
    for (int j = 0; j < Dv4; j += 4) {
      float4 ov[4], rv[4], us[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        ov[x] = *reinterpret_cast<const float4*>(Os + (t0 + 16 * x) * kRow + j);
        rv[x] = *reinterpret_cast<const float4*>(Rs + (t0 + 16 * x) * kRow + j);
        us[x] = *reinterpret_cast<const float4*>(Us + (s0 + 16 * x) * kRow + j);
      }
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          dp[x][y] = fmaf(ov[x].x, us[y].x, fmaf(ov[x].y, us[y].y, fmaf(ov[x].z, us[y].z, fmaf(ov[x].w, us[y].w, dp[x][y]))));
          da[x][y] = fmaf(rv[x].x, us[y].x, fmaf(rv[x].y, us[y].y, fmaf(rv[x].z, us[y].z, fmaf(rv[x].w, us[y].w, da[x][y]))));
        }
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int t = t0 + 16 * x;
      float rowsum = 0.f, rowb = 0.f;
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const int ss = s0 + 16 * y;
        float fp = 0.f, fa = 0.f, m1 = 0.f;
        if (t < L && ss <= t) {
          const float f = expf(lg[t] - lg[ss]);
          fp = dp[x][y] * f;
          m1 = fp * qk[x][y];                      // dP o P
          if (ss < t) {
            const float dav = -da[x][y];
            fa = dav * bs[t] * f;
            m1 = fmaf(fa, kk[x][y], m1);           // dA o A
            rowb = fmaf(dav * f, kk[x][y], rowb);  // dA o f o KK (dbeta)
          }
        }
        Fp[t * kSq + ss] = fp;
        Fa[t * kSq + ss] = fa;
        M1[t * kSq + ss] = m1;
        rowsum += m1;
      }
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) {  // over the 16 lanes that share row t
        rowsum += __shfl_xor_sync(0xffffffffu, rowsum, o);
        rowb += __shfl_xor_sync(0xffffffffu, rowb, o);
      }
      if (s0 == 0) {
        dlg[t] = rowsum;
        dbt[t] = rowb;
      }
    }
  }
  __syncthreads();
  if (tid < kChunk) {  // column sums of M1, in row order
    float x = 0.f;
    for (int t = 0; t < kChunk; ++t) x += M1[t * kSq + tid];
    dlg[tid] -= x;
  }
  // dQ, dK: four consecutive columns c4 and rows warp + 8 m per thread, in two passes of
  // four rows; h0 and dh_end are staged 16 state columns at a time, transposed ([j][i])
  const int c4 = lane * 4;
  constexpr int kHt = kMaxD + 4;        // row stride of the transposed staging
  static_assert(2 * 16 * kHt <= kChunk * kSq, "h0 / dh_end staging must fit in the M1 buffer");
  float* hst = M1;                      // [16][kHt] h0 columns j0..j0+15, transposed
  float* dst = M1 + 16 * kHt;           // [16][kHt] the same columns of dh_end
  Tin* dq = static_cast<Tin*>(a.dq);
  Tin* dk = static_cast<Tin*>(a.dk);
  for (int pass = 0; pass < 2; ++pass) {
    float4 qa[4], ka[4], z1[4], z2[4], z3[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) qa[m] = ka[m] = z1[m] = z2[m] = z3[m] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int tb = warp + 32 * pass;    // rows tb + 8 m, m < 4
    for (int q = 0; q < kChunk; ++q) {
      const float4 k4 = *reinterpret_cast<const float4*>(Ks + q * kRow + c4);
      const float4 q4 = *reinterpret_cast<const float4*>(Qs + q * kRow + c4);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int t = tb + 8 * m;
        const float a1 = Fp[t * kSq + q], a2 = Fp[q * kSq + t], a3 = Fa[t * kSq + q] + Fa[q * kSq + t];
        qa[m].x = fmaf(a1, k4.x, qa[m].x); qa[m].y = fmaf(a1, k4.y, qa[m].y);         // (dP o f) K
        qa[m].z = fmaf(a1, k4.z, qa[m].z); qa[m].w = fmaf(a1, k4.w, qa[m].w);
        ka[m].x = fmaf(a2, q4.x, fmaf(a3, k4.x, ka[m].x));                              // (dP o f)^T Q
        ka[m].y = fmaf(a2, q4.y, fmaf(a3, k4.y, ka[m].y));                              // + (dA o b f) K
        ka[m].z = fmaf(a2, q4.z, fmaf(a3, k4.z, ka[m].z));                              //   and transpose
        ka[m].w = fmaf(a2, q4.w, fmaf(a3, k4.w, ka[m].w));
      }
    }
    for (int j0 = 0; j0 < ns * kSlice; j0 += 16) {
      const int sl = j0 / kSlice, off = j0 % kSlice;
      __syncthreads();
      const float* hg = pred >= 0 ? slice_block(w.states, pred, h, sl, H, ns, Dk) : nullptr;
      const float* dg = slice_block(w.dend, c, h, sl, H, ns, Dk);
      for (int idx = tid; idx < kMaxD * 16; idx += kThreads) {
        const int ii = idx / 16, jj = idx % 16;
        if (ii < Dk) {
          if (hg) cp4(hst + jj * kHt + ii, hg + ii * kSlice + off + jj);
          else hst[jj * kHt + ii] = 0.f;
          cp4(dst + jj * kHt + ii, dg + ii * kSlice + off + jj);
        } else {
          hst[jj * kHt + ii] = 0.f;
          dst[jj * kHt + ii] = 0.f;
        }
      }
      cp_wait();
      __syncthreads();
      const int jn = min(16, Dv - j0);
      for (int jj = 0; jj < jn; ++jj) {
        const float4 h4 = *reinterpret_cast<const float4*>(hst + jj * kHt + c4);
        const float4 d4 = *reinterpret_cast<const float4*>(dst + jj * kHt + c4);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int t = tb + 8 * m;
          const float o = Os[t * kRow + j0 + jj], rr = Rs[t * kRow + j0 + jj], u = Us[t * kRow + j0 + jj];
          z1[m].x = fmaf(o, h4.x, z1[m].x); z1[m].y = fmaf(o, h4.y, z1[m].y);       // (dO h0^T)_ti
          z1[m].z = fmaf(o, h4.z, z1[m].z); z1[m].w = fmaf(o, h4.w, z1[m].w);
          z2[m].x = fmaf(rr, h4.x, z2[m].x); z2[m].y = fmaf(rr, h4.y, z2[m].y);     // (dr h0^T)_ti
          z2[m].z = fmaf(rr, h4.z, z2[m].z); z2[m].w = fmaf(rr, h4.w, z2[m].w);
          z3[m].x = fmaf(u, d4.x, z3[m].x); z3[m].y = fmaf(u, d4.y, z3[m].y);       // (u dh_end^T)_ti
          z3[m].z = fmaf(u, d4.z, z3[m].z); z3[m].w = fmaf(u, d4.w, z3[m].w);
        }
      }
    }
    // rows tb + 8 m: dq, dk, and the d lg / dbeta terms E_t q_t . (dO h0^T)_t,
    // -beta_t E_t k_t . (dr h0^T)_t and -E_t k_t . (dr h0^T)_t (a row lives in one warp)
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int t = tb + 8 * m;
      const float4 qv = *reinterpret_cast<const float4*>(Qs + t * kRow + c4);
      const float4 kv = *reinterpret_cast<const float4*>(Ks + t * kRow + c4);
      float cq = 0.f, ck2 = 0.f;
      if (c4 < Dk4) {  // columns past Dk hold zeros in Q and K; columns past Dk4 hold no data
        cq = qv.x * z1[m].x + qv.y * z1[m].y + qv.z * z1[m].z + qv.w * z1[m].w;
        ck2 = kv.x * z2[m].x + kv.y * z2[m].y + kv.z * z2[m].z + kv.w * z2[m].w;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        cq += __shfl_xor_sync(0xffffffffu, cq, o);
        ck2 += __shfl_xor_sync(0xffffffffu, ck2, o);
      }
      if (lane == 0) {
        dlg[t] += E[t] * cq - bs[t] * E[t] * ck2;
        dbt[t] -= E[t] * ck2;
      }
      if (t < L) {
        const float e = E[t], wt = wv[t], be = bs[t] * E[t];
        const float qo[4] = {qa[m].x + e * z1[m].x, qa[m].y + e * z1[m].y, qa[m].z + e * z1[m].z,
                             qa[m].w + e * z1[m].w};
        const float ko[4] = {ka[m].x + wt * z3[m].x - be * z2[m].x, ka[m].y + wt * z3[m].y - be * z2[m].y,
                             ka[m].z + wt * z3[m].z - be * z2[m].z, ka[m].w + wt * z3[m].w - be * z2[m].w};
        const int64_t base = (static_cast<int64_t>(r0 + t) * H + h) * Dk + c4;
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2)
          if (c4 + e2 < Dk) {
            dq[base + e2] = from_f32<Tin>(qo[e2]);
            dk[base + e2] = from_f32<Tin>(ko[e2]);
          }
      }
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
              bool bwd, bool saved, bool outs_ok, const char* name, cudaStream_t st, int64_t* mc_out, bool* empty) {
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
  // stamp of the inputs: FNV-1a over the shapes, the dtype and the input addresses (never 0)
  uint32_t stamp = 2166136261u;
  auto mix = [&](uint64_t x) {
    for (int b = 0; b < 8; ++b) stamp = (stamp ^ static_cast<uint32_t>((x >> (8 * b)) & 0xffu)) * 16777619u;
  };
  for (const void* ptr : {q, k, v, static_cast<const void*>(g), static_cast<const void*>(beta),
                          static_cast<const void*>(node_start), static_cast<const void*>(node_end),
                          static_cast<const void*>(node_parent)})
    mix(reinterpret_cast<uintptr_t>(ptr));
  for (int64_t x : {T, n_nodes, static_cast<int64_t>(H), static_cast<int64_t>(Dk), static_cast<int64_t>(Dv),
                    static_cast<int64_t>(dtype)})
    mix(static_cast<uint64_t>(x));
  stamp |= 1u;
  gdn_setup_kernel<<<1, kSetupThreads, fits ? setup_bytes : 0, st>>>(
      node_start, node_end, node_parent, static_cast<int>(n_nodes), static_cast<int>(T), n_flags, a.w,
      static_cast<int>(mc), fits, static_cast<int>(stamp), saved ? kStampUse : kStampWrite, a.err);
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

// saved: the forward's factors, corrections and end states are in the workspace already
// (checked by the set-up kernel's stamp); otherwise they are recomputed first.
template <typename Tin>
int gdn_backward(GdnArgs& a, int64_t mc, bool saved, cudaStream_t st) {
  int n_sm = 0, rc;
  if ((rc = sm_count(&n_sm))) return rc;
  if (!saved && (rc = run_forward_chain<Tin>(a, mc, n_sm, st))) return rc;
  if ((rc = smem_opt_in(reinterpret_cast<const void*>(gdn_bprep_kernel<Tin>), static_cast<int>(kBprepSmem))))
    return rc;
  gdn_bprep_kernel<Tin><<<dim3(static_cast<unsigned>(mc), static_cast<unsigned>(a.H)), kThreads, kBprepSmem, st>>>(a);
  TREE_LAUNCH_CHECK("gdn_bprep_kernel");
  if ((rc = smem_opt_in(reinterpret_cast<const void*>(gdn_bchain_kernel<Tin>), static_cast<int>(kBchainSmem))) ||
      (rc = smem_opt_in(reinterpret_cast<const void*>(gdn_grads_kernel<Tin>), static_cast<int>(kGradsSmem))))
    return rc;
  gdn_bchain_kernel<Tin><<<std::min(n_sm, kMaxCtas), kBThreads, kBchainSmem, st>>>(a);
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
                     workspace, workspace_bytes, false, false, o != nullptr, "tree_gdn_fwd", st, &mc, &empty);
  if (rc || empty) return rc;
  a.o = o;
  return dtype == TREE_DTYPE_BF16 ? gdn_forward<__nv_bfloat16>(a, mc, st) : gdn_forward<float>(a, mc, st);
}

static int gdn_bwd_call(const char* name, bool saved, const void* q, const void* k, const void* v, const float* g,
                        const float* beta, const void* dout, void* dq, void* dk, void* dv, float* dg, float* dbeta,
                        const int32_t* node_start, const int32_t* node_end, const int32_t* node_parent, int64_t T,
                        int64_t n_nodes, int H, int Dk, int Dv, int dtype, void* workspace, size_t workspace_bytes,
                        tree_stream_t stream) {
  clear_error();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  GdnArgs a{};
  int64_t mc = 0;
  bool empty = false;
  // the alignment of dout is checked before anything is enqueued (a saved call's set-up
  // consumes the stamp)
  if (dout && !aligned16(dout)) return fail(TREE_ERR_ALIGNMENT, "%s: dout not 16-byte aligned", name);
  int rc = gdn_begin(a, q, k, v, g, beta, node_start, node_end, node_parent, T, n_nodes, H, Dk, Dv, dtype,
                     workspace, workspace_bytes, true, saved, dout && dq && dk && dv && dg && dbeta, name, st,
                     &mc, &empty);
  if (rc || empty) return rc;
  a.dout = dout; a.dq = dq; a.dk = dk; a.dv = dv; a.dg = dg; a.dbeta = dbeta;
  return dtype == TREE_DTYPE_BF16 ? gdn_backward<__nv_bfloat16>(a, mc, saved, st)
                                  : gdn_backward<float>(a, mc, saved, st);
}

extern "C" int tree_gdn_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                            const void* dout, void* dq, void* dk, void* dv, float* dg, float* dbeta,
                            const int32_t* node_start, const int32_t* node_end, const int32_t* node_parent,
                            int64_t T, int64_t n_nodes, int H, int Dk, int Dv, int dtype, void* workspace,
                            size_t workspace_bytes, tree_stream_t stream) {
  return gdn_bwd_call("tree_gdn_bwd", false, q, k, v, g, beta, dout, dq, dk, dv, dg, dbeta, node_start, node_end,
                      node_parent, T, n_nodes, H, Dk, Dv, dtype, workspace, workspace_bytes, stream);
}

extern "C" int tree_gdn_bwd_saved(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                  const void* dout, void* dq, void* dk, void* dv, float* dg, float* dbeta,
                                  const int32_t* node_start, const int32_t* node_end, const int32_t* node_parent,
                                  int64_t T, int64_t n_nodes, int H, int Dk, int Dv, int dtype, void* workspace,
                                  size_t workspace_bytes, tree_stream_t stream) {
  return gdn_bwd_call("tree_gdn_bwd_saved", true, q, k, v, g, beta, dout, dq, dk, dv, dg, dbeta, node_start,
                      node_end, node_parent, T, n_nodes, H, Dk, Dv, dtype, workspace, workspace_bytes, stream);
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
