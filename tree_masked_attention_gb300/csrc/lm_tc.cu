// Shared-logit log-probs on tcgen05 tensor cores (bf16 in, fp32 accumulate).
//
// Trie packing (agillm.io), "Share logits, preserve every prediction": z_r = h_r W_LM
// for every packed row; each original prediction (occurrence) reads the log-softmax of
// its source row at its target; "The training-loop change is small": gathering the
// target log-probs avoids materialising the logits. "Same chain rule, shared
// computation graph", Step 1: G_z = p - e_y per occurrence, summed at shared rows. With
// g_o = dL/dlogp_o and c_r = sum of g_o over row r's occurrences:
//   G_z[r, v] = -c_r softmax(z_r)_v + sum_{o at r, y_o = v} g_o,
//   dH = G_z W^T,   dW = H^T G_z.
//
// One persistent GEMM kernel (output tiles 128 x 256, K blocks of 64, four-stage TMA
// ring, two TMEM accumulators so the epilogue of one tile overlaps the MMAs of the next)
// runs four products:
//   z (forward)   A = H (K-major), B = W (MN-major); epilogue: per-row max and sum of exp
//                 of the tile (online over 32-column chunks) and the target logits of the
//                 row's occurrences that fall in the tile (logits never reach memory);
//   z (backward)  same operands; epilogue writes G_z (bf16) to the workspace;
//   dH            A = G_z (K-major), B = W (K-major: rows of W are the N index);
//   dW            A = H^T (MN-major view of H), B = G_z (MN-major).
// Warps: 0 TMA, 1 MMA (and TMEM owner), 2-5 epilogue (one accumulator row per thread).
#include <algorithm>
#include <cmath>

#include "attn_internal.h"
#include "common.h"
#include "device_common.cuh"
#include "sm100.cuh"
#include "tmap.h"

namespace tree {
using namespace sm100;

namespace lmtc {

constexpr int BM = 128, BN = 256, BK = 64, NST = 4;
constexpr int kThreads = 192;
constexpr uint32_t kABytes = BM * BK * 2;  // 16 KB
constexpr uint32_t kBBytes = BN * BK * 2;  // 32 KB

enum Epi { EPI_LSE = 0, EPI_GZ = 1, EPI_STORE = 2, EPI_DW = 3 };

struct Smem {
  uint8_t a[NST][kABytes];
  uint8_t b[NST][kBBytes];
  uint64_t full[NST], empty[NST], acc_full[2], acc_empty[2];
  uint32_t tmem_base;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

// Tiles walk slabs of this many 128-row M blocks, M fastest within a slab. Measured on the
// 8192 x 4096 x 128256 log-prob step (4 steps per point, about +-1 % between runs): the
// forward at 32 blocks (a 32 MB band of H per pass over W) took 4.81-4.87 ms against
// 5.08 ms with one slab over all 64 blocks; G_z at 32 and dH at 16 gave the backward
// 16.05 ms against 16.1-16.2 (dW at 8 or 32 was no better than 16).
#ifndef LM_RASTER_GROUP_DEFAULT
#define LM_RASTER_GROUP_DEFAULT 32  // z with the online LSE (forward)
#endif
#ifndef LM_RASTER_GROUP_DW
#define LM_RASTER_GROUP_DW 16  // dW = H^T G_z: 16 M blocks (32 MB of H) stay in L2 per pass over G_z
#endif
#ifndef LM_RASTER_GROUP_DH
#define LM_RASTER_GROUP_DH 16  // dH = G_z W^T
#endif
#ifndef LM_RASTER_GROUP_GZ
#define LM_RASTER_GROUP_GZ 32  // z again for G_z
#endif

struct Params {
  int M, N, K;
  int a_mn, b_mn;        // operand majorness (1 = MN-major)
  int raster_group;      // tiles walk slabs of this many M blocks, M fastest within a slab
                         // (0: N fastest over the whole grid)
  int epi;
  // EPI_LSE / EPI_GZ
  const int32_t* row_ptr;
  const int32_t* perm;
  const int32_t* targets;
  int n_occ;
  float* part_max;       // [n_nb, M]
  float* part_sum;
  float* logp;           // EPI_LSE: target logits
  const float* lse;      // EPI_GZ
  const float* crow;
  const float* grad;
  __nv_bfloat16* out;    // EPI_GZ: G_z [M, N]; EPI_STORE / EPI_DW: C [M, N]
  float* out_f32;        // EPI_DW: when set, C [M, N] is written in fp32 here instead of `out`
  float* occ_delta;      // EPI_GZ writes, EPI_DW reads: exact - stored G_z at target cells
  const int32_t* blk_ptr;  // EPI_DW: occurrences grouped by 256-column target block
  const int32_t* blk_ent;  //         {source row, occurrence}
  const __nv_bfloat16* h;  // EPI_DW: hidden [rows, M]
  int* err;
};

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
  uint32_t v;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(v) : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  return v;
}

// Loads the A and B blocks of k-block kb of tile (mb, nb) into stage buffers.
__device__ __forceinline__ void load_stage(const Params& p, const CUtensorMap* ta, const CUtensorMap* tb,
                                           uint8_t* a, uint8_t* b, uint64_t* bar, int mb, int nb, int kb) {
  const int k0 = kb * BK;
  if (!p.a_mn) {
    tma_load_2d(a, ta, bar, k0, mb * BM);                       // box {64 K, 128 M}
  } else {
    tma_load_2d(a, ta, bar, mb * BM, k0);                       // box {64 M, 64 K}, twice
    tma_load_2d(a + kABytes / 2, ta, bar, mb * BM + 64, k0);
  }
  if (!p.b_mn) {
    tma_load_2d(b, tb, bar, k0, nb * BN);                       // box {64 K, 256 N}
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) tma_load_2d(b + q * (kBBytes / 4), tb, bar, nb * BN + 64 * q, k0);
  }
}

__device__ __forceinline__ void tile_coords(const Params& p, int t, int n_mb, int n_nb, int* mb, int* nb) {
  const int g = min(p.raster_group, n_mb);
  if (g <= 0) {
    *mb = t / n_nb;
    *nb = t % n_nb;
    return;
  }
  const int slab = t / (g * n_nb), local = t - slab * g * n_nb;
  const int rows = min(g, n_mb - slab * g);  // the last slab may be shorter
  *mb = slab * g + local % rows;
  *nb = local / rows;
}

// Occurrence range of row m, or an empty range (and the error flag) when the CSR is bad.
__device__ __forceinline__ void row_occ(const Params& p, int m, int* b, int* e) {
  *b = p.row_ptr[m];
  *e = p.row_ptr[m + 1];
  if (*b < 0 || *e < *b || *e > p.n_occ) {
    raise_error(p.err, TREE_ERR_DEVICE_CHECK);
    *b = *e = 0;
  }
}

// Next occurrence (cursor k in [k, e)) of the row whose target lies in [n0, n0 + BN):
// returns the column within the tile, or -1. Sets *o to the occurrence id.
__device__ __forceinline__ int next_in_tile(const Params& p, int* k, int e, int n0, int* o) {
  while (*k < e) {
    const int oo = p.perm[*k];
    if (oo < 0 || oo >= p.n_occ) {
      raise_error(p.err, TREE_ERR_DEVICE_CHECK);
      ++*k;
      continue;
    }
    const int y = p.targets[oo];
    if (y < 0 || y >= p.N) {
      raise_error(p.err, TREE_ERR_DEVICE_CHECK);
      ++*k;
      continue;
    }
    if (y >= n0 && y < n0 + BN) {
      *o = oo;
      return y - n0;
    }
    ++*k;
  }
  return -1;
}

__global__ void __launch_bounds__(kThreads, 1)
lm_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, Params p) {
  extern __shared__ uint8_t smem_raw[];
  if (p.err && (*reinterpret_cast<volatile int*>(p.err) & (1 << TREE_ERR_TIMEOUT))) return;
  Smem& S = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_mb = (p.M + BM - 1) / BM, n_nb = (p.N + BN - 1) / BN, n_kb = (p.K + BK - 1) / BK;
  const int n_tiles = n_mb * n_nb;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.acc_full[s], 1);
      mbar_init(&S.acc_empty[s], 4);
    }
    fence_mbarrier_init();
  }
  if (warp == 1) tmem_alloc(&S.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
        int mb, nb;
        tile_coords(p, t, n_mb, n_nb, &mb, &nb);
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int st = it % NST;
          if (it >= NST && !(ok = mbar_wait(&S.empty[st], ((it / NST) - 1) & 1, p.err))) break;
          mbar_arrive_expect_tx(&S.full[st], kABytes + kBBytes);
          load_stage(p, &tmA, &tmB, S.a[st], S.b[st], &S.full[st], mb, nb, kb);
        }
      }
      // no copy left in flight
      for (int j = (it > NST ? it - NST : 0); j < it; ++j) mbar_wait(&S.full[j % NST], (j / NST) & 1, p.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(BM, BN, p.a_mn, p.b_mn);
      int it = 0, ai = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x, ++ai) {
        const int buf = ai & 1;
        if (ai >= 2 && !(ok = mbar_wait(&S.acc_empty[buf], ((ai >> 1) - 1) & 1, p.err))) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * BN;
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int st = it % NST;
          if (!(ok = mbar_wait(&S.full[st], (it / NST) & 1, p.err))) break;
          tc_fence_after();
          const uint32_t ab = smem_u32(S.a[st]), bb = smem_u32(S.b[st]);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = p.a_mn ? desc_sw128(ab + kk * 2048, kABytes / 2, 1024) : desc_sw128(ab + kk * 32, 16, 1024);
            const uint64_t bd = p.b_mn ? desc_sw128(bb + kk * 2048, kBBytes / 4, 1024) : desc_sw128(bb + kk * 32, 16, 1024);
            mma_ss(d, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&S.empty[st]);
        }
        if (ok) mma_commit(&S.acc_full[buf]);
      }
      // wait for the last MMAs before TMEM is freed
      if (ai > 0) mbar_wait(&S.acc_full[(ai - 1) & 1], ((ai - 1) >> 1) & 1, p.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue warps 2-5
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const uint32_t lanes = static_cast<uint32_t>(q4 * 32) << 16;
    int ai = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++ai) {
      int mb, nb;
      tile_coords(p, t, n_mb, n_nb, &mb, &nb);
      const int buf = ai & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&S.acc_full[buf], (ai >> 1) & 1, p.err))) break;
      tc_fence_after();
      const uint32_t acc = tmem + lanes + buf * BN;
      const int m = mb * BM + r, n0 = nb * BN;
      const bool row_ok = m < p.M;
      const int ncols = min(BN, p.N - n0);
      if (p.epi == EPI_STORE || p.epi == EPI_DW) {
        if (p.epi == EPI_DW) {
          // dW only: add back, in fp32, what storing G_z in bf16 dropped at target cells:
          // dW[m, y] += H[r, m] * (exact - stored) for every occurrence cell (r, y) of this
          // vocabulary block, straight into the accumulator column, in the block's entry order
          const int lb = p.blk_ptr[nb], le = p.blk_ptr[nb + 1];
          for (int q = lb; q < le; ++q) {  // warp-uniform
            const int oo = p.blk_ent[2 * q + 1];
            const int col = p.targets[oo] - n0;
            const float dlt = p.occ_delta[oo];
            if (dlt == 0.f || col < 0 || col >= BN) continue;
            const float x =
                row_ok ? dlt * __bfloat162float(p.h[static_cast<int64_t>(p.blk_ent[2 * q]) * p.M + m]) : 0.f;
            const uint32_t cur = tmem_ld1(acc + col);
            tmem_st1(acc + col, __float_as_uint(__uint_as_float(cur) + x));
            tmem_st_wait();  // a later entry may hit the same column
          }
        }
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32], pk[16];
          tmem_ld32(acc + c * 32, v);
          tmem_ld_wait();
          if (p.out_f32) {  // fp32 dW: the accumulator as it is
            if (row_ok && c * 32 < ncols) {
              float* dst = p.out_f32 + static_cast<int64_t>(m) * p.N + n0 + c * 32;
              if (c * 32 + 32 <= ncols && (p.N % 4) == 0) {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                  reinterpret_cast<float4*>(dst)[u] =
                      make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                                  __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3]));
              } else {
                for (int u = 0; u < 32 && c * 32 + u < ncols; ++u) dst[u] = __uint_as_float(v[u]);
              }
            }
            continue;
          }
#pragma unroll
          for (int u = 0; u < 16; ++u) pk[u] = pack_bf16(__uint_as_float(v[2 * u]), __uint_as_float(v[2 * u + 1]));
          if (row_ok && c * 32 < ncols) {
            __nv_bfloat16* dst = p.out + static_cast<int64_t>(m) * p.N + n0 + c * 32;
            if (c * 32 + 32 <= ncols && (p.N % 8) == 0) {
#pragma unroll
              for (int u = 0; u < 4; ++u)
                reinterpret_cast<uint4*>(dst)[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
            } else {
              for (int u = 0; u < 32 && c * 32 + u < ncols; ++u)
                dst[u] = __float2bfloat16_rn(__uint_as_float(v[u]));
            }
          }
        }
      } else if (p.epi == EPI_LSE) {
        float mx = -INFINITY, sm = 0.f;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(acc + c * 32, v);
          tmem_ld_wait();
          const int valid = min(32, ncols - c * 32);  // same for the whole warp
          if (valid <= 0) continue;
          float cm = -INFINITY;
#pragma unroll
          for (int u = 0; u < 32; ++u)
            if (u < valid) cm = fmaxf(cm, __uint_as_float(v[u]));
          const float nm = fmaxf(mx, cm);
          float cs = 0.f;
#pragma unroll
          for (int u = 0; u < 32; ++u)
            if (u < valid) cs += exp2f((__uint_as_float(v[u]) - nm) * 1.4426950408889634f);
          sm = sm * exp2f((mx - nm) * 1.4426950408889634f) + cs;
          mx = nm;
        }
        if (row_ok) {
          p.part_max[static_cast<int64_t>(nb) * p.M + m] = mx;
          p.part_sum[static_cast<int64_t>(nb) * p.M + m] = sm;
        }
        // target logits of this row's occurrences in this tile (one TMEM column per round)
        int k = 0, e = 0, o = -1;
        if (row_ok) row_occ(p, m, &k, &e);
        int col = row_ok ? next_in_tile(p, &k, e, n0, &o) : -1;
        while (true) {
          const unsigned want = __ballot_sync(0xffffffffu, col >= 0);
          if (!want) break;
          const int c = __shfl_sync(0xffffffffu, col, __ffs(want) - 1);
          const float z = __uint_as_float(tmem_ld1(acc + c));
          if (col == c) {
            p.logp[o] = z;
            ++k;
            col = next_in_tile(p, &k, e, n0, &o);
          }
        }
      } else {  // EPI_GZ
        const float l = row_ok ? p.lse[m] : 0.f, cr = row_ok ? p.crow[m] : 0.f;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32], pk[16];
          tmem_ld32(acc + c * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const float g0 = -cr * exp2f((__uint_as_float(v[2 * u]) - l) * 1.4426950408889634f);
            const float g1 = -cr * exp2f((__uint_as_float(v[2 * u + 1]) - l) * 1.4426950408889634f);
            pk[u] = pack_bf16(g0, g1);
          }
          if (row_ok && c * 32 < ncols) {
            __nv_bfloat16* dst = p.out + static_cast<int64_t>(m) * p.N + n0 + c * 32;
            if (c * 32 + 32 <= ncols && (p.N % 8) == 0) {
#pragma unroll
              for (int u = 0; u < 4; ++u)
                reinterpret_cast<uint4*>(dst)[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
            } else {
              for (int u = 0; u < 32 && c * 32 + u < ncols; ++u) {
                const __nv_bfloat162 h2 = *reinterpret_cast<const __nv_bfloat162*>(&pk[u / 2]);
                dst[u] = (u & 1) ? h2.y : h2.x;
              }
            }
          }
        }
        // target entries: -c p_y + sum of g over the row's occurrences with target y
        int k = 0, e = 0, o = -1;
        if (row_ok) row_occ(p, m, &k, &e);
        const int kb0 = k;
        int col = row_ok ? next_in_tile(p, &k, e, n0, &o) : -1;
        while (true) {
          const unsigned want = __ballot_sync(0xffffffffu, col >= 0);
          if (!want) break;
          const int c = __shfl_sync(0xffffffffu, col, __ffs(want) - 1);
          const float z = __uint_as_float(tmem_ld1(acc + c));
          if (col == c) {
            float gsum = 0.f;
            bool first = true;  // the cell's first occurrence (in CSR order) carries its residual
            for (int kk = kb0; kk < e; ++kk) {
              const int oo = p.perm[kk];
              if (oo >= 0 && oo < p.n_occ && p.targets[oo] == n0 + c) {
                gsum += p.grad[oo];
                if (kk < k) first = false;
              }
            }
            const float val = -cr * exp2f((z - l) * 1.4426950408889634f) + gsum;
            const __nv_bfloat16 stored = __float2bfloat16_rn(val);
            p.out[static_cast<int64_t>(m) * p.N + n0 + c] = stored;
            if (first) p.occ_delta[o] = val - __bfloat162float(stored);
            // skip the row's further occurrences of the same target (already summed)
            do {
              ++k;
              col = next_in_tile(p, &k, e, n0, &o);
            } while (col == c);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.acc_empty[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Occurrences grouped by the 256-column vocabulary block of their target, for the dW
// epilogue's correction: a stable counting sort in one CTA. Block b's entries are
// blk_ent[2 e .. 2 e + 1] = {source row, occurrence} for e in [blk_ptr[b], blk_ptr[b + 1]),
// in increasing CSR position k (the order the dW epilogue adds them in, so the sums are
// reproducible). Counts with shared atomics, an exclusive scan, then, chunk by chunk, one
// warp hands out positions in k order (lanes with the same block take consecutive slots).
// Occurrences with an out-of-range id or target are left out (the GEMM epilogues flag them).
// Also zeroes occ_delta.
constexpr int kGroupThreads = 1024;

__global__ void __launch_bounds__(kGroupThreads) lm_group_occ_kernel(
    const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ perm, const int32_t* __restrict__ targets, int T,
    int n_occ, int V, int n_blk, int chunk, int32_t* __restrict__ blk_ptr, int32_t* __restrict__ blk_ent,
    float* __restrict__ occ_delta) {
  extern __shared__ int gsm[];
  int* cur = gsm;            // [n_blk] counts, then the next free slot of each block
  int* sb = cur + n_blk;     // [chunk] block of each occurrence of the chunk (-1: none)
  int* so = sb + chunk;      // [chunk] occurrence id
  int* sr = so + chunk;      // [chunk] source row
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  auto block_of = [&](int k, int* o_out) {
    const int o = perm[k];
    int b = -1;
    if (o >= 0 && o < n_occ) {
      const int y = targets[o];
      if (y >= 0 && y < V) b = y / BN;
    }
    *o_out = o;
    return b;
  };
  for (int i = tid; i < n_occ; i += kGroupThreads) occ_delta[i] = 0.f;
  for (int b = tid; b < n_blk; b += kGroupThreads) cur[b] = 0;
  __syncthreads();
  for (int k = tid; k < n_occ; k += kGroupThreads) {
    int o;
    const int b = block_of(k, &o);
    if (b >= 0) atomicAdd(&cur[b], 1);
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the counts
    int run = 0;
    for (int b0 = 0; b0 < n_blk; b0 += 32) {
      const int b = b0 + lane;
      const int x = b < n_blk ? cur[b] : 0;
      int incl = x;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
      }
      if (b < n_blk) {
        cur[b] = run + incl - x;
        blk_ptr[b] = run + incl - x;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) blk_ptr[n_blk] = run;
  }
  __syncthreads();
  for (int c0 = 0; c0 < n_occ; c0 += chunk) {
    const int len = min(chunk, n_occ - c0);
    for (int i = tid; i < len; i += kGroupThreads) {
      int o;
      sb[i] = block_of(c0 + i, &o);
      so[i] = o;
      sr[i] = 0;
    }
    __syncthreads();
    for (int r = tid; r < T; r += kGroupThreads) {  // the row holding each position of the chunk
      const int lo = max(row_ptr[r], c0), hi = min(row_ptr[r + 1], c0 + len);
      for (int k = lo; k < hi; ++k) sr[k - c0] = r;
    }
    __syncthreads();
    if (warp == 0) {
      for (int i0 = 0; i0 < len; i0 += 32) {
        const int i = i0 + lane;
        const int b = i < len ? sb[i] : -1;
        const unsigned mask = __match_any_sync(0xffffffffu, b >= 0 ? b : -1 - lane);
        const int leader = __ffs(mask) - 1;
        int base = 0;
        if (b >= 0 && lane == leader) {
          base = cur[b];
          cur[b] = base + __popc(mask);
        }
        base = __shfl_sync(0xffffffffu, base, leader);
        if (b >= 0) {
          const int pos = base + __popc(mask & ((1u << lane) - 1u));
          blk_ent[2 * pos] = sr[i];
          blk_ent[2 * pos + 1] = so[i];
        }
      }
    }
    __syncthreads();
  }
}

}  // namespace lmtc

bool logprob_tc_supported(int dtype) { return dtype == TREE_DTYPE_BF16; }

static int map2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                 uint32_t box_rows) {
  const uint64_t dims[2] = {inner, rows};
  const uint64_t strides[1] = {inner * 2};
  const uint32_t box[2] = {box_inner, box_rows};
  return make_tmap(m, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dims, strides, box, true);
}

static int n_sms(int* n) {
  static int cached[128] = {0};
  int dev = 0;
  TREE_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 128) return fail(TREE_ERR_CUDA, "device ordinal %d out of range", dev);
  if (!cached[dev]) TREE_CUDA_TRY(cudaDeviceGetAttribute(&cached[dev], cudaDevAttrMultiProcessorCount, dev));
  *n = cached[dev];
  return TREE_OK;
}

static int launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const lmtc::Params& p, cudaStream_t st,
                       const char* name) {
  using namespace lmtc;
  if (int rc_ = smem_opt_in(reinterpret_cast<const void*>(lm_gemm_kernel), static_cast<int>(kSmemBytes))) return rc_;
  int sms = 0;
  int rc = n_sms(&sms);
  if (rc) return rc;
  const int64_t tiles = static_cast<int64_t>((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN);
  const int grid = static_cast<int>(std::min<int64_t>(sms, tiles));
  lm_gemm_kernel<<<grid, kThreads, kSmemBytes, st>>>(ta, tb, p);
  TREE_LAUNCH_CHECK(name);
  return TREE_OK;
}

int logprob_fwd_tc(const LogprobArgs& a, cudaStream_t st) {
  using namespace lmtc;
  CUtensorMap ta, tb;
  int rc;
  if ((rc = map2d(&ta, a.h, a.K, a.T, 64, BM)) || (rc = map2d(&tb, a.w, a.V, a.K, 64, 64))) return rc;
  Params p{};
  p.M = static_cast<int>(a.T);
  p.N = static_cast<int>(a.V);
  p.K = static_cast<int>(a.K);
  p.a_mn = 0;
  p.b_mn = 1;
  p.raster_group = LM_RASTER_GROUP_DEFAULT;
  p.epi = EPI_LSE;
  p.row_ptr = a.row_ptr;
  p.perm = a.perm;
  p.targets = a.targets;
  p.n_occ = static_cast<int>(a.n_occ);
  p.part_max = a.ws.part_max;
  p.part_sum = a.ws.part_sum;
  p.logp = a.logp;
  p.err = device_error_word();
  if ((rc = launch_gemm(ta, tb, p, st, "lm_gemm_kernel<lse>"))) return rc;
  const int n_nb = static_cast<int>((a.V + BN - 1) / BN);
  return lse_combine_launch(a.ws.part_max, a.ws.part_sum, n_nb, a.T, a.row_ptr, a.perm, a.n_occ, a.lse, a.logp, st);
}

int logprob_bwd_tc(const LogprobArgs& a, cudaStream_t st) {
  using namespace lmtc;
  int rc = row_grad_sum_launch(a.row_ptr, a.perm, a.grad, a.T, a.n_occ, a.ws.crow, st);
  if (rc) return rc;
  const int n_blk = static_cast<int>((a.V + BN - 1) / BN);
  {
    // the counting sort's shared memory: block counters, then three arrays per chunk
    const int budget = 200 * 1024 / 4;
    if (n_blk > budget / 2)
      return fail(TREE_ERR_SHAPE, "tree_logprob_bwd: V = %lld has too many 256-column blocks", (long long)a.V);
    const int chunk = std::min(8192, (budget - n_blk) / 3);
    const size_t smem = sizeof(int) * (static_cast<size_t>(n_blk) + 3 * static_cast<size_t>(chunk));
    if ((rc = smem_opt_in(reinterpret_cast<const void*>(lm_group_occ_kernel), static_cast<int>(smem)))) return rc;
    lm_group_occ_kernel<<<1, kGroupThreads, smem, st>>>(a.row_ptr, a.perm, a.targets, static_cast<int>(a.T),
                                                        static_cast<int>(a.n_occ), static_cast<int>(a.V), n_blk, chunk,
                                                        a.ws.blk_ptr, a.ws.blk_ent, a.ws.occ_delta);
    TREE_LAUNCH_CHECK("lm_group_occ_kernel");
  }
  __nv_bfloat16* gz = static_cast<__nv_bfloat16*>(a.ws.gz);
  // 1) G_z = recomputed softmax terms and target terms, bf16 [T, V]
  {
    CUtensorMap ta, tb;
    if ((rc = map2d(&ta, a.h, a.K, a.T, 64, BM)) || (rc = map2d(&tb, a.w, a.V, a.K, 64, 64))) return rc;
    Params p{};
    p.M = static_cast<int>(a.T);
    p.N = static_cast<int>(a.V);
    p.K = static_cast<int>(a.K);
    p.a_mn = 0;
    p.b_mn = 1;
    p.raster_group = LM_RASTER_GROUP_GZ;
    p.epi = EPI_GZ;
    p.row_ptr = a.row_ptr;
    p.perm = a.perm;
    p.targets = a.targets;
    p.n_occ = static_cast<int>(a.n_occ);
    p.lse = a.lse;
    p.crow = a.ws.crow;
    p.grad = a.grad;
    p.out = gz;
    p.occ_delta = a.ws.occ_delta;
    p.err = device_error_word();
    if ((rc = launch_gemm(ta, tb, p, st, "lm_gemm_kernel<gz>"))) return rc;
  }
  // 2) dH [T, K_h] = G_z W^T: A = G_z (K-major over V), B = W rows (K-major over V)
  {
    CUtensorMap ta, tb;
    if ((rc = map2d(&ta, gz, a.V, a.T, 64, BM)) || (rc = map2d(&tb, a.w, a.V, a.K, 64, BN))) return rc;
    Params p{};
    p.M = static_cast<int>(a.T);
    p.N = static_cast<int>(a.K);
    p.K = static_cast<int>(a.V);
    p.a_mn = 0;
    p.b_mn = 0;
    p.raster_group = LM_RASTER_GROUP_DH;
    p.epi = EPI_STORE;
    p.out = static_cast<__nv_bfloat16*>(a.dh);
    p.err = device_error_word();
    if ((rc = launch_gemm(ta, tb, p, st, "lm_gemm_kernel<dh>"))) return rc;
  }
  // 3) dW [K_h, V] = H^T G_z: A = H viewed MN-major, B = G_z MN-major
  {
    CUtensorMap ta, tb;
    if ((rc = map2d(&ta, a.h, a.K, a.T, 64, 64)) || (rc = map2d(&tb, gz, a.V, a.T, 64, 64))) return rc;
    Params p{};
    p.M = static_cast<int>(a.K);
    p.N = static_cast<int>(a.V);
    p.K = static_cast<int>(a.T);
    p.a_mn = 1;
    p.b_mn = 1;
    p.raster_group = LM_RASTER_GROUP_DW;
    p.epi = EPI_DW;
    if (a.dw_fp32) p.out_f32 = static_cast<float*>(a.dw);
    else p.out = static_cast<__nv_bfloat16*>(a.dw);
    p.targets = a.targets;
    p.occ_delta = a.ws.occ_delta;
    p.blk_ptr = a.ws.blk_ptr;
    p.blk_ent = a.ws.blk_ent;
    p.h = static_cast<const __nv_bfloat16*>(a.h);
    p.err = device_error_word();
    if ((rc = launch_gemm(ta, tb, p, st, "lm_gemm_kernel<dw>"))) return rc;
  }
  return TREE_OK;
}

}  // namespace tree
