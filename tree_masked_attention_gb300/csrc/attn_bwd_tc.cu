// Tree attention backward on tcgen05 tensor cores (bf16 in, fp32 accumulate, d = 128).
//
// Trie packing, "Same chain rule, shared computation graph", Step 3: a key collects
// the gradients of every descendant query that sees it. With key j visible to query
// i iff j <= i <= subtree_end[j], the queries of a 128-key tile are exactly the
// contiguous rows [first key, max subtree_end of the tile] (every row in between lies
// in some key's subtree), so the CTA of one key tile and one KV head walks that range
// in 64-row query tiles, for every query head of the GQA group, and keeps dK and dV
// in TMEM for the whole walk.
//
// Per step (key tile K/V resident; query tile Q_i, dO_i, LSE_i, Delta_i from a TMA ring):
//   S^T  = K Q_i^T          (M=128 keys, N=64 queries)      -> TMEM
//   dP^T = V dO_i^T         (M=128, N=64)                   -> TMEM
//   P^T  = exp2(S^T scale log2e - LSE_i log2e) on visible pairs, 0 elsewhere
//   dS^T = P^T (dP^T - Delta_i)                              (compute warps, one key row each)
//   dV  += P^T dO_i         (A = P^T bf16 from TMEM, B = dO_i MN-major)
//   dK  += dS^T Q_i         (A = dS^T bf16 from TMEM, B = Q_i MN-major)
//   dQ_i^T = K^T dS^T       (M=128 dims, N=64 queries; A = K MN-major, B = dS^T MN-major)
//   dQ_i += scale dQ_i^T    (fp32 reductions into the workspace accumulator, coalesced
//                            along the head dimension; a final kernel converts to bf16)
// Both compute warpgroups work on the same step, warpgroup w on queries 32w..32w+31 of
// the tile, so a step's softmax backward takes half as long. TMEM (512 columns): two
// slots used by alternate steps (S^T, then P^T and dS^T as bf16 pairs), one dP^T slot,
// one dQ^T slot (64 each), dV and dK (128 each). While the warps work on step g, the
// tensor core already computes S^T and dP^T of step g+1 into the free slots, and dQ^T
// of step g-1 drains through a warpgroup of its own into the fp32 accumulator.
//   warps 0-7    compute (0-3 and 4-7: query halves); at the end of a unit 0-3 add dK, 4-7 dV
//   warp 8       TMA producer, and issues dK
//   warp 9       issues dP^T (owns TMEM)
//   warp 10      issues dV, then S^T two steps ahead into the slot that dV and dK have read
//   warp 11      issues dQ^T
//   warps 12-15  dQ^T drain, staging and TMA reduce
// A tcgen05.mma issue occupies its thread for about as long as an N<=128 MMA runs, so the
// four issuing threads share a step's 32 MMAs. The operands that stay in TMEM (P^T and
// dS^T) spare shared-memory bandwidth, which the MMAs' operand reads otherwise saturate.
#include <algorithm>
#include <cmath>

#include "attn_internal.h"
#include "attn_mask.cuh"
#include "common.h"
#include "device_common.cuh"
#include "sm100.cuh"
#include "tmap.h"

namespace tree {
using namespace sm100;

namespace tcbwd {

constexpr int BN = 128, BQ = 64, D = 128, NST = 3;
constexpr int kThreads = 512;
constexpr int kWarpProducer = 8, kWarpMma = 9, kWarpMma2 = 10, kWarpMma3 = 11, kWarpDq = 12;
constexpr uint32_t kKSub = 128 * 128;          // 128 key rows x 128 B
constexpr uint32_t kKTile = 2 * kKSub;         // K or V: 128 x 128 bf16
constexpr uint32_t kQSub = BQ * 128;           // 64 query rows x 128 B
constexpr uint32_t kQTile = 2 * kQSub;         // Q_i or dO_i: 64 x 128 bf16
constexpr uint32_t kDsTile = BN * 128;         // dS^T: 128 key rows x 64 bf16

struct Smem {
  uint8_t k[kKTile];
  uint8_t v[kKTile];
  uint8_t q[NST][kQTile];
  uint8_t dout[NST][kQTile];
  uint8_t ds[2][kDsTile];
  // scale * dQ of half a query tile, row-major [32 queries][128 dims], for the TMA reduce;
  // the two halves alternate so that one is written while the other is being read
  float dq_stage[2][(BQ / 2) * D];
  float lse2[NST][BQ];
  float delta[NST][BQ];
  uint64_t stage_read, kv_full, qdo_full[NST], qdo_empty[NST], s_full[2], dp_full, ld_done, ds_ready[2], dk_done[2],
      dq_full[2], drain_done, mma_done, fin[4];
  uint32_t tmem_base;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
// dK and dV staging at the end of a unit, 64 KB each, over q, dout and ds (contiguous)
constexpr uint32_t kEpiBytes = BN * D * 4;
static_assert(offsetof(Smem, dout) == offsetof(Smem, q) + sizeof(Smem::q) &&
                  offsetof(Smem, ds) == offsetof(Smem, dout) + sizeof(Smem::dout) &&
                  sizeof(Smem::q) + sizeof(Smem::dout) + sizeof(Smem::ds) >= 2 * kEpiBytes &&
                  offsetof(Smem, q) % 1024 == 0,
              "dK / dV staging needs q, dout and ds contiguous and 1024-byte aligned");
static_assert(kSmemBytes + 64 <= 232448, "backward shared memory exceeds the 227 KB per-block limit");

struct Params {
  int T, T_pad, Hq, Hkv;  // T: key rows; T_pad: query rows rounded up to 64
  int Tq, q_off;          // query rows, key rows before the first query
  float scale_log2, scale;
  const int32_t* kmax;
  const int32_t* endp;
  const float* lse2;    // [Hq, T_pad] LSE * log2(e), +inf past T
  const float* delta;   // [Hq, T_pad] dO . O, 0 past T
  float* dq_acc;        // [T, Hq, d] fp32, zeroed by the preprocess kernel
  float* dk_acc;        // [T, Hkv, d] fp32 (scaled), zeroed by the preprocess kernel
  float* dv_acc;        // [T, Hkv, d] fp32, zeroed by the preprocess kernel
  const int4* units;    // work units {key tile, KV head, first step, end step}
  const int* n_units;
  int* counter;         // next unit to hand out
  int* err;
};


__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void red_add(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

__device__ __forceinline__ void red_add4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// Query tiles of 64 rows seen by key tile kt: [qt_lo, qt_lo + nq). The queries that can
// see the tile are the key rows [max(first key, q_off), max subtree_end]; query tile t
// holds key rows q_off + 64 t ...
__device__ __forceinline__ int query_tiles_of(int kt, int kmax, int T, int q_off, int* qt_lo) {
  const int first = max(kt * BN, q_off);
  const int last_row = min(kmax, T - 1);
  *qt_lo = (first - q_off) / BQ;
  return last_row >= first ? (last_row - q_off) / BQ - *qt_lo + 1 : 0;
}
__device__ __forceinline__ int key_tile_queries(const Params& p, int kt, int* qt_lo) {
  return query_tiles_of(kt, p.kmax[kt], p.T, p.q_off, qt_lo);
}

// Persistent: each CTA takes work units {key tile, KV head, steps [b, e)} from a counter.
// Step t of a key tile is query tile qt_lo + t / G and query head kvh*G + t % G (query
// position outermost, so a unit covers whole query tiles for every head of the group).
// Barrier phases run on over the CTA's whole life: g counts its steps, uit its units.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct Unit {
  int kt, kvh, b, L, qt_lo;
};

// Takes the next work unit (thread `fetcher` draws it; every thread of the CTA calls this).
// Returns 0 to run it, 1 for a malformed unit (reported; the caller skips it after a CTA
// barrier), 2 when there is no more work or the CTA is aborting.
__device__ __forceinline__ int fetch_unit(const Params& p, int G, int* s_unit, int* s_abort, bool fetcher, Unit& U) {
  if (fetcher) *s_unit = atomicAdd(p.counter, 1);
  __syncthreads();
  const int u = *reinterpret_cast<volatile int*>(s_unit);
  if (u >= *p.n_units || *reinterpret_cast<volatile int*>(s_abort)) return 2;
  const int4 W = p.units[u];
  U.kt = W.x;
  U.kvh = W.y;
  U.b = W.z;
  U.L = W.w - W.z;
  U.qt_lo = 0;
  const bool unit_ok = U.kt >= 0 && U.kt * BN < p.T && U.kvh >= 0 && U.kvh < p.Hkv && U.b >= 0 && U.L > 0;
  const int nq = unit_ok ? key_tile_queries(p, U.kt, &U.qt_lo) : 0;
  if (!unit_ok || W.w > G * nq) {
    if (fetcher) raise_error(p.err, TREE_ERR_DEVICE_CHECK);
    return 1;
  }
  return 0;
}

__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                   const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ CUtensorMap tmDK,
                   const __grid_constant__ CUtensorMap tmDV, Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_unit, s_abort;
  if (p.err && (*reinterpret_cast<volatile int*>(p.err) & (1 << TREE_ERR_TIMEOUT))) return;
  Smem& S = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int G = p.Hq / p.Hkv;

  // Barrier phases run over the CTA's whole life, indexed by its step counter g; those
  // with two copies alternate between steps, so that a step's arrival can never land on
  // the phase of the step before it before every waiter has seen that one.
  if (threadIdx.x == 0) {
    mbar_init(&S.kv_full, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&S.qdo_full[s], 1);
      mbar_init(&S.qdo_empty[s], 2);  // dV (warp 10) and dK (warp 8) read Q_i / dO_i last
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.s_full[s], 1);
      mbar_init(&S.ds_ready[s], 8);
      mbar_init(&S.dk_done[s], 1);
      mbar_init(&S.dq_full[s], 1);
    }
    mbar_init(&S.dp_full, 1);
    mbar_init(&S.ld_done, 8);
    mbar_init(&S.drain_done, 4);
    mbar_init(&S.mma_done, 2);  // dV (warp 10) and dK (warp 8) accumulation of a unit
    mbar_init(&S.stage_read, 2);  // the dK / dV reduces of a unit have read their staging
    for (int w = 0; w < 4; ++w) mbar_init(&S.fin[w], 1);
    fence_mbarrier_init();
    s_abort = 0;
  }
  if (warp == kWarpMma) tmem_alloc(&S.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  // TMEM columns: S^T/P^T of even steps at 0, of odd steps at 64; dP^T 128; dQ^T 192
  constexpr uint32_t kColDP = 128, kColDQ = 192, kColDV = 256, kColDK = 384;
  int g0 = 0, uit = 0;  // steps and units this CTA has run (every role counts them)
  int g_loaded = 0;     // producer: steps whose Q_i / dO_i loads were issued
  int last_stage = -1;  // dQ drain leader: staging half of the most recent reduce

  // Each role runs its own copy of the unit loop; all meet at two CTA barriers per unit.
  if (warp < 8) {
    // ------------------------------------------------------------ compute warps
    const int wg = warp >> 2, q4 = warp & 3;
    const int r = q4 * 32 + lane;  // key row of S^T, dP^T, dK, dV
    const uint32_t lanes = static_cast<uint32_t>(q4 * 32) << 16;
    const float sl2 = p.scale_log2;
    while (true) {
      Unit U;
      const int fu = fetch_unit(p, G, &s_unit, &s_abort, threadIdx.x == 0, U);
      if (fu == 2) break;
      if (fu == 1) {
        __syncthreads();
        continue;
      }
      const int b = U.b, L = U.L;
      const int j = U.kt * BN + r;
      const int ej = p.endp[j];  // -1 past T
      // the previous unit's dK / dV reduces must have read their staging (the Q / dO / dS
      // buffers) before this unit's loads reuse them; the producer waits for this
      if (uit > 0 && q4 == 0 && lane == 0) {
        bulk_wait_read0();
        mbar_arrive(&S.stage_read);
      }
      bool ok = true;
      for (int l = 0; l < L; ++l) {
        const int g = g0 + l, st = g % NST, t = b + l;
        const int i0 = p.q_off + (U.qt_lo + t / G) * BQ + wg * 32;  // first query of this half, among the keys
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&S.s_full[g & 1], (g >> 1) & 1, p.err) &&
                                               mbar_wait(&S.dp_full, g & 1, p.err) &&
                                               mbar_wait(&S.qdo_full[st], (g / NST) & 1, p.err))))
          break;
        tc_fence_after();
        const uint32_t tS = tmem + lanes + (g & 1) * 64 + wg * 32, tD = tmem + lanes + kColDP + wg * 32;
        uint32_t sv[32], dp[32];
        tmem_ld32(tS, sv);
        tmem_ld32(tD, dp);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.ld_done);  // dP^T of the next step may overwrite its slot
        if (!__all_sync(0xffffffffu, j <= i0 && ej >= i0 + 31)) {
#pragma unroll
          for (int t2 = 0; t2 < 32; ++t2) {
            const int i = i0 + t2;
            if (!((j <= i) && (i <= ej))) sv[t2] = 0xff800000u;  // -inf: p = 0
          }
        }
        const float4* l4 = reinterpret_cast<const float4*>(S.lse2[st] + wg * 32);
        const float4* d4 = reinterpret_cast<const float4*>(S.delta[st] + wg * 32);
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int t4 = 0; t4 < 8; ++t4) {
          const float4 L4 = l4[t4], D4 = d4[t4];
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int t2 = t4 * 4 + h2 * 2;
            const float2 lv = h2 ? make_float2(L4.z, L4.w) : make_float2(L4.x, L4.y);
            const float2 dv = h2 ? make_float2(D4.z, D4.w) : make_float2(D4.x, D4.y);
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[t2]), __uint_as_float(sv[t2 + 1])),
                                        make_float2(sl2, sl2), make_float2(-lv.x, -lv.y));
            const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            const float2 dd = __fmul2_rn(pp, __fadd2_rn(make_float2(__uint_as_float(dp[t2]), __uint_as_float(dp[t2 + 1])),
                                                        make_float2(-dv.x, -dv.y)));
            pk[t2 / 2] = pack_bf16(pp.x, pp.y);
            dk[t2 / 2] = pack_bf16(dd.x, dd.y);
          }
        }
        // P^T and dS^T (bf16 pairs) over this half's S^T columns, which only this warp has
        // read: P^T (the A operand of dV) in the first 16, dS^T (that of dK) in the last 16
        tmem_st16(tS, pk);
        tmem_st16(tS + 16, dk);
        // dS^T into shared memory too (the B operand of dQ^T) once dQ^T of step g-2 has
        // read the buffer
        if (g >= 2 && !(ok = __all_sync(0xffffffffu, mbar_wait(&S.dq_full[g & 1], ((g >> 1) - 1) & 1, p.err))))
          break;
        uint8_t* dsrow = S.ds[g & 1] + r * 128;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const int chunk = (wg * 4 + w) ^ (r & 7);
          *reinterpret_cast<uint4*>(dsrow + chunk * 16) = make_uint4(dk[4 * w], dk[4 * w + 1], dk[4 * w + 2], dk[4 * w + 3]);
        }
        tmem_st_wait();
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.ds_ready[g & 1]);
      }
      // Unit epilogue: warps 0-3 add scale * dK, warps 4-7 add dV into the fp32
      // accumulators (one key row per thread). The rows are staged in the Q_i / dO_i / dS^T
      // buffers, idle now, as four [128 keys][32 dims] tiles with the 128-byte swizzle, and
      // added by TMA reduces. dQ^T of the unit's last two steps must have read dS^T first.
      const int g_end = g0 + L;
      ok = __all_sync(0xffffffffu, ok && mbar_wait(&S.mma_done, uit & 1, p.err) &&
                                       mbar_wait(&S.dq_full[(g_end - 1) & 1], ((g_end - 1) >> 1) & 1, p.err) &&
                                       (L < 2 || mbar_wait(&S.dq_full[g_end & 1], ((g_end - 2) >> 1) & 1, p.err)));
      tc_fence_after();
      if (ok) {
        uint8_t* stage = S.q[0] + wg * kEpiBytes;
        const float mul = wg == 0 ? p.scale : 1.f;
        const uint32_t tacc = tmem + lanes + (wg == 0 ? kColDK : kColDV);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tacc + c * 32, v);
          tmem_ld_wait();
          uint8_t* row = stage + c * (kEpiBytes / 4) + r * 128;
#pragma unroll
          for (int w = 0; w < 8; ++w)
            *reinterpret_cast<float4*>(row + ((w ^ (r & 7)) * 16)) =
                make_float4(__uint_as_float(v[4 * w]) * mul, __uint_as_float(v[4 * w + 1]) * mul,
                            __uint_as_float(v[4 * w + 2]) * mul, __uint_as_float(v[4 * w + 3]) * mul);
        }
        fence_proxy_async_smem();
        named_bar_sync(2 + wg, 128);
        if (q4 == 0 && lane == 0) {
          for (int c = 0; c < 4; ++c)
            tma_reduce_add_3d(wg == 0 ? &tmDK : &tmDV, stage + c * (kEpiBytes / 4), c * 32, U.kvh, U.kt * BN);
          bulk_commit();  // read completion is waited for at the next unit's start
        }
      } else {
        s_abort = 1;
      }
      g0 += L;
      ++uit;
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    }
    // the last unit's dK / dV reduces must have read their staging before the CTA exits
    if (q4 == 0 && lane == 0) bulk_wait_read0();
  } else if (warp < kWarpDq) {
    // ---------------------------------------------------- producer and MMA issuers
    constexpr uint32_t id_s = idesc_bf16(BN, BQ, 0, 0);  // S^T, dP^T
    constexpr uint32_t id_kv = idesc_bf16(BN, D, 0, 1);  // dV, dK (B MN-major)
    constexpr uint32_t id_dq = idesc_bf16(D, BQ, 1, 1);  // dQ^T (A and B MN-major)
    const uint32_t kb = smem_u32(S.k), vb = smem_u32(S.v);
    // S^T = K Q_i^T into the step's slot, or dP^T = V dO_i^T into the dP^T slot
    auto issue_sdp = [&](int g, bool is_s) -> bool {
      const int st = g % NST;
      if (!mbar_wait(&S.qdo_full[st], (g / NST) & 1, p.err)) return false;
      tc_fence_after();
      const uint32_t xb = smem_u32(is_s ? S.q[st] : S.dout[st]), ab = is_s ? kb : vb;
      const uint32_t d = tmem + (is_s ? (g & 1) * 64 : kColDP);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ka = (kk >> 2) * kKSub + (kk & 3) * 32, qa = (kk >> 2) * kQSub + (kk & 3) * 32;
        mma_ss(d, desc_sw128(ab + ka, 16, 1024), desc_sw128(xb + qa, 16, 1024), id_s, kk > 0);
      }
      mma_commit(is_s ? &S.s_full[g & 1] : &S.dp_full);
      return true;
    };
    while (true) {
      Unit U;
      const int fu = fetch_unit(p, G, &s_unit, &s_abort, false, U);
      if (fu == 2) break;
      if (fu == 1) {
        __syncthreads();
        continue;
      }
      const int kvh = U.kvh, b = U.b, L = U.L, j0 = U.kt * BN;
      if (lane == 0) {
        bool ok = true;
        if (warp == kWarpProducer) {
          if (uit == 0) {
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmDO);
          }
          mbar_arrive_expect_tx(&S.kv_full, 2 * kKTile);
          tma_load_3d(S.k, &tmK, &S.kv_full, 0, kvh, j0);
          tma_load_3d(S.k + kKSub, &tmK, &S.kv_full, 64, kvh, j0);
          tma_load_3d(S.v, &tmV, &S.kv_full, 0, kvh, j0);
          tma_load_3d(S.v + kKSub, &tmV, &S.kv_full, 64, kvh, j0);
          // Q_i, dO_i, LSE_i, Delta_i of step g once step g - NST no longer reads the stage
          auto load_step = [&](int g) -> bool {
            const int st = g % NST, t = b + (g - g0);
            if (g >= NST && !mbar_wait(&S.qdo_empty[st], ((g / NST) - 1) & 1, p.err)) return false;
            const int h = kvh * G + t % G;
            const int i0 = (U.qt_lo + t / G) * BQ;
            mbar_arrive_expect_tx(&S.qdo_full[st], 2 * kQTile + 2 * BQ * 4);
            tma_load_3d(S.q[st], &tmQ, &S.qdo_full[st], 0, h, i0);
            tma_load_3d(S.q[st] + kQSub, &tmQ, &S.qdo_full[st], 64, h, i0);
            tma_load_3d(S.dout[st], &tmDO, &S.qdo_full[st], 0, h, i0);
            tma_load_3d(S.dout[st] + kQSub, &tmDO, &S.qdo_full[st], 64, h, i0);
            bulk_load(S.lse2[st], p.lse2 + static_cast<int64_t>(h) * p.T_pad + i0, BQ * 4, &S.qdo_full[st]);
            bulk_load(S.delta[st], p.delta + static_cast<int64_t>(h) * p.T_pad + i0, BQ * 4, &S.qdo_full[st]);
            g_loaded = g + 1;
            return true;
          };
          // Q / dO go where the previous unit's dK / dV were staged
          if (uit > 0) ok = mbar_wait(&S.stage_read, (uit - 1) & 1, p.err);
          for (int l = 0; ok && l < min(NST, L); ++l) ok = load_step(g0 + l);
          for (int l = 0; ok && l < L; ++l) {
            const int g = g0 + l, st = g % NST;
            if (!(ok = mbar_wait(&S.ds_ready[g & 1], (g >> 1) & 1, p.err))) break;
            tc_fence_after();
            const uint32_t qb = smem_u32(S.q[st]), tDS = tmem + (g & 1) * 64 + 16;
#pragma unroll
            for (int kk = 0; kk < BQ / 16; ++kk)  // dK += dS^T Q; dS^T of query half w at column 32w + 16
              mma_ts(tmem + kColDK, tDS + (kk >> 1) * 32 + (kk & 1) * 8, desc_sw128(qb + kk * 2048, kQSub, 1024),
                     id_kv, (l > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&S.qdo_empty[st]);
            mma_commit(&S.dk_done[g & 1]);
            if (l + NST < L) ok = load_step(g + NST);
          }
          mma_commit(&S.mma_done);
        } else if (warp == kWarpMma) {
          // dP^T of step g+1 as soon as every compute warp has read step g's
          ok = mbar_wait(&S.kv_full, uit & 1, p.err) && issue_sdp(g0, false);
          for (int l = 0; ok && l + 1 < L; ++l) {
            const int g = g0 + l;
            if (!(ok = mbar_wait(&S.ld_done, g & 1, p.err))) break;
            tc_fence_after();
            ok = issue_sdp(g + 1, false);
          }
        } else if (warp == kWarpMma2) {
          ok = mbar_wait(&S.kv_full, uit & 1, p.err);
          for (int l = 0; ok && l < min(2, L); ++l) ok = issue_sdp(g0 + l, true);
          for (int l = 0; ok && l < L; ++l) {
            const int g = g0 + l, st = g % NST;
            if (!(ok = mbar_wait(&S.ds_ready[g & 1], (g >> 1) & 1, p.err))) break;
            tc_fence_after();
            const uint32_t ob = smem_u32(S.dout[st]), tP = tmem + (g & 1) * 64;
#pragma unroll
            for (int kk = 0; kk < BQ / 16; ++kk)  // dV += P^T dO; P^T of query half w at column 32w
              mma_ts(tmem + kColDV, tP + (kk >> 1) * 32 + (kk & 1) * 8, desc_sw128(ob + kk * 2048, kQSub, 1024),
                     id_kv, (l > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&S.qdo_empty[st]);
            // S^T of step g+2 into the slot whose P^T the dV above reads (same issuer:
            // ordered) and whose dS^T dK (warp 8) reads
            if (l + 2 < L) {
              if (!(ok = mbar_wait(&S.dk_done[g & 1], (g >> 1) & 1, p.err))) break;
              tc_fence_after();
              if (!(ok = issue_sdp(g + 2, true))) break;
            }
          }
          mma_commit(&S.mma_done);
        } else {
          ok = mbar_wait(&S.kv_full, uit & 1, p.err);
          for (int l = 0; ok && l < L; ++l) {
            const int g = g0 + l;
            if (!(ok = mbar_wait(&S.ds_ready[g & 1], (g >> 1) & 1, p.err))) break;
            // the dQ^T columns must have been drained (step g-1)
            if (g >= 1 && !(ok = mbar_wait(&S.drain_done, (g - 1) & 1, p.err))) break;
            tc_fence_after();
            const uint32_t db = smem_u32(S.ds[g & 1]);
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)  // dQ^T = K^T dS^T
              mma_ss(tmem + kColDQ, desc_sw128(kb + kk * 2048, kKSub, 1024), desc_sw128(db + kk * 2048, kQSub, 1024),
                     id_dq, kk > 0);
            mma_commit(&S.dq_full[g & 1]);
          }
        }
        if (!ok) s_abort = 1;
      }
      __syncwarp();
      g0 += L;
      ++uit;
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    }
  } else {
    // ------------------------------------------------------ dQ drain (warps 12-15)
    // TMEM lane = head dimension r, column = query. Free the columns once they are in
    // registers, then per half tile write scale * dQ row-major into a staging buffer and
    // add it into the fp32 accumulator with one TMA reduce (one thread issues them all).
    const int q4 = warp & 3, r = q4 * 32 + lane;
    const uint32_t lanes = static_cast<uint32_t>(q4 * 32) << 16;
    const bool leader = warp == kWarpDq && lane == 0;
    while (true) {
      Unit U;
      const int fu = fetch_unit(p, G, &s_unit, &s_abort, false, U);
      if (fu == 2) break;
      if (fu == 1) {
        __syncthreads();
        continue;
      }
      const int kvh = U.kvh, b = U.b, L = U.L;
      bool ok = true;
      for (int l = 0; l < L; ++l) {
        const int g = g0 + l, t = b + l;
        const int h = kvh * G + t % G;
        const int i0 = (U.qt_lo + t / G) * BQ;
        // one decision for the four warps: they meet at the staging barriers below
        if (!(ok = named_bar_and(1, 128, mbar_wait(&S.dq_full[g & 1], (g >> 1) & 1, p.err)))) break;
        tc_fence_after();
        uint32_t v[2][32];
        tmem_ld32(tmem + lanes + kColDQ, v[0]);
        tmem_ld32(tmem + lanes + kColDQ + 32, v[1]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.drain_done);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          // the reduce that last read this half's buffer must be done reading it
          if (leader) {
            if (last_stage == half) bulk_wait_read0(); else bulk_wait_read1();
          }
          named_bar_sync(1, 128);
          float* buf = S.dq_stage[half];
#pragma unroll
          for (int t2 = 0; t2 < 32; ++t2) buf[t2 * D + r] = __uint_as_float(v[half][t2]) * p.scale;
          fence_proxy_async_smem();
          named_bar_sync(1, 128);
          if (leader && i0 + half * (BQ / 2) < p.Tq) {
            tma_reduce_add_3d(&tmDQ, buf, 0, h, i0 + half * (BQ / 2));
            bulk_commit();
            last_stage = half;
          }
        }
      }
      if (!ok) s_abort = 1;
      g0 += L;
      ++uit;
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    }
  }
  // The last dQ reduces must have read their staging before the CTA exits.
  if (warp == kWarpDq && lane == 0) bulk_wait_read0();
  // On an early exit, leave no TMA copy or MMA in flight.
  if (s_abort && warp >= kWarpProducer && warp <= kWarpMma3 && lane == 0) {
    if (warp == kWarpProducer) {
      if (uit > 0) mbar_wait(&S.kv_full, (uit - 1) & 1, p.err);
      for (int g = max(0, g_loaded - NST); g < g_loaded; ++g) mbar_wait(&S.qdo_full[g % NST], (g / NST) & 1, p.err);
    }
    mma_commit(&S.fin[warp - kWarpProducer]);
    mbar_wait(&S.fin[warp - kWarpProducer], 0, p.err);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

struct PrepParams {
  const int32_t* end;  // subtree_end [T] (of the key rows)
  int T, T_pad, n_kt, Hq, Hkv, max_units;  // T: key rows; T_pad: query rows rounded up to 64
  int Tq, q_off, n_rows;                   // query rows, keys before them, rows the blocks cover
  int one_unit_per_tile;                   // deterministic mode: every key tile is one unit
  int32_t* kmax;       // [n_kt] max subtree_end of each 128-key tile
  int32_t* kmin;       // [n_kt] min subtree_end of each 128-key tile
  int32_t* endp;       // [n_kt * 128] subtree_end, -1 past T
  int4* units;
  int* n_units;
  int* counter;
  int* bucket;         // [T_pad / 64 + 1]
  const __nv_bfloat16* o;
  const __nv_bfloat16* dout;
  const float* lse;    // [Hq, T]
  float* lse2;         // [Hq, T_pad]
  float* delta;        // [Hq, T_pad]
  float* dq_acc;
  float* dk_acc;
  float* dv_acc;
  int* err;
};

// Block 0 (the planner): per-128-key-tile bounds of subtree_end (checked to lie in
// [j, T)), the padded copy the main kernel reads, and the work units. Every key tile's
// steps (its 64-row query tiles x the G query heads of the group) are cut into chunks of
// chunk_q whole query tiles, chunk_q growing with the total work so that there are at
// most about 1216 + Hkv * n_kt units; the units of all key tiles are then ordered by the
// first query tile they cover (a counting sort), so that the CTAs running at the same
// time work on nearby query rows and share the Q / dO tiles and the dQ accumulator lines
// in L2.
// Blocks 1..: Delta = dO . O and LSE * log2(e) per (row, head), padded to T_pad with
// (0, +inf), and zeroed fp32 dQ, dK and dV accumulators; one warp per (row, head).
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const PrepParams q) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (blockIdx.x > 0) {
    const int64_t w = static_cast<int64_t>(blockIdx.x - 1) * 8 + warp;
    if (w >= static_cast<int64_t>(q.n_rows) * q.Hq) return;
    const int64_t i = w / q.Hq;
    const int h = static_cast<int>(w % q.Hq);
    if (i < q.T && i >= q.Tq && h < q.Hkv) {  // key rows past the query rows: zero dK, dV only
      const int64_t kv = (i * q.Hkv + h) * 128 + lane * 4;
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(q.dk_acc + kv) = z;
      *reinterpret_cast<float4*>(q.dv_acc + kv) = z;
    }
    if (i >= q.T_pad) return;
    float dl = 0.f, l2 = INFINITY;
    if (i < q.Tq) {
      const int64_t off = w * 128 + lane * 4;
      const uint2 a = *reinterpret_cast<const uint2*>(q.o + off);
      const uint2 b = *reinterpret_cast<const uint2*>(q.dout + off);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
      const float2 a0 = __bfloat1622float2(a2[0]), a1 = __bfloat1622float2(a2[1]);
      const float2 b0 = __bfloat1622float2(b2[0]), b1 = __bfloat1622float2(b2[1]);
      dl = a0.x * b0.x + a0.y * b0.y + a1.x * b1.x + a1.y * b1.y;
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) dl += __shfl_xor_sync(0xffffffffu, dl, s);
      l2 = q.lse[static_cast<int64_t>(h) * q.Tq + i] * 1.4426950408889634f;
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(q.dq_acc + off) = z;
      if (h < q.Hkv) {
        const int64_t kv = (i * q.Hkv + h) * 128 + lane * 4;
        *reinterpret_cast<float4*>(q.dk_acc + kv) = z;
        *reinterpret_cast<float4*>(q.dv_acc + kv) = z;
      }
    }
    if (lane == 0) {
      q.lse2[static_cast<int64_t>(h) * q.T_pad + i] = l2;
      q.delta[static_cast<int64_t>(h) * q.T_pad + i] = dl;
    }
    return;
  }
  // ---------------------------------------------------------------- planner
  __shared__ long long s_total;
  __shared__ int s_units;
  const int T = q.T, n_q64 = q.T_pad / BQ, G = q.Hq / q.Hkv;
  if (threadIdx.x == 0) {
    s_total = 0;
    s_units = 0;
    *q.counter = 0;
  }
  for (int b = threadIdx.x; b <= n_q64; b += blockDim.x) q.bucket[b] = 0;
  for (int kt = warp; kt < q.n_kt; kt += blockDim.x / 32) {
    int mx = -1, mn = INT32_MAX;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int j = kt * BN + c * 32 + lane;
      const bool in = j < T;
      const int e = in ? q.end[j] : -1;
      if (in && (e < j || e >= T)) raise_error(q.err, TREE_ERR_DEVICE_CHECK);
      q.endp[j] = e;
      if (in) {
        mx = max(mx, e);
        mn = min(mn, e);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    }
    if (lane == 0) {
      q.kmax[kt] = mx;
      q.kmin[kt] = mn;
    }
  }
  __syncthreads();
  auto tiles_of = [&](int kt, int* lo) -> int { return query_tiles_of(kt, q.kmax[kt], T, q.q_off, lo); };
  long long local = 0;
  for (int kt = threadIdx.x; kt < q.n_kt; kt += blockDim.x) {
    int lo;
    local += tiles_of(kt, &lo);
  }
  atomicAdd(reinterpret_cast<unsigned long long*>(&s_total), static_cast<unsigned long long>(local));
  __syncthreads();
  const long long steps_all = s_total * G * q.Hkv;
  // ~8 units per SM on large trees; on small ones the 16-step floor keeps units short
  const int chunk_steps = static_cast<int>(max(16LL, (steps_all + 1215) / 1216));
  const int chunk_q = q.one_unit_per_tile ? (INT32_MAX / 4) : (chunk_steps + G - 1) / G;
  for (int kt = threadIdx.x; kt < q.n_kt; kt += blockDim.x) {  // units per first query tile
    int lo;
    const int nq = tiles_of(kt, &lo);
    for (int c = 0; c * chunk_q < nq; ++c) atomicAdd(&q.bucket[lo + c * chunk_q], 1);
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan, in units of (key tile, chunk) pairs
    int run = 0;
    for (int b0 = 0; b0 <= n_q64; b0 += 32) {
      const int b = b0 + lane;
      const int x = b < n_q64 ? q.bucket[b] : 0;
      int incl = x;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (b <= n_q64) q.bucket[b] = run + incl - x;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_units = run;
  }
  __syncthreads();
  for (int kt = threadIdx.x; kt < q.n_kt; kt += blockDim.x) {
    int lo;
    const int nq = tiles_of(kt, &lo);
    for (int c = 0; c * chunk_q < nq; ++c) {
      const int pos = atomicAdd(&q.bucket[lo + c * chunk_q], 1);
      const int b0 = c * chunk_q * G, b1 = min((c + 1) * chunk_q, nq) * G;
      for (int kvh = 0; kvh < q.Hkv; ++kvh) {
        const int idx = pos * q.Hkv + kvh;
        if (idx < q.max_units) q.units[idx] = make_int4(kt, kvh, b0, b1);
      }
    }
  }
  if (threadIdx.x == 0) *q.n_units = min(s_units * q.Hkv, q.max_units);
}

}  // namespace tcbwd

// ------------------------------------------------------------------------------------
// Deterministic dQ (the backward's deterministic mode): query-stationary. One CTA owns 128
// query rows of one query head and walks the key tiles its rows can see in increasing
// order, with dQ accumulating in TMEM, so every dQ element is one fixed-order sum:
//   S = Q K^T, dP = dO V^T                  (M = 128 queries, N = 128 keys, K = d; TMEM)
//   P = exp2(S scale log2e - LSE log2e) on visible pairs, dS = P (dP - Delta)   (4 warps,
//                                           one query row per thread, 64 keys at a time)
//   dQ += dS K                               (A = dS bf16 from TMEM over S's columns,
//                                           B = the K tile MN-major)
// and scale * dQ is stored (not added) into the fp32 accumulator the conversion reads.
// Warps 0-3 compute, warp 4 TMA, warp 5 MMA. TMEM: S [0, 128), dP [128, 256), dQ [256, 384).
namespace tcdq {
using tcbwd::ex2_approx;

constexpr int BM = 128, BN = 128, D = 128;
constexpr int kThreads = 192;
constexpr int kWarpProducer = 4, kWarpMma = 5;
constexpr uint32_t kSub = 128 * 128;   // 128 rows x 128 B: one swizzle-128 sub-tile
constexpr uint32_t kTile = 2 * kSub;   // 128 rows x 128 bf16

struct Smem {
  uint8_t q[kTile];
  uint8_t dout[kTile];
  uint8_t k[2][kTile];
  uint8_t v[2][kTile];
  uint64_t qdo_full, k_full[2], v_full[2], kv_empty[2], sd_full, ds_full, mma_done;
  uint32_t tmem_base;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 232448, "dQ kernel shared memory exceeds the per-block limit");

struct Params {
  int T, Tq, T_pad, Hq, Hkv, n_qt, n_kt;
  float scale_log2, scale;
  const int32_t* kmax;
  const int32_t* kmin;
  const int32_t* endp;
  const float* lse2;    // [Hq, T_pad] LSE * log2(e)
  const float* delta;   // [Hq, T_pad]
  float* dq_acc;        // [Tq, Hq, d] fp32, written
  int* err;
};

__global__ void __launch_bounds__(kThreads, 1)
attn_dq_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                  const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, Params p) {
  extern __shared__ uint8_t smem_raw[];
  if (p.err && (*reinterpret_cast<volatile int*>(p.err) & (1 << TREE_ERR_TIMEOUT))) return;
  Smem& S = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int h = blockIdx.y;
  const int qt = p.n_qt - 1 - blockIdx.x;  // longest query tiles first
  const int i0 = qt * BM;
  const int kt_hi = min((i0 + BM - 1) / BN, p.n_kt - 1);
  const int kvh = h / (p.Hq / p.Hkv);
  if (threadIdx.x == 0) {
    mbar_init(&S.qdo_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.k_full[s], 1);
      mbar_init(&S.v_full[s], 1);
      mbar_init(&S.kv_empty[s], 1);
    }
    mbar_init(&S.sd_full, 1);
    mbar_init(&S.ds_full, 4);
    mbar_init(&S.mma_done, 1);
    fence_mbarrier_init();
  }
  if (warp == kWarpMma) tmem_alloc(&S.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  constexpr uint32_t kColDP = 128, kColDQ = 256;

  if (warp == kWarpProducer) {
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmDO);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      mbar_arrive_expect_tx(&S.qdo_full, 2 * kTile);
      for (int sub = 0; sub < 2; ++sub) {
        tma_load_3d(S.q + sub * kSub, &tmQ, &S.qdo_full, sub * 64, h, i0);
        tma_load_3d(S.dout + sub * kSub, &tmDO, &S.qdo_full, sub * 64, h, i0);
      }
      int n = 0;
      for (int kt = 0; kt <= kt_hi; ++kt) {
        if (p.kmax[kt] < i0) continue;
        const int s = n & 1;
        if (n >= 2 && !mbar_wait(&S.kv_empty[s], ((n >> 1) - 1) & 1, p.err)) break;
        mbar_arrive_expect_tx(&S.k_full[s], kTile);
        tma_load_3d(S.k[s], &tmK, &S.k_full[s], 0, kvh, kt * BN);
        tma_load_3d(S.k[s] + kSub, &tmK, &S.k_full[s], 64, kvh, kt * BN);
        mbar_arrive_expect_tx(&S.v_full[s], kTile);
        tma_load_3d(S.v[s], &tmV, &S.v_full[s], 0, kvh, kt * BN);
        tma_load_3d(S.v[s] + kSub, &tmV, &S.v_full[s], 64, kvh, kt * BN);
        ++n;
      }
      for (int m = (n >= 2 ? n - 2 : 0); m < n; ++m) {
        mbar_wait(&S.k_full[m & 1], (m >> 1) & 1, p.err);
        mbar_wait(&S.v_full[m & 1], (m >> 1) & 1, p.err);
      }
      mbar_wait(&S.qdo_full, 0, p.err);
    }
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(BM, BN, 0, 0);   // S, dP: both operands K-major
      constexpr uint32_t idesc_q = idesc_bf16(BM, D, 0, 1);    // dQ: B = K tile MN-major
      int N = 0;
      for (int kt = 0; kt <= kt_hi; ++kt) N += p.kmax[kt] >= i0;
      const uint32_t qa = smem_u32(S.q), oa = smem_u32(S.dout);
      bool ok = mbar_wait(&S.qdo_full, 0, p.err);
      for (int n = 0; ok && n < N; ++n) {
        const int s = n & 1;
        if (!(ok = mbar_wait(&S.k_full[s], (n >> 1) & 1, p.err) && mbar_wait(&S.v_full[s], (n >> 1) & 1, p.err)))
          break;
        tc_fence_after();
        const uint32_t kb = smem_u32(S.k[s]), vb = smem_u32(S.v[s]);
        // S over the columns dS(n-1) occupied: the MMAs run in issue order, so dQ(n-1),
        // issued before, has read them
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kSub + (kk & 3) * 32;
          mma_ss(tmem, desc_sw128(qa + off, 16, 1024), desc_sw128(kb + off, 16, 1024), idesc_s, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kSub + (kk & 3) * 32;
          mma_ss(tmem + kColDP, desc_sw128(oa + off, 16, 1024), desc_sw128(vb + off, 16, 1024), idesc_s, kk > 0);
        }
        mma_commit(&S.sd_full);
        if (!(ok = mbar_wait(&S.ds_full, n & 1, p.err))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)  // dQ += dS K: dS (bf16 pairs) at columns 0..63
          mma_ts(tmem + kColDQ, tmem + kk * 8, desc_sw128(kb + kk * 2048, kSub, 1024), idesc_q,
                 (n > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&S.kv_empty[s]);
      }
      mma_commit(&S.mma_done);
      mbar_wait(&S.mma_done, 0, p.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute warps 0-3
    const int r = warp * 32 + lane, i = i0 + r;
    const uint32_t lanes = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    const bool row_ok = i < p.Tq;
    const float l2 = row_ok ? p.lse2[static_cast<int64_t>(h) * p.T_pad + i] : INFINITY;
    const float dl = row_ok ? p.delta[static_cast<int64_t>(h) * p.T_pad + i] : 0.f;
    int n = 0;
    bool ok = true;
    for (int kt = 0; kt <= kt_hi; ++kt) {
      if (p.kmax[kt] < i0) continue;
      const int j0 = kt * BN;
      const bool partial = !(j0 + BN - 1 <= i0 && p.kmin[kt] >= i0 + BM - 1);
      uint32_t vis[4] = {~0u, ~0u, ~0u, ~0u};
      if (partial) {
#pragma unroll
        for (int c = 0; c < 4; ++c) vis[c] = visible32(p.endp, j0 + 32 * c, i);
      }
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&S.sd_full, n & 1, p.err)))) break;
      tc_fence_after();
      // 64 keys at a time: S and dP of those keys, then dS (bf16 pairs) over S's first
      // columns (half 0 -> columns 0..31, half 1 -> 32..63: both already read)
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t sv[64], dp[64];
        tmem_ld32(tmem + lanes + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tmem_ld32(tmem + lanes + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        tmem_ld32(tmem + lanes + kColDP + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
        tmem_ld32(tmem + lanes + kColDP + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
        tmem_ld_wait();
        uint32_t pk[32];
#pragma unroll
        for (int t = 0; t < 64; t += 2) {
          const int key = half * 64 + t;
          const bool v0 = (vis[key >> 5] >> (key & 31)) & 1u, v1 = (vis[(key + 1) >> 5] >> ((key + 1) & 31)) & 1u;
          const float p0 = v0 ? ex2_approx(fmaf(__uint_as_float(sv[t]), sl2, -l2)) : 0.f;
          const float p1 = v1 ? ex2_approx(fmaf(__uint_as_float(sv[t + 1]), sl2, -l2)) : 0.f;
          pk[t / 2] = pack_bf16(p0 * (__uint_as_float(dp[t]) - dl), p1 * (__uint_as_float(dp[t + 1]) - dl));
        }
        tmem_st32(tmem + lanes + half * 32, pk);
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.ds_full);
      ++n;
    }
    // epilogue: scale * dQ (fp32) into the accumulator rows of this head
    ok = __all_sync(0xffffffffu, ok && mbar_wait(&S.mma_done, 0, p.err));
    tc_fence_after();
    if (ok) {
      float4* dst = reinterpret_cast<float4*>(p.dq_acc + (static_cast<int64_t>(i) * p.Hq + h) * D);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        if (n > 0) {
          tmem_ld32(tmem + lanes + kColDQ + c * 32, o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t) o[t] = 0u;
        }
        if (row_ok) {
#pragma unroll
          for (int u = 0; u < 8; ++u)
            dst[8 * c + u] = make_float4(__uint_as_float(o[4 * u]) * p.scale, __uint_as_float(o[4 * u + 1]) * p.scale,
                                         __uint_as_float(o[4 * u + 2]) * p.scale, __uint_as_float(o[4 * u + 3]) * p.scale);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace tcdq

// dQ, dK and dV (bf16) from their fp32 accumulators in one launch, 4 elements per thread.
__global__ void attn_grads_to_bf16_kernel(const float* __restrict__ aq, __nv_bfloat16* __restrict__ oq, int64_t nq4,
                                          const float* __restrict__ ak, __nv_bfloat16* __restrict__ ok, int64_t nk4,
                                          const float* __restrict__ av, __nv_bfloat16* __restrict__ ov) {
  int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const float* a;
  __nv_bfloat16* o;
  if (t < nq4) {
    a = aq; o = oq;
  } else if ((t -= nq4) < nk4) {
    a = ak; o = ok;
  } else if ((t -= nk4) < nk4) {
    a = av; o = ov;
  } else {
    return;
  }
  const float4 v = reinterpret_cast<const float4*>(a)[t];
  uint2 u;
  u.x = sm100::pack_bf16(v.x, v.y);
  u.y = sm100::pack_bf16(v.z, v.w);
  reinterpret_cast<uint2*>(o)[t] = u;
}

// The same conversion with the backward of the depth rotation (tree_rope, inverse) on dQ
// and dK, applied to the fp32 sums before the one rounding: rotate-half pairs
// (x[f], x[f + 64]) turned by -pos * theta^(-2f/128). One thread owns one row, 4
// consecutive frequencies and 4 heads (of dQ, then dK), so each (cos, sin) serves 4
// heads; then dV, 4 elements per thread.
__global__ void attn_grads_rope_to_bf16_kernel(const float* __restrict__ aq, __nv_bfloat16* __restrict__ oq,
                                               const float* __restrict__ ak, __nv_bfloat16* __restrict__ ok,
                                               const float* __restrict__ av, __nv_bfloat16* __restrict__ ov,
                                               const int32_t* __restrict__ pos, int64_t T, int Hq, int Hkv,
                                               float neg2_log2base_over_d, int* err) {
  constexpr int kGroups = 16, kHeads = 4;  // 16 groups of 4 frequencies per 128-wide row
  const int n_heads = Hq + Hkv, chunks = (n_heads + kHeads - 1) / kHeads;
  const int64_t n_rot = T * chunks * kGroups;
  int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= n_rot) {  // dV: plain conversion
    t -= n_rot;
    if (t >= T * Hkv * 32) return;
    const float4 v = reinterpret_cast<const float4*>(av)[t];
    uint2 u;
    u.x = sm100::pack_bf16(v.x, v.y);
    u.y = sm100::pack_bf16(v.z, v.w);
    reinterpret_cast<uint2*>(ov)[t] = u;
    return;
  }
  const int g = static_cast<int>(t % kGroups);
  const int chunk = static_cast<int>((t / kGroups) % chunks);
  const int64_t row = t / (kGroups * chunks);
  const int p0 = pos[row];
  if (p0 < 0) {
    raise_error(err, TREE_ERR_DEVICE_CHECK);
    return;
  }
  // all of the thread's loads first (8 in flight), then the rotation and the stores
  float4 x1[kHeads], x2[kHeads];
  int64_t off[kHeads];
  bool isq[kHeads], valid[kHeads];
#pragma unroll
  for (int u = 0; u < kHeads; ++u) {
    const int hh = chunk * kHeads + u;
    valid[u] = hh < n_heads;
    isq[u] = hh < Hq;
    const int H = isq[u] ? Hq : Hkv, h = isq[u] ? hh : hh - Hq;
    off[u] = (row * H + h) * 128 + g * 4;
    if (valid[u]) {
      const float* a = (isq[u] ? aq : ak) + off[u];
      x1[u] = *reinterpret_cast<const float4*>(a);
      x2[u] = *reinterpret_cast<const float4*>(a + 64);
    }
  }
  float c[4], s[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float inv_freq = exp2f(static_cast<float>(g * 4 + i) * neg2_log2base_over_d);
    sincosf(static_cast<float>(p0) * inv_freq, &s[i], &c[i]);
  }
#pragma unroll
  for (int u = 0; u < kHeads; ++u) {
    if (!valid[u]) continue;
    __nv_bfloat16* o = (isq[u] ? oq : ok) + off[u];
    const float4 a1 = x1[u], a2 = x2[u];
    // inverse rotation: y1 = x1 c + x2 s, y2 = x2 c - x1 s
    uint2 u1, u2;
    u1.x = sm100::pack_bf16(a1.x * c[0] + a2.x * s[0], a1.y * c[1] + a2.y * s[1]);
    u1.y = sm100::pack_bf16(a1.z * c[2] + a2.z * s[2], a1.w * c[3] + a2.w * s[3]);
    u2.x = sm100::pack_bf16(a2.x * c[0] - a1.x * s[0], a2.y * c[1] - a1.y * s[1]);
    u2.y = sm100::pack_bf16(a2.z * c[2] - a1.z * s[2], a2.w * c[3] - a1.w * s[3]);
    *reinterpret_cast<uint2*>(o) = u1;
    *reinterpret_cast<uint2*>(o + 64) = u2;
  }
}

static int rows_map(CUtensorMap* m, const void* base, int64_t T, int H, uint32_t rows) {
  const uint64_t dims[3] = {128, static_cast<uint64_t>(H), static_cast<uint64_t>(T)};
  const uint64_t strides[2] = {128 * 2, static_cast<uint64_t>(H) * 128 * 2};
  const uint32_t box[3] = {64, 1, rows};
  return make_tmap(m, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, dims, strides, box, true);
}

bool attn_bwd_tc_supported(int dtype, int d, int deterministic) {
  (void)deterministic;  // both modes run on the tensor-core kernels
  return dtype == TREE_DTYPE_BF16 && d == 128;
}

int64_t attn_bwd_max_units(int64_t T, int Hkv) { return 4096 + static_cast<int64_t>(Hkv) * ((T + 127) / 128) + 64; }

static int sm_count(int* n) {
  static int cached[128] = {0};
  int dev = 0;
  TREE_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 128) return fail(TREE_ERR_CUDA, "device ordinal %d out of range", dev);
  if (!cached[dev]) TREE_CUDA_TRY(cudaDeviceGetAttribute(&cached[dev], cudaDevAttrMultiProcessorCount, dev));
  *n = cached[dev];
  return TREE_OK;
}

// Gateway keys' gradients (the key rows before the queries): fp32 sums added into the
// caller's accumulators, so that several child partitions sharing a gateway add up
// without bf16 rounding between them.
__global__ void gateway_past_grads_kernel(const float* __restrict__ dk_acc, const float* __restrict__ dv_acc,
                                          int64_t n4, float* __restrict__ dk_past, float* __restrict__ dv_past) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= 2 * n4) return;
  const bool is_v = t >= n4;
  const int64_t u = is_v ? t - n4 : t;
  const float4 g = reinterpret_cast<const float4*>(is_v ? dv_acc : dk_acc)[u];
  float4* o = reinterpret_cast<float4*>(is_v ? dv_past : dk_past) + u;
  float4 x = *o;
  x.x += g.x; x.y += g.y; x.z += g.z; x.w += g.w;
  *o = x;
}

int attn_bwd_tc(const AttnArgs& a, cudaStream_t st) {
  using namespace tcbwd;
  const int64_t Tq = a.T - a.q_off;  // queries: the last Tq key rows
  const int64_t T_pad = (Tq + BQ - 1) / BQ * BQ;
  const int n_kt = static_cast<int>((a.T + BN - 1) / BN);
  const int max_units = static_cast<int>(attn_bwd_max_units(a.T, a.Hkv));
  {
    PrepParams q{};
    q.end = a.end;
    q.T = static_cast<int>(a.T);
    q.T_pad = static_cast<int>(T_pad);
    q.Tq = static_cast<int>(Tq);
    q.q_off = static_cast<int>(a.q_off);
    q.n_rows = static_cast<int>(std::max<int64_t>(T_pad, a.T));
    q.n_kt = n_kt;
    q.Hq = a.Hq;
    q.Hkv = a.Hkv;
    q.max_units = max_units;
    q.kmax = a.ws.kmax128;
    q.kmin = a.ws.kmin128;
    q.endp = a.ws.end_pad;
    q.units = reinterpret_cast<int4*>(a.ws.units);
    q.n_units = a.ws.n_units;
    q.counter = a.ws.counter;
    q.bucket = a.ws.bucket;
    q.o = static_cast<const __nv_bfloat16*>(a.o);
    q.dout = static_cast<const __nv_bfloat16*>(a.dout);
    q.lse = a.lse;
    q.lse2 = a.ws.lse2_pad;
    q.delta = a.ws.delta_pad;
    q.dq_acc = a.ws.dq_acc;
    q.dk_acc = a.ws.dk_acc;
    q.dv_acc = a.ws.dv_acc;
    q.err = device_error_word();
    q.one_unit_per_tile = a.deterministic;
    const int64_t pre_blocks = (static_cast<int64_t>(q.n_rows) * a.Hq + 7) / 8;
    attn_bwd_prep_kernel<<<static_cast<unsigned>(1 + pre_blocks), 256, 0, st>>>(q);
    TREE_LAUNCH_CHECK("attn_bwd_prep_kernel");
  }
  int rc = TREE_OK;
  CUtensorMap mk, mv, mq, mdo, mdq;
  if ((rc = rows_map(&mk, a.k, a.T, a.Hkv, 128)) || (rc = rows_map(&mv, a.v, a.T, a.Hkv, 128)) ||
      (rc = rows_map(&mq, a.q, Tq, a.Hq, BQ)) || (rc = rows_map(&mdo, a.dout, Tq, a.Hq, BQ)))
    return rc;
  {
    // fp32 dQ accumulator [Tq, Hq, 128] as {d, head, row}, box {128, 1, 64}, no swizzle
    const uint64_t dims[3] = {128, static_cast<uint64_t>(a.Hq), static_cast<uint64_t>(Tq)};
    const uint64_t strides[2] = {128 * 4, static_cast<uint64_t>(a.Hq) * 128 * 4};
    const uint32_t box[3] = {128, 1, BQ / 2};
    if ((rc = make_tmap(&mdq, a.ws.dq_acc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dims, strides, box, false))) return rc;
  }
  CUtensorMap mdk, mdv;
  {
    // fp32 dK / dV accumulators [T, Hkv, 128] as {d, head, row}, box {32, 1, 128}, 128-byte swizzle
    const uint64_t dims[3] = {128, static_cast<uint64_t>(a.Hkv), static_cast<uint64_t>(a.T)};
    const uint64_t strides[2] = {128 * 4, static_cast<uint64_t>(a.Hkv) * 128 * 4};
    const uint32_t box[3] = {32, 1, BN};
    if ((rc = make_tmap(&mdk, a.ws.dk_acc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dims, strides, box, true)) ||
        (rc = make_tmap(&mdv, a.ws.dv_acc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dims, strides, box, true)))
      return rc;
  }
  if (int rc_ = smem_opt_in(reinterpret_cast<const void*>(attn_bwd_tc_kernel), static_cast<int>(kSmemBytes))) return rc_;
  int n_sm = 0;
  if ((rc = sm_count(&n_sm))) return rc;
  Params p{};
  p.T = static_cast<int>(a.T);
  p.T_pad = static_cast<int>(T_pad);
  p.Tq = static_cast<int>(Tq);
  p.q_off = static_cast<int>(a.q_off);
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.scale = a.scale;
  p.kmax = a.ws.kmax128;
  p.endp = a.ws.end_pad;
  p.lse2 = a.ws.lse2_pad;
  p.delta = a.ws.delta_pad;
  p.dq_acc = a.ws.dq_acc;
  p.dk_acc = a.ws.dk_acc;
  p.dv_acc = a.ws.dv_acc;
  p.units = reinterpret_cast<const int4*>(a.ws.units);
  p.n_units = a.ws.n_units;
  p.counter = a.ws.counter;
  p.err = device_error_word();
  const int grid = static_cast<int>(std::min<int64_t>(n_sm, max_units));
  timing_begin(1, st);
  attn_bwd_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(mk, mv, mq, mdo, mdq, mdk, mdv, p);
  TREE_LAUNCH_CHECK("attn_bwd_tc_kernel");
  timing_end(1, st);
  if (a.deterministic) {
    // dQ again, query-stationary in a fixed order, over the accumulator the kernel above
    // added into in whatever order its units ran
    using namespace tcdq;
    CUtensorMap mq2, mdo2, mk2, mv2;
    if ((rc = rows_map(&mq2, a.q, Tq, a.Hq, 128)) || (rc = rows_map(&mdo2, a.dout, Tq, a.Hq, 128)) ||
        (rc = rows_map(&mk2, a.k, a.T, a.Hkv, 128)) || (rc = rows_map(&mv2, a.v, a.T, a.Hkv, 128)))
      return rc;
    if ((rc = smem_opt_in(reinterpret_cast<const void*>(attn_dq_tc_kernel), static_cast<int>(tcdq::kSmemBytes))))
      return rc;
    tcdq::Params d{};
    d.T = static_cast<int>(a.T);
    d.Tq = static_cast<int>(Tq);
    d.T_pad = static_cast<int>(T_pad);
    d.Hq = a.Hq;
    d.Hkv = a.Hkv;
    d.n_qt = static_cast<int>((Tq + 127) / 128);
    d.n_kt = n_kt;
    d.scale_log2 = a.scale * 1.4426950408889634f;
    d.scale = a.scale;
    d.kmax = a.ws.kmax128;
    d.kmin = a.ws.kmin128;
    d.endp = a.ws.end_pad;
    d.lse2 = a.ws.lse2_pad;
    d.delta = a.ws.delta_pad;
    d.dq_acc = a.ws.dq_acc;
    d.err = device_error_word();
    attn_dq_tc_kernel<<<dim3(d.n_qt, a.Hq), tcdq::kThreads, tcdq::kSmemBytes, st>>>(mq2, mdo2, mk2, mv2, d);
    TREE_LAUNCH_CHECK("attn_dq_tc_kernel");
  }
  if (a.rope_pos) {
    const int64_t n = a.T * ((a.Hq + a.Hkv + 3) / 4) * 16 + a.T * a.Hkv * 32;
    const float e = static_cast<float>(-2.0 * std::log2(static_cast<double>(a.rope_theta)) / a.d);
    attn_grads_rope_to_bf16_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(
        a.ws.dq_acc, static_cast<__nv_bfloat16*>(a.dq), a.ws.dk_acc, static_cast<__nv_bfloat16*>(a.dk),
        a.ws.dv_acc, static_cast<__nv_bfloat16*>(a.dv), a.rope_pos, a.T, a.Hq, a.Hkv, e, device_error_word());
    TREE_LAUNCH_CHECK("attn_grads_rope_to_bf16_kernel");
    return TREE_OK;
  }
  // dQ of the queries; dK and dV of the key rows that are queries too (all of them but for
  // gateway calls, whose leading q_off key rows go to the fp32 gateway sums instead)
  const int64_t kv_off = a.q_off * a.Hkv * a.d;
  const int64_t nq4 = Tq * a.Hq * a.d / 4, nk4 = Tq * a.Hkv * a.d / 4;
  attn_grads_to_bf16_kernel<<<static_cast<unsigned>((nq4 + 2 * nk4 + 255) / 256), 256, 0, st>>>(
      a.ws.dq_acc, static_cast<__nv_bfloat16*>(a.dq), nq4, a.ws.dk_acc + kv_off, static_cast<__nv_bfloat16*>(a.dk),
      nk4, a.ws.dv_acc + kv_off, static_cast<__nv_bfloat16*>(a.dv));
  TREE_LAUNCH_CHECK("attn_grads_to_bf16_kernel");
  if (a.q_off > 0) {
    const int64_t n4 = kv_off / 4;
    gateway_past_grads_kernel<<<static_cast<unsigned>((2 * n4 + 255) / 256), 256, 0, st>>>(
        a.ws.dk_acc, a.ws.dv_acc, n4, a.dk_past, a.dv_past);
    TREE_LAUNCH_CHECK("gateway_past_grads_kernel");
  }
  return TREE_OK;
}

}  // namespace tree
