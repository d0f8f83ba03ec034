// Tree attention forward on tcgen05 tensor cores (bf16 in, fp32 accumulate, d = 128).
//
// Visibility (Tree Training, arXiv 2511.00413, §3.2 "Attention Mask"; Trie packing
// "Step 2 - Allow only ancestors and self"): key j is visible to query i iff
// j <= i <= subtree_end[j]. Per 128-key tile the metadata kernel stores the max
// and min of subtree_end; a (query tile, key tile) pair is
//   skipped  when max_end < first query (no key of the tile sees any query),
//   full     when the tile lies wholly before the query tile and min_end >= last query,
//   partial  otherwise (the interval test is applied to every score in registers).
//
// One CTA owns 128 query rows of two query heads that share one KV head (GQA), so
// every K/V tile fetched by TMA feeds two independent softmax streams, and the
// tensor core alternates between them:
//   warp 8  (TMA)     Q of both heads once; K and V of each visible key tile into a
//                     two-stage ring (128-byte swizzle, zero fill past T).
//   warp 9  (MMA)     S_h = Q_h K^T (SS, M=N=128, K=16 x 8) into TMEM; after the softmax
//                     of head h wrote P_h (bf16) over its S columns, O_h += P_h V
//                     (A operand from TMEM, V MN-major in shared memory).
//   warps 0-3 / 4-7   softmax of head A / head B, one thread per query row: row max
//                     (masked, in the base-2 domain), lazy rescaling of O in TMEM only
//                     when the max grows by more than 2^8, P = exp2(s - m) to TMEM,
//                     then the epilogue O / l -> bf16 -> swizzled smem -> TMA store.
// TMEM: S_A [0,128) S_B [128,256) O_A [256,384) O_B [384,512) fp32 columns.
// When the GQA group is odd, neighbouring query heads may read different KV heads: each
// CTA then owns one query head (head B's columns, MMAs and softmax warps stay idle).
#include <cmath>

#include "attn_internal.h"
#include "attn_mask.cuh"
#include "common.h"
#include "device_common.cuh"
#include "sm100.cuh"
#include "tmap.h"

namespace tree {
using namespace sm100;

namespace tcfwd {

constexpr int BM = 128, BN = 128, D = 128;
constexpr int kThreads = 320;  // 8 softmax warps, TMA warp, MMA warp
constexpr int kWarpProducer = 8, kWarpMma = 9;
constexpr uint32_t kSub = 128 * 128;   // 128 rows x 128 B (64 bf16): one swizzle-128 sub-tile
constexpr uint32_t kTile = 2 * kSub;   // 128 rows x 128 bf16
constexpr float kRescaleLog2 = 8.0f;   // rescale O only when the row max grows by > 2^8

struct Smem {
  uint8_t q[2][kTile];
  uint8_t k[2][kTile];
  uint8_t v[2][kTile];
  uint64_t q_full, k_full[2], v_full[2], kv_empty[2], s_full[2], p_full[2], o_done[2], mma_done;
  uint32_t tmem_base;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

struct Params {
  int T, Hq, Hkv, n_qt;  // T: key rows
  int nh;                // query heads per CTA: 2 (even GQA group), or 1 (odd group: head B idles)
  int Tq, q_off, n_kt;   // query rows, key rows before the first query, key tiles
  float scale_log2;
  const int32_t* kmax;
  const int32_t* kmin;
  const int32_t* kmax32;  // per 32-key chunk: max and min subtree_end (ceil(T / 32) entries)
  const int32_t* kmin32;
  const int32_t* endp;  // subtree_end padded with -1 to a multiple of 128
  float* lse;
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

// 2^x on the SFU (ex2.approx.ftz: ~2 ulp, flushes subnormal results to zero).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO, Params p) {
  extern __shared__ uint8_t smem_raw[];
  // A CTA that finds a timeout already reported does no work: one lost arrival must
  // not make every later CTA wait out its own limits.
  if (p.err && (*reinterpret_cast<volatile int*>(p.err) & (1 << TREE_ERR_TIMEOUT))) return;
  Smem& S = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int h0 = p.nh * blockIdx.x;
  const int qt = p.n_qt - 1 - blockIdx.y;  // longest query tiles first
  const int i0 = qt * BM;                  // first query row of the tile (query buffers)
  const int iq0 = p.q_off + i0;            // the same row among the keys
  const int kt_hi = min((iq0 + BM - 1) / BN, p.n_kt - 1);  // last key tile before the tile's last query
  const int kvh = h0 / (p.Hq / p.Hkv);

  if (threadIdx.x == 0) {
    mbar_init(&S.q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.k_full[s], 1);
      mbar_init(&S.v_full[s], 1);
      mbar_init(&S.kv_empty[s], 1);
      mbar_init(&S.s_full[s], 1);
      mbar_init(&S.p_full[s], 4);
      mbar_init(&S.o_done[s], 1);
    }
    mbar_init(&S.mma_done, 1);
    fence_mbarrier_init();
  }
  if (warp == kWarpMma) tmem_alloc(&S.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == kWarpProducer) {
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      mbar_arrive_expect_tx(&S.q_full, p.nh * kTile);
      for (int hh = 0; hh < p.nh; ++hh)
        for (int sub = 0; sub < 2; ++sub) tma_load_3d(S.q[hh] + sub * kSub, &tmQ, &S.q_full, sub * 64, h0 + hh, i0);
      int n = 0;
      for (int kt = 0; kt <= kt_hi; ++kt) {
        if (p.kmax[kt] < iq0) continue;
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
      // Leave no copy in flight: wait for the loads of the last (up to) two tiles.
      for (int m = (n >= 2 ? n - 2 : 0); m < n; ++m) {
        mbar_wait(&S.k_full[m & 1], (m >> 1) & 1, p.err);
        mbar_wait(&S.v_full[m & 1], (m >> 1) & 1, p.err);
      }
    }
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16(BM, D, 0, 1);
      auto issue_s = [&](int h, int s) {
        const uint32_t qa = smem_u32(S.q[h]), kb = smem_u32(S.k[s]);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kSub + (kk & 3) * 32;
          mma_ss(tmem + h * 128, desc_sw128(qa + off, 16, 1024), desc_sw128(kb + off, 16, 1024), idesc_qk,
                 kk > 0);
        }
        mma_commit(&S.s_full[h]);
      };
      auto issue_pv = [&](int h, int s, int n) {
        const uint32_t vb = smem_u32(S.v[s]);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(tmem + 256 + h * 128, tmem + h * 128 + kk * 8, desc_sw128(vb + kk * 2048, kSub, 1024),
                 idesc_pv, (n > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&S.o_done[h]);
      };
      int N = 0;
      for (int kt = 0; kt <= kt_hi; ++kt) N += p.kmax[kt] >= iq0;
      bool ok = N > 0 && mbar_wait(&S.q_full, 0, p.err) && mbar_wait(&S.k_full[0], 0, p.err);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        if (p.nh == 2) issue_s(1, 0);
      }
      for (int n = 0; ok && n < N; ++n) {
        const int s = n & 1;
        if (!(ok = mbar_wait(&S.p_full[0], n & 1, p.err) && mbar_wait(&S.v_full[s], (n >> 1) & 1, p.err))) break;
        tc_fence_after();
        issue_pv(0, s, n);
        const bool more = n + 1 < N;
        if (more) {
          if (!(ok = mbar_wait(&S.k_full[s ^ 1], ((n + 1) >> 1) & 1, p.err))) break;
          tc_fence_after();
          issue_s(0, s ^ 1);
        }
        if (p.nh == 2) {
          if (!(ok = mbar_wait(&S.p_full[1], n & 1, p.err))) break;
          tc_fence_after();
          issue_pv(1, s, n);
        }
        mma_commit(&S.kv_empty[s]);
        if (more && p.nh == 2) issue_s(1, s ^ 1);
      }
      mma_commit(&S.mma_done);
      mbar_wait(&S.mma_done, 0, p.err);
    }
    __syncwarp();
  } else if (warp < 4 * p.nh) {
    // ------------------------------------------------------------ softmax warps
    const int h = warp >> 2, q4 = warp & 3;
    const int r = q4 * 32 + lane, ik = iq0 + r;  // the thread's query row, as a key row
    const uint32_t lanes = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t tS = tmem + lanes + h * 128, tO = tmem + lanes + 256 + h * 128;
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY, l = 0.f;
    int n = 0;
    bool ok = true;
    const float rescale_raw = kRescaleLog2 / sl2;  // the 2^8 threshold in raw score units
    for (int kt = 0; kt <= kt_hi; ++kt) {
      if (p.kmax[kt] < iq0) continue;
      const int j0 = kt * BN;
      const bool partial = !(j0 + BN - 1 <= iq0 && p.kmin[kt] >= iq0 + BM - 1);
      // visibility bits of this row's 128 keys, formed while the MMA of S runs. A 32-key
      // chunk lying wholly at or before the row, whose smallest subtree_end reaches the row,
      // is visible whole; one after the row, or whose largest subtree_end stops short of
      // it, is hidden whole; only the rest is tested key by key.
      uint32_t vis[4] = {~0u, ~0u, ~0u, ~0u};
      if (partial) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int jb = j0 + 32 * c;
          if (jb >= p.T || ik < jb) {
            vis[c] = 0u;
          } else {
            const int kx = __ldg(p.kmax32 + (jb >> 5)), kn = __ldg(p.kmin32 + (jb >> 5));
            if (ik > kx) vis[c] = 0u;
            else if (jb + 31 <= ik && ik <= kn) vis[c] = ~0u;
            else vis[c] = visible32(p.endp, jb, ik);
          }
        }
      }
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&S.s_full[h], n & 1, p.err)))) break;
      tc_fence_after();
      // one pass over the row's 128 scores: all four TMEM loads in flight, one wait
      uint32_t sr[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
      tmem_ld_wait();
      if (partial && (vis[0] & vis[1] & vis[2] & vis[3]) != ~0u) {
#pragma unroll
        for (int t = 0; t < 128; ++t)
          if (!((vis[t >> 5] >> (t & 31)) & 1u)) sr[t] = 0xff800000u;  // -inf: p = 0
      }
      // row max with eight independent chains (short dependency chains, not one of 128)
      float m8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) m8[u] = __uint_as_float(sr[u]);
#pragma unroll
      for (int t = 8; t < 128; ++t) m8[t & 7] = fmaxf(m8[t & 7], __uint_as_float(sr[t]));
      const float mt = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      // lazy rescaling (raw score units): move the running max only when it grows by > 2^8
      float new_m = m_run;
      bool need = false;
      if (mt > m_run + rescale_raw) {
        new_m = mt;
        need = m_run != -INFINITY;
      }
      const float corr = need ? ex2_approx((m_run - new_m) * sl2) : 1.f;
      if (need) l *= corr;
      m_run = new_m;
      // p = 2^(s * scale * log2(e) - m2): one packed FFMA and one ex2 per score
      const float m2 = m_run == -INFINITY ? 0.f : m_run * sl2;
      const float2 scl = make_float2(sl2, sl2), off = make_float2(-m2, -m2);
      float2 ls[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int t = 0; t < 64; ++t) {
        const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[2 * t]), __uint_as_float(sr[2 * t + 1])), scl, off);
        const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        ls[t & 3] = __fadd2_rn(ls[t & 3], pp);
        sr[t] = pack_bf16(pp.x, pp.y);  // P packed over the front half (already consumed)
      }
      const float2 lsum = __fadd2_rn(__fadd2_rn(ls[0], ls[1]), __fadd2_rn(ls[2], ls[3]));
      l += lsum.x + lsum.y;
      tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      // rescale O (after PV of the previous tile completed) before PV of this tile is issued
      if (__any_sync(0xffffffffu, need)) {
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&S.o_done[h], (n - 1) & 1, p.err)))) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * corr);
          tmem_st32(tO + c * 32, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.p_full[h]);
      ++n;
    }
    if (ok && n > 0) ok = mbar_wait(&S.o_done[h], (n - 1) & 1, p.err);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    // epilogue: O / l -> bf16 -> swizzled staging (this head's Q buffer) -> TMA store.
    // Every warp of the group reaches the named barrier; a warp whose waits gave up
    // (error already flagged) writes nothing.
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    uint8_t* stage = S.q[h];
    if (ok) {
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 32; t += 2)
          pk[t / 2] = pack_bf16(__uint_as_float(o[t]) * inv_l, __uint_as_float(o[t + 1]) * inv_l);
        uint8_t* row = stage + (c >> 1) * kSub + r * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int chunk = ((c & 1) * 4 + u) ^ (r & 7);
          *reinterpret_cast<uint4*>(row + chunk * 16) = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
      const int i = i0 + r;
      if (i < p.Tq) p.lse[static_cast<int64_t>(h0 + h) * p.Tq + i] = (m_run * sl2 + log2f(l)) * 0.6931471805599453f;
    }
    fence_proxy_async_smem();
    asm volatile("bar.sync %0, 128;" ::"r"(1 + h) : "memory");
    if (q4 == 0 && lane == 0) {
      tma_store_3d(&tmO, stage, 0, h0 + h, i0);
      tma_store_3d(&tmO, stage + kSub, 64, h0 + h, i0);
      bulk_commit();
      bulk_wait_read0();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace tcfwd

// Per 128-key tile: max / min subtree_end, plus subtree_end padded with -1.
__global__ void tile_meta128_kernel(const int32_t* __restrict__ end, int64_t n, int32_t* __restrict__ kmax,
                                    int32_t* __restrict__ kmin, int32_t* __restrict__ kmax32,
                                    int32_t* __restrict__ kmin32, int32_t* __restrict__ endp, int* err) {
  __shared__ int smax[4], smin[4];
  const int64_t j = static_cast<int64_t>(blockIdx.x) * 128 + threadIdx.x;
  const bool in = j < n;
  const int e = in ? end[j] : -1;
  if (in && (e < j || e >= n)) raise_error(err, TREE_ERR_DEVICE_CHECK);
  endp[j] = e;
  int mx = in ? e : -1, mn = in ? e : INT32_MAX;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  }
  if (threadIdx.x % 32 == 0) {
    smax[threadIdx.x / 32] = mx;
    smin[threadIdx.x / 32] = mn;
    if (in) {  // this warp's 32-key chunk starts inside the tree
      kmax32[j / 32] = mx;
      kmin32[j / 32] = mn;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    kmax[blockIdx.x] = max(max(smax[0], smax[1]), max(smax[2], smax[3]));
    kmin[blockIdx.x] = min(min(smin[0], smin[1]), min(smin[2], smin[3]));
  }
}

int tile_meta128_launch(const AttnArgs& a, cudaStream_t st) {
  const int64_t n_tiles = (a.T + 127) / 128;
  tile_meta128_kernel<<<static_cast<unsigned>(n_tiles), 128, 0, st>>>(
      a.end, a.T, a.ws.kmax128, a.ws.kmin128, a.ws.kmax32, a.ws.kmin32, a.ws.end_pad, device_error_word());
  TREE_LAUNCH_CHECK("tile_meta128_kernel");
  return TREE_OK;
}

// [T, H, 128] bf16 as a 3-D tensor map {d, H, T}, box {64, 1, 128}, 128-byte swizzle.
static int qkv_map(CUtensorMap* m, const void* base, int64_t T, int H) {
  const uint64_t dims[3] = {128, static_cast<uint64_t>(H), static_cast<uint64_t>(T)};
  const uint64_t strides[2] = {128 * 2, static_cast<uint64_t>(H) * 128 * 2};
  const uint32_t box[3] = {64, 1, 128};
  return make_tmap(m, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, dims, strides, box, true);
}

bool attn_fwd_tc_supported(int dtype, int d, int Hq, int Hkv) {
  (void)Hq;  // an odd GQA group runs one query head per CTA
  (void)Hkv;
  return dtype == TREE_DTYPE_BF16 && d == 128;
}

int attn_fwd_tc(const AttnArgs& a, cudaStream_t st) {
  using namespace tcfwd;
  int rc = tile_meta128_launch(a, st);
  if (rc) return rc;
  const int64_t Tq = a.T - a.q_off;  // queries: the last Tq key rows
  CUtensorMap mq, mk, mv, mo;
  if ((rc = qkv_map(&mq, a.q, Tq, a.Hq)) || (rc = qkv_map(&mk, a.k, a.T, a.Hkv)) ||
      (rc = qkv_map(&mv, a.v, a.T, a.Hkv)) || (rc = qkv_map(&mo, a.o, Tq, a.Hq)))
    return rc;
  if (int rc_ = smem_opt_in(reinterpret_cast<const void*>(attn_fwd_tc_kernel), static_cast<int>(kSmemBytes))) return rc_;
  Params p{};
  p.T = static_cast<int>(a.T);
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Tq = static_cast<int>(Tq);
  p.q_off = static_cast<int>(a.q_off);
  p.n_qt = static_cast<int>((Tq + BM - 1) / BM);
  p.n_kt = static_cast<int>((a.T + BN - 1) / BN);
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.kmax = a.ws.kmax128;
  p.kmin = a.ws.kmin128;
  p.kmax32 = a.ws.kmax32;
  p.kmin32 = a.ws.kmin32;
  p.endp = a.ws.end_pad;
  p.lse = a.lse;
  p.err = device_error_word();
  p.nh = (a.Hq / a.Hkv) % 2 == 0 ? 2 : 1;
  dim3 grid(a.Hq / p.nh, p.n_qt);
  timing_begin(0, st);
  attn_fwd_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(mq, mk, mv, mo, p);
  TREE_LAUNCH_CHECK("attn_fwd_tc_kernel");
  timing_end(0, st);
  return TREE_OK;
}

}  // namespace tree
