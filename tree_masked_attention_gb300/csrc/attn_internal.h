// Internal interface between the C ABI and the attention kernels.
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace tree {

// Scratch carved out of the caller's workspace (every region 256-byte aligned).
struct AttnWs {
  int32_t* kmax32;   // [ceil(T/32)]  per 32-key tile: max subtree_end
  int32_t* kmin32;   // [ceil(T/32)]  per 32-key tile: min subtree_end
  int32_t* kmax128;  // [ceil(T/128)] per 128-key tile: max subtree_end
  int32_t* kmin128;  // [ceil(T/128)] per 128-key tile: min subtree_end
  int32_t* end_pad;  // [ceil(T/128)*128] subtree_end, -1 past T
  float* delta;      // [Hq, T]       dO . O per query row and head
  float* dq_acc;     // [T, Hq, d]    fp32 dQ accumulator (tensor-core backward)
  float* lse2_pad;   // [Hq, T_pad]   LSE * log2(e), +inf past T (T_pad = T rounded up to 64)
  float* delta_pad;  // [Hq, T_pad]   dO . O, 0 past T
  float* dk_acc;     // [T, Hkv, d]   fp32 dK accumulator (tensor-core backward)
  float* dv_acc;     // [T, Hkv, d]   fp32 dV accumulator
  int32_t* units;    // [max_units * 4] backward work units {key tile, KV head, first step, end step}
  int32_t* n_units;  // [1]
  int32_t* counter;  // [1] next unit to hand out
  int32_t* bucket;   // [ceil(T/64) + 1] planner: units per first query tile
};

struct AttnArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;             // forward output / backward input
  float* lse;          // forward output / backward input, [Hq, T]
  const void* dout;
  void* dq;
  void* dk;
  void* dv;
  const int32_t* end;  // subtree_end [T]
  int64_t T;           // key rows; query rows are [q_off, T) of the same key space
  int64_t q_off;       // rows of keys before the first query (0 but for gateway calls)
  int Hq, Hkv, d, dtype;
  float scale;
  int deterministic;
  float* dk_past;      // gateway backward: fp32 [q_off, Hkv, d] sums the past keys' dK is added to
  float* dv_past;      // gateway backward: the same for dV
  const int32_t* rope_pos;  // backward only: when set, dq/dk get the inverse depth rotation
  float rope_theta;
  AttnWs ws;
};

// Bytes of workspace, and the carve-up of `base` when it is non-null.
size_t attn_ws_layout(int64_t T, int Hq, int Hkv, int d, int dtype, void* base, AttnWs* ws);

int tile_meta_launch(const int32_t* end, int64_t n, int tile, int32_t* kmax, int32_t* kmin,
                     cudaStream_t st);
// CUDA-core kernels: fp32 storage with head size 128, the one shape no tensor-core kernel serves
int attn_fwd_simt(const AttnArgs& a, cudaStream_t st);
int attn_bwd_simt(const AttnArgs& a, cudaStream_t st);

// tcgen05 kind::tf32 kernels with a two-term split (head size 64, fp32 or bf16 storage)
bool attn_tc32_supported(int dtype, int d);
int attn_fwd_tc32(const AttnArgs& a, cudaStream_t st);
int attn_bwd_tc32(const AttnArgs& a, cudaStream_t st);

// tcgen05 / TMA kernels (bf16, d = 128, even GQA group)
bool attn_fwd_tc_supported(int dtype, int d, int Hq, int Hkv);
int tile_meta128_launch(const AttnArgs& a, cudaStream_t st);
int attn_fwd_tc(const AttnArgs& a, cudaStream_t st);
bool attn_bwd_tc_supported(int dtype, int d, int deterministic);
int64_t attn_bwd_max_units(int64_t T, int Hkv);
int attn_bwd_tc(const AttnArgs& a, cudaStream_t st);

int rope_launch(void* q, void* k, const int32_t* pos, int64_t T, int Hq, int Hkv, int d,
                float theta_base, int dtype, int inverse, cudaStream_t st);

// ---- log-prob path ----
struct LogprobWs {
  float* part_max;   // [n_vtiles, T] per vocabulary tile: row max of the logits
  float* part_sum;   // [n_vtiles, T] per vocabulary tile: sum exp(z - max)
  float* crow;       // [T]           sum of grad_logp over the row's occurrences
  void* gz;          // [T, V]        G_z (fp32 on the fp32 path, bf16 on the bf16 path)
  float* occ_delta;  // [n_occ]       exact minus bf16-stored G_z at each occurrence's target cell
  int32_t* blk_ptr;  // [ceil(V/256)+1] occurrences grouped by 256-column target block
  int32_t* blk_ent;  // [2 * n_occ]   {source row, occurrence} per group entry
};

struct LogprobArgs {
  const void* h;
  const void* w;
  const int32_t* row_ptr;
  const int32_t* perm;
  const int32_t* targets;
  const float* grad;   // grad_logp (backward)
  float* lse;
  float* logp;
  void* dh;
  void* dw;
  int64_t T, K, V, n_occ;
  int dtype;
  int dw_fp32;         // backward: d_w in fp32 whatever dtype is
  LogprobWs ws;
};

size_t logprob_ws_layout(int64_t T, int64_t K, int64_t V, int64_t n_occ, int dtype, void* base, LogprobWs* ws);
// fp32: tcgen05 kind::tf32 GEMMs with a two-term split
int logprob_fwd_tc32(const LogprobArgs& a, cudaStream_t st);
int logprob_bwd_tc32(const LogprobArgs& a, cudaStream_t st);
int lse_combine_launch(const float* part_max, const float* part_sum, int n_tiles, int64_t T, const int32_t* row_ptr,
                       const int32_t* perm, int64_t n_occ, float* lse, float* logp, cudaStream_t st);
int row_grad_sum_launch(const int32_t* row_ptr, const int32_t* perm, const float* grad, int64_t T, int64_t n_occ,
                        float* crow, cudaStream_t st);
// bf16: the kind::f16 GEMM with fused epilogues
bool logprob_tc_supported(int dtype);
int logprob_fwd_tc(const LogprobArgs& a, cudaStream_t st);
int logprob_bwd_tc(const LogprobArgs& a, cudaStream_t st);

}  // namespace tree
