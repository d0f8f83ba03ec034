// The C ABI (include/tree_attn.h): argument checks, workspace carve-up and dispatch
// to the kernel families. Nothing here allocates device memory.
#include <cuda_runtime.h>

#include <cmath>

#include "attn_internal.h"
#include "common.h"

namespace tree {

namespace {

struct Carver {
  char* base;
  size_t off = 0;
  template <typename T>
  T* take(size_t count) {
    off = round_up(off, 256);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

bool dtype_ok(int dtype) { return dtype == TREE_DTYPE_F32 || dtype == TREE_DTYPE_BF16; }

}  // namespace

size_t attn_ws_layout(int64_t T, int Hq, int Hkv, int d, int dtype, void* base, AttnWs* ws) {
  (void)dtype;
  Carver c{static_cast<char*>(base)};
  AttnWs w{};
  const size_t t32 = static_cast<size_t>((T + 31) / 32), t128 = static_cast<size_t>((T + 127) / 128);
  w.kmax32 = c.take<int32_t>(t32);
  w.kmin32 = c.take<int32_t>(t32);
  w.kmax128 = c.take<int32_t>(t128);
  w.kmin128 = c.take<int32_t>(t128);
  w.end_pad = c.take<int32_t>(t128 * 128);
  w.delta = c.take<float>(static_cast<size_t>(Hq) * T);
  w.dq_acc = c.take<float>(static_cast<size_t>(T) * Hq * d);
  const size_t t_pad = static_cast<size_t>((T + 63) / 64 * 64);
  w.lse2_pad = c.take<float>(static_cast<size_t>(Hq) * t_pad);
  w.delta_pad = c.take<float>(static_cast<size_t>(Hq) * t_pad);
  w.dk_acc = c.take<float>(static_cast<size_t>(T) * Hkv * d);
  w.dv_acc = c.take<float>(static_cast<size_t>(T) * Hkv * d);
  w.units = c.take<int32_t>(static_cast<size_t>(attn_bwd_max_units(T, Hkv)) * 4);
  w.n_units = c.take<int32_t>(1);
  w.counter = c.take<int32_t>(1);
  w.bucket = c.take<int32_t>(static_cast<size_t>((T + 63) / 64) + 1);
  if (ws) *ws = w;
  return round_up(c.off, 256);
}

size_t logprob_ws_layout(int64_t T, int64_t K, int64_t V, int64_t n_occ, int dtype, void* base, LogprobWs* ws) {
  (void)K;
  (void)dtype;
  Carver c{static_cast<char*>(base)};
  LogprobWs w{};
  const size_t n_vt = static_cast<size_t>((V + 63) / 64);
  w.part_max = c.take<float>(n_vt * T);
  w.part_sum = c.take<float>(n_vt * T);
  w.crow = c.take<float>(static_cast<size_t>(T));
  w.gz = c.take<float>(static_cast<size_t>(T) * V);
  w.occ_delta = c.take<float>(static_cast<size_t>(n_occ) + 1);
  w.blk_ptr = c.take<int32_t>(static_cast<size_t>((V + 255) / 256) + 1);
  w.blk_ent = c.take<int32_t>(2 * static_cast<size_t>(n_occ) + 2);
  if (ws) *ws = w;
  return round_up(c.off, 256);
}

static int check_attn_shape(int64_t T, int Hq, int Hkv, int d, int dtype) {
  if (!dtype_ok(dtype)) return fail(TREE_ERR_DTYPE, "dtype %d is not TREE_DTYPE_F32/BF16", dtype);
  if (T < 1 || T > INT32_MAX - 256) return fail(TREE_ERR_SHAPE, "T = %lld outside [1, 2^31)", (long long)T);
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Hq > 65535)
    return fail(TREE_ERR_SHAPE, "Hq = %d, Hkv = %d: need Hkv >= 1, Hq %% Hkv == 0, Hq <= 65535", Hq, Hkv);
  if (d != 64 && d != 128) return fail(TREE_ERR_SHAPE, "head size %d: supported 64, 128", d);
  return TREE_OK;
}

static int check_ws(void* ws, size_t have, size_t need) {
  if (need > have) return fail(TREE_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", have, need);
  if (!ws) return fail(TREE_ERR_INVALID_ARG, "workspace is null");
  if (!aligned256(ws)) return fail(TREE_ERR_ALIGNMENT, "workspace not 256-byte aligned");
  return TREE_OK;
}

}  // namespace tree

using namespace tree;

extern "C" int tree_rope(void* q, void* k, const int32_t* position_ids, int64_t T, int Hq, int Hkv, int d,
                         float theta_base, int dtype, int inverse, tree_stream_t stream) {
  clear_error();
  if (!dtype_ok(dtype)) return fail(TREE_ERR_DTYPE, "tree_rope: bad dtype %d", dtype);
  if (T < 0 || Hq < 0 || Hkv < 0 || d < 2 || d > 256 || d % 2)
    return fail(TREE_ERR_SHAPE, "tree_rope: T=%lld Hq=%d Hkv=%d d=%d", (long long)T, Hq, Hkv, d);
  if (!(theta_base > 1.f) || !std::isfinite(theta_base))
    return fail(TREE_ERR_INVALID_ARG, "tree_rope: theta_base must be finite and > 1");
  if (T == 0 || (!q && !k)) return TREE_OK;
  if (!position_ids) return fail(TREE_ERR_INVALID_ARG, "tree_rope: position_ids is null");
  if ((q && !aligned16(q)) || (k && !aligned16(k)))
    return fail(TREE_ERR_ALIGNMENT, "tree_rope: q/k not 16-byte aligned");
  return rope_launch(q, k, position_ids, T, Hq, Hkv, d, theta_base, dtype, inverse,
                     reinterpret_cast<cudaStream_t>(stream));
}

extern "C" size_t tree_attn_workspace_size(int64_t T, int Hq, int Hkv, int d, int dtype) {
  if (T < 1 || Hq < 1 || d < 1) return 0;
  return attn_ws_layout(T, Hq, Hkv, d, dtype, nullptr, nullptr);
}

extern "C" int tree_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                             const int32_t* subtree_end, int64_t T, int Hq, int Hkv, int d, int dtype,
                             float softmax_scale, void* workspace, size_t workspace_bytes,
                             tree_stream_t stream) {
  clear_error();
  int rc = check_attn_shape(T, Hq, Hkv, d, dtype);
  if (rc) return rc;
  if (!q || !k || !v || !o || !lse || !subtree_end)
    return fail(TREE_ERR_INVALID_ARG, "tree_attn_fwd: null tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(TREE_ERR_ALIGNMENT, "tree_attn_fwd: q/k/v/o not 16-byte aligned");
  const size_t need = attn_ws_layout(T, Hq, Hkv, d, dtype, nullptr, nullptr);
  if ((rc = check_ws(workspace, workspace_bytes, need))) return rc;
  AttnArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse; a.end = subtree_end;
  a.T = T; a.Hq = Hq; a.Hkv = Hkv; a.d = d; a.dtype = dtype;
  a.scale = softmax_scale > 0.f ? softmax_scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  attn_ws_layout(T, Hq, Hkv, d, dtype, workspace, &a.ws);
  if (attn_fwd_tc_supported(dtype, d, Hq, Hkv)) return attn_fwd_tc(a, reinterpret_cast<cudaStream_t>(stream));
  if (attn_tc32_supported(dtype, d)) return attn_fwd_tc32(a, reinterpret_cast<cudaStream_t>(stream));
  return attn_fwd_simt(a, reinterpret_cast<cudaStream_t>(stream));
}

static int attn_bwd_common(const char* name, const void* q, const void* k, const void* v, const void* o,
                           const void* dout, const float* lse, void* dq, void* dk, void* dv,
                           const int32_t* subtree_end, int64_t T, int Hq, int Hkv, int d, int dtype,
                           float softmax_scale, int deterministic, const int32_t* rope_pos, float rope_theta,
                           void* workspace, size_t workspace_bytes, tree_stream_t stream) {
  clear_error();
  int rc = check_attn_shape(T, Hq, Hkv, d, dtype);
  if (rc) return rc;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !subtree_end)
    return fail(TREE_ERR_INVALID_ARG, "%s: null tensor pointer", name);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(TREE_ERR_ALIGNMENT, "%s: tensors not 16-byte aligned", name);
  if (deterministic != 0 && deterministic != 1)
    return fail(TREE_ERR_INVALID_ARG, "%s: deterministic must be 0 or 1", name);
  const size_t need = attn_ws_layout(T, Hq, Hkv, d, dtype, nullptr, nullptr);
  if ((rc = check_ws(workspace, workspace_bytes, need))) return rc;
  AttnArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = const_cast<void*>(o); a.lse = const_cast<float*>(lse);
  a.dout = dout; a.dq = dq; a.dk = dk; a.dv = dv; a.end = subtree_end;
  a.T = T; a.Hq = Hq; a.Hkv = Hkv; a.d = d; a.dtype = dtype; a.deterministic = deterministic;
  a.scale = softmax_scale > 0.f ? softmax_scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  attn_ws_layout(T, Hq, Hkv, d, dtype, workspace, &a.ws);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (attn_bwd_tc_supported(dtype, d, deterministic)) {
    a.rope_pos = rope_pos;  // fused into the conversion of the fp32 sums
    a.rope_theta = rope_theta;
    return attn_bwd_tc(a, st);
  }
  if ((rc = attn_tc32_supported(dtype, d) ? attn_bwd_tc32(a, st) : attn_bwd_simt(a, st)) || !rope_pos) return rc;
  return tree_rope(dq, dk, rope_pos, T, Hq, Hkv, d, rope_theta, dtype, 1, stream);
}

extern "C" int tree_attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                             const float* lse, void* dq, void* dk, void* dv, const int32_t* subtree_end,
                             int64_t T, int Hq, int Hkv, int d, int dtype, float softmax_scale,
                             int deterministic, void* workspace, size_t workspace_bytes,
                             tree_stream_t stream) {
  return attn_bwd_common("tree_attn_bwd", q, k, v, o, dout, lse, dq, dk, dv, subtree_end, T, Hq, Hkv, d, dtype,
                         softmax_scale, deterministic, nullptr, 0.f, workspace, workspace_bytes, stream);
}

extern "C" int tree_attn_bwd_rope(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                  const float* lse, void* dq, void* dk, void* dv, const int32_t* subtree_end,
                                  const int32_t* position_ids, int64_t T, int Hq, int Hkv, int d, int dtype,
                                  float softmax_scale, float theta_base, int deterministic, void* workspace,
                                  size_t workspace_bytes, tree_stream_t stream) {
  if (!position_ids) {
    clear_error();
    return fail(TREE_ERR_INVALID_ARG, "tree_attn_bwd_rope: position_ids is null");
  }
  if (!(theta_base > 1.f) || !std::isfinite(theta_base)) {
    clear_error();
    return fail(TREE_ERR_INVALID_ARG, "tree_attn_bwd_rope: theta_base must be finite and > 1");
  }
  return attn_bwd_common("tree_attn_bwd_rope", q, k, v, o, dout, lse, dq, dk, dv, subtree_end, T, Hq, Hkv, d,
                         dtype, softmax_scale, deterministic, position_ids, theta_base, workspace,
                         workspace_bytes, stream);
}

static int check_lm(const void* h, const void* w, const int32_t* row_ptr, const int32_t* perm,
                    const int32_t* targets, int64_t T, int64_t K, int64_t V, int64_t n_occ, int dtype) {
  if (!dtype_ok(dtype)) return fail(TREE_ERR_DTYPE, "bad dtype %d", dtype);
  if (T < 1 || K < 1 || V < 1 || n_occ < 0 || T > INT32_MAX || n_occ > INT32_MAX || V > INT32_MAX)
    return fail(TREE_ERR_SHAPE, "T=%lld K_h=%lld V=%lld n_occ=%lld", (long long)T, (long long)K,
                (long long)V, (long long)n_occ);
  if (K % 64 || V % 8) return fail(TREE_ERR_SHAPE, "need K_h %% 64 == 0 and V %% 8 == 0 (K_h=%lld V=%lld)",
                                   (long long)K, (long long)V);
  if (!h || !w || !row_ptr || (n_occ > 0 && (!perm || !targets)))
    return fail(TREE_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(h) || !aligned16(w)) return fail(TREE_ERR_ALIGNMENT, "hidden / w_lm not 16-byte aligned");
  return TREE_OK;
}

extern "C" size_t tree_logprob_workspace_size(int64_t T, int64_t K_h, int64_t V, int64_t n_occ, int dtype) {
  if (T < 1 || K_h < 1 || V < 1 || n_occ < 0) return 0;
  return logprob_ws_layout(T, K_h, V, n_occ, dtype, nullptr, nullptr);
}

extern "C" int tree_logprob_fwd(const void* hidden, const void* w_lm, const int32_t* occ_row_ptr,
                                const int32_t* occ_perm, const int32_t* occ_targets, int64_t T, int64_t K_h,
                                int64_t V, int64_t n_occ, float* lse, float* logp, int dtype, void* workspace,
                                size_t workspace_bytes, tree_stream_t stream) {
  clear_error();
  int rc = check_lm(hidden, w_lm, occ_row_ptr, occ_perm, occ_targets, T, K_h, V, n_occ, dtype);
  if (rc) return rc;
  if (!lse || (n_occ > 0 && !logp)) return fail(TREE_ERR_INVALID_ARG, "tree_logprob_fwd: null output");
  const size_t need = logprob_ws_layout(T, K_h, V, n_occ, dtype, nullptr, nullptr);
  if ((rc = check_ws(workspace, workspace_bytes, need))) return rc;
  LogprobArgs a{};
  a.h = hidden; a.w = w_lm; a.row_ptr = occ_row_ptr; a.perm = occ_perm; a.targets = occ_targets;
  a.lse = lse; a.logp = logp; a.T = T; a.K = K_h; a.V = V; a.n_occ = n_occ; a.dtype = dtype;
  logprob_ws_layout(T, K_h, V, n_occ, dtype, workspace, &a.ws);
  if (logprob_tc_supported(dtype)) return logprob_fwd_tc(a, reinterpret_cast<cudaStream_t>(stream));
  return logprob_fwd_tc32(a, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int tree_logprob_bwd(const void* hidden, const void* w_lm, const float* lse,
                                const int32_t* occ_row_ptr, const int32_t* occ_perm,
                                const int32_t* occ_targets, const float* grad_logp, int64_t T, int64_t K_h,
                                int64_t V, int64_t n_occ, void* d_hidden, void* d_w, int dw_fp32, int dtype,
                                void* workspace, size_t workspace_bytes, tree_stream_t stream) {
  clear_error();
  int rc = check_lm(hidden, w_lm, occ_row_ptr, occ_perm, occ_targets, T, K_h, V, n_occ, dtype);
  if (rc) return rc;
  if (!lse || !d_hidden || !d_w || (n_occ > 0 && !grad_logp))
    return fail(TREE_ERR_INVALID_ARG, "tree_logprob_bwd: null pointer");
  if (dw_fp32 != 0 && dw_fp32 != 1) return fail(TREE_ERR_INVALID_ARG, "tree_logprob_bwd: dw_fp32 = %d", dw_fp32);
  if (!aligned16(d_hidden) || !aligned16(d_w))
    return fail(TREE_ERR_ALIGNMENT, "tree_logprob_bwd: d_hidden / d_w not 16-byte aligned");
  const size_t need = logprob_ws_layout(T, K_h, V, n_occ, dtype, nullptr, nullptr);
  if ((rc = check_ws(workspace, workspace_bytes, need))) return rc;
  LogprobArgs a{};
  a.h = hidden; a.w = w_lm; a.row_ptr = occ_row_ptr; a.perm = occ_perm; a.targets = occ_targets;
  a.grad = grad_logp; a.lse = const_cast<float*>(lse); a.dh = d_hidden; a.dw = d_w;
  a.T = T; a.K = K_h; a.V = V; a.n_occ = n_occ; a.dtype = dtype;
  a.dw_fp32 = dtype == TREE_DTYPE_F32 ? 1 : dw_fp32;
  logprob_ws_layout(T, K_h, V, n_occ, dtype, workspace, &a.ws);
  if (logprob_tc_supported(dtype)) return logprob_bwd_tc(a, reinterpret_cast<cudaStream_t>(stream));
  return logprob_bwd_tc32(a, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int tree_kernel_path(int op, int dtype, int d) {
  if (op == 0 || op == 1) {
    if (op == 0 ? attn_fwd_tc_supported(dtype, d, 2, 1) : attn_bwd_tc_supported(dtype, d, 0)) return 1;
    return attn_tc32_supported(dtype, d) ? 2 : 0;
  }
  if (op == 2 || op == 3) return logprob_tc_supported(dtype) ? 1 : 2;
  return 0;
}
