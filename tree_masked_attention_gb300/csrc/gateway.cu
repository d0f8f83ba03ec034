// tree_attn_fwd_gateway / tree_attn_bwd_gateway: attention of a child partition through
// its partition gateway.
//
// Tree Training (arXiv 2511.00413) §3.3 "Differentiable partition boundaries" and
// Appendix B.2-B.5: a child partition C runs on its own rows and attends to the keys and
// values its parent partition accumulated up to the cut node (the past), under an
// additive bias that is 0 at the cut node's ancestors and -inf elsewhere (eq. 15-16),
// combined with the ordinary tree mask inside C (eq. 14). Gradients reaching the past
// keys and values from several child partitions are summed in fp32 (B.5).
//
// The tensor-core kernels run unchanged on one key space: the past rows [0, P) followed
// by C's rows [P, P + T), with C's queries at key rows P..P+T-1. The interval rule
// (key j visible to query i iff j <= i <= subtree_end[j]) expresses eq. 14 exactly:
//   past key j, bias 0     -> subtree_end = P + T - 1 (visible to every query of C)
//   past key j, bias -inf  -> subtree_end = j         (no query of C lies in [j, j])
//   own key P + j          -> subtree_end = P + subtree_end_C[j]
// This kernel writes that array into the workspace; the forward's tile metadata and the
// backward's planner then read it in place.
#include <cmath>

#include "attn_internal.h"
#include "common.h"
#include "device_common.cuh"

namespace tree {

__global__ void gateway_end_kernel(const float* __restrict__ bias, const int32_t* __restrict__ child_end,
                                   int64_t P, int64_t T, int32_t* __restrict__ out, int* err) {
  const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j >= P + T) return;
  int64_t e;
  if (j < P) {
    const float b = bias[j];
    if (b == 0.f) {
      e = P + T - 1;
    } else {
      if (!(isinf(b) && b < 0.f)) raise_error(err, TREE_ERR_DEVICE_CHECK);  // eq. 16: 0 or -inf only
      e = j;
    }
  } else {
    const int64_t r = j - P;
    int64_t c = child_end[r];
    if (c < r || c >= T) {  // not a preorder subtree interval: report, keep the row to itself
      raise_error(err, TREE_ERR_DEVICE_CHECK);
      c = r;
    }
    e = P + c;
  }
  out[j] = static_cast<int32_t>(e);
}

namespace {

int check_gateway(const char* who, int64_t P, int64_t T, int Hq, int Hkv, int d, int dtype, bool bwd) {
  if (dtype != TREE_DTYPE_BF16 && dtype != TREE_DTYPE_F32) return fail(TREE_ERR_DTYPE, "%s: bad dtype %d", who, dtype);
  if (P < 0 || T < 1 || P + T > INT32_MAX - 256)
    return fail(TREE_ERR_SHAPE, "%s: past_len = %lld, T = %lld", who, (long long)P, (long long)T);
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Hq > 65535)
    return fail(TREE_ERR_SHAPE, "%s: Hq = %d, Hkv = %d", who, Hq, Hkv);
  const bool tc = bwd ? attn_bwd_tc_supported(dtype, d, 0) && attn_fwd_tc_supported(dtype, d, Hq, Hkv)
                      : attn_fwd_tc_supported(dtype, d, Hq, Hkv);
  if (!tc)
    return fail(dtype == TREE_DTYPE_BF16 ? TREE_ERR_SHAPE : TREE_ERR_DTYPE,
                "%s: gateway attention runs on the tensor-core kernels: bf16, d = 128", who);
  return TREE_OK;
}

int gateway_end(const float* bias, const int32_t* child_end, int64_t P, int64_t T, int32_t* out, cudaStream_t st) {
  const int64_t n = P + T;
  gateway_end_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(bias, child_end, P, T, out,
                                                                           device_error_word());
  TREE_LAUNCH_CHECK("gateway_end_kernel");
  return TREE_OK;
}

}  // namespace
}  // namespace tree

using namespace tree;

extern "C" size_t tree_attn_gateway_workspace_size(int64_t past_len, int64_t T, int Hq, int Hkv, int d, int dtype) {
  if (past_len < 0 || T < 1 || Hq < 1 || d < 1) return 0;
  return attn_ws_layout(past_len + T, Hq, Hkv, d, dtype, nullptr, nullptr);
}

extern "C" int tree_attn_fwd_gateway(const void* q, const void* k, const void* v, void* o, float* lse,
                                     const float* attn_bias, const int32_t* subtree_end, int64_t past_len,
                                     int64_t T, int Hq, int Hkv, int d, int dtype, float softmax_scale,
                                     void* workspace, size_t workspace_bytes, tree_stream_t stream) {
  clear_error();
  int rc = check_gateway("tree_attn_fwd_gateway", past_len, T, Hq, Hkv, d, dtype, false);
  if (rc) return rc;
  if (!q || !k || !v || !o || !lse || !subtree_end || (past_len > 0 && !attn_bias))
    return fail(TREE_ERR_INVALID_ARG, "tree_attn_fwd_gateway: null pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(TREE_ERR_ALIGNMENT, "tree_attn_fwd_gateway: q/k/v/o not 16-byte aligned");
  const int64_t Tk = past_len + T;
  const size_t need = attn_ws_layout(Tk, Hq, Hkv, d, dtype, nullptr, nullptr);
  if (workspace_bytes < need)
    return fail(TREE_ERR_WORKSPACE, "tree_attn_fwd_gateway: workspace of %zu bytes, %zu needed", workspace_bytes, need);
  if (!workspace || !aligned256(workspace))
    return fail(TREE_ERR_ALIGNMENT, "tree_attn_fwd_gateway: workspace null or not 256-byte aligned");
  AttnArgs a{};
  attn_ws_layout(Tk, Hq, Hkv, d, dtype, workspace, &a.ws);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if ((rc = gateway_end(attn_bias, subtree_end, past_len, T, a.ws.end_pad, st))) return rc;
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
  a.end = a.ws.end_pad;  // read in place by the tile metadata kernel
  a.T = Tk; a.q_off = past_len; a.Hq = Hq; a.Hkv = Hkv; a.d = d; a.dtype = dtype;
  a.scale = softmax_scale > 0.f ? softmax_scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  return attn_fwd_tc(a, st);
}

extern "C" int tree_attn_bwd_gateway(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                     const float* lse, void* dq, void* dk, void* dv, float* dk_past, float* dv_past,
                                     const float* attn_bias, const int32_t* subtree_end, int64_t past_len, int64_t T,
                                     int Hq, int Hkv, int d, int dtype, float softmax_scale, void* workspace,
                                     size_t workspace_bytes, tree_stream_t stream) {
  clear_error();
  int rc = check_gateway("tree_attn_bwd_gateway", past_len, T, Hq, Hkv, d, dtype, true);
  if (rc) return rc;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !subtree_end ||
      (past_len > 0 && (!attn_bias || !dk_past || !dv_past)))
    return fail(TREE_ERR_INVALID_ARG, "tree_attn_bwd_gateway: null pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || (past_len > 0 && (!aligned16(dk_past) || !aligned16(dv_past))))
    return fail(TREE_ERR_ALIGNMENT, "tree_attn_bwd_gateway: tensors not 16-byte aligned");
  const int64_t Tk = past_len + T;
  const size_t need = attn_ws_layout(Tk, Hq, Hkv, d, dtype, nullptr, nullptr);
  if (workspace_bytes < need)
    return fail(TREE_ERR_WORKSPACE, "tree_attn_bwd_gateway: workspace of %zu bytes, %zu needed", workspace_bytes, need);
  if (!workspace || !aligned256(workspace))
    return fail(TREE_ERR_ALIGNMENT, "tree_attn_bwd_gateway: workspace null or not 256-byte aligned");
  AttnArgs a{};
  attn_ws_layout(Tk, Hq, Hkv, d, dtype, workspace, &a.ws);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if ((rc = gateway_end(attn_bias, subtree_end, past_len, T, a.ws.end_pad, st))) return rc;
  a.q = q; a.k = k; a.v = v; a.o = const_cast<void*>(o); a.lse = const_cast<float*>(lse);
  a.dout = dout; a.dq = dq; a.dk = dk; a.dv = dv; a.dk_past = dk_past; a.dv_past = dv_past;
  a.end = a.ws.end_pad;  // read in place by the backward's planner
  a.T = Tk; a.q_off = past_len; a.Hq = Hq; a.Hkv = Hkv; a.d = d; a.dtype = dtype;
  a.scale = softmax_scale > 0.f ? softmax_scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  return attn_bwd_tc(a, st);
}
