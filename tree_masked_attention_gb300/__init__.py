"""Tree-packed training hot path on GB300 (sm_103a): Python binding of libtreeattn.so.

Thin argument marshalling over the C ABI in include/tree_attn.h. Every step of
the path runs in the library's CUDA kernels (or, for tree_pack, its C++ host
code); PyTorch provides device memory and the current stream only. There is no
CPU fallback: calls raise when the library is missing or a tensor is not on a
CUDA device.

Functions (same names as the C ABI):
  tree_pack(seqs, seq_weights=None)                 -> dict of numpy arrays
  tree_rope(q, k, position_ids, theta_base, inverse) -> rotates q, k in place
  tree_attn_fwd(q, k, v, subtree_end, ...)          -> (o, lse)
  tree_attn_bwd(q, k, v, o, dout, lse, subtree_end, ...) -> (dq, dk, dv)
  tree_logprob_fwd(hidden, w_lm, occ_row_ptr, occ_perm, occ_targets, ...) -> (lse, logp)
  tree_logprob_bwd(hidden, w_lm, lse, occ_row_ptr, occ_perm, occ_targets, grad_logp, ...)
                                                    -> (d_hidden, d_w)
  tree_policy_loss(logp, old_logp, advantage, ...)  -> (loss, grad_logp, loss_sum)
  tree_attn_fwd_gateway(q, k, v, attn_bias, subtree_end) -> (o, lse)
  tree_attn_bwd_gateway(q, k, v, o, dout, lse, attn_bias, subtree_end, dk_past, dv_past)
                                                    -> (dq, dk, dv, dk_past, dv_past)
  tree_gdn_fwd(q, k, v, g, beta, node_start, node_end, node_parent) -> o
  tree_gdn_bwd(q, k, v, g, beta, dout, node_start, node_end, node_parent, saved=False)
                                                    -> (dq, dk, dv, dg, dbeta)
  tree_conv1d_fwd(x, w, parent_row, bias)           -> y
  tree_conv1d_bwd(x, w, dy, subtree_end, position_ids) -> (dx, dw, dbias)
"""
from __future__ import annotations

import ctypes as C

import numpy as np

from ._lib import PackOut, PackSizes, TreeError, check, lib

__all__ = [
    "tree_pack", "tree_validate_subtree_end", "tree_rope", "tree_attn_workspace_size",
    "tree_attn_fwd", "tree_attn_bwd", "tree_attn_bwd_rope", "tree_kernel_timing", "tree_kernel_last_ms", "tree_logprob_workspace_size", "tree_logprob_fwd", "tree_policy_loss",
    "tree_conv1d_fwd", "tree_conv1d_bwd", "tree_conv1d_workspace_size", "tree_attn_fwd_gateway",
    "tree_attn_bwd_gateway", "tree_attn_gateway_workspace_size", "tree_gdn_fwd", "tree_gdn_workspace_size",
    "tree_gdn_bwd", "tree_gdn_bwd_saved", "tree_gdn_bwd_workspace_size",
    "tree_logprob_bwd", "tree_check_device_status", "tree_kernel_path", "tree_launch_count", "TreeError", "lib",
    "DTYPE_F32", "DTYPE_BF16",
]

DTYPE_F32 = 0
DTYPE_BF16 = 1

_PACK_T = ("packed_ids", "position_ids", "subtree_end", "path_count", "parent_row", "node_of_token")
_PACK_NODE = ("node_start", "node_end", "node_parent")
_PACK_OCC = ("occ_source_rows", "occ_targets", "occ_seq", "occ_perm")


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(C.POINTER(ctype))


def tree_pack(seqs, seq_weights=None, fields=None) -> dict:
    """Pack host token sequences (iterables of ints) into a preorder trie.

    Returns numpy arrays named as in tree_pack_out (include/tree_attn.h), plus
    T, n_nodes, n_occ, n_roots and ``paths`` (packed rows of every sequence).
    ``fields`` (an iterable of those names, "paths" included) limits the arrays
    computed and returned to the ones named; the library skips the work of the rest.
    """
    L = lib()
    seqs = [np.asarray(s, dtype=np.int32).reshape(-1) for s in seqs]
    offs = np.zeros(len(seqs) + 1, dtype=np.int64)
    offs[1:] = np.cumsum([len(s) for s in seqs])
    toks = np.ascontiguousarray(np.concatenate(seqs) if seqs else np.zeros(0, np.int32), dtype=np.int32)
    plan = C.c_void_p()
    sizes = PackSizes()
    check(L.tree_pack_plan(_ptr(toks, C.c_int32), _ptr(offs, C.c_int64), len(seqs), C.byref(plan),
                           C.byref(sizes)), "tree_pack_plan")
    try:
        T, nn, no = sizes.T, sizes.n_nodes, sizes.n_occ
        res = {n: np.empty(T, np.int32) for n in _PACK_T}
        res.update({n: np.empty(nn, np.int32) for n in _PACK_NODE})
        res.update({n: np.empty(no, np.int32) for n in _PACK_OCC})
        res["occ_weights"] = np.empty(no, np.float32)
        res["occ_row_ptr"] = np.empty(T + 1, np.int32)
        res["token_rows"] = np.empty(sizes.n_tokens, np.int32)
        if fields is not None:
            want = set(fields)
            unknown = want - set(res) - {"paths"}
            if unknown:
                raise ValueError(f"tree_pack: unknown fields {sorted(unknown)}")
            if "paths" in want:
                want.add("token_rows")
            res = {n: a for n, a in res.items() if n in want}
        out = PackOut()
        for name, _ in PackOut._fields_:
            if name in res:
                setattr(out, name, _ptr(res[name], C.c_float if name == "occ_weights" else C.c_int32))
        w = None
        if seq_weights is not None:
            w = np.ascontiguousarray(seq_weights, dtype=np.float32)
            if w.shape != (len(seqs),):
                raise ValueError("seq_weights must have one entry per sequence")
        check(L.tree_pack_emit(plan, _ptr(w, C.c_float) if w is not None else None, C.byref(out)),
              "tree_pack_emit")
    finally:
        L.tree_plan_free(plan)
    res.update(T=T, n_nodes=nn, n_occ=no, n_roots=sizes.n_roots)
    if "token_rows" in res:
        res["paths"] = [res["token_rows"][offs[k]:offs[k + 1]] for k in range(len(seqs))]
    return res


def tree_validate_subtree_end(subtree_end) -> None:
    a = np.ascontiguousarray(subtree_end, dtype=np.int32)
    check(lib().tree_validate_subtree_end(_ptr(a, C.c_int32), a.size), "tree_validate_subtree_end")


# ---------------------------------------------------------------- device calls
def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}: bfloat16 or float32")


def _dev(t, name, dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return C.c_void_p(t.data_ptr())


def _stream(t):
    torch = _torch()
    return C.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _workspace(nbytes, device, workspace):
    torch = _torch()
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError(f"workspace too small: {nbytes} bytes needed")
        return workspace
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def tree_rope(q, k, position_ids, theta_base: float = 10000.0, inverse: bool = False) -> None:
    """Rotate q [T,Hq,d] and k [T,Hkv,d] in place by depth positions (int32 [T])."""
    torch = _torch()
    ref = q if q is not None else k
    T, d = ref.shape[0], ref.shape[2]
    Hq = q.shape[1] if q is not None else 0
    Hkv = k.shape[1] if k is not None else 0
    check(lib().tree_rope(_dev(q, "q", ref.dtype), _dev(k, "k", ref.dtype),
                          _dev(position_ids, "position_ids", torch.int32), T, Hq, Hkv, d,
                          float(theta_base), _dtype_code(ref), int(bool(inverse)), _stream(ref)),
          "tree_rope")


def tree_attn_workspace_size(T, Hq, Hkv, d, dtype_code) -> int:
    return int(lib().tree_attn_workspace_size(T, Hq, Hkv, d, dtype_code))


def tree_attn_fwd(q, k, v, subtree_end, softmax_scale: float = 0.0, workspace=None, out=None, lse=None):
    """Tree attention forward; returns (o [T,Hq,d], lse [Hq,T] fp32)."""
    torch = _torch()
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    dt = _dtype_code(q)
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device) if lse is None else lse
    nbytes = tree_attn_workspace_size(T, Hq, Hkv, d, dt)
    ws = _workspace(nbytes, q.device, workspace)
    check(lib().tree_attn_fwd(_dev(q, "q"), _dev(k, "k", q.dtype), _dev(v, "v", q.dtype),
                              _dev(o, "o", q.dtype), _dev(lse, "lse", torch.float32),
                              _dev(subtree_end, "subtree_end", torch.int32), T, Hq, Hkv, d, dt,
                              float(softmax_scale), C.c_void_p(ws.data_ptr()),
                              ws.numel() * ws.element_size(), _stream(q)), "tree_attn_fwd")
    return o, lse


def tree_attn_bwd(q, k, v, o, dout, lse, subtree_end, softmax_scale: float = 0.0,
                  deterministic: bool = False, workspace=None, grads=None):
    """Tree attention backward; returns (dq, dk, dv) in the input dtype."""
    torch = _torch()
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    dt = _dtype_code(q)
    if grads is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    else:
        dq, dk, dv = grads
    nbytes = tree_attn_workspace_size(T, Hq, Hkv, d, dt)
    ws = _workspace(nbytes, q.device, workspace)
    check(lib().tree_attn_bwd(_dev(q, "q"), _dev(k, "k", q.dtype), _dev(v, "v", q.dtype),
                              _dev(o, "o", q.dtype), _dev(dout, "dout", q.dtype),
                              _dev(lse, "lse", torch.float32), _dev(dq, "dq", q.dtype),
                              _dev(dk, "dk", q.dtype), _dev(dv, "dv", q.dtype),
                              _dev(subtree_end, "subtree_end", torch.int32), T, Hq, Hkv, d, dt,
                              float(softmax_scale), int(bool(deterministic)),
                              C.c_void_p(ws.data_ptr()), ws.numel() * ws.element_size(), _stream(q)),
          "tree_attn_bwd")
    return dq, dk, dv


def tree_attn_bwd_rope(q, k, v, o, dout, lse, subtree_end, position_ids, theta_base: float = 10000.0,
                       softmax_scale: float = 0.0, deterministic: bool = False, workspace=None, grads=None):
    """tree_attn_bwd followed by the inverse depth rotation on dq and dk (one fused pass):
    for q, k rotated by tree_rope, returns the gradients of the unrotated q, k, and dv."""
    torch = _torch()
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    dt = _dtype_code(q)
    if grads is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    else:
        dq, dk, dv = grads
    nbytes = tree_attn_workspace_size(T, Hq, Hkv, d, dt)
    ws = _workspace(nbytes, q.device, workspace)
    check(lib().tree_attn_bwd_rope(_dev(q, "q"), _dev(k, "k", q.dtype), _dev(v, "v", q.dtype),
                                   _dev(o, "o", q.dtype), _dev(dout, "dout", q.dtype),
                                   _dev(lse, "lse", torch.float32), _dev(dq, "dq", q.dtype),
                                   _dev(dk, "dk", q.dtype), _dev(dv, "dv", q.dtype),
                                   _dev(subtree_end, "subtree_end", torch.int32),
                                   _dev(position_ids, "position_ids", torch.int32), T, Hq, Hkv, d, dt,
                                   float(softmax_scale), float(theta_base), int(bool(deterministic)),
                                   C.c_void_p(ws.data_ptr()), ws.numel() * ws.element_size(), _stream(q)),
          "tree_attn_bwd_rope")
    return dq, dk, dv


def tree_kernel_timing(enable: bool) -> None:
    """Bracket each attention call's main kernel with CUDA events (for benchmarks)."""
    lib().tree_kernel_timing(int(bool(enable)))


def tree_selftest_exp2(x):
    """The library's FMA-pipe 2^x on a device fp32 tensor (for tests)."""
    torch = _torch()
    y = torch.empty_like(x)
    check(lib().tree_selftest_exp2(_dev(x, "x", torch.float32), _dev(y, "y", torch.float32), x.numel(), _stream(x)),
          "tree_selftest_exp2")
    return y


def tree_kernel_last_ms(which: int) -> float:
    """Duration of the latest bracketed main kernel (0: forward, 1: backward), or -1."""
    return float(lib().tree_kernel_last_ms(int(which)))


def tree_policy_loss(logp, old_logp, advantage, weight=None, mask=None, eps_low: float = 0.2,
                     eps_high=None, grad=None):
    """Per-occurrence clipped policy objective: returns (loss [n_occ], grad_logp [n_occ],
    loss_sum [1]), all fp32 on the device; grad_logp feeds tree_logprob_bwd."""
    torch = _torch()
    n = logp.shape[0]
    f32 = torch.float32
    loss = torch.empty(n, dtype=f32, device=logp.device)
    g = torch.empty(n, dtype=f32, device=logp.device) if grad is None else grad
    total = torch.empty(1, dtype=f32, device=logp.device)
    check(lib().tree_policy_loss(_dev(logp, "logp", f32), _dev(old_logp, "old_logp", f32),
                                 _dev(advantage, "advantage", f32), _dev(weight, "weight", f32),
                                 _dev(mask, "mask", torch.uint8), n, float(eps_low),
                                 float(eps_low if eps_high is None else eps_high),
                                 _dev(loss, "loss", f32), _dev(g, "grad_logp", f32),
                                 _dev(total, "loss_sum", f32), _stream(logp)),
          "tree_policy_loss")
    return loss, g, total


def tree_attn_gateway_workspace_size(past_len, T, Hq, Hkv, d, dtype_code) -> int:
    return int(lib().tree_attn_gateway_workspace_size(past_len, T, Hq, Hkv, d, dtype_code))


def tree_attn_fwd_gateway(q, k, v, attn_bias, subtree_end, softmax_scale: float = 0.0, workspace=None, out=None,
                          lse=None):
    """Child-partition attention through a gateway: q [T,Hq,d]; k, v [past_len+T,Hkv,d]
    (past rows first); attn_bias fp32 [past_len] (0 / -inf); subtree_end int32 [T] local
    to the partition. Returns (o [T,Hq,d], lse [Hq,T])."""
    torch = _torch()
    T, Hq, d = q.shape
    Tk, Hkv = k.shape[0], k.shape[1]
    P = Tk - T
    dt = _dtype_code(q)
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device) if lse is None else lse
    ws = _workspace(tree_attn_gateway_workspace_size(P, T, Hq, Hkv, d, dt), q.device, workspace)
    check(lib().tree_attn_fwd_gateway(_dev(q, "q"), _dev(k, "k", q.dtype), _dev(v, "v", q.dtype), _dev(o, "o", q.dtype),
                                      _dev(lse, "lse", torch.float32), _dev(attn_bias, "attn_bias", torch.float32),
                                      _dev(subtree_end, "subtree_end", torch.int32), P, T, Hq, Hkv, d, dt,
                                      float(softmax_scale), C.c_void_p(ws.data_ptr()), ws.numel() * ws.element_size(),
                                      _stream(q)), "tree_attn_fwd_gateway")
    return o, lse


def tree_attn_bwd_gateway(q, k, v, o, dout, lse, attn_bias, subtree_end, dk_past=None, dv_past=None,
                          softmax_scale: float = 0.0, workspace=None):
    """Backward of tree_attn_fwd_gateway: returns (dq [T,Hq,d], dk [T,Hkv,d], dv [T,Hkv,d]) for
    the partition's own rows and (dk_past, dv_past) fp32 [past_len,Hkv,d], to which the past
    rows' gradients were added (new zeroed tensors when not given)."""
    torch = _torch()
    T, Hq, d = q.shape
    Tk, Hkv = k.shape[0], k.shape[1]
    P = Tk - T
    dt = _dtype_code(q)
    f32 = torch.float32
    dq = torch.empty_like(q)
    dk = torch.empty((T, Hkv, d), dtype=q.dtype, device=q.device)
    dv = torch.empty((T, Hkv, d), dtype=q.dtype, device=q.device)
    if dk_past is None:
        dk_past = torch.zeros((P, Hkv, d), dtype=f32, device=q.device)
    if dv_past is None:
        dv_past = torch.zeros((P, Hkv, d), dtype=f32, device=q.device)
    ws = _workspace(tree_attn_gateway_workspace_size(P, T, Hq, Hkv, d, dt), q.device, workspace)
    check(lib().tree_attn_bwd_gateway(_dev(q, "q"), _dev(k, "k", q.dtype), _dev(v, "v", q.dtype), _dev(o, "o", q.dtype),
                                      _dev(dout, "dout", q.dtype), _dev(lse, "lse", f32), _dev(dq, "dq", q.dtype),
                                      _dev(dk, "dk", q.dtype), _dev(dv, "dv", q.dtype),
                                      _dev(dk_past, "dk_past", f32) if P > 0 else None,
                                      _dev(dv_past, "dv_past", f32) if P > 0 else None,
                                      _dev(attn_bias, "attn_bias", f32), _dev(subtree_end, "subtree_end", torch.int32),
                                      P, T, Hq, Hkv, d, dt, float(softmax_scale), C.c_void_p(ws.data_ptr()),
                                      ws.numel() * ws.element_size(), _stream(q)), "tree_attn_bwd_gateway")
    return dq, dk, dv, dk_past, dv_past


def tree_gdn_workspace_size(T, n_nodes, H, Dk, Dv) -> int:
    return int(lib().tree_gdn_workspace_size(T, n_nodes, H, Dk, Dv))


def tree_gdn_fwd(q, k, v, g, beta, node_start, node_end, node_parent, workspace=None, out=None):
    """Gated DeltaNet forward with tree state routing: q, k [T,H,Dk]; v [T,H,Dv]; g, beta
    fp32 [T,H]; node arrays int32 [n_nodes]. Returns o [T,H,Dv] in q's dtype."""
    torch = _torch()
    T, H, Dk = q.shape
    Dv = v.shape[2]
    n_nodes = node_start.shape[0]
    o = torch.empty((T, H, Dv), dtype=q.dtype, device=q.device) if out is None else out
    f32, i32 = torch.float32, torch.int32
    ws = _workspace(tree_gdn_workspace_size(T, n_nodes, H, Dk, Dv), q.device, workspace)
    check(lib().tree_gdn_fwd(_dev(q, "q"), _dev(k, "k", q.dtype), _dev(v, "v", q.dtype), _dev(g, "g", f32),
                             _dev(beta, "beta", f32), _dev(o, "o", q.dtype), _dev(node_start, "node_start", i32),
                             _dev(node_end, "node_end", i32), _dev(node_parent, "node_parent", i32), T, n_nodes,
                             H, Dk, Dv, _dtype_code(q), C.c_void_p(ws.data_ptr()), ws.numel() * ws.element_size(),
                             _stream(q)), "tree_gdn_fwd")
    return o


def tree_gdn_bwd_workspace_size(T, n_nodes, H, Dk, Dv) -> int:
    return int(lib().tree_gdn_bwd_workspace_size(T, n_nodes, H, Dk, Dv))


def tree_gdn_bwd(q, k, v, g, beta, dout, node_start, node_end, node_parent, workspace=None, grads=None,
                 saved=False):
    """Gradients of sum(dout * o) for tree_gdn_fwd: returns (dq, dk, dv, dg, dbeta), dq, dk
    [T,H,Dk] and dv [T,H,Dv] in q's dtype, dg, dbeta fp32 [T,H]. grads: optional
    preallocated tuple of the five outputs. saved=True (tree_gdn_bwd_saved) takes the
    forward's states from `workspace`, which must be the tree_gdn_bwd_workspace_size()
    buffer the last tree_gdn_fwd on these inputs ran with, instead of recomputing them."""
    if saved and workspace is None:
        raise ValueError("tree_gdn_bwd(saved=True) needs the workspace the forward ran with")
    torch = _torch()
    T, H, Dk = q.shape
    Dv = v.shape[2]
    n_nodes = node_start.shape[0]
    if grads is None:
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
                 torch.empty((T, H), dtype=torch.float32, device=q.device),
                 torch.empty((T, H), dtype=torch.float32, device=q.device))
    dq, dk, dv, dg, db = grads
    f32, i32 = torch.float32, torch.int32
    ws = _workspace(tree_gdn_bwd_workspace_size(T, n_nodes, H, Dk, Dv), q.device, workspace)
    name = "tree_gdn_bwd_saved" if saved else "tree_gdn_bwd"
    check(getattr(lib(), name)(_dev(q, "q"), _dev(k, "k", q.dtype), _dev(v, "v", q.dtype), _dev(g, "g", f32),
                               _dev(beta, "beta", f32), _dev(dout, "dout", q.dtype), _dev(dq, "dq", q.dtype),
                               _dev(dk, "dk", q.dtype), _dev(dv, "dv", q.dtype), _dev(dg, "dg", f32),
                               _dev(db, "dbeta", f32), _dev(node_start, "node_start", i32),
                               _dev(node_end, "node_end", i32), _dev(node_parent, "node_parent", i32), T,
                               n_nodes, H, Dk, Dv, _dtype_code(q), C.c_void_p(ws.data_ptr()),
                               ws.numel() * ws.element_size(), _stream(q)), name)
    return dq, dk, dv, dg, db


def tree_gdn_bwd_saved(q, k, v, g, beta, dout, node_start, node_end, node_parent, workspace, grads=None):
    """tree_gdn_bwd taking the forward's states from `workspace` (the
    tree_gdn_bwd_workspace_size() buffer the last tree_gdn_fwd on these inputs ran with)."""
    return tree_gdn_bwd(q, k, v, g, beta, dout, node_start, node_end, node_parent, workspace=workspace,
                        grads=grads, saved=True)


def tree_conv1d_fwd(x, w, parent_row, bias=None, out=None):
    """Tree-correct causal depthwise conv1d: x [T, C], w [C, K] (x's dtype), parent_row
    int32 [T], bias [C] or None; returns y [T, C] in x's dtype."""
    torch = _torch()
    T, Cc = x.shape
    K = w.shape[1]
    y = torch.empty_like(x) if out is None else out
    check(lib().tree_conv1d_fwd(_dev(x, "x"), _dev(w, "w", x.dtype), _dev(bias, "bias", x.dtype),
                                _dev(y, "y", x.dtype), _dev(parent_row, "parent_row", torch.int32), T, Cc, K,
                                _dtype_code(x), _stream(x)), "tree_conv1d_fwd")
    return y


def tree_conv1d_workspace_size(T, C_, K) -> int:
    return int(lib().tree_conv1d_workspace_size(T, C_, K))


def tree_conv1d_bwd(x, w, dy, subtree_end, position_ids, workspace=None, grads=None, want_dw: bool = True,
                    want_dbias: bool = True):
    """Gradients of tree_conv1d_fwd: returns (dx [T, C] in x's dtype, dw [C, K] fp32 or None,
    dbias [C] fp32 or None)."""
    torch = _torch()
    T, Cc = x.shape
    K = w.shape[1]
    f32 = torch.float32
    if grads is None:
        dx = torch.empty_like(x)
        dw = torch.empty((Cc, K), dtype=f32, device=x.device) if want_dw else None
        db = torch.empty(Cc, dtype=f32, device=x.device) if want_dbias else None
    else:
        dx, dw, db = grads
    ws = _workspace(tree_conv1d_workspace_size(T, Cc, K), x.device, workspace)
    i32 = torch.int32
    check(lib().tree_conv1d_bwd(_dev(x, "x"), _dev(w, "w", x.dtype), _dev(dy, "dy", x.dtype),
                                _dev(dx, "dx", x.dtype), _dev(dw, "dw", f32), _dev(db, "dbias", f32),
                                _dev(subtree_end, "subtree_end", i32), _dev(position_ids, "position_ids", i32),
                                T, Cc, K, _dtype_code(x), C.c_void_p(ws.data_ptr()),
                                ws.numel() * ws.element_size(), _stream(x)), "tree_conv1d_bwd")
    return dx, dw, db


def tree_logprob_workspace_size(T, K_h, V, n_occ, dtype_code) -> int:
    return int(lib().tree_logprob_workspace_size(T, K_h, V, n_occ, dtype_code))


def tree_logprob_fwd(hidden, w_lm, occ_row_ptr, occ_perm, occ_targets, workspace=None, lse=None, logp=None):
    """Shared-logit log-probs; returns (lse [T] fp32, logp [n_occ] fp32)."""
    torch = _torch()
    T, K = hidden.shape
    V = w_lm.shape[1]
    n_occ = occ_targets.shape[0]
    dt = _dtype_code(hidden)
    lse = torch.empty(T, dtype=torch.float32, device=hidden.device) if lse is None else lse
    logp = torch.empty(n_occ, dtype=torch.float32, device=hidden.device) if logp is None else logp
    ws = _workspace(tree_logprob_workspace_size(T, K, V, n_occ, dt), hidden.device, workspace)
    i32 = torch.int32
    check(lib().tree_logprob_fwd(_dev(hidden, "hidden"), _dev(w_lm, "w_lm", hidden.dtype),
                                 _dev(occ_row_ptr, "occ_row_ptr", i32), _dev(occ_perm, "occ_perm", i32),
                                 _dev(occ_targets, "occ_targets", i32), T, K, V, n_occ,
                                 _dev(lse, "lse", torch.float32), _dev(logp, "logp", torch.float32), dt,
                                 C.c_void_p(ws.data_ptr()), ws.numel() * ws.element_size(),
                                 _stream(hidden)), "tree_logprob_fwd")
    return lse, logp


def tree_logprob_bwd(hidden, w_lm, lse, occ_row_ptr, occ_perm, occ_targets, grad_logp, workspace=None,
                     grads=None, dw_fp32: bool = False):
    """Backward of the shared-logit log-probs; returns (d_hidden, d_w): d_hidden in the
    input dtype, d_w in the input dtype or, with dw_fp32, in fp32."""
    torch = _torch()
    T, K = hidden.shape
    V = w_lm.shape[1]
    n_occ = occ_targets.shape[0]
    dt = _dtype_code(hidden)
    dw_dtype = torch.float32 if dw_fp32 else hidden.dtype
    if grads is None:
        dh, dw = torch.empty_like(hidden), torch.empty((K, V), dtype=dw_dtype, device=hidden.device)
    else:
        dh, dw = grads
    ws = _workspace(tree_logprob_workspace_size(T, K, V, n_occ, dt), hidden.device, workspace)
    i32 = torch.int32
    check(lib().tree_logprob_bwd(_dev(hidden, "hidden"), _dev(w_lm, "w_lm", hidden.dtype),
                                 _dev(lse, "lse", torch.float32), _dev(occ_row_ptr, "occ_row_ptr", i32),
                                 _dev(occ_perm, "occ_perm", i32), _dev(occ_targets, "occ_targets", i32),
                                 _dev(grad_logp, "grad_logp", torch.float32), T, K, V, n_occ,
                                 _dev(dh, "d_hidden", hidden.dtype), _dev(dw, "d_w", dw_dtype), int(bool(dw_fp32)), dt,
                                 C.c_void_p(ws.data_ptr()), ws.numel() * ws.element_size(),
                                 _stream(hidden)), "tree_logprob_bwd")
    return dh, dw


def tree_check_device_status(stream=None) -> None:
    """Synchronise and raise TreeError if a kernel flagged a range error or a timeout."""
    torch = _torch()
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    check(lib().tree_check_device_status(C.c_void_p(s)), "tree_check_device_status")


def tree_launch_count() -> int:
    """Kernel launches the library has enqueued in this process."""
    return int(lib().tree_launch_count())


def tree_kernel_path(op: int, dtype_code: int, d: int) -> int:
    return int(lib().tree_kernel_path(op, dtype_code, d))
