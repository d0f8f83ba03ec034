"""Oracle shared-logit log-probs: per-occurrence logits, log-softmax, gather; and the
gradient scattered back into shared rows.

Test infrastructure only (see the package docstring).

Trie packing (agillm.io):
* "Share logits, preserve every prediction": the LM head gives z_u = h_u W_LM
  at every packed node; each original next-token prediction is one occurrence
  (source row, target), and several occurrences may read the same row.
* "The training-loop change is small": log_softmax over the vocabulary, then
  the log-prob of each occurrence's target; differentiable indexing scatters and
  adds the gradients of repeated rows.
* "Same chain rule, shared computation graph", Step 1: for one target,
  d(-log p_y)/dz = p - e_y; at a shared row the contributions of different
  targets add.
Tree Training (arXiv 2511.00413) §3.1 eq. 4-5 and §3.2 "Loss Weights": a
per-token weight multiplies each loss term before the reduction.

The oracle computes one full logits row per OCCURRENCE (the unpacked,
per-branch amount of work), in float64. The incoming gradient is g_o =
dL/dlogp_o (for the weighted NLL L = -sum_o w_o logp_o, g_o = -w_o), so
  G_z[r] = sum_{o at r} g_o (e_{y_o} - softmax(z_r)),  dH = G_z W^T,  dW = H^T G_z.
"""
from __future__ import annotations

import numpy as np


def _logsumexp(z):
    m = z.max(axis=-1, keepdims=True)
    return (m + np.log(np.exp(z - m).sum(axis=-1, keepdims=True)))[..., 0]


def logprob_ref_fwd(h, w, src, tgt, T=None, chunk: int = 64):
    """logp [n_occ] and LSE [T] (NaN on rows without an occurrence), float64."""
    h = np.asarray(h, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    src = np.asarray(src, dtype=np.int64)
    tgt = np.asarray(tgt, dtype=np.int64)
    T = h.shape[0] if T is None else T
    logp = np.empty(len(src))
    lse = np.full(T, np.nan)
    for o0 in range(0, len(src), chunk):
        sl = slice(o0, o0 + chunk)
        z = h[src[sl]] @ w                    # one logits row per occurrence
        l_ = _logsumexp(z)
        logp[sl] = z[np.arange(z.shape[0]), tgt[sl]] - l_
        lse[src[sl]] = l_
    return logp, lse


def logprob_ref_gz(h, w, src, tgt, grad_logp, rows, chunk: int = 64):
    """G_z for the listed rows [n, V]: the sum over the row's occurrences of
    g_o (e_{y_o} - softmax(z))."""
    h = np.asarray(h, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    src = np.asarray(src, dtype=np.int64)
    tgt = np.asarray(tgt, dtype=np.int64)
    g = np.asarray(grad_logp, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.int64)
    where = {int(r): n for n, r in enumerate(rows)}
    sel = np.nonzero(np.isin(src, rows))[0]
    gz = np.zeros((len(rows), w.shape[1]))
    for o0 in range(0, len(sel), chunk):
        os_ = sel[o0:o0 + chunk]
        z = h[src[os_]] @ w
        p = np.exp(z - _logsumexp(z)[:, None])
        go = -g[os_, None] * p
        go[np.arange(len(os_)), tgt[os_]] += g[os_]
        for n, o in enumerate(os_):
            gz[where[int(src[o])]] += go[n]
    return gz


def logprob_ref_bwd(h, w, src, tgt, grad_logp, chunk: int = 64):
    """dH [T,K_h] and dW [K_h,V] (float64) of the per-occurrence loss."""
    h = np.asarray(h, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    src = np.asarray(src, dtype=np.int64)
    tgt = np.asarray(tgt, dtype=np.int64)
    g = np.asarray(grad_logp, dtype=np.float64)
    dh = np.zeros_like(h)
    dw = np.zeros_like(w)
    for o0 in range(0, len(src), chunk):
        sl = slice(o0, o0 + chunk)
        hs = h[src[sl]]
        z = hs @ w
        p = np.exp(z - _logsumexp(z)[:, None])
        go = -g[sl, None] * p                     # g_o * (e_y - p): the -p part
        go[np.arange(z.shape[0]), tgt[sl]] += g[sl]
        np.add.at(dh, src[sl], go @ w.T)          # scatter-add into shared rows
        dw += hs.T @ go
    return dh, dw
