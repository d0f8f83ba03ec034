"""Oracle tree-correct causal depthwise conv1d (the SSM layers' short convolution).

Test infrastructure only (see the package docstring).

Tree Training (arXiv 2511.00413) §3.2 "(ii) Causal convolution", eq. 11 and Fig. 4: a
causal conv1d with kernel size K needs the preceding K-1 tokens as left context; in
the DFS order the tokens just before a child chunk belong to a sibling branch, so each
chunk takes the last K-1 effective tokens of its parent chunk as its left context,
which replicates what each token sees in an independent per-branch pass.

Readings taken: the context is the conv's input x at the K-1 nearest ancestors of a
row along its path (reaching past a short parent chunk into the grandparent), zero
above the root, as in a per-branch pass with zero left padding; the weights w[c, k]
apply tap k to the token K-1-k steps back (w[c, K-1] to the token itself), plus an
optional bias; no activation (it is a separate step of the layer).

The oracle unpacks the tree into its root-to-node paths and runs an ordinary causal
depthwise convolution on each path (every path through a row gives that row the same
output, which the oracle checks); the backward hands each row's output gradient to
exactly one path containing it and adds the per-path gradients back into packed rows.
"""
from __future__ import annotations

import numpy as np


def _causal_conv_path(xp, w, b):
    """Causal depthwise conv of one path: xp [L, C], w [C, K] -> [L, C]."""
    L, C = xp.shape
    K = w.shape[1]
    pad = np.concatenate([np.zeros((K - 1, C)), xp], axis=0)
    y = np.zeros((L, C)) if b is None else np.tile(np.asarray(b, dtype=np.float64), (L, 1))
    for k in range(K):
        y += w[:, k][None, :] * pad[k:k + L]
    return y


def conv1d_ref_fwd(x, w, paths, bias=None):
    """y [T, C] (float64): per-path causal conv, read back into packed rows."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    T, C = x.shape
    y = np.full((T, C), np.nan)
    for path in paths:
        p = np.asarray(path, dtype=np.int64)
        yp = _causal_conv_path(x[p], w, bias)
        seen = ~np.isnan(y[p, 0])
        if seen.any():
            assert np.allclose(y[p][seen], yp[seen], rtol=1e-12, atol=1e-12), "paths disagree on a shared row"
        y[p] = yp
    assert not np.isnan(y).any(), "a row lies on no path"
    return y


def conv1d_ref_bwd(x, w, dy, paths, bias=None):
    """dx [T, C], dw [C, K], dbias [C] (float64) for L = sum(dy * y)."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    T, C = x.shape
    K = w.shape[1]
    owner = np.full(T, -1)
    for pi, path in enumerate(paths):
        for r in path:
            if owner[r] < 0:
                owner[r] = pi
    dx = np.zeros((T, C))
    dw = np.zeros((C, K))
    for pi, path in enumerate(paths):
        p = np.asarray(path, dtype=np.int64)
        g = np.where((owner[p] == pi)[:, None], dy[p], 0.0)  # this path's share of dy
        L = p.shape[0]
        pad = np.concatenate([np.zeros((K - 1, C)), x[p]], axis=0)
        gpad = np.zeros((L + K - 1, C))
        for k in range(K):
            dw[:, k] += (g * pad[k:k + L]).sum(axis=0)
            gpad[k:k + L] += w[:, k][None, :] * g
        dx[p] += gpad[K - 1:]
    dbias = dy.sum(axis=0)
    return dx, dw, dbias


def conv1d_ref_rows(x, w, parent_row, bias=None):
    """The same forward written row by row over the parent links (the definition the
    kernels restate), for cross-checking the per-path oracle."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    T, C = x.shape
    K = w.shape[1]
    y = np.zeros((T, C)) if bias is None else np.tile(np.asarray(bias, dtype=np.float64), (T, 1))
    for i in range(T):
        a = i
        for m in range(K):  # a is the m-th ancestor of i (0: i itself)
            if a < 0:
                break
            y[i] += w[:, K - 1 - m] * x[a]
            a = int(parent_row[a])
    return y
