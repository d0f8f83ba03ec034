"""Oracle tree-routed Gated DeltaNet (GDN) recurrence.

Test infrastructure only (see the package docstring).

Tree Training (arXiv 2511.00413) §3.2 "SSM Layers (GDN)", eq. 10, and Appendix A.2: a
GDN layer carries a recurrent state from one token to the next; in the preorder
serialisation the token before a child chunk belongs to a sibling branch, so each chunk
(tree node) starts from the end state of its parent chunk, and a root chunk from zero.
At the token level that is: the state a row starts from is the state after its parent
row (parent_row), zero above a root -- exactly the state of an independent per-branch
pass.

The recurrence (gated delta rule; per head, state S of shape [Dv, Dk]):
    S_t = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   alpha_t = exp(g_t)
    o_t = S_t q_t
The appendix's chunked listing computes the same thing blockwise (a WY correction inside
the chunk, the parent's state across it); the oracle is the token recurrence itself.

Readings taken: g is the per-token log-decay (alpha = exp(g), g <= 0), beta the write
strength; q and k are used as given (any L2 normalisation or 1/sqrt(Dk) scaling of q is
the caller's, as the listing takes q, k as inputs); heads are independent and q/k/v/g/beta
all have the same number of heads.

The oracle unpacks the tree into its root-to-node paths and runs the recurrence along
each one from a zero state (every path through a row gives it the same output, which the
oracle checks). The backward hands each row's output gradient to exactly one path
containing it and adds the per-path gradients into packed rows (a row's output depends
only on its ancestors, so the loss splits over paths this way exactly).
"""
from __future__ import annotations

import numpy as np


def _path_fwd(q, k, v, g, beta):
    """One path, one head: q, k [L, Dk]; v [L, Dv]; g, beta [L] -> o [L, Dv], states [L+1, Dv, Dk]."""
    L, Dk = k.shape
    Dv = v.shape[1]
    S = np.zeros((Dv, Dk))
    states = [S]
    o = np.zeros((L, Dv))
    eye = np.eye(Dk)
    for t in range(L):
        a = np.exp(g[t])
        S = a * S @ (eye - beta[t] * np.outer(k[t], k[t])) + beta[t] * np.outer(v[t], k[t])
        states.append(S)
        o[t] = S @ q[t]
    return o, states


def gdn_ref_fwd(q, k, v, g, beta, paths):
    """o [T, H, Dv] (float64). q, k [T, H, Dk]; v [T, H, Dv]; g, beta [T, H]."""
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    T, H, _ = q.shape
    Dv = v.shape[2]
    o = np.full((T, H, Dv), np.nan)
    for path in paths:
        p = np.asarray(path, dtype=np.int64)
        for h in range(H):
            op, _ = _path_fwd(q[p, h], k[p, h], v[p, h], g[p, h], beta[p, h])
            seen = ~np.isnan(o[p, h, 0])
            if seen.any():
                assert np.allclose(o[p, h][seen], op[seen], rtol=1e-10, atol=1e-10), "paths disagree on a shared row"
            o[p, h] = op
    assert not np.isnan(o).any(), "a row lies on no path"
    return o


def _path_bwd(q, k, v, g, beta, do):
    """Reverse pass of one path and head: gradients of sum(do * o)."""
    L, Dk = k.shape
    _, states = _path_fwd(q, k, v, g, beta)
    eye = np.eye(Dk)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dg, dbeta = np.zeros(L), np.zeros(L)
    dS = np.zeros_like(states[0])
    for t in range(L - 1, -1, -1):
        S_prev, S_t = states[t], states[t + 1]
        a = np.exp(g[t])
        dS = dS + np.outer(do[t], q[t])          # o_t = S_t q_t
        dq[t] = S_t.T @ do[t]
        P = eye - beta[t] * np.outer(k[t], k[t])
        A = a * P
        # S_t = S_prev A + beta v k^T
        dA = S_prev.T @ dS
        dv[t] = beta[t] * dS @ k[t]
        dk[t] += beta[t] * dS.T @ v[t]
        dbeta[t] += v[t] @ dS @ k[t]
        # A = a (I - beta k k^T)
        da = np.sum(dA * P)
        dbeta[t] += -a * (k[t] @ dA @ k[t])
        dk[t] += -a * beta[t] * (dA + dA.T) @ k[t]
        dg[t] = da * a
        dS = dS @ A.T
    return dq, dk, dv, dg, dbeta


def gdn_ref_bwd(q, k, v, g, beta, do, paths):
    """dq, dk [T, H, Dk], dv [T, H, Dv], dg, dbeta [T, H] (float64) for L = sum(do * o)."""
    q, k, v, g, beta, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta, do))
    T, H, _ = q.shape
    owner = np.full(T, -1)
    for pi, path in enumerate(paths):
        for r in path:
            if owner[r] < 0:
                owner[r] = pi
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dg, dbeta = np.zeros_like(g), np.zeros_like(beta)
    for pi, path in enumerate(paths):
        p = np.asarray(path, dtype=np.int64)
        mine = (owner[p] == pi)[:, None]
        for h in range(H):
            a, b, c, e, f = _path_bwd(q[p, h], k[p, h], v[p, h], g[p, h], beta[p, h], np.where(mine, do[p, h], 0.0))
            np.add.at(dq[:, h], p, a)
            np.add.at(dk[:, h], p, b)
            np.add.at(dv[:, h], p, c)
            np.add.at(dg[:, h], p, e)
            np.add.at(dbeta[:, h], p, f)
    return dq, dk, dv, dg, dbeta
