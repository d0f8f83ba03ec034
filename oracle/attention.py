"""Oracle tree attention: unpack into paths, run ordinary causal attention per path.

Test infrastructure only (see the package docstring).

Definition followed (Tree Training, arXiv 2511.00413, §3.1 eq. 6 "forward
equivalence"): the packed result at a token must equal what a standalone
per-branch forward computes. So the oracle does not use any mask encoding at
all: it walks each input path (the packed rows of one original sequence, root
first) and runs textbook causal softmax attention on it,
  S = Q K^T * scale,  P = softmax(S + causal),  O = P V,  LSE = log sum exp(S),
with scale = 1/sqrt(d) (Trie packing, "Step 3 - Attention collects descendant
contributions": S = QK^T/sqrt(d_k) + M_tree). There is no softcap and no dropout
(Trie packing, "Verify equivalence before measuring speed", item 1).

Backward (Trie packing, "Same chain rule, shared computation graph", Step 3):
each packed query's output gradient dO_i is handed to exactly one path holding
the row (the first in input order); every other path gets zero for that row.
Ordinary causal attention backward then runs per path,
  dV = P^T dO, dP = dO V^T, Delta = rowsum(P o dP), dS = P o (dP - Delta),
  dQ = scale dS K, dK = scale dS^T Q,
and the per-path gradients are added back into the packed rows, so a shared key
collects the contributions of all its descendants.

Readings: GQA query head h uses KV head h // (Hq / Hkv) (contiguous groups);
LSE is the natural log; K/V gradients of a KV head sum over its query heads.
"""
from __future__ import annotations

import numpy as np


def _kv_of(Hq: int, Hkv: int) -> np.ndarray:
    assert Hq % Hkv == 0
    return np.arange(Hq) // (Hq // Hkv)


def _scale(d: int, scale) -> float:
    return 1.0 / np.sqrt(d) if scale is None or scale <= 0 else float(scale)


def _path_softmax(qp, kp, scale):
    """Causal attention probabilities along one path. qp,kp: [L,H,d] -> P [H,L,L], lse [H,L]."""
    L = qp.shape[0]
    s = np.matmul(qp.transpose(1, 0, 2), kp.transpose(1, 2, 0)) * scale     # [H, L, L]
    causal = np.triu(np.ones((L, L), dtype=bool), k=1)
    s[:, causal] = -np.inf
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=-1, keepdims=True)
    return e / l, (m + np.log(l))[..., 0]


def attn_ref_fwd(q, k, v, paths, scale=None, head_chunk: int = 8):
    """O [T,Hq,d] and LSE [Hq,T] (float64) of causal attention along every path.

    A row lying on several paths gets the same value from each (eq. 6); the
    oracle checks that to 1e-12 and keeps the first.
    """
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    kv = _kv_of(Hq, Hkv)
    sc = _scale(d, scale)
    o = np.full((T, Hq, d), np.nan)
    lse = np.full((Hq, T), np.nan)
    done = np.zeros(T, dtype=bool)
    for path in paths:
        path = np.asarray(path, dtype=np.int64)
        if path.size == 0:
            continue
        for h0 in range(0, Hq, head_chunk):
            hs = np.arange(h0, min(Hq, h0 + head_chunk))
            p, l_ = _path_softmax(q[path][:, hs], k[path][:, kv[hs]], sc)
            op = np.matmul(p, v[path][:, kv[hs]].transpose(1, 0, 2)).transpose(1, 0, 2)
            old = done[path]
            if old.any():
                ref_o = o[path[old]][:, hs]
                assert np.allclose(op[old], ref_o, rtol=0, atol=1e-12), "path invariance violated"
            o[path[~old][:, None], hs[None, :]] = op[~old]
            lse[hs[:, None], path[~old][None, :]] = l_[:, ~old]
        done[path] = True
    return o, lse


def attn_ref_bwd(q, k, v, dout, paths, scale=None, head_chunk: int = 8):
    """dQ [T,Hq,d], dK/dV [T,Hkv,d] (float64) by per-path causal backward."""
    q, k, v, dout = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dout))
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    kv = _kv_of(Hq, Hkv)
    sc = _scale(d, scale)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    owner = np.full(T, -1)
    for pi, path in enumerate(paths):
        for r in path:
            if owner[r] < 0:
                owner[r] = pi
    for pi, path in enumerate(paths):
        path = np.asarray(path, dtype=np.int64)
        if path.size == 0:
            continue
        assigned = (owner[path] == pi).astype(np.float64)
        for h0 in range(0, Hq, head_chunk):
            hs = np.arange(h0, min(Hq, h0 + head_chunk))
            qp, kp, vp = q[path][:, hs], k[path][:, kv[hs]], v[path][:, kv[hs]]
            p, _ = _path_softmax(qp, kp, sc)
            dop = dout[path][:, hs] * assigned[:, None, None]
            qh, kh, vh, doh = (x.transpose(1, 0, 2) for x in (qp, kp, vp, dop))   # [H, L, d]
            dvp = np.matmul(p.transpose(0, 2, 1), doh).transpose(1, 0, 2)          # P^T dO
            dpp = np.matmul(doh, vh.transpose(0, 2, 1))                            # dO V^T
            delta = (p * dpp).sum(axis=-1, keepdims=True)
            ds = p * (dpp - delta)
            dqp = np.matmul(ds, kh).transpose(1, 0, 2) * sc                        # dS K
            dkp = np.matmul(ds.transpose(0, 2, 1), qh).transpose(1, 0, 2) * sc     # dS^T Q
            dq[path[:, None], hs[None, :]] += dqp
            for hi, h in enumerate(hs):
                np.add.at(dk, (path, kv[h]), dkp[:, hi])
                np.add.at(dv, (path, kv[h]), dvp[:, hi])
    return dq, dk, dv


def _chains(paths) -> dict:
    """row -> rows from its root to itself, read off the first path that holds it."""
    chain = {}
    for path in paths:
        path = np.asarray(path, dtype=np.int64)
        for t, r in enumerate(path):
            if int(r) not in chain:
                chain[int(r)] = path[:t + 1]
    return chain


def _row_softmax(q, k, chain, r, kv, sc):
    """Attention probabilities [Hq, len(chain)] and lse [Hq] of query row r."""
    s = np.einsum("hd,jhd->hj", q[r], k[chain][:, kv]) * sc
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=-1, keepdims=True)
    return e / l, (m + np.log(l))[:, 0]


def attn_ref_rows(q, k, v, paths, rows, scale=None):
    """O [n,Hq,d] and LSE [Hq,n] for the listed query rows only (each row's own chain)."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    Hq, d = q.shape[1], q.shape[2]
    kv = _kv_of(Hq, k.shape[1])
    sc = _scale(d, scale)
    ch = _chains(paths)
    o = np.empty((len(rows), Hq, d))
    lse = np.empty((Hq, len(rows)))
    for n, r in enumerate(rows):
        c = ch[int(r)]
        p, l_ = _row_softmax(q, k, c, int(r), kv, sc)
        o[n] = np.einsum("hj,jhd->hd", p, v[c][:, kv])
        lse[:, n] = l_
    return o, lse


def attn_ref_dq_rows(q, k, v, dout, paths, rows, scale=None):
    """dQ [n,Hq,d] for the listed query rows (each depends only on its own chain)."""
    q, k, v, dout = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dout))
    Hq, d = q.shape[1], q.shape[2]
    kv = _kv_of(Hq, k.shape[1])
    sc = _scale(d, scale)
    ch = _chains(paths)
    dq = np.empty((len(rows), Hq, d))
    for n, r in enumerate(rows):
        c = ch[int(r)]
        p, _ = _row_softmax(q, k, c, int(r), kv, sc)
        dp = np.einsum("hd,jhd->hj", dout[int(r)], v[c][:, kv])
        delta = (p * dp).sum(axis=-1, keepdims=True)
        ds = p * (dp - delta)
        dq[n] = np.einsum("hj,jhd->hd", ds, k[c][:, kv]) * sc
    return dq


def attn_ref_dkdv_rows(q, k, v, dout, paths, keys, scale=None):
    """dK, dV [n,Hkv,d] for the listed key rows: sum over every descendant-or-self
    query (every row whose path runs through the key) and every query head of the group."""
    q, k, v, dout = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dout))
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    kv = _kv_of(Hq, Hkv)
    sc = _scale(d, scale)
    ch = _chains(paths)
    desc: dict = {}
    want = {int(j) for j in keys}
    for path in paths:
        path = [int(r) for r in path]
        for t, r in enumerate(path):
            if r in want:
                desc.setdefault(r, set()).update(path[t:])
    dk = np.zeros((len(keys), Hkv, d))
    dv = np.zeros((len(keys), Hkv, d))
    for n, j in enumerate(keys):
        j = int(j)
        for i in sorted(desc.get(j, ())):
            c = ch[i]
            p, _ = _row_softmax(q, k, c, i, kv, sc)
            dp = np.einsum("hd,jhd->hj", dout[i], v[c][:, kv])
            delta = (p * dp).sum(axis=-1)
            t = int(np.nonzero(c == j)[0][0])
            pj = p[:, t]
            dsj = pj * (dp[:, t] - delta)
            for h in range(Hq):
                dv[n, kv[h]] += pj[h] * dout[i, h]
                dk[n, kv[h]] += sc * dsj[h] * q[i, h]
    return dk, dv


def dense_mask_from_chunks(node_start, node_end, node_parent, T) -> np.ndarray:
    """Dense [T,T] boolean mask built as Tree Training Appendix A.1 describes it:
    a token sees the whole of every ancestor chunk, and within its own chunk
    the tokens at or before itself (brute force; tiny trees only)."""
    m = np.zeros((T, T), dtype=bool)
    n = len(node_start)
    for c in range(n):
        anc = []
        a = c
        while a >= 0:
            anc.append(a)
            a = int(node_parent[a])
        c0, c1 = int(node_start[c]), int(node_end[c])
        for a in anc:
            a0, a1 = int(node_start[a]), int(node_end[a])
            for i in range(c0, c1 + 1):
                if a == c:
                    m[i, c0:i + 1] = True
                else:
                    m[i, a0:a1 + 1] = True
    return m


def mask_from_paths(paths, T) -> np.ndarray:
    """Dense [T,T] boolean mask: query i sees key j iff j is on i's own path at or before i."""
    m = np.zeros((T, T), dtype=bool)
    for path in paths:
        path = np.asarray(path, dtype=np.int64)
        for t in range(len(path)):
            m[path[t], path[:t + 1]] = True
    return m


def leaf_paths_from_parents(parent_row) -> list:
    """Root-to-leaf row lists of a forest given each row's parent (-1 for roots)."""
    parent_row = np.asarray(parent_row)
    T = len(parent_row)
    has_child = np.zeros(T, dtype=bool)
    has_child[parent_row[parent_row >= 0]] = True
    out = []
    for leaf in np.nonzero(~has_child)[0]:
        chain = [int(leaf)]
        while parent_row[chain[-1]] >= 0:
            chain.append(int(parent_row[chain[-1]]))
        out.append(np.array(chain[::-1], dtype=np.int32))
    return out
