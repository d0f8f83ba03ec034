"""Pins of the tree-routed Gated DeltaNet oracle (oracle/gdn.py).

Tree Training §3.2 "SSM Layers (GDN)", eq. 10 and Appendix A.2: each chunk (tree node)
starts from its parent chunk's end state. The oracle's token recurrence is pinned to a
chunked solution written independently here (per node, the delta-rule corrections of
the whole node from one lower-triangular solve, started from the parent node's end
state, as eq. 10 routes it), to closed forms, to the delta rule's retrieval property and
to finite differences.
"""
import numpy as np
import pytest

import oracle
import synth

rng = np.random.default_rng(31)


def _inputs(T, H=2, Dk=6, Dv=5, seed=0):
    r = np.random.default_rng(seed)
    k = r.normal(size=(T, H, Dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    return (r.normal(size=(T, H, Dk)), k, r.normal(size=(T, H, Dv)), -r.uniform(0.0, 0.5, size=(T, H)),
            r.uniform(0.1, 0.9, size=(T, H)))


def _chunked_tree(q, k, v, g, beta, ref):
    """Per node: with h0 the parent node's end state (zero at a root), cumulative decay
    G_t = exp(sum_{r<=t} g_r) inside the node, the corrected values u solve
        u_t + beta_t sum_{s<t} (G_t / G_s) (k_t . k_s) u_s = beta_t (v_t - G_t h0^T k_t),
    the outputs are o_t = G_t h0^T q_t + sum_{s<=t} (G_t / G_s) (q_t . k_s) u_s and the end
    state is G_L h0 + sum_s (G_L / G_s) k_s u_s^T (state h = S^T, [Dk, Dv])."""
    T, H, Dk = q.shape
    Dv = v.shape[2]
    o = np.zeros((T, H, Dv))
    end_state = {}
    for n in range(len(ref["node_start"])):
        s0, s1 = int(ref["node_start"][n]), int(ref["node_end"][n]) + 1
        par = int(ref["node_parent"][n])
        for h in range(H):
            h0 = end_state[(par, h)] if par >= 0 else np.zeros((Dk, Dv))
            K, V, Q = k[s0:s1, h], v[s0:s1, h], q[s0:s1, h]
            G = np.exp(np.cumsum(g[s0:s1, h]))
            b = beta[s0:s1, h]
            L = s1 - s0
            ratio = G[:, None] / G[None, :]
            M = np.eye(L) + np.tril(b[:, None] * ratio * (K @ K.T), -1)
            u = np.linalg.solve(M, b[:, None] * (V - G[:, None] * (K @ h0)))
            o[s0:s1, h] = G[:, None] * (Q @ h0) + np.tril(ratio * (Q @ K.T)) @ u
            end_state[(n, h)] = G[-1] * h0 + (K * (G[-1] / G)[:, None]).T @ u
    return o


@pytest.mark.parametrize("seed", range(4))
def test_recurrence_matches_chunked_tree_solution(seed):
    r = np.random.default_rng(seed)
    seqs = synth.random_sequences(r, 10, 25, vocab=3, min_len=1)
    ref = oracle.pack_ref(seqs)
    q, k, v, g, beta = _inputs(ref["T"], seed=seed)
    o = oracle.gdn_ref_fwd(q, k, v, g, beta, ref["paths"])
    assert np.allclose(o, _chunked_tree(q, k, v, g, beta, ref), atol=1e-10)


def test_sibling_starts_from_the_parent_state():
    """Eq. 10 / Fig. 2: the second sibling continues the shared prefix's state, not the
    first sibling's: its outputs equal a pass over [prefix, second sibling] alone."""
    ref = oracle.pack_ref([[1, 2, 3, 4, 5], [1, 2, 3, 6, 7]])
    q, k, v, g, beta = _inputs(ref["T"], seed=4)
    o = oracle.gdn_ref_fwd(q, k, v, g, beta, ref["paths"])
    alone = [0, 1, 2, 5, 6]
    solo = oracle.pack_ref([[1, 2, 3, 6, 7]])
    o2 = oracle.gdn_ref_fwd(q[alone], k[alone], v[alone], g[alone], beta[alone], solo["paths"])
    assert np.allclose(o[alone], o2, atol=1e-12)
    # the sequential (DFS-order) routing gives something else at the second sibling
    chain = oracle.pack_ref([[1, 2, 3, 4, 5, 6, 7]])
    o_seq = oracle.gdn_ref_fwd(q, k, v, g, beta, chain["paths"])
    assert not np.allclose(o_seq[5], o[5])


def test_no_decay_full_write_overwrites():
    """alpha -> 0, beta = 1: the state is v_t k_t^T, so o_t = v_t (k_t . q_t)."""
    seqs = synth.random_sequences(rng, 6, 12, vocab=3)
    ref = oracle.pack_ref(seqs)
    q, k, v, g, beta = _inputs(ref["T"], seed=5)
    o = oracle.gdn_ref_fwd(q, k, v, np.full_like(g, -60.0), np.ones_like(beta), ref["paths"])
    want = v * np.sum(k * q, axis=-1, keepdims=True)
    assert np.allclose(o, want, atol=1e-12)


def test_zero_write_strength_is_zero():
    seqs = synth.random_sequences(rng, 6, 12, vocab=3)
    ref = oracle.pack_ref(seqs)
    q, k, v, g, beta = _inputs(ref["T"], seed=6)
    assert np.abs(oracle.gdn_ref_fwd(q, k, v, g, np.zeros_like(beta), ref["paths"])).max() == 0.0


def test_delta_rule_retrieves_the_last_write():
    """alpha = 1, beta = 1, unit keys: S_t k_t = v_t whatever the earlier state, so reading
    with q_t = k_t returns v_t."""
    seqs = synth.random_sequences(rng, 8, 20, vocab=3)
    ref = oracle.pack_ref(seqs)
    _, k, v, g, beta = _inputs(ref["T"], seed=7)
    o = oracle.gdn_ref_fwd(k, k, v, np.zeros_like(g), np.ones_like(beta), ref["paths"])
    assert np.allclose(o, v, atol=1e-10)


def test_backward_matches_finite_differences():
    ref = oracle.pack_ref([[1, 2, 3, 4], [1, 2, 5], [1, 6, 7, 8, 9]])
    T = ref["T"]
    q, k, v, g, beta = _inputs(T, H=1, Dk=3, Dv=2, seed=8)
    do = np.random.default_rng(9).normal(size=(T, 1, 2))
    grads = oracle.gdn_ref_bwd(q, k, v, g, beta, do, ref["paths"])
    args = [q, k, v, g, beta]
    Lf = lambda a: float((do * oracle.gdn_ref_fwd(*a, ref["paths"])).sum())
    eps = 1e-6
    for which in range(5):
        x = args[which]
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            fd = (Lf(plus) - Lf(minus)) / (2 * eps)
            assert fd == pytest.approx(grads[which][idx], abs=1e-6, rel=1e-5), (which, idx)


def test_backward_tree_equals_sum_over_branches():
    """Gradients of a tree = gradients of the per-branch passes, each row's output
    gradient counted once: checked against the chunked solution by finite differences on
    a random tree (the backward never runs the chunked form, so the two are independent)."""
    r = np.random.default_rng(10)
    seqs = synth.random_sequences(r, 5, 8, vocab=2, min_len=2)
    ref = oracle.pack_ref(seqs)
    T = ref["T"]
    q, k, v, g, beta = _inputs(T, H=1, Dk=3, Dv=2, seed=10)
    do = r.normal(size=(T, 1, 2))
    dq, dk, dv, dg, dbeta = oracle.gdn_ref_bwd(q, k, v, g, beta, do, ref["paths"])
    eps = 1e-6
    for name, x, gx in (("v", v, dv), ("g", g, dg), ("beta", beta, dbeta)):
        for idx in [(i,) + (0,) * (x.ndim - 1) for i in range(T)]:
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            sub = {"v": (q, k, xp, g, beta), "g": (q, k, v, xp, beta), "beta": (q, k, v, g, xp)}[name]
            sbm = {"v": (q, k, xm, g, beta), "g": (q, k, v, xm, beta), "beta": (q, k, v, g, xm)}[name]
            fd = ((do * _chunked_tree(*sub, ref)).sum() - (do * _chunked_tree(*sbm, ref)).sum()) / (2 * eps)
            assert fd == pytest.approx(gx[idx], abs=1e-6, rel=1e-5), (name, idx)


def _chunked_tree_bwd(q, k, v, g, beta, do, ref):
    """Reverse-mode of the per-node chunked solution (_chunked_tree), node by node from
    the leaves up: a node's end-state gradient is the sum of its children's start-state
    gradients (siblings share their parent's end state), and within the node
        u = M^{-1} r,  r = beta (V - E (K h0)),  O = E (Q h0) + P u,
        h_end = E_{L-1} h0 + sum_s (E_{L-1}/E_s) k_s u_s^T,   E = exp(cumsum g),
    are differentiated through the triangular solve (dr = M^{-T} du, dM = -dr u^T)."""
    T, H, Dk = q.shape
    Dv = v.shape[2]
    n_nodes = len(ref["node_start"])
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dg, dbeta = np.zeros_like(g), np.zeros_like(beta)
    # forward pass once, keeping every node's start state
    start = {}
    end_state = {}
    for n in range(n_nodes):
        s0, s1 = int(ref["node_start"][n]), int(ref["node_end"][n]) + 1
        par = int(ref["node_parent"][n])
        for h in range(H):
            h0 = end_state[(par, h)] if par >= 0 else np.zeros((Dk, Dv))
            start[(n, h)] = h0
            K, V = k[s0:s1, h], v[s0:s1, h]
            lg = np.cumsum(g[s0:s1, h])
            E, b = np.exp(lg), beta[s0:s1, h]
            f = np.exp(lg[:, None] - lg[None, :])
            M = np.eye(s1 - s0) + np.tril(b[:, None] * f * (K @ K.T), -1)
            u = np.linalg.solve(M, b[:, None] * (V - E[:, None] * (K @ h0)))
            end_state[(n, h)] = E[-1] * h0 + (K * np.exp(lg[-1] - lg)[:, None]).T @ u
    dh_end = {(n, h): np.zeros((Dk, Dv)) for n in range(n_nodes) for h in range(H)}
    for n in range(n_nodes - 1, -1, -1):          # children come after their parent in preorder
        s0, s1 = int(ref["node_start"][n]), int(ref["node_end"][n]) + 1
        par = int(ref["node_parent"][n])
        L = s1 - s0
        for h in range(H):
            h0, dhe = start[(n, h)], dh_end[(n, h)]
            K, Q, V, dO = k[s0:s1, h], q[s0:s1, h], v[s0:s1, h], do[s0:s1, h]
            lg = np.cumsum(g[s0:s1, h])
            E, b = np.exp(lg), beta[s0:s1, h]
            f = np.exp(lg[:, None] - lg[None, :])
            low, strict = np.tril(np.ones((L, L))), np.tril(np.ones((L, L)), -1)
            KK, QK = K @ K.T, Q @ K.T
            A = strict * b[:, None] * f * KK
            P = low * f * QK
            kh, qh = K @ h0, Q @ h0
            r = b[:, None] * (V - E[:, None] * kh)
            u = np.linalg.solve(np.eye(L) + A, r)
            w = np.exp(lg[-1] - lg)
            dK, dQ, dlg = np.zeros_like(K), np.zeros_like(Q), np.zeros(L)
            dh0 = E[-1] * dhe
            dlg[-1] += E[-1] * np.sum(dhe * h0)
            # h_end = ... + sum_s w_s k_s u_s^T
            du = w[:, None] * (K @ dhe)
            dK += w[:, None] * (u @ dhe.T)
            dw = np.sum((K @ dhe) * u, axis=1) * w
            dlg[-1] += dw.sum()
            dlg -= dw
            # O = E qh + P u
            dqh = E[:, None] * dO
            dh0 += Q.T @ dqh
            dQ += dqh @ h0.T
            dlg += E * np.sum(dO * qh, axis=1)
            du += P.T @ dO
            dP = low * (dO @ u.T)
            dQ += (dP * f) @ K
            dK += (dP * f).T @ Q
            dlg += np.sum(dP * P, axis=1) - np.sum(dP * P, axis=0)
            # u = M^{-1} r
            dr = np.linalg.solve((np.eye(L) + A).T, du)
            dA = -strict * (dr @ u.T)
            dbeta[s0:s1, h] += np.sum(dA * f * KK, axis=1)
            dK += (dA * b[:, None] * f) @ K + (dA * b[:, None] * f).T @ K
            dlg += np.sum(dA * A, axis=1) - np.sum(dA * A, axis=0)
            # r = beta (V - E kh)
            dbeta[s0:s1, h] += np.sum(dr * (V - E[:, None] * kh), axis=1)
            dv[s0:s1, h] += b[:, None] * dr
            dkh = -(b * E)[:, None] * dr
            dh0 += K.T @ dkh
            dK += dkh @ h0.T
            dlg += -b * E * np.sum(dr * kh, axis=1)
            dg[s0:s1, h] += np.cumsum(dlg[::-1])[::-1]
            dq[s0:s1, h] += dQ
            dk[s0:s1, h] += dK
            if par >= 0:
                dh_end[(par, h)] += dh0
    return dq, dk, dv, dg, dbeta


@pytest.mark.parametrize("seed", range(3))
def test_backward_matches_chunked_reverse_mode(seed):
    """The oracle's token-by-token reverse pass against the reverse mode of the per-node
    chunked solution (a triangular solve per node, end-state gradients summed over the
    children): two independent computations of the same gradients."""
    r = np.random.default_rng(40 + seed)
    seqs = synth.random_sequences(r, 9, 20, vocab=3, min_len=2)
    ref = oracle.pack_ref(seqs)
    T = ref["T"]
    q, k, v, g, beta = _inputs(T, seed=40 + seed)
    do = r.normal(size=(T, q.shape[1], v.shape[2]))
    want = _chunked_tree_bwd(q, k, v, g, beta, do, ref)
    got = oracle.gdn_ref_bwd(q, k, v, g, beta, do, ref["paths"])
    for name, a, b in zip(("dq", "dk", "dv", "dg", "dbeta"), got, want):
        assert np.allclose(a, b, atol=1e-9), (name, float(np.abs(a - b).max()))
