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
