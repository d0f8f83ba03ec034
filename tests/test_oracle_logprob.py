"""Pins for oracle.logprob: library log_softmax/gather/autograd (the pages' own
training-loop sketch), cross-entropy special case, the printed gradient at a
shared row, the branch-average identity (eq. 1-5) and finite differences."""
import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import golden


def _torch_ref(h, w, src, tgt, grad_logp):
    th = torch.tensor(h, dtype=torch.float64, requires_grad=True)
    tw = torch.tensor(w, dtype=torch.float64, requires_grad=True)
    logits = th @ tw
    lp = torch.nn.functional.log_softmax(logits, dim=-1)
    tok = lp[torch.tensor(src, dtype=torch.long), torch.tensor(tgt, dtype=torch.long)]
    tok.backward(torch.tensor(grad_logp, dtype=torch.float64))
    return (tok.detach().numpy(), torch.logsumexp(logits, -1).detach().numpy(),
            th.grad.numpy(), tw.grad.numpy())


@pytest.mark.parametrize("seed", range(5))
def test_against_library_gather(seed):
    rng = np.random.default_rng(seed)
    T, K, V = 11, 7, 23
    h = rng.standard_normal((T, K))
    w = rng.standard_normal((K, V)) * 0.5
    n_occ = 30
    src = rng.integers(0, T - 2, size=n_occ)        # rows T-2, T-1 carry no occurrence
    tgt = rng.integers(0, V, size=n_occ)
    g = rng.standard_normal(n_occ)
    logp, lse = oracle.logprob_ref_fwd(h, w, src, tgt)
    dh, dw = oracle.logprob_ref_bwd(h, w, src, tgt, g)
    rl, rlse, rdh, rdw = _torch_ref(h, w, src, tgt, g)
    np.testing.assert_allclose(logp, rl, atol=1e-12)
    used = np.unique(src)
    np.testing.assert_allclose(lse[used], rlse[used], atol=1e-12)
    assert np.isnan(lse[T - 2:]).all()
    np.testing.assert_allclose(dh, rdh, atol=1e-12)
    np.testing.assert_allclose(dw, rdw, atol=1e-12)
    gz = oracle.logprob_ref_gz(h, w, src, tgt, g, np.arange(T))
    np.testing.assert_allclose(gz @ w.T, dh, atol=1e-12)
    np.testing.assert_allclose(h.T @ gz, dw, atol=1e-12)


def test_one_occurrence_per_row_is_cross_entropy():
    rng = np.random.default_rng(9)
    T, K, V = 13, 5, 17
    h, w = rng.standard_normal((T, K)), rng.standard_normal((K, V))
    tgt = rng.integers(0, V, size=T)
    logp, _ = oracle.logprob_ref_fwd(h, w, np.arange(T), tgt)
    ce = torch.nn.functional.cross_entropy(torch.tensor(h @ w), torch.tensor(tgt), reduction="sum")
    np.testing.assert_allclose(-logp.sum(), ce.item(), rtol=1e-13)


def test_shared_row_gradient_trie_packing():
    """At row C the gradients for targets D and E add: (p_C - e_D) + (p_C - e_E)."""
    g = golden("trie_packing_example.json")
    p = oracle.pack_ref(g["sequences"])
    rng = np.random.default_rng(1)
    h, w = rng.standard_normal((7, 6)), rng.standard_normal((6, 7))
    src, tgt = p["occ_source_rows"], p["occ_targets"]
    gz = oracle.logprob_ref_gz(h, w, src, tgt, -np.ones(len(src)), [2])   # L = sum of NLL
    z = h[2] @ w
    pc = np.exp(z - z.max()) / np.exp(z - z.max()).sum()
    e = np.eye(7)
    np.testing.assert_allclose(gz[0], (pc - e[3]) + (pc - e[4]), atol=1e-14)


def test_branch_average_equals_weighted_unique_tokens():
    """Tree Training eq. 1-5: (1/K) sum over paths of per-token losses equals
    sum over unique tokens of (g_t / K) * loss_t, value and gradient."""
    t = synth.galton_watson(seed=3, budget=300, seg=(3, 12), vocab=50)
    p = oracle.pack_ref(t.seqs)
    K = len(t.seqs)
    rng = np.random.default_rng(2)
    h, w = rng.standard_normal((p["T"], 6)), rng.standard_normal((6, 50)) * 0.3
    src, tgt = p["occ_source_rows"], p["occ_targets"]
    logp, _ = oracle.logprob_ref_fwd(h, w, src, tgt)
    sep_avg = -logp.sum() / K                             # every path, every position
    # unique tokens t (non-root rows) predicted from their parent row, weight g_t / K;
    # g_t counted by brute force over the input sequences
    bf = oracle.brute_force_prefixes(t.seqs)
    pre = {}
    for s, path in zip(t.seqs, p["paths"]):
        for j, r in enumerate(path):
            pre[int(r)] = tuple(int(x) for x in s[:j + 1])
    rows = [r for r in range(p["T"]) if p["parent_row"][r] >= 0]
    u_src = np.array([p["parent_row"][r] for r in rows])
    u_tgt = np.array([p["packed_ids"][r] for r in rows])
    lam = np.array([bf[pre[r]] / K for r in rows])
    ulogp, _ = oracle.logprob_ref_fwd(h, w, u_src, u_tgt)
    np.testing.assert_allclose(sep_avg, -(lam * ulogp).sum(), rtol=1e-12)
    dh1, dw1 = oracle.logprob_ref_bwd(h, w, src, tgt, -np.ones(len(src)) / K)
    dh2, dw2 = oracle.logprob_ref_bwd(h, w, u_src, u_tgt, -lam)
    np.testing.assert_allclose(dh1, dh2, atol=1e-12)
    np.testing.assert_allclose(dw1, dw2, atol=1e-12)


def test_finite_differences():
    rng = np.random.default_rng(4)
    T, K, V = 4, 3, 6
    h, w = rng.standard_normal((T, K)), rng.standard_normal((K, V))
    src = np.array([0, 0, 1, 2, 2, 2])
    tgt = rng.integers(0, V, size=6)
    wt = rng.random(6)
    loss = lambda hh, ww: -(wt * oracle.logprob_ref_fwd(hh, ww, src, tgt)[0]).sum()
    dh, dw = oracle.logprob_ref_bwd(h, w, src, tgt, -wt)
    eps = 1e-6
    for idx in np.ndindex(h.shape):
        hp, hm = h.copy(), h.copy()
        hp[idx] += eps
        hm[idx] -= eps
        assert abs((loss(hp, w) - loss(hm, w)) / (2 * eps) - dh[idx]) < 1e-7
    for idx in np.ndindex(w.shape):
        wp, wm = w.copy(), w.copy()
        wp[idx] += eps
        wm[idx] -= eps
        assert abs((loss(h, wp) - loss(h, wm)) / (2 * eps) - dw[idx]) < 1e-7
