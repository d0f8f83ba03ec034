"""Pins of the tree-correct causal depthwise conv1d oracle (oracle/conv.py).

Tree Training §3.2 "(ii) Causal convolution", eq. 11, Fig. 4: each chunk uses its
parent's last K-1 effective tokens as left context, which replicates the context of an
independent per-branch pass.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

rng = np.random.default_rng(21)


def _torch_causal_conv(x, w, b=None):
    """torch.nn.functional.conv1d, float64, depthwise, left padding K-1: [L, C] -> [L, C]."""
    L, C = x.shape
    K = w.shape[1]
    xt = torch.from_numpy(np.ascontiguousarray(x.T))[None]            # [1, C, L]
    wt = torch.from_numpy(np.ascontiguousarray(w))[:, None, :]        # [C, 1, K]
    bt = None if b is None else torch.from_numpy(np.asarray(b, dtype=np.float64))
    y = torch.nn.functional.conv1d(torch.nn.functional.pad(xt, (K - 1, 0)), wt, bt, groups=C)
    return y[0].numpy().T


def _tree(seed, n_seqs=12, max_len=30, vocab=4):
    r = np.random.default_rng(seed)
    seqs = synth.random_sequences(r, n_seqs, max_len, vocab, min_len=1)
    return seqs, oracle.pack_ref(seqs)


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_chain_is_plain_causal_conv(K):
    """One sequence: the tree conv is the ordinary causal conv (torch conv1d)."""
    seqs = [np.arange(37, dtype=np.int32)]
    ref = oracle.pack_ref(seqs)
    x = rng.normal(size=(37, 5))
    w = rng.normal(size=(5, K))
    b = rng.normal(size=5)
    assert np.allclose(oracle.conv1d_ref_fwd(x, w, ref["paths"], b), _torch_causal_conv(x, w, b), atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_every_sequence_sees_its_own_branch(seed):
    """Eq. 11's claim: on every input sequence the packed output equals the conv of that
    sequence alone (torch conv1d on the sequence's own rows)."""
    seqs, ref = _tree(seed)
    T, C, K = ref["T"], 6, 4
    x = rng.normal(size=(T, C))
    w = rng.normal(size=(C, K))
    y = oracle.conv1d_ref_fwd(x, w, ref["paths"])
    for path in ref["paths"]:
        p = np.asarray(path)
        assert np.allclose(y[p], _torch_causal_conv(x[p], w), atol=1e-12)


def test_figure4_sibling_tokens_are_not_context():
    """Fig. 4 (K = 3): a child chunk that follows a sibling branch in DFS order takes its
    left context from the parent's last two tokens, not from the sibling."""
    # root chain 0-1-2 (tokens 10, 11, 12); child A = 3-4 (tokens 20, 21); child B = 5-6
    seqs = [np.array([10, 11, 12, 20, 21], dtype=np.int32), np.array([10, 11, 12, 30, 31], dtype=np.int32)]
    ref = oracle.pack_ref(seqs)
    assert ref["T"] == 7 and list(ref["parent_row"]) == [-1, 0, 1, 2, 3, 2, 5]
    x = np.eye(7)  # one channel per row: y[i, j] = weight given to row j at row i
    w = np.tile(np.array([[1.0, 10.0, 100.0]]), (7, 1))  # taps: 2 back, 1 back, self
    y = oracle.conv1d_ref_fwd(x, w, ref["paths"])
    # row 5 (first token of B) sees rows 1, 2 (parent chain) and itself, never 3, 4 (A)
    assert y[5, 5] == 100.0 and y[5, 2] == 10.0 and y[5, 1] == 1.0
    assert y[5, 3] == 0.0 and y[5, 4] == 0.0
    assert y[6, 6] == 100.0 and y[6, 5] == 10.0 and y[6, 2] == 1.0


@pytest.mark.parametrize("seed", [3, 4])
def test_parent_link_form_agrees(seed):
    seqs, ref = _tree(seed)
    T = ref["T"]
    x = rng.normal(size=(T, 3))
    w = rng.normal(size=(3, 3))
    b = rng.normal(size=3)
    assert np.allclose(oracle.conv1d_ref_rows(x, w, ref["parent_row"], b),
                       oracle.conv1d_ref_fwd(x, w, ref["paths"], b), atol=1e-12)


def test_backward_matches_finite_differences():
    """L = sum(dy * y) is linear in x, w and the bias, so central differences are exact
    up to rounding."""
    seqs, ref = _tree(5, n_seqs=6, max_len=12)
    T, C, K = ref["T"], 3, 3
    x = rng.normal(size=(T, C))
    w = rng.normal(size=(C, K))
    b = rng.normal(size=C)
    dy = rng.normal(size=(T, C))
    dx, dw, db = oracle.conv1d_ref_bwd(x, w, dy, ref["paths"], b)
    L = lambda x_, w_, b_: float((dy * oracle.conv1d_ref_fwd(x_, w_, ref["paths"], b_)).sum())
    h = 1e-3
    for j in range(T):
        for c in range(C):
            e = np.zeros_like(x)
            e[j, c] = h
            assert (L(x + e, w, b) - L(x - e, w, b)) / (2 * h) == pytest.approx(dx[j, c], abs=1e-8)
    for c in range(C):
        for k in range(K):
            e = np.zeros_like(w)
            e[c, k] = h
            assert (L(x, w + e, b) - L(x, w - e, b)) / (2 * h) == pytest.approx(dw[c, k], abs=1e-8)
    assert np.allclose(db, dy.sum(axis=0))


def test_backward_matches_autograd_on_each_branch():
    """torch autograd through conv1d on every sequence, each row's output gradient given
    to one sequence through it, summed back into packed rows."""
    seqs, ref = _tree(6)
    T, C, K = ref["T"], 4, 4
    x = rng.normal(size=(T, C))
    w = rng.normal(size=(C, K))
    dy = rng.normal(size=(T, C))
    dx, dw, _ = oracle.conv1d_ref_bwd(x, w, dy, ref["paths"])
    xt = torch.from_numpy(x).requires_grad_()
    wt = torch.from_numpy(w).requires_grad_()
    used = np.zeros(T, dtype=bool)
    total = 0.0
    for path in ref["paths"]:
        p = torch.from_numpy(np.asarray(path, dtype=np.int64))
        xp = xt[p].T[None]
        yp = torch.nn.functional.conv1d(torch.nn.functional.pad(xp, (K - 1, 0)), wt[:, None, :], groups=C)[0].T
        mask = torch.from_numpy(~used[np.asarray(path)]).double()[:, None]
        total = total + (yp * torch.from_numpy(dy[np.asarray(path)]) * mask).sum()
        used[np.asarray(path)] = True
    total.backward()
    assert np.allclose(dx, xt.grad.numpy(), atol=1e-10)
    assert np.allclose(dw, wt.grad.numpy(), atol=1e-10)


def test_kernel_size_one_is_pointwise():
    seqs, ref = _tree(7)
    T = ref["T"]
    x = rng.normal(size=(T, 4))
    w = rng.normal(size=(4, 1))
    b = rng.normal(size=4)
    assert np.allclose(oracle.conv1d_ref_fwd(x, w, ref["paths"], b), x * w[:, 0] + b)
