"""Pins for oracle.attention: printed visibility, the pages' dense-mask builder,
library attention (torch scaled_dot_product_attention, float64 CPU) on special
cases and on brute-force dense masks, and gradient identities."""
import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import golden


def _sdpa(q, k, v, mask=None, causal=False, dout=None):
    """Library attention in float64 with autograd; q [T,Hq,d], k/v [T,Hkv,d]."""
    Hq, Hkv = q.shape[1], k.shape[1]
    tq = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    tk = torch.tensor(k, dtype=torch.float64, requires_grad=True)
    tv = torch.tensor(v, dtype=torch.float64, requires_grad=True)
    rep = Hq // Hkv
    kk = tk.repeat_interleave(rep, dim=1).transpose(0, 1)
    vv = tv.repeat_interleave(rep, dim=1).transpose(0, 1)
    m = None if mask is None else torch.tensor(mask)
    o = torch.nn.functional.scaled_dot_product_attention(
        tq.transpose(0, 1), kk, vv, attn_mask=m, is_causal=causal).transpose(0, 1)
    res = [o.detach().numpy()]
    if dout is not None:
        o.backward(torch.tensor(dout, dtype=torch.float64))
        res += [tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()]
    return res


def test_visibility_statements_trie_packing():
    g = golden("trie_packing_example.json")
    p = oracle.pack_ref(g["sequences"])
    m = oracle.mask_from_paths(p["paths"], p["T"])
    vs = g["visibility_statements"]
    E, G = 4, 6
    assert sorted(np.nonzero(m[E])[0].tolist()) == vs["E_sees"]
    assert not m[E, vs["E_never"]].any()
    assert sorted(np.nonzero(m[G])[0].tolist()) == vs["G_sees"]
    assert not m[G, vs["G_never"]].any()
    assert int(m.sum()) == g["allowed_pairs_packed"]
    # differs from the ordinary lower-triangular mask of a length-7 sequence
    assert not np.array_equal(m, np.tril(np.ones((7, 7), dtype=bool)))


def test_visibility_rows_prefix_tree_merge():
    g = golden("prefix_tree_merge_example.json")
    p = oracle.pack_ref(g["sequences"])
    m = oracle.mask_from_paths(p["paths"], p["T"])
    for path in g["sequence_paths"]:
        leaf = path[-1]
        assert sorted(np.nonzero(m[leaf])[0].tolist()) == path


@pytest.mark.parametrize("seed", range(25))
def test_three_mask_readings_agree(seed):
    """Path unpacking == the chunk builder of the paper's appendix A.1 == the
    per-key interval rule j <= i <= subtree_end[j] (the encoding the kernels use)."""
    rng = np.random.default_rng(100 + seed)
    seqs = synth.random_sequences(rng, int(rng.integers(1, 8)), 12, vocab=int(rng.integers(2, 4)))
    p = oracle.pack_ref(seqs)
    T = p["T"]
    if T == 0:
        return
    m_path = oracle.mask_from_paths(p["paths"], T)
    m_chunk = oracle.dense_mask_from_chunks(p["node_start"], p["node_end"], p["node_parent"], T)
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    m_int = (j <= i) & (i <= p["subtree_end"][None, :])
    assert np.array_equal(m_path, m_chunk)
    assert np.array_equal(m_path, m_int)
    assert int(m_path.sum()) == int((p["position_ids"].astype(np.int64) + 1).sum())


def _rand_qkv(rng, T, Hq, Hkv, d):
    return (rng.standard_normal((T, Hq, d)), rng.standard_normal((T, Hkv, d)),
            rng.standard_normal((T, Hkv, d)), rng.standard_normal((T, Hq, d)))


def test_chain_is_ordinary_causal_attention():
    rng = np.random.default_rng(1)
    T, Hq, Hkv, d = 37, 4, 2, 16
    q, k, v, do = _rand_qkv(rng, T, Hq, Hkv, d)
    paths = [np.arange(T)]
    o, lse = oracle.attn_ref_fwd(q, k, v, paths)
    dq, dk, dv = oracle.attn_ref_bwd(q, k, v, do, paths)
    ro, rdq, rdk, rdv = _sdpa(q, k, v, causal=True, dout=do)
    for a, b in [(o, ro), (dq, rdq), (dk, rdk), (dv, rdv)]:
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)
    # LSE against the library log-sum-exp of the causal scores
    s = torch.einsum("ihd,jhd->hij", torch.tensor(q), torch.tensor(np.repeat(k, 2, axis=1))) / np.sqrt(d)
    s = s.masked_fill(torch.triu(torch.ones(T, T, dtype=torch.bool), 1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-11)


@pytest.mark.parametrize("seed", range(8))
def test_tree_against_library_dense_mask(seed):
    """Random trees (forests included): oracle == library attention under the
    appendix-A.1 dense mask, forward and all three gradients."""
    rng = np.random.default_rng(200 + seed)
    seqs = synth.random_sequences(rng, int(rng.integers(2, 7)), 14, vocab=3, min_len=1)
    p = oracle.pack_ref(seqs)
    T = p["T"]
    Hq, Hkv, d = [(2, 1, 8), (4, 2, 16), (4, 4, 8), (8, 2, 32)][seed % 4]
    q, k, v, do = _rand_qkv(rng, T, Hq, Hkv, d)
    m = oracle.dense_mask_from_chunks(p["node_start"], p["node_end"], p["node_parent"], T)
    o, lse = oracle.attn_ref_fwd(q, k, v, p["paths"])
    dq, dk, dv = oracle.attn_ref_bwd(q, k, v, do, p["paths"])
    ro, rdq, rdk, rdv = _sdpa(q, k, v, mask=m, dout=do)
    for a, b in [(o, ro), (dq, rdq), (dk, rdk), (dv, rdv)]:
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)


def test_forest_of_chains_is_packed_varlen():
    """A forest of chains is plain sequence packing: block-diagonal causal attention."""
    rng = np.random.default_rng(3)
    lens = [5, 9, 1, 7]
    seqs, tok = [], 0
    for L in lens:
        seqs.append(list(range(tok, tok + L)))
        tok += L
    p = oracle.pack_ref(seqs)
    T = p["T"]
    assert T == sum(lens)
    q, k, v, do = _rand_qkv(rng, T, 2, 2, 8)
    o, _ = oracle.attn_ref_fwd(q, k, v, p["paths"])
    s0 = 0
    for L in lens:
        sl = slice(s0, s0 + L)
        (ro,) = _sdpa(q[sl], k[sl], v[sl], causal=True)
        np.testing.assert_allclose(o[sl], ro, rtol=0, atol=1e-12)
        assert (p["position_ids"][sl] == np.arange(L)).all()
        s0 += L


def test_value_gradient_reaches_only_ancestors():
    """dV_j collects only from queries that see j: with dO nonzero at one row, every
    key off that row's path gets exactly zero gradient."""
    g = golden("trie_packing_example.json")
    p = oracle.pack_ref(g["sequences"])
    rng = np.random.default_rng(4)
    q, k, v, _ = _rand_qkv(rng, 7, 1, 1, 8)
    for i in range(7):
        do = np.zeros((7, 1, 8))
        do[i] = rng.standard_normal((1, 8))
        _, dk, dv = oracle.attn_ref_bwd(q, k, v, do, p["paths"])
        chain = [r for r in range(7) if oracle.mask_from_paths(p["paths"], 7)[i, r]]
        off = [r for r in range(7) if r not in chain]
        assert np.abs(dv[off]).max(initial=0) == 0 and np.abs(dk[off]).max(initial=0) == 0
        assert np.abs(dv[chain]).min() > 0


def test_row_sampled_functions_match_full():
    t = synth.tiny_tree()
    p = oracle.pack_ref(t.seqs)
    rng = np.random.default_rng(5)
    q, k, v, do = _rand_qkv(rng, p["T"], 4, 2, 16)
    o, lse = oracle.attn_ref_fwd(q, k, v, p["paths"])
    dq, dk, dv = oracle.attn_ref_bwd(q, k, v, do, p["paths"])
    rows = [0, 5, 23, 24, 31, 43, 44, 60, 75]
    so, slse = oracle.attn_ref_rows(q, k, v, p["paths"], rows)
    np.testing.assert_allclose(so, o[rows], atol=1e-12)
    np.testing.assert_allclose(slse, lse[:, rows], atol=1e-12)
    np.testing.assert_allclose(oracle.attn_ref_dq_rows(q, k, v, do, p["paths"], rows), dq[rows], atol=1e-11)
    sdk, sdv = oracle.attn_ref_dkdv_rows(q, k, v, do, p["paths"], rows)
    np.testing.assert_allclose(sdk, dk[rows], atol=1e-11)
    np.testing.assert_allclose(sdv, dv[rows], atol=1e-11)
    # identities that hold at any size: sum_j dV_j = sum_i dO_i per KV group, sum_j dK_j = 0
    np.testing.assert_allclose(dv.sum(0), do.reshape(p["T"], 2, 2, 16).sum(axis=(0, 2)), atol=1e-10)
    np.testing.assert_allclose(dk.sum(0), 0, atol=1e-10)


def test_leaf_paths_cover_rows():
    t = synth.tiny_tree()
    p = oracle.pack_ref(t.seqs)
    lp = oracle.leaf_paths_from_parents(p["parent_row"])
    assert len(lp) == 3
    assert [x.tolist() for x in lp] == [x.tolist() for x in p["paths"]]
