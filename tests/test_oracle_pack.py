"""Pins for oracle.pack_ref: the pages' worked examples and a brute-force restatement."""
import numpy as np
import pytest

import oracle
import synth
from conftest import golden


def test_trie_packing_example():
    g = golden("trie_packing_example.json")
    p = oracle.pack_ref(g["sequences"])
    assert p["T"] == 7
    assert p["packed_ids"].tolist() == g["packed_tokens"]
    assert p["position_ids"].tolist() == g["position_ids"]
    assert p["occ_source_rows"].tolist() == g["source_rows"]
    assert p["occ_targets"].tolist() == g["targets"]
    assert p["n_occ"] == g["n_occurrences"]
    assert len(set(p["occ_source_rows"].tolist())) == g["n_logit_rows"]
    assert p["T"] == g["ffn_rows_packed"]
    assert sum(len(s) for s in g["sequences"]) == g["ffn_rows_unpacked"]
    # derived from the trie: C's subtree is C D E, B's is everything after A
    assert p["subtree_end"].tolist() == [6, 6, 4, 3, 4, 6, 6]
    assert p["path_count"].tolist() == [3, 3, 2, 1, 1, 1, 1]


def test_prefix_tree_merge_example():
    g = golden("prefix_tree_merge_example.json")
    p = oracle.pack_ref(g["sequences"])
    assert p["packed_ids"].tolist() == g["packed_sequence"]
    assert p["T"] == g["packed_tokens"]
    assert sum(len(s) for s in g["sequences"]) == g["original_tokens"]
    assert round(100 * oracle.token_ratio(p["T"], g["sequences"]), 1) == g["token_ratio_percent"]
    assert p["n_nodes"] == len(g["nodes"])
    for c, node in enumerate(g["nodes"]):
        assert [int(p["node_start"][c]), int(p["node_end"][c])] == node["pos"]
        assert int(p["node_parent"][c]) == node["parent"]
        toks = p["packed_ids"][node["pos"][0]:node["pos"][1] + 1].tolist()
        assert toks == node["tokens"]
        members = [k for k, path in enumerate(p["paths"]) if node["pos"][0] in path.tolist()]
        assert members == node["seqs"]
    assert [x.tolist() for x in p["paths"]] == g["sequence_paths"]
    # derived: depth positions and subtree ends of the 9 packed rows
    assert p["position_ids"].tolist() == [0, 1, 2, 3, 4, 3, 4, 5, 6]
    assert p["subtree_end"].tolist() == [8, 8, 8, 4, 4, 8, 8, 8, 8]
    assert p["n_occ"] == 4 + 4 + 6


def _check_against_prefixes(seqs):
    p = oracle.pack_ref(seqs)
    bf = oracle.brute_force_prefixes(seqs)
    T = p["T"]
    assert T == len(bf)
    # reconstruct every row's prefix from its path
    prefix = [None] * T
    for s, path in zip(seqs, p["paths"]):
        for t, r in enumerate(path):
            pre = tuple(int(x) for x in s[:t + 1])
            assert prefix[r] is None or prefix[r] == pre
            prefix[r] = pre
    assert set(prefix) == set(bf.keys())
    for i in range(T):
        assert p["packed_ids"][i] == prefix[i][-1]
        assert p["position_ids"][i] == len(prefix[i]) - 1
        assert p["path_count"][i] == bf[prefix[i]]
        # subtree interval <=> prefix relation (preorder contiguity)
        for j in range(T):
            in_sub = i <= j <= p["subtree_end"][i]
            assert in_sub == (prefix[j][:len(prefix[i])] == prefix[i])
    # siblings appear in order of first insertion
    first_seen = {}
    for s in seqs:
        for t in range(len(s)):
            first_seen.setdefault(tuple(int(x) for x in s[:t + 1]), len(first_seen))
    for i in range(T):
        for j in range(i + 1, T):
            if prefix[i][:-1] == prefix[j][:-1]:
                assert first_seen[prefix[i]] < first_seen[prefix[j]]
    # occurrences: sequence-major next-token predictions
    o = 0
    for k, s in enumerate(seqs):
        for t in range(len(s) - 1):
            assert prefix[p["occ_source_rows"][o]] == tuple(int(x) for x in s[:t + 1])
            assert p["occ_targets"][o] == s[t + 1]
            assert p["occ_seq"][o] == k
            o += 1
    assert o == p["n_occ"]
    # CSR by row, stable
    perm = p["occ_perm"]
    rp = p["occ_row_ptr"]
    assert rp[0] == 0 and rp[-1] == p["n_occ"]
    for r in range(T):
        seg = perm[rp[r]:rp[r + 1]]
        assert (p["occ_source_rows"][seg] == r).all()
        assert (np.diff(seg) > 0).all()
    # nodes: consecutive chains; a boundary exactly at roots, forks and sequence ends
    ends = {tuple(int(x) for x in s) for s in seqs if len(s)}
    nchild = {}
    for pre in prefix:
        if len(pre) > 1:
            nchild[pre[:-1]] = nchild.get(pre[:-1], 0) + 1
    for i in range(T):
        par = prefix[i][:-1]
        boundary = len(par) == 0 or nchild.get(par, 0) != 1 or par in ends
        assert (p["node_start"] == i).any() == boundary
    return p


@pytest.mark.parametrize("seed", range(40))
def test_random_against_brute_force(seed):
    rng = np.random.default_rng(seed)
    seqs = synth.random_sequences(rng, int(rng.integers(1, 7)), 9, vocab=int(rng.integers(2, 4)))
    _check_against_prefixes(seqs)


def test_duplicates_and_prefix_sequences():
    seqs = [[5, 6, 7], [5, 6, 7], [5, 6], [], [9], [5, 6, 7, 8]]
    p = _check_against_prefixes(seqs)
    assert p["n_roots"] == 2
    assert p["path_count"][0] == 4


def test_agentic_short_closed_form():
    """Short-prompt agentic tree: 256 + 16*128 packed rows; allowed pairs in closed
    form sum_i (pos_i + 1) over the prompt and four 512-token chains."""
    t = synth.agentic_short()
    p = oracle.pack_ref(t.seqs)
    assert p["T"] == 256 + 16 * 128
    P = oracle.allowed_pairs_from_paths(p["paths"], p["T"])
    closed = 256 * 257 // 2 + 4 * sum(range(257, 769))
    assert P == closed == 1082496
    assert P == int((p["position_ids"].astype(np.int64) + 1).sum())


def test_tiny_tree_shape():
    t = synth.tiny_tree()
    p = oracle.pack_ref(t.seqs)
    assert p["T"] == 76 and p["n_occ"] == 129
    assert oracle.allowed_pairs_from_paths(p["paths"], p["T"]) == 2142
    assert len(set(p["occ_source_rows"].tolist())) == 73
