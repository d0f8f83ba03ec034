"""Pins of the partition-gateway attention oracle (oracle/gateway.py).

Tree Training §3.3 "Differentiable partition boundaries": with gateways, every token
is computed exactly once and the partitioned pass equals the unpartitioned one. So the
gateway oracle, run partition by partition, must reproduce the whole-tree per-path
oracle: outputs and LSE at every row, and -- with the gradients that reach each
gateway row summed over the child partitions (B.5) -- dQ, dK and dV at every row.
Appendix B.3's example fixes the bias; eq. 17 fixes the positions.
"""
import numpy as np
import pytest

import oracle
import synth

rng = np.random.default_rng(77)


def _qkv(T, Hq=4, Hkv=2, d=8, seed=0):
    r = np.random.default_rng(seed)
    return (r.normal(size=(T, Hq, d)), r.normal(size=(T, Hkv, d)), r.normal(size=(T, Hkv, d)),
            r.normal(size=(T, Hq, d)))


def _cut_candidates(ref):
    """Nodes with at least one child node: (cut node, its child nodes' first rows)."""
    kids = {}
    for n in range(len(ref["node_start"])):
        p = int(ref["node_parent"][n])
        if p >= 0:
            kids.setdefault(p, []).append(int(ref["node_start"][n]))
    return kids


def _partitioned(ref, q, k, v, do, parent_rows, children, with_bwd=True):
    """Run the parent partition (its own rows, no past) and every child partition through
    its gateway; return whole-tree O, LSE and the summed gradients."""
    T, Hq, d = q.shape
    o = np.full((T, Hq, d), np.nan)
    lse = np.full((Hq, T), np.nan)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    pr = np.asarray(parent_rows)
    pe = oracle.local_subtree_end(pr, ref["subtree_end"])
    po, pl = oracle.gateway_attn_ref_fwd(q[pr], k[pr], v[pr], 0, np.zeros(0, bool), pe)
    o[pr], lse[:, pr] = po, pl
    if with_bwd:
        a, b, c = oracle.gateway_attn_ref_bwd(q[pr], k[pr], v[pr], do[pr], 0, np.zeros(0, bool), pe)
        dq[pr] += a
        dk[pr] += b
        dv[pr] += c
    for ch in children:
        g = ch if isinstance(ch, dict) else oracle.gateway_for_child(ref, parent_rows, ch)
        rows = np.concatenate([g["past_rows"], g["child_rows"]])
        cr = g["child_rows"]
        P = len(g["past_rows"])
        co, cl = oracle.gateway_attn_ref_fwd(q[cr], k[rows], v[rows], P, g["past_visible"], g["child_end"])
        o[cr], lse[:, cr] = co, cl
        if with_bwd:
            a, b, c = oracle.gateway_attn_ref_bwd(q[cr], k[rows], v[rows], do[cr], P, g["past_visible"],
                                                  g["child_end"])
            dq[cr] += a
            np.add.at(dk, rows, b)     # gateway rows collect every child's gradient (B.5)
            np.add.at(dv, rows, c)
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("seed", range(6))
def test_partitioned_pass_equals_whole_tree(seed):
    """Cut at a random node with children; each child subtree is a child partition."""
    r = np.random.default_rng(seed)
    seqs = synth.random_sequences(r, 14, 24, vocab=3, min_len=2)
    ref = oracle.pack_ref(seqs)
    cands = _cut_candidates(ref)
    assert cands
    cut = sorted(cands)[int(r.integers(0, len(cands)))]
    children = cands[cut]
    T = ref["T"]
    cut_rows = set()
    for c in children:
        cut_rows.update(range(c, int(ref["subtree_end"][c]) + 1))
    parent_rows = [i for i in range(T) if i not in cut_rows]
    q, k, v, do = _qkv(T, seed=seed)
    o, lse, dq, dk, dv = _partitioned(ref, q, k, v, do, parent_rows, children)
    ro, rl = oracle.attn_ref_fwd(q, k, v, ref["paths"])
    rdq, rdk, rdv = oracle.attn_ref_bwd(q, k, v, do, ref["paths"])
    assert np.allclose(o, ro, atol=1e-12) and np.allclose(lse, rl, atol=1e-12)
    assert np.allclose(dq, rdq, atol=1e-10)
    assert np.allclose(dk, rdk, atol=1e-10) and np.allclose(dv, rdv, atol=1e-10)


def test_two_level_partition_equals_whole_tree():
    """A child partition that is itself cut: the grandchild's past is the child's
    accumulated sequence (its own past, then its rows), ancestor-filtered."""
    for seed in range(4):
        r = np.random.default_rng(100 + seed)
        seqs = synth.random_sequences(r, 16, 30, vocab=2, min_len=3)
        ref = oracle.pack_ref(seqs)
        cands = _cut_candidates(ref)
        # a cut node whose child subtree holds another cut node
        pairs = [(c, g) for n, cs in cands.items() for c in cs for m, gs in cands.items()
                 for g in gs if c < int(ref["node_start"][m]) <= int(ref["subtree_end"][c]) and m != n]
        if not pairs:
            continue
        c, g = pairs[int(r.integers(0, len(pairs)))]
        T = ref["T"]
        c_rows = set(range(c, int(ref["subtree_end"][c]) + 1))
        g_rows = set(range(g, int(ref["subtree_end"][g]) + 1))
        parent_rows = [i for i in range(T) if i not in c_rows]
        gc = oracle.gateway_for_child(ref, parent_rows, c)
        own_c = np.array([i for i in gc["child_rows"] if i not in g_rows])
        gc = dict(gc, child_rows=own_c, child_end=oracle.local_subtree_end(own_c, ref["subtree_end"]))
        c_seq = list(gc["past_rows"]) + list(own_c)
        gg = oracle.gateway_for_child(ref, c_seq, g)
        q, k, v, do = _qkv(T, seed=seed)
        o, lse, dq, dk, dv = _partitioned(ref, q, k, v, do, parent_rows, [gc, gg])
        ro, rl = oracle.attn_ref_fwd(q, k, v, ref["paths"])
        rdq, rdk, rdv = oracle.attn_ref_bwd(q, k, v, do, ref["paths"])
        assert np.allclose(o, ro, atol=1e-12) and np.allclose(lse, rl, atol=1e-12)
        assert np.allclose(dq, rdq, atol=1e-10) and np.allclose(dk, rdk, atol=1e-10)
        assert np.allclose(dv, rdv, atol=1e-10)
        return
    pytest.fail("no two-level cut found")


def test_appendix_b3_example_masks_the_sibling():
    """B.3: the parent's sequence is [a, b, c1, c2] with siblings c1, c2 and the cut at
    c2; the gateway holds c1's token, which c2's children must not see. B.4: then the
    child's position offset (3) differs from the past length (4)."""
    a, b, c1, c2, dd = 10, 11, 12, 13, 14
    ref = oracle.pack_ref([[a, b, c1], [a, b, c2, dd]])
    assert ref["packed_ids"].tolist() == [a, b, c1, c2, dd]
    g = oracle.gateway_for_child(ref, [0, 1, 2, 3], 4)
    assert g["past_rows"].tolist() == [0, 1, 2, 3]
    assert g["past_visible"].tolist() == [True, True, False, True]
    assert g["pos_offset"] == 3 and len(g["past_rows"]) == 4


def test_position_offset_continues_the_depth():
    """Eq. 17: pos_offset plus the depth inside the child partition is the row's depth in
    the whole tree, for every possible cut."""
    seqs = synth.random_sequences(rng, 20, 30, vocab=3, min_len=2)
    ref = oracle.pack_ref(seqs)
    for cut, children in _cut_candidates(ref).items():
        for c in children:
            g = oracle.gateway_for_child(ref, list(range(ref["T"])), c)
            rows = g["child_rows"]
            local_depth = ref["position_ids"][rows] - ref["position_ids"][c]
            assert np.array_equal(g["pos_offset"] + local_depth, ref["position_ids"][rows])


def test_no_past_is_plain_tree_attention():
    seqs = synth.random_sequences(rng, 10, 20, vocab=3)
    ref = oracle.pack_ref(seqs)
    T = ref["T"]
    q, k, v, _ = _qkv(T, seed=3)
    o, l = oracle.gateway_attn_ref_fwd(q, k, v, 0, np.zeros(0, bool), ref["subtree_end"])
    ro, rl = oracle.attn_ref_fwd(q, k, v, ref["paths"])
    assert np.allclose(o, ro, atol=1e-12) and np.allclose(l, rl, atol=1e-12)


def test_interval_encoding_of_eq14():
    """The kernels' reading of eq. 14: in one key space [past; own rows], with own row i
    at index past_len + i, a past key is visible to every own row (subtree end = last
    row) or to none (end = itself, no query there), and an own key keeps its subtree
    interval shifted by past_len. Brute force against the dense mask."""
    for _ in range(20):
        P = int(rng.integers(0, 40))
        seqs = synth.random_sequences(rng, 8, 16, vocab=3)
        ref = oracle.pack_ref(seqs)
        Tc = ref["T"]
        if Tc == 0:
            continue
        vis = rng.random(P) < 0.5
        end = np.concatenate([np.where(vis, P + Tc - 1, np.arange(P)), P + ref["subtree_end"]])
        i = P + np.arange(Tc)[:, None]
        j = np.arange(P + Tc)[None, :]
        enc = (j <= i) & (i <= end[None, :])
        assert np.array_equal(enc, oracle.gateway_mask_ref(vis, ref["subtree_end"]))
