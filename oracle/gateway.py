"""Oracle partition-gateway attention.

Test infrastructure only (see the package docstring).

Tree Training (arXiv 2511.00413) §3.3 "Differentiable partition boundaries" and
Appendix B.1-B.5: a tree too large for one pass is cut into partitions. At a cut
node n_c, a child partition C runs on its own rows only and reads the keys and values
its parent partition P has accumulated, through a gateway:

* the past: P's key/value rows up to and including n_c's last token (B.2 step 1),
  possibly preceded by P's own inherited past;
* an additive bias over the past, 0 where the row is an ancestor of n_c and -inf
  elsewhere (eq. 15-16): P's preorder sequence can hold sibling subtrees of n_c
  before it, which C must not see;
* the combined mask of eq. 14: the bias on past columns, the ordinary tree mask on
  C's own columns;
* positions continuing from pos_offset(C) = pos_offset(P) + pos(n_c) + |T_{n_c}|
  (eq. 17), i.e. one past the depth of n_c's last token;
* gradients that reach the gateway keys and values from several child partitions
  are summed (B.5 keeps that sum in float32; here everything is float64).

Readings taken: the past holds P's rows through n_c's last token (B.1's shape
[1, H, e_nc, d]); a past row is visible iff it is an ancestor of the child
partition's first row. For a partition whose own past was already ancestor-filtered
(eq. 16's [0, past_len_P) term) the two agree; the ancestor rule is the one that keeps
the exactness of eq. 6 when an inherited past still holds masked rows.

The attention itself is written out densely: a boolean mask over [C's rows] x
[past + C's rows] and an ordinary masked softmax, forward and backward, so it
depends on no mask encoding.
"""
from __future__ import annotations

import numpy as np


def _kv_of(Hq: int, Hkv: int) -> np.ndarray:
    assert Hq % Hkv == 0
    return np.arange(Hq) // (Hq // Hkv)


def gateway_mask_ref(past_visible, child_end) -> np.ndarray:
    """Eq. 14 as a boolean matrix [Tc, past_len + Tc]: past column j visible iff
    past_visible[j]; own column past_len + j visible to own row i iff j <= i <=
    child_end[j] (j an ancestor-or-self of i inside C)."""
    pv = np.asarray(past_visible, dtype=bool)
    ce = np.asarray(child_end, dtype=np.int64)
    P, Tc = pv.shape[0], ce.shape[0]
    m = np.zeros((Tc, P + Tc), dtype=bool)
    m[:, :P] = pv[None, :]
    i = np.arange(Tc)[:, None]
    j = np.arange(Tc)[None, :]
    m[:, P:] = (j <= i) & (i <= ce[None, :])
    return m


def _softmax_rows(q, k_all, mask, scale):
    """Per query head: scores [Hq, Tc, Tk], probabilities and LSE under `mask`."""
    s = np.einsum("ihd,jhd->hij", q, k_all) * scale
    s = np.where(mask[None], s, -np.inf)
    mx = s.max(axis=-1, keepdims=True)
    e = np.where(mask[None], np.exp(s - mx), 0.0)
    l = e.sum(axis=-1, keepdims=True)
    return e / l, (mx + np.log(l))[..., 0]


def gateway_attn_ref_fwd(q, k_all, v_all, past_len, past_visible, child_end, scale=None):
    """O [Tc, Hq, d] and LSE [Hq, Tc] of the child partition's queries q [Tc, Hq, d]
    over the keys/values k_all, v_all [past_len + Tc, Hkv, d] (past rows first)."""
    q, k_all, v_all = (np.asarray(x, dtype=np.float64) for x in (q, k_all, v_all))
    Tc, Hq, d = q.shape
    Hkv = k_all.shape[1]
    assert k_all.shape[0] == past_len + Tc
    sc = 1.0 / np.sqrt(d) if scale is None or scale <= 0 else float(scale)
    kv = _kv_of(Hq, Hkv)
    mask = gateway_mask_ref(past_visible, child_end)
    p, lse = _softmax_rows(q, k_all[:, kv], mask, sc)
    o = np.einsum("hij,jhd->ihd", p, v_all[:, kv])
    return o, lse


def gateway_attn_ref_bwd(q, k_all, v_all, dout, past_len, past_visible, child_end, scale=None):
    """dq [Tc, Hq, d], dk_all and dv_all [past_len + Tc, Hkv, d] for L = sum(dout * O):
    dV = P^T dO, dP = dO V^T, dS = P (dP - rowsum(P dP)), dQ = scale dS K, dK = scale dS^T Q,
    K/V gradients summed over each KV head's query heads."""
    q, k_all, v_all, dout = (np.asarray(x, dtype=np.float64) for x in (q, k_all, v_all, dout))
    Tc, Hq, d = q.shape
    Tk, Hkv = k_all.shape[0], k_all.shape[1]
    sc = 1.0 / np.sqrt(d) if scale is None or scale <= 0 else float(scale)
    kv = _kv_of(Hq, Hkv)
    mask = gateway_mask_ref(past_visible, child_end)
    kq, vq = k_all[:, kv], v_all[:, kv]                      # [Tk, Hq, d]
    p, _ = _softmax_rows(q, kq, mask, sc)                    # [Hq, Tc, Tk]
    dv_h = np.einsum("hij,ihd->jhd", p, dout)
    dp = np.einsum("ihd,jhd->hij", dout, vq)
    ds = p * (dp - (p * dp).sum(axis=-1, keepdims=True))
    dq = np.einsum("hij,jhd->ihd", ds, kq) * sc
    dk_h = np.einsum("hij,ihd->jhd", ds, q) * sc
    dk = np.zeros((Tk, Hkv, d))
    dv = np.zeros((Tk, Hkv, d))
    for h in range(Hq):
        dk[:, kv[h]] += dk_h[:, h]
        dv[:, kv[h]] += dv_h[:, h]
    return dq, dk, dv


def is_ancestor_or_self(parent_row, a: int, r: int) -> bool:
    """True iff row a lies on the root-to-r path of the tree given by parent links."""
    while r >= 0:
        if r == a:
            return True
        r = int(parent_row[r])
    return False


def local_subtree_end(rows, subtree_end) -> np.ndarray:
    """subtree_end of a partition's rows, renumbered 0..len-1: rows is an increasing
    list of whole-tree rows (a preorder subsequence closed under taking ancestors
    inside it), and row rows[i]'s local subtree ends at the last listed row of its
    whole-tree subtree."""
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty(rows.shape[0], dtype=np.int64)
    for i, r in enumerate(rows):
        out[i] = np.searchsorted(rows, subtree_end[r], side="right") - 1
    return out


def gateway_for_child(ref, parent_seq, child_first_row: int):
    """The gateway of the child partition rooted at whole-tree row c = child_first_row.

    parent_seq: the whole-tree rows whose keys/values the parent partition holds, in
    its own order (its inherited past first, then its own rows in preorder). The cut
    node's last token is c's parent row; the past is parent_seq through it (B.2), each
    past row visible iff it is an ancestor of c (eq. 15-16). Returns past_rows,
    past_visible, the child's rows, their local subtree_end, and pos_offset (eq. 17:
    the depth of the cut node's first token plus its token count, i.e. one past the
    depth of its last token)."""
    c = int(child_first_row)
    cut_last = int(ref["parent_row"][c])
    assert cut_last >= 0, "a child partition starts below some cut node"
    parent_seq = [int(r) for r in parent_seq]
    past_rows = parent_seq[: parent_seq.index(cut_last) + 1]
    pv = np.array([is_ancestor_or_self(ref["parent_row"], r, cut_last) for r in past_rows], dtype=bool)
    child_rows = np.arange(c, int(ref["subtree_end"][c]) + 1)
    # eq. 17: the depth of the cut node's first token plus its token count, the cut
    # node's tokens running from its chunk's first token through c's parent row
    first = int(ref["node_start"][int(ref["node_of_token"][cut_last])])
    pos_offset = int(ref["position_ids"][first]) + (cut_last - first + 1)
    return dict(past_rows=np.array(past_rows, dtype=np.int64), past_visible=pv, child_rows=child_rows,
                child_end=local_subtree_end(child_rows, ref["subtree_end"]), pos_offset=pos_offset)
