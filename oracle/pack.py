"""Oracle packing: sequences -> token trie -> preorder rows, positions, nodes, occurrences.

Test infrastructure only (see the package docstring).

Sources:
* Trie packing (agillm.io), "Step 1 - Store each node once": a token is shared
  only when its whole preceding context is identical; packed tokens, packed index
  and position IDs (depth on the original path) of the ABCD/ABCE/ABFG example.
* Tree Training (arXiv 2511.00413) §3.1 eq. 8: the DFS serialisation visits a
  node's token, then each child subtree in turn; §3.2 eq. 9: a token's position
  is the length of its ancestor segments plus its offset in its own segment,
  which is its depth in the trie.
* Claw-R1 "Prefix Tree Merge", "1. build and compress": insert every sequence
  into a trie, merge single-child chains into nodes, number the nodes in preorder
  with inclusive [start, end] positions.
* Trie packing, "Share logits, preserve every prediction" and "The training-loop
  change is small": one occurrence (source row, target) per original next-token
  prediction, listed sequence by sequence.

Readings taken where the pages are silent:
* children (and roots) are ordered by first insertion, as both worked examples do;
* several roots make a forest, each root restarting positions at 0;
* a node (chunk) also ends where an input sequence ends, as the Claw-R1 example's
  node list does ([6,7] ends at seq1's end even though 7 has a single child);
* a duplicated sequence is a separate path: it counts in path_count and emits its
  own occurrences; no EOS target is appended.
"""
from __future__ import annotations

import numpy as np


def pack_ref(seqs, seq_weights=None) -> dict:
    """Pack token sequences into a prefix trie serialised in preorder.

    Returns a dict of numpy arrays:
      packed_ids[T], position_ids[T], subtree_end[T] (last preorder row of the
      row's subtree), path_count[T] (input sequences whose path holds the row),
      parent_row[T] (-1 for a root), node_of_token[T], node_start/node_end
      (inclusive)/node_parent[n_nodes], occ_source_rows/occ_targets/occ_seq
      (int32) and occ_weights (float32) [n_occ], occ_row_ptr[T+1] and
      occ_perm[n_occ] (occurrences stably sorted by source row), and
      ``paths``: per input sequence, the packed rows along it.
    """
    n_seqs = len(seqs)
    if seq_weights is None:
        seq_weights = [1.0] * n_seqs
    # --- insert every sequence into a dict trie (insertion-ordered children) ---
    tok: list[int] = []
    kids: list[dict] = []
    through: list[int] = []      # sequences whose path contains the trie node
    ends: list[int] = []         # sequences that end at the trie node
    roots: dict = {}
    trie_paths = []
    for s in seqs:
        level = roots
        path = []
        for t in s:
            t = int(t)
            node = level.get(t)
            if node is None:
                node = len(tok)
                tok.append(t)
                kids.append({})
                through.append(0)
                ends.append(0)
                level[t] = node
            through[node] += 1
            path.append(node)
            level = kids[node]
        if path:
            ends[path[-1]] += 1
        trie_paths.append(path)

    # --- preorder DFS (eq. 8), children in insertion order; explicit stack ---
    order, depth, tparent = [], [], []
    stack = [(r, 0, -1) for r in reversed(list(roots.values()))]
    while stack:
        n, dep, par = stack.pop()
        order.append(n)
        depth.append(dep)
        tparent.append(par)
        for c in reversed(list(kids[n].values())):
            stack.append((c, dep + 1, n))
    T = len(order)
    row_of = {n: i for i, n in enumerate(order)}
    packed_ids = np.array([tok[n] for n in order], dtype=np.int32)
    position_ids = np.array(depth, dtype=np.int32)
    parent_row = np.array([row_of[p] if p >= 0 else -1 for p in tparent], dtype=np.int32)
    path_count = np.array([through[n] for n in order], dtype=np.int32)

    # subtree sizes from children (reverse preorder visits children before parents)
    size = np.ones(T, dtype=np.int64)
    for i in range(T - 1, -1, -1):
        if parent_row[i] >= 0:
            size[parent_row[i]] += size[i]
    subtree_end = (np.arange(T) + size - 1).astype(np.int32)

    # --- nodes: maximal single-child chains, broken at forks, roots and sequence ends ---
    starts = []
    for i in range(T):
        p = parent_row[i]
        if p < 0 or len(kids[order[p]]) != 1 or ends[order[p]] > 0:
            starts.append(i)
    n_nodes = len(starts)
    node_start = np.array(starts, dtype=np.int32)
    node_end = (np.array(starts[1:] + [T], dtype=np.int32) - 1) if starts else np.zeros(0, np.int32)
    node_of_token = np.empty(T, dtype=np.int32)
    for c in range(n_nodes):
        node_of_token[node_start[c]:node_end[c] + 1] = c
    node_parent = np.array([node_of_token[parent_row[s]] if parent_row[s] >= 0 else -1
                            for s in starts], dtype=np.int32)

    # --- occurrences: sequence-major, then position along the sequence ---
    src, tgt, wts, sq = [], [], [], []
    paths = []
    for k, (s, path) in enumerate(zip(seqs, trie_paths)):
        rows = [row_of[n] for n in path]
        paths.append(np.array(rows, dtype=np.int32))
        for t in range(len(rows) - 1):
            src.append(rows[t])
            tgt.append(int(s[t + 1]))
            wts.append(seq_weights[k])
            sq.append(k)
    occ_source_rows = np.array(src, dtype=np.int32)
    occ_targets = np.array(tgt, dtype=np.int32)
    occ_weights = np.array(wts, dtype=np.float32)
    occ_seq = np.array(sq, dtype=np.int32)
    counts = np.bincount(occ_source_rows, minlength=T) if len(src) else np.zeros(T, np.int64)
    occ_row_ptr = np.zeros(T + 1, dtype=np.int32)
    occ_row_ptr[1:] = np.cumsum(counts)
    occ_perm = np.argsort(occ_source_rows, kind="stable").astype(np.int32)

    return dict(T=T, n_nodes=n_nodes, n_occ=len(src), n_roots=len(roots),
                packed_ids=packed_ids, position_ids=position_ids, subtree_end=subtree_end,
                path_count=path_count, parent_row=parent_row, node_of_token=node_of_token,
                node_start=node_start, node_end=node_end, node_parent=node_parent,
                occ_source_rows=occ_source_rows, occ_targets=occ_targets,
                occ_weights=occ_weights, occ_seq=occ_seq, occ_row_ptr=occ_row_ptr,
                occ_perm=occ_perm, paths=paths)


def brute_force_prefixes(seqs) -> dict:
    """Independent restatement of "shareable iff the whole preceding context is
    identical": every distinct non-empty prefix of an input sequence is one packed
    token. Returns {prefix tuple: number of sequences having that prefix}."""
    count: dict = {}
    for s in seqs:
        s = tuple(int(t) for t in s)
        for L in range(1, len(s) + 1):
            count[s[:L]] = count.get(s[:L], 0) + 1
    return count
