"""Oracle workload statistics.

Test infrastructure only (see the package docstring).

* Potential overlap ratio, Tree Training (arXiv 2511.00413) §4.1 eq. 12:
  POR = 1 - N_tree / N_base, N_base the token count of the baseline
  serialisation (every path on its own, eq. 7), N_tree the tokens in the tree.
* Token ratio, Claw-R1 "Prefix Tree Merge", performance table: packed tokens
  divided by the tokens of all original sequences.
* Allowed (query, key) pairs: Trie packing, "Memory: a dense mask is not
  enough" counts the visible pairs of the packed tree (21 in the example).
"""
from __future__ import annotations

import numpy as np


def por(n_tree: float, n_base: float) -> float:
    return 1.0 - float(n_tree) / float(n_base)


def token_ratio(n_packed: int, seqs) -> float:
    return float(n_packed) / float(sum(len(s) for s in seqs))


def allowed_pairs_from_paths(paths, T) -> int:
    """Number of (query, key) pairs with key on the query's path at or before it,
    counted by enumerating every packed row's chain once."""
    seen = np.zeros(T, dtype=bool)
    total = 0
    for path in paths:
        for t, r in enumerate(path):
            if not seen[r]:
                seen[r] = True
                total += t + 1
    return int(total)
