"""Oracle rotary position embedding on depth positions.

Test infrastructure only (see the package docstring).

Tree Training (arXiv 2511.00413) §3.2 "Position Embedding", eq. 9: every token
gets the position it has in its own per-path sequence, so RoPE gives the packed
token exactly the rotation it gets in the standalone branch. Trie packing,
"Step 1 - Store each node once": position IDs are the node's depth on its
original path ("use these positions for RoPE").

The oracle does not read any packed position array: it walks every path and uses
the row's index on that path (checking that all paths agree).

Reading taken (the pages name RoPE but not its variant): the rotate-half pairing
(element k with element k + d/2), frequencies theta_k = base^(-2k/d) with
base = 10000 by default; the inverse (backward) is the rotation by the negated
angle, the transpose of the forward rotation.
"""
from __future__ import annotations

import numpy as np


def rope_ref(x, paths, theta_base: float = 10000.0, inverse: bool = False):
    """Rotate x [T,H,d] (float64 result) by each row's index on its path."""
    x = np.asarray(x, dtype=np.float64)
    T, H, d = x.shape
    pos = np.full(T, -1, dtype=np.int64)
    for path in paths:
        for t, r in enumerate(path):
            if pos[r] < 0:
                pos[r] = t
            else:
                assert pos[r] == t, "a row has two different depths"
    assert (pos >= 0).all(), "a row lies on no path"
    half = d // 2
    freq = theta_base ** (-2.0 * np.arange(half) / d)          # [half]
    ang = pos[:, None].astype(np.float64) * freq[None, :]     # [T, half]
    if inverse:
        ang = -ang
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)
