"""Oracle: a plain, slow, CPU-only statement of what tree-packed training computes.

TEST INFRASTRUCTURE ONLY. The test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only code that may import, call or run
anything in this package. The library (``tree_masked_attention_gb300``) never
touches it, and the two share no code: no kernels, headers, helpers, tables or
pre/post-processing. The only module both sides use is ``synth`` (seeded input
generators, none of the method's arithmetic).

Everything floating point is float64 NumPy on the (possibly bf16-rounded) inputs.
The oracle follows the plain definitions on the pages:

* ``pack``      -- token trie, preorder (DFS) serialisation, depth positions,
                   nodes (chunks), next-token occurrences.
                   Trie packing, "Step 1 - Store each node once" and
                   "Share logits, preserve every prediction"; Tree Training
                   (arXiv 2511.00413) §3.1 eq. 8 and §3.2 eq. 9; Claw-R1
                   "Prefix Tree Merge", "1. build and compress".
* ``attention`` -- unpack the tree into its root-to-node paths and run ordinary
                   causal attention on each path, forward and backward
                   (Tree Training §3.1 eq. 6 forward equivalence; Trie
                   packing "Step 2 - Allow only ancestors and self" and
                   "Step 3 - Attention collects descendant contributions").
* ``rope``      -- rotary position embedding at each token's index on its own
                   path (Tree Training §3.2 "Position Embedding", eq. 9).
* ``logprob``   -- per-occurrence logits row, log-softmax, gather, and the
                   gradient of the weighted loss scattered back to rows
                   (Trie packing "Share logits, preserve every prediction" and
                   "Same chain rule, shared computation graph", Step 1).
* ``policy``    -- the per-occurrence clipped policy objective and its gradient
                   with respect to each occurrence's log-probability (Trie
                   packing, "The training-loop change is small"; Tree Training
                   §3.1 eq. 1).
* ``conv``      -- tree-correct causal depthwise conv1d: per-path convolution with
                   the parent's tokens as left context (Tree Training §3.2
                   "(ii) Causal convolution", eq. 11, Fig. 4).
* ``gateway``   -- partition-gateway attention: a child partition's queries over the
                   parent's accumulated keys (ancestor bias) and its own rows (tree
                   mask), dense masked softmax forward and backward (Tree Training
                   §3.3 "Differentiable partition boundaries", Appendix B.1-B.5,
                   eq. 14-17).
* ``gdn``       -- tree-routed Gated DeltaNet recurrence: each chunk starts from its
                   parent chunk's end state; per-path token recurrence, forward and
                   backward (Tree Training §3.2 "SSM Layers (GDN)", eq. 10, A.2).
* ``metrics``   -- potential overlap ratio (Tree Training §4.1 eq. 12).

Pins (tests/test_oracle_*.py) tie every function to values printed on the
pages, closed forms, library routines on special cases and brute force.
No function here is "parity unpinned".
"""
from .pack import pack_ref, brute_force_prefixes
from .attention import (attn_ref_fwd, attn_ref_bwd, attn_ref_rows, attn_ref_dq_rows,
                        attn_ref_dkdv_rows, dense_mask_from_chunks, mask_from_paths,
                        leaf_paths_from_parents)
from .rope import rope_ref
from .logprob import logprob_ref_fwd, logprob_ref_bwd, logprob_ref_gz
from .metrics import por, token_ratio, allowed_pairs_from_paths

from .policy import policy_loss_ref
from .conv import conv1d_ref_fwd, conv1d_ref_bwd, conv1d_ref_rows
from .gdn import gdn_ref_fwd, gdn_ref_bwd
from .gateway import (gateway_mask_ref, gateway_attn_ref_fwd, gateway_attn_ref_bwd, gateway_for_child,
                      local_subtree_end, is_ancestor_or_self)

__all__ = [
    "pack_ref", "brute_force_prefixes", "attn_ref_fwd", "attn_ref_bwd", "attn_ref_rows",
    "attn_ref_dq_rows", "attn_ref_dkdv_rows", "dense_mask_from_chunks", "mask_from_paths",
    "leaf_paths_from_parents", "rope_ref", "logprob_ref_fwd", "logprob_ref_bwd",
    "logprob_ref_gz", "por", "token_ratio", "allowed_pairs_from_paths", "policy_loss_ref",
    "conv1d_ref_fwd", "conv1d_ref_bwd", "conv1d_ref_rows", "gateway_mask_ref", "gateway_attn_ref_fwd",
    "gateway_attn_ref_bwd", "gateway_for_child", "local_subtree_end", "is_ancestor_or_self",
    "gdn_ref_fwd", "gdn_ref_bwd",
]
