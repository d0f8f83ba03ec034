"""CPU tests of the native library: it loads, exports every declared symbol,
packs bit-exactly like the oracle and rejects bad arguments on the host."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import oracle
import synth
from conftest import ROOT


@pytest.fixture(scope="module")
def tma():
    import __graft_entry__
    __graft_entry__.build()
    import tree_masked_attention_gb300 as m
    return m


def _declared():
    src = open(os.path.join(ROOT, "include", "tree_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tree_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(tma):
    names = _declared()
    assert "tree_attn_fwd" in names and "tree_logprob_bwd" in names
    L = tma.lib()
    for n in names:
        assert hasattr(L, n), n
    from tree_masked_attention_gb300._lib import SIGNATURES
    assert sorted(SIGNATURES) == names


KEYS = ("packed_ids", "position_ids", "subtree_end", "path_count", "parent_row", "node_of_token",
        "node_start", "node_end", "node_parent", "occ_source_rows", "occ_targets", "occ_seq",
        "occ_weights", "occ_row_ptr", "occ_perm")


def _same(a, b):
    for k in KEYS:
        assert np.array_equal(a[k], b[k]), k
    assert [x.tolist() for x in a["paths"]] == [x.tolist() for x in b["paths"]]
    for k in ("T", "n_nodes", "n_occ", "n_roots"):
        assert a[k] == b[k], k


@pytest.mark.parametrize("seed", range(60))
def test_pack_bit_exact_random(tma, seed):
    rng = np.random.default_rng(1000 + seed)
    seqs = synth.random_sequences(rng, int(rng.integers(0, 9)), 12, vocab=int(rng.integers(1, 5)))
    w = rng.random(len(seqs)).astype(np.float32)
    _same(tma.tree_pack(seqs, w), oracle.pack_ref(seqs, w))


@pytest.mark.parametrize("gen", ["tiny_tree", "agentic_short", "agentic_long", "galton_watson", "lm_head_tree"])
def test_pack_bit_exact_workloads(tma, gen):
    t = getattr(synth, gen)()
    _same(tma.tree_pack(t.seqs), oracle.pack_ref(t.seqs))


@pytest.mark.parametrize("fields", [("position_ids", "subtree_end"), ("paths", "node_parent"),
                                    ("occ_row_ptr", "occ_perm", "occ_targets"), ()])
def test_pack_field_subsets(tma, fields):
    """tree_pack(fields=...) returns exactly the named arrays, bit-equal to the oracle's."""
    t = synth.galton_watson(seed=2, budget=900, seg=(5, 60), vocab=50)
    got = tma.tree_pack(t.seqs, fields=fields)
    ref = oracle.pack_ref(t.seqs)
    arrays = {k for k, v in got.items() if not isinstance(v, int)}
    assert arrays == set(fields) | ({"token_rows"} if "paths" in fields else set())
    for f in fields:
        if f == "paths":
            assert all(np.array_equal(a, b) for a, b in zip(got["paths"], ref["paths"]))
        else:
            assert np.array_equal(got[f], ref[f]), f
    with pytest.raises(ValueError):
        tma.tree_pack(t.seqs, fields=("no_such_field",))


def test_pack_pages_examples(tma):
    from conftest import golden
    g = golden("trie_packing_example.json")
    p = tma.tree_pack(g["sequences"])
    assert p["position_ids"].tolist() == g["position_ids"]
    assert p["occ_source_rows"].tolist() == g["source_rows"]
    g3 = golden("prefix_tree_merge_example.json")
    p3 = tma.tree_pack(g3["sequences"])
    assert [[int(a), int(b)] for a, b in zip(p3["node_start"], p3["node_end"])] == [n["pos"] for n in g3["nodes"]]


def test_pack_edge_cases(tma):
    p = tma.tree_pack([])
    assert p["T"] == 0 and p["n_occ"] == 0
    p = tma.tree_pack([[], [7]])
    assert p["T"] == 1 and p["occ_row_ptr"].tolist() == [0, 0]


def test_validate_subtree_end(tma):
    tma.tree_validate_subtree_end([6, 6, 4, 3, 4, 6, 6])
    with pytest.raises(tma.TreeError):
        tma.tree_validate_subtree_end([1, 2, 2])       # row 1's subtree leaves row 0's
    with pytest.raises(tma.TreeError):
        tma.tree_validate_subtree_end([0, 0])          # end < i


def test_host_argument_errors(tma):
    L = tma.lib()
    # bad shapes / dtypes are refused before any CUDA call
    assert L.tree_attn_fwd(None, None, None, None, None, None, 16, 4, 3, 64, 1, 0.0, None, 0, None) == 2
    assert L.tree_attn_fwd(None, None, None, None, None, None, 16, 4, 2, 96, 1, 0.0, None, 0, None) == 2
    assert L.tree_attn_fwd(None, None, None, None, None, None, 16, 4, 2, 64, 7, 0.0, None, 0, None) == 3
    assert L.tree_attn_fwd(None, None, None, None, None, None, 16, 4, 2, 64, 1, 0.0, None, 0, None) == 1
    assert b"null" in L.tree_last_error()
    assert L.tree_logprob_fwd(None, None, None, None, None, 8, 60, 512, 4, None, None, 1, None, 0, None) == 2
    assert L.tree_rope(None, None, None, 4, 1, 1, 7, 10000.0, 1, 0, None) == 2
    assert L.tree_attn_workspace_size(4096, 32, 8, 128, 1) > 0
    assert L.tree_logprob_workspace_size(64, 64, 512, 100, 0) > 0


def test_every_workload_runs_on_tensor_cores(tma):
    """Kernel family per call (0 CUDA cores, 1 tcgen05 kind::f16, 2 tcgen05 kind::tf32 with
    the two-term split): the tiny fp32 tree (head size 64, fp32 LM head) takes the tf32
    kernels, the bf16 trees at head size 128 and the bf16 LM head the kind::f16 kernels; bf16
    at head size 64 runs on the tf32 kernels; only fp32 at head size 128 is left on CUDA
    cores."""
    F32, BF16 = 0, 1
    for op in (0, 1, 2, 3):
        assert tma.tree_kernel_path(op, F32, 64) == 2
    for op in (0, 1):
        assert tma.tree_kernel_path(op, BF16, 128) == 1
        assert tma.tree_kernel_path(op, BF16, 64) == 2
        assert tma.tree_kernel_path(op, F32, 128) == 0
    for op in (2, 3):
        assert tma.tree_kernel_path(op, BF16, 128) == 1


def test_kernel_timing_without_brackets(tma):
    """Without a recorded bracket (or a device) the timing query answers -1."""
    tma.tree_kernel_timing(False)
    assert tma.tree_kernel_last_ms(5) == -1
    assert tma.tree_kernel_last_ms(-1) == -1


def test_policy_loss_rejects_bad_clip_range(tma):
    """Argument checks run before any device work."""
    L = tma.lib()
    assert L.tree_policy_loss(None, None, None, None, None, 4, 1.5, 0.2, None, None, None, None) != 0
    assert L.tree_policy_loss(None, None, None, None, None, 4, 0.2, float("inf"), None, None, None, None) != 0
    assert L.tree_policy_loss(None, None, None, None, None, -1, 0.2, 0.2, None, None, None, None) != 0


def test_conv1d_rejects_bad_sizes(tma):
    """Channel count, kernel size, dtype and workspace are checked before any device work."""
    L = tma.lib()
    assert L.tree_conv1d_fwd(None, None, None, None, None, 16, 12, 4, 1, None) == 2   # C not a multiple of 8
    assert L.tree_conv1d_fwd(None, None, None, None, None, 16, 16, 9, 1, None) == 2   # K > 8
    assert L.tree_conv1d_fwd(None, None, None, None, None, 16, 16, 4, 5, None) == 3   # dtype
    assert L.tree_conv1d_fwd(None, None, None, None, None, 16, 16, 4, 1, None) == 1   # null pointers
    assert L.tree_conv1d_bwd(None, None, None, None, None, None, None, None, 16, 16, 0, 1, None, 0, None) == 2
    # one fp32 partial of dw (K) and dbias (1) per row group: 38 groups of 432 rows here
    assert L.tree_conv1d_workspace_size(16384, 8192, 4) == 38 * 5 * 8192 * 4
    assert L.tree_conv1d_workspace_size(16, 16, 9) == 0


def test_gateway_and_gdn_reject_bad_arguments(tma):
    """Host-side checks of the gateway and GDN calls run before any device work."""
    L = tma.lib()
    # gateway: tensor-core kernels only (bf16, d = 128), T >= 1, past_len >= 0
    assert L.tree_attn_fwd_gateway(None, None, None, None, None, None, None, 10, 16, 4, 2, 64, 1, 0.0,
                                   None, 0, None) == 2
    assert L.tree_attn_fwd_gateway(None, None, None, None, None, None, None, 10, 16, 4, 2, 128, 0, 0.0,
                                   None, 0, None) == 3
    assert L.tree_attn_fwd_gateway(None, None, None, None, None, None, None, -1, 16, 4, 2, 128, 1, 0.0,
                                   None, 0, None) == 2
    assert L.tree_attn_fwd_gateway(None, None, None, None, None, None, None, 10, 16, 4, 2, 128, 1, 0.0,
                                   None, 0, None) == 1
    assert L.tree_attn_bwd_gateway(None, None, None, None, None, None, None, None, None, None, None, None,
                                   None, 10, 0, 4, 2, 128, 1, 0.0, None, 0, None) == 2
    assert L.tree_attn_gateway_workspace_size(100, 200, 4, 2, 128, 1) == L.tree_attn_workspace_size(300, 4, 2, 128, 1)
    # GDN: Dk, Dv <= 128, nodes for the rows, dtype
    assert L.tree_gdn_fwd(None, None, None, None, None, None, None, None, None, 64, 4, 2, 256, 64, 1,
                          None, 0, None) == 2
    assert L.tree_gdn_fwd(None, None, None, None, None, None, None, None, None, 64, 4, 2, 64, 64, 9,
                          None, 0, None) == 3
    assert L.tree_gdn_fwd(None, None, None, None, None, None, None, None, None, 64, 0, 2, 64, 64, 1,
                          None, 0, None) == 2
    assert L.tree_gdn_fwd(None, None, None, None, None, None, None, None, None, 64, 4, 2, 64, 64, 1,
                          None, 0, None) == 1
    # GDN backward: the same checks, and every gradient pointer
    assert L.tree_gdn_bwd(*([None] * 14), 64, 4, 2, 256, 64, 1, None, 0, None) == 2
    assert L.tree_gdn_bwd(*([None] * 14), 64, 4, 2, 64, 64, 9, None, 0, None) == 3
    assert L.tree_gdn_bwd(*([None] * 14), 64, 4, 2, 64, 64, 1, None, 0, None) == 1
    assert L.tree_gdn_bwd_workspace_size(16384, 55, 16, 128, 128) > L.tree_gdn_workspace_size(16384, 55, 16, 128, 128)
    # the wait-limit test hook rejects limits outside (0, 2] s and sub-chunks below -1
    assert L.tree_gdn_test_withhold(0, 0.0) == 1
    assert L.tree_gdn_test_withhold(0, 3.0) == 1
    assert L.tree_gdn_test_withhold(-2, 0.1) == 1
    # workspace: sub-chunk table, schedule and one 64-row sub-chunk end state per (sub-chunk, head)
    ws = L.tree_gdn_workspace_size(16384, 55, 16, 128, 128)
    assert ws >= (55 + 16384 // 64 + 1) * 16 * 128 * 128 * 4
