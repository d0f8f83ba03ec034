"""Pins for oracle.metrics against the pages' printed numbers."""
import oracle
from conftest import golden


def test_por_figure5():
    g = golden("por_figure5.json")
    assert round(100 * oracle.por(g["n_tree"], g["n_base"]), 1) == g["por_percent"]


def test_token_ratio_and_pairs_examples():
    g = golden("trie_packing_example.json")
    p = oracle.pack_ref(g["sequences"])
    assert oracle.allowed_pairs_from_paths(p["paths"], p["T"]) == g["allowed_pairs_packed"]
    assert sum(len(s) * (len(s) + 1) // 2 for s in g["sequences"]) == g["allowed_pairs_unpacked"]
    assert p["T"] ** 2 == g["dense_scores_packed"]
    assert sum(len(s) ** 2 for s in g["sequences"]) == g["dense_scores_unpacked"]
    g3 = golden("prefix_tree_merge_example.json")
    p3 = oracle.pack_ref(g3["sequences"])
    assert oracle.allowed_pairs_from_paths(p3["paths"], p3["T"]) == 37
