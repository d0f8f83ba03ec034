"""Pins for oracle.rope_ref: printed positions, complex-number rotation, the
relative-position property, invertibility."""
import numpy as np

import oracle
import synth
from conftest import golden


def _positions(paths, T):
    x = np.zeros((T, 1, 4))
    x[..., 1] = 1.0
    # d = 4, base 1e8: pair 1 (elements 1 and 3) turns by theta_1 = 1e-4 per position
    y = oracle.rope_ref(x, paths, theta_base=1e8)
    return np.rint(np.arctan2(y[:, 0, 3], y[:, 0, 1]) / 1e-4).astype(int)


def test_positions_from_paths_match_printed():
    g = golden("trie_packing_example.json")
    p = oracle.pack_ref(g["sequences"])
    assert _positions(p["paths"], 7).tolist() == g["position_ids"]


def test_complex_rotation_and_relative_property():
    rng = np.random.default_rng(0)
    T, H, d = 29, 3, 16
    paths = [np.arange(T)]
    x = rng.standard_normal((T, H, d))
    y = oracle.rope_ref(x, paths, theta_base=500.0)
    half = d // 2
    # library complex arithmetic: (x1 + i x2) * exp(i * pos * theta_k)
    theta = 500.0 ** (-np.arange(half) * 2.0 / d)
    z = (x[..., :half] + 1j * x[..., half:]) * np.exp(1j * np.arange(T)[:, None, None] * theta)
    np.testing.assert_allclose(y, np.concatenate([z.real, z.imag], -1), atol=1e-12)
    # norms kept; inverse undoes; position 0 is the identity
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), atol=1e-12)
    np.testing.assert_allclose(oracle.rope_ref(y, paths, 500.0, inverse=True), x, atol=1e-12)
    np.testing.assert_allclose(y[0], x[0], atol=0)
    # <R_m q, R_n k> depends only on m - n
    q = rng.standard_normal((1, 1, d))
    k = rng.standard_normal((1, 1, d))
    qq = oracle.rope_ref(np.repeat(q, T, 0), paths, 500.0)
    kk = oracle.rope_ref(np.repeat(k, T, 0), paths, 500.0)
    dots = np.einsum("ihd,jhd->ij", qq, kk)
    for off in range(-5, 6):
        diag = np.diagonal(dots, offset=off)
        np.testing.assert_allclose(diag, diag[0], atol=1e-10)


def test_siblings_share_positions():
    t = synth.tiny_tree()
    p = oracle.pack_ref(t.seqs)
    pos = _positions(p["paths"], p["T"])
    assert (pos[24:44] == np.arange(24, 44)).all()        # child A
    assert (pos[44:52] == np.arange(24, 32)).all()        # child B
    assert (pos[52:64] == pos[64:76]).all()               # the two 12-token leaves
