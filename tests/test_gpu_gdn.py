"""GPU parity of the tree-routed Gated DeltaNet forward (Tree Training §3.2 "SSM Layers
(GDN)", eq. 10, Appendix A.2) with the per-branch recurrence oracle: random forests,
nodes longer than one 64-row sub-chunk, fp32 and bf16."""
import numpy as np
import pytest

import oracle
import synth
from gpu_common import BF16_TOL, F32_TOL, assert_close, dev, host, need_cuda, tma, torch

pytestmark = pytest.mark.gpu


def _inputs(T, H, Dk, Dv, seed, bf16):
    r = np.random.default_rng(seed)
    q = r.normal(size=(T, H, Dk)) / np.sqrt(Dk)
    k = r.normal(size=(T, H, Dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.normal(size=(T, H, Dv))
    g = -r.uniform(0.0, 0.2, size=(T, H))
    beta = r.uniform(0.05, 0.95, size=(T, H))
    q, k, v = (x.astype(np.float32) for x in (q, k, v))
    if bf16:
        q, k, v = (synth.bf16_round(x) for x in (q, k, v))
    return q, k, v, g.astype(np.float32), beta.astype(np.float32)


def _check(m, seqs, H, Dk, Dv, seed, bf16):
    pk = m.tree_pack(seqs)
    ref = oracle.pack_ref(seqs)
    T = pk["T"]
    q, k, v, g, beta = _inputs(T, H, Dk, Dv, seed, bf16)
    td = torch.bfloat16 if bf16 else torch.float32
    o = m.tree_gdn_fwd(dev(q, td), dev(k, td), dev(v, td), dev(g), dev(beta), dev(pk["node_start"]),
                       dev(pk["node_end"]), dev(pk["node_parent"]))
    m.tree_check_device_status()
    ro = oracle.gdn_ref_fwd(q, k, v, g, beta, ref["paths"])
    assert_close("o", o, ro, BF16_TOL if bf16 else F32_TOL)
    return pk


@pytest.mark.parametrize("seed,Dk,Dv,bf16", [(0, 64, 64, False), (1, 32, 96, False), (2, 128, 128, True)])
def test_gdn_random_forests(seed, Dk, Dv, bf16):
    """Short random sequences over a small vocabulary: many forks and several roots."""
    need_cuda()
    m = tma()
    rng = np.random.default_rng(700 + seed)
    seqs = synth.random_sequences(rng, 20, 90, vocab=2, min_len=1)
    pk = _check(m, seqs, 2, Dk, Dv, seed, bf16)
    assert pk["n_roots"] >= 2


@pytest.mark.parametrize("bf16", [False, True])
def test_gdn_galton_watson(bf16):
    """Segments of 20-300 rows: nodes of several 64-row sub-chunks, fanout up to 3."""
    need_cuda()
    m = tma()
    t = synth.galton_watson(seed=3, budget=2000, seg=(20, 300), vocab=1000)
    _check(m, t.seqs, 3, 128, 128, 3, bf16)


def test_gdn_long_chain_and_wide_fork():
    """A 700-row chain (eleven sub-chunks in one node) and a root with 30 children."""
    need_cuda()
    m = tma()
    seqs = [list(range(700))] + [[0, 5000 + i, 6000 + i] for i in range(30)]
    _check(m, seqs, 2, 64, 64, 5, False)


def test_gdn_bad_nodes_set_device_flag():
    """Node arrays that do not tile the rows in preorder are reported through the device
    error word; nothing is computed."""
    need_cuda()
    m = tma()
    T, H, D = 10, 1, 32
    x = torch.zeros((T, H, D), dtype=torch.float32, device="cuda")
    gb = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    ns = torch.tensor([0, 6], dtype=torch.int32, device="cuda")
    ne = torch.tensor([4, 9], dtype=torch.int32, device="cuda")   # row 5 belongs to no node
    npar = torch.tensor([-1, 0], dtype=torch.int32, device="cuda")
    m.tree_gdn_fwd(x, x, x, gb, gb, ns, ne, npar)
    with pytest.raises(m.TreeError) as ei:
        m.tree_check_device_status()
    assert ei.value.status == 7
    m.tree_check_device_status()
