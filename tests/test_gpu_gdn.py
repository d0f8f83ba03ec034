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


# ------------------------------------------------------------------------------ backward
def _check_bwd(m, seqs, H, Dk, Dv, seed, bf16):
    """Every gradient of sum(dO * o) against the oracle's per-branch reverse pass."""
    pk = m.tree_pack(seqs)
    ref = oracle.pack_ref(seqs)
    T = pk["T"]
    q, k, v, g, beta = _inputs(T, H, Dk, Dv, seed, bf16)
    r = np.random.default_rng(seed + 50)
    do = r.normal(size=(T, H, Dv)).astype(np.float32)
    if bf16:
        do = synth.bf16_round(do)
    td = torch.bfloat16 if bf16 else torch.float32
    nodes = [dev(pk[n]) for n in ("node_start", "node_end", "node_parent")]
    got = m.tree_gdn_bwd(dev(q, td), dev(k, td), dev(v, td), dev(g), dev(beta), dev(do, td), *nodes)
    m.tree_check_device_status()
    want = oracle.gdn_ref_bwd(q, k, v, g, beta, do, ref["paths"])
    tol = BF16_TOL if bf16 else F32_TOL
    for name, a, b in zip(("dq", "dk", "dv"), got[:3], want[:3]):
        assert_close(name, a, b, tol)
    # dg and dbeta are fp32 outputs of fp32 arithmetic on the same (rounded) inputs
    for name, a, b in zip(("dg", "dbeta"), got[3:], want[3:]):
        assert_close(name, a, b, F32_TOL)
    return pk


@pytest.mark.parametrize("seed,Dk,Dv,bf16", [(0, 64, 64, False), (1, 32, 96, False), (2, 128, 128, True)])
def test_gdn_bwd_random_forests(seed, Dk, Dv, bf16):
    """Many forks and several roots: sibling state gradients summed at the parent's end."""
    need_cuda()
    m = tma()
    rng = np.random.default_rng(800 + seed)
    seqs = synth.random_sequences(rng, 20, 90, vocab=2, min_len=1)
    pk = _check_bwd(m, seqs, 2, Dk, Dv, seed, bf16)
    assert pk["n_roots"] >= 2


@pytest.mark.parametrize("bf16", [False, True])
def test_gdn_bwd_galton_watson(bf16):
    """Nodes of several 64-row sub-chunks and fanout up to 3 (a sub-chunk's end-state
    gradient comes from the next sub-chunk of its node or from every child)."""
    need_cuda()
    m = tma()
    t = synth.galton_watson(seed=4, budget=1500, seg=(20, 300), vocab=1000)
    _check_bwd(m, t.seqs, 2, 128, 128, 4, bf16)


def test_gdn_bwd_long_chain_and_wide_fork():
    """A 700-row chain (eleven sub-chunks in one node) and a root with 30 children, whose
    start-state gradients all add into the root's end state."""
    need_cuda()
    m = tma()
    seqs = [list(range(700))] + [[0, 5000 + i, 6000 + i] for i in range(30)]
    _check_bwd(m, seqs, 2, 64, 64, 6, False)


@pytest.mark.parametrize("case", ["single_token", "forest_of_singletons", "exactly_64_rows", "65_rows"])
def test_gdn_degenerate_trees(case):
    """One row; 200 one-row roots (every node starts from zero); a node of exactly one
    64-row sub-chunk; one row past it (a one-row second sub-chunk). Forward and backward."""
    need_cuda()
    m = tma()
    seqs = {"single_token": [[7]], "forest_of_singletons": [[i] for i in range(200)],
            "exactly_64_rows": [list(range(64))], "65_rows": [list(range(65))]}[case]
    _check(m, seqs, 2, 64, 64, 8, False)
    _check_bwd(m, seqs, 2, 64, 64, 8, False)


def test_gdn_bwd_repeats_bitwise():
    """Fixed summation orders: two backward calls give identical bits."""
    need_cuda()
    m = tma()
    t = synth.galton_watson(seed=5, budget=1200, seg=(20, 200), vocab=1000)
    pk = m.tree_pack(t.seqs)
    T = pk["T"]
    q, k, v, g, beta = _inputs(T, 2, 64, 64, 7, False)
    do = np.random.default_rng(8).normal(size=(T, 2, 64)).astype(np.float32)
    args = [dev(x) for x in (q, k, v, g, beta, do)] + [dev(pk[n]) for n in ("node_start", "node_end", "node_parent")]
    a = m.tree_gdn_bwd(*args)
    b = m.tree_gdn_bwd(*args)
    m.tree_check_device_status()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


# ------------------------------------------------------------------------------ saved forward
def _gdn_case(m, seed, H, D, bf16):
    t = synth.galton_watson(seed=seed, budget=1500, seg=(20, 300), vocab=1000)
    pk = m.tree_pack(t.seqs)
    T = pk["T"]
    q, k, v, g, beta = _inputs(T, H, D, D, seed + 20, bf16)
    do = np.random.default_rng(seed + 21).normal(size=(T, H, D)).astype(np.float32)
    if bf16:
        do = synth.bf16_round(do)
    return t, pk, (q, k, v, g, beta, do)


def test_gdn_bwd_saved_matches_recompute_and_oracle():
    """tree_gdn_bwd_saved after tree_gdn_fwd on the backward-sized workspace takes the
    forward's factors, corrections and end states from it: the same bits as tree_gdn_bwd,
    which recomputes them from the inputs, and the oracle's gradients."""
    need_cuda()
    m = tma()
    H, D = 2, 128
    t, pk, (q, k, v, g, beta, do) = _gdn_case(m, 6, H, D, True)
    ref = oracle.pack_ref(t.seqs)
    T, td = pk["T"], torch.bfloat16
    nodes = [dev(pk[n]) for n in ("node_start", "node_end", "node_parent")]
    ins = [dev(q, td), dev(k, td), dev(v, td), dev(g), dev(beta)]
    d_o = dev(do, td)
    ws = torch.empty(m.tree_gdn_bwd_workspace_size(T, len(pk["node_start"]), H, D, D), dtype=torch.uint8,
                     device="cuda")
    m.tree_gdn_fwd(*ins, *nodes, workspace=ws)
    saved = m.tree_gdn_bwd_saved(*ins, d_o, *nodes, workspace=ws)
    recomputed = m.tree_gdn_bwd(*ins, d_o, *nodes)
    m.tree_check_device_status()
    for name, a, b in zip(("dq", "dk", "dv", "dg", "dbeta"), saved, recomputed):
        assert torch.equal(a, b), name
    want = oracle.gdn_ref_bwd(q, k, v, g, beta, do, ref["paths"])
    for name, a, b in zip(("dq", "dk", "dv"), saved[:3], want[:3]):
        assert_close(name, a, b, BF16_TOL)
    for name, a, b in zip(("dg", "dbeta"), saved[3:], want[3:]):
        assert_close(name, a, b, F32_TOL)


def test_gdn_bwd_saved_needs_the_forward_of_its_inputs():
    """The workspace stamp: a second saved backward without a new forward, one after a
    forward of other inputs, and one on a workspace no forward ran with each set
    TREE_ERR_DEVICE_CHECK and schedule nothing; a matched pair afterwards runs normally."""
    need_cuda()
    m = tma()
    H, D = 2, 64
    t, pk, (q, k, v, g, beta, do) = _gdn_case(m, 7, H, D, False)
    T = pk["T"]
    nodes = [dev(pk[n]) for n in ("node_start", "node_end", "node_parent")]
    ins = [dev(x) for x in (q, k, v, g, beta)]
    d_o = dev(do)
    size = m.tree_gdn_bwd_workspace_size(T, len(pk["node_start"]), H, D, D)
    ws = torch.empty(size, dtype=torch.uint8, device="cuda")

    def rejected(workspace, inputs=ins):
        m.tree_gdn_bwd_saved(*inputs, d_o, *nodes, workspace=workspace)
        with pytest.raises(m.TreeError) as ei:
            m.tree_check_device_status()
        assert ei.value.status == 7   # TREE_ERR_DEVICE_CHECK
        m.tree_check_device_status()  # cleared

    m.tree_gdn_fwd(*ins, *nodes, workspace=ws)
    first = m.tree_gdn_bwd_saved(*ins, d_o, *nodes, workspace=ws)
    m.tree_check_device_status()
    rejected(ws)                                          # the stamp was consumed
    other = [dev(x) for x in (q, k, v, g, beta)]          # same values, other buffers
    m.tree_gdn_fwd(*other, *nodes, workspace=ws)
    rejected(ws)                                          # the forward was of other inputs
    rejected(torch.zeros(size, dtype=torch.uint8, device="cuda"))  # no forward on this workspace
    m.tree_gdn_fwd(*ins, *nodes, workspace=ws)
    again = m.tree_gdn_bwd_saved(*ins, d_o, *nodes, workspace=ws)
    m.tree_check_device_status()
    for a, b in zip(first, again):
        assert torch.equal(a, b)


# ------------------------------------------------------------------------------ bounded waits
def _withheld_call(m, fn, args, sub_chunk):
    rc = m.lib().tree_gdn_test_withhold(sub_chunk, 0.05)
    assert rc == 0, m.lib().tree_last_error()
    fn(*args)
    with pytest.raises(m.TreeError) as ei:
        m.tree_check_device_status()
    return ei.value.status


@pytest.mark.parametrize("which", ["fwd", "bwd"])
def test_gdn_wait_runs_out_when_a_publication_is_withheld(which):
    """The first sub-chunk never publishes its state (test hook), so the waits of the
    sub-chunks that continue from it run out after 50 ms: the call ends with
    TREE_ERR_TIMEOUT in the device error word, every CTA leaves, and the next call runs
    normally and matches the oracle."""
    need_cuda()
    m = tma()
    t = synth.galton_watson(seed=3, budget=600, seg=(20, 150), vocab=1000)
    pk = m.tree_pack(t.seqs)
    ref = oracle.pack_ref(t.seqs)
    T = pk["T"]
    q, k, v, g, beta = _inputs(T, 2, 64, 64, 9, False)
    do = np.random.default_rng(10).normal(size=(T, 2, 64)).astype(np.float32)
    nodes = [dev(pk[n]) for n in ("node_start", "node_end", "node_parent")]
    ins = [dev(x) for x in (q, k, v, g, beta)]
    if which == "fwd":
        fn, args = m.tree_gdn_fwd, ins + nodes
    else:
        fn, args = m.tree_gdn_bwd, ins + [dev(do)] + nodes
    assert _withheld_call(m, fn, args, 0) == 6          # TREE_ERR_TIMEOUT
    m.tree_check_device_status()                          # cleared, context usable
    if which == "fwd":
        assert_close("o after a timeout", fn(*args), oracle.gdn_ref_fwd(q, k, v, g, beta, ref["paths"]), F32_TOL)
    else:
        want = oracle.gdn_ref_bwd(q, k, v, g, beta, do, ref["paths"])
        for name, a, b in zip(("dq", "dk", "dv", "dg", "dbeta"), fn(*args), want):
            assert_close(name + " after a timeout", a, b, F32_TOL)
    m.tree_check_device_status()


def test_gdn_full_size_two_heads():
    """The bench's GDN configuration at full size (the 16,384-row Galton-Watson tree,
    16 heads, Dk = Dv = 128, bf16 q / k / v / dO, fp32 gates): forward and backward of all
    16 heads on the GPU, heads 3 and 12 against the per-branch oracle element by element
    (heads are independent, so two heads of the same call stand for all of them)."""
    need_cuda()
    m = tma()
    t = synth.galton_watson()
    pk = m.tree_pack(t.seqs)
    ref = oracle.pack_ref(t.seqs)
    T, H, D = pk["T"], 16, 128
    q, k, v, g, beta = _inputs(T, H, D, D, 31, True)
    r = np.random.default_rng(32)
    do = synth.bf16_round(r.normal(size=(T, H, D)).astype(np.float32))
    td = torch.bfloat16
    nodes = [dev(pk[n]) for n in ("node_start", "node_end", "node_parent")]
    args = (dev(q, td), dev(k, td), dev(v, td), dev(g), dev(beta))
    o = m.tree_gdn_fwd(*args, *nodes)
    got = m.tree_gdn_bwd(*args, dev(do, td), *nodes)
    m.tree_check_device_status()
    hs = [3, 12]
    sub = lambda x: np.ascontiguousarray(x[:, hs])
    ro = oracle.gdn_ref_fwd(sub(q), sub(k), sub(v), sub(g), sub(beta), ref["paths"])
    assert_close("o", host(o)[:, hs], ro, BF16_TOL)
    want = oracle.gdn_ref_bwd(sub(q), sub(k), sub(v), sub(g), sub(beta), sub(do), ref["paths"])
    for name, a, b in zip(("dq", "dk", "dv"), got[:3], want[:3]):
        assert_close(name, host(a)[:, hs], b, BF16_TOL)
    for name, a, b in zip(("dg", "dbeta"), got[3:], want[3:]):
        assert_close(name, host(a)[:, hs], b, F32_TOL)
