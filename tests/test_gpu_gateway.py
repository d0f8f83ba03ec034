"""GPU parity of partition-gateway attention (Tree Training §3.3 "Differentiable partition
boundaries", Appendix B.2-B.5) with the oracle: each child partition's O, LSE, dQ and its
own dK / dV through the tensor-core kernels, and the gateway rows' dK / dV summed over the
sibling child partitions in fp32 (B.5); the partitioned pass also matches the
whole-tree kernels."""
import numpy as np
import pytest

import oracle
import synth
from gpu_common import BF16_TOL, F32_TOL, assert_close, dev, host, need_cuda, tma, torch

pytestmark = pytest.mark.gpu

Hq, Hkv, D = 4, 2, 128


def _cut(ref, min_children=2):
    """The node with >= min_children child nodes that ends last in preorder (so that the
    rows before it hold sibling subtrees the gateway must hide); its children's first rows."""
    kids = {}
    for n in range(len(ref["node_start"])):
        p = int(ref["node_parent"][n])
        if p >= 0:
            kids.setdefault(p, []).append(int(ref["node_start"][n]))
    cands = [(int(ref["node_end"][p]), cs) for p, cs in kids.items() if len(cs) >= min_children]
    assert cands
    return max(cands)[1]


def _partition(ref, children):
    T = ref["T"]
    cut = set()
    for c in children:
        cut.update(range(c, int(ref["subtree_end"][c]) + 1))
    return [i for i in range(T) if i not in cut]


def _inputs(T, seed):
    return (synth.normal(seed * 10 + 1, (T, Hq, D), bf16=True), synth.normal(seed * 10 + 2, (T, Hkv, D), bf16=True),
            synth.normal(seed * 10 + 3, (T, Hkv, D), bf16=True), synth.normal(seed * 10 + 4, (T, Hq, D), bf16=True))


@pytest.mark.parametrize("seed,budget", [(0, 700), (1, 1300), (2, 2100)])
def test_gateway_children_match_oracle(seed, budget):
    need_cuda()
    m = tma()
    t = synth.galton_watson(seed=seed, budget=budget, seg=(20, 160), vocab=1000)
    ref = oracle.pack_ref(t.seqs)
    children = _cut(ref)
    parent_rows = _partition(ref, children)
    q, k, v, do = _inputs(ref["T"], seed)
    bf = torch.bfloat16
    dkp = dvp = None
    sum_dk = sum_dv = None
    hidden_seen = False
    for c in children:
        g = oracle.gateway_for_child(ref, parent_rows, c)
        rows = np.concatenate([g["past_rows"], g["child_rows"]])
        cr, P, pv, ce = g["child_rows"], len(g["past_rows"]), g["past_visible"], g["child_end"]
        hidden_seen |= not pv.all()
        bias = np.where(pv, 0.0, -np.inf).astype(np.float32)
        tq, tk, tv, tdo = dev(q[cr], bf), dev(k[rows], bf), dev(v[rows], bf), dev(do[cr], bf)
        o, lse = m.tree_attn_fwd_gateway(tq, tk, tv, dev(bias), dev(ce.astype(np.int32)))
        if dkp is None:
            dkp = torch.zeros((P, Hkv, D), dtype=torch.float32, device="cuda")
            dvp = torch.zeros((P, Hkv, D), dtype=torch.float32, device="cuda")
        # siblings share the gateway: the same past rows, gradients added in fp32
        dq, dk, dv, dkp, dvp = m.tree_attn_bwd_gateway(tq, tk, tv, o, tdo, lse, dev(bias), dev(ce.astype(np.int32)),
                                                       dk_past=dkp, dv_past=dvp)
        m.tree_check_device_status()
        ro, rl = oracle.gateway_attn_ref_fwd(q[cr], k[rows], v[rows], P, pv, ce)
        rdq, rdk, rdv = oracle.gateway_attn_ref_bwd(q[cr], k[rows], v[rows], do[cr], P, pv, ce)
        assert_close("O", o, ro, BF16_TOL)
        assert_close("LSE", lse, rl, F32_TOL)
        assert_close("dQ", dq, rdq, BF16_TOL)
        assert_close("dK own", dk, rdk[P:], BF16_TOL)
        assert_close("dV own", dv, rdv[P:], BF16_TOL)
        sum_dk = rdk[:P] if sum_dk is None else sum_dk + rdk[:P]
        sum_dv = rdv[:P] if sum_dv is None else sum_dv + rdv[:P]
    assert hidden_seen, "the cut should hide some earlier sibling rows"
    # B.5: the gateway rows' gradients, summed over the children in fp32 (P, dS enter the
    # MMAs in bf16, so the bf16 bound applies to the sum as to dK itself)
    assert_close("dK past (sum over children)", dkp, sum_dk, BF16_TOL)
    assert_close("dV past (sum over children)", dvp, sum_dv, BF16_TOL)


def test_gateway_without_past_is_tree_attention():
    """past_len = 0: the same kernels on the same rows as tree_attn_fwd / tree_attn_bwd."""
    need_cuda()
    m = tma()
    t = synth.galton_watson(seed=4, budget=900, seg=(5, 90), vocab=1000)
    pk = m.tree_pack(t.seqs)
    q, k, v, do = (dev(x, torch.bfloat16) for x in _inputs(pk["T"], 4))
    end = dev(pk["subtree_end"])
    e0 = torch.empty(0, dtype=torch.float32, device="cuda")
    o1, l1 = m.tree_attn_fwd(q, k, v, end)
    o2, l2 = m.tree_attn_fwd_gateway(q, k, v, e0, end)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    g1 = m.tree_attn_bwd(q, k, v, o1, do, l1, end)
    g2 = m.tree_attn_bwd_gateway(q, k, v, o1, do, l1, e0, end)
    m.tree_check_device_status()
    for a, b, name in zip(g1, g2[:3], ("dq", "dk", "dv")):
        assert_close(name, a, host(b), BF16_TOL)


@pytest.mark.parametrize("P,frac", [(1, 1.0), (128, 0.5), (300, 0.3), (513, 0.0)])
def test_gateway_past_lengths(P, frac):
    """Past lengths on and off the 128-row tiles, all visible, some or none visible; a
    synthetic past in front of a random child tree."""
    need_cuda()
    m = tma()
    rng = np.random.default_rng(P)
    t = synth.galton_watson(seed=P % 7, budget=450, seg=(5, 90), vocab=1000)
    ref = oracle.pack_ref(t.seqs)
    Tc = ref["T"]
    q, k, v, do = _inputs(P + Tc, P)
    q, do = q[P:], do[P:]
    pv = rng.random(P) < frac
    bias = np.where(pv, 0.0, -np.inf).astype(np.float32)
    ce = ref["subtree_end"].astype(np.int32)
    bf = torch.bfloat16
    tq, tk, tv, tdo = dev(q, bf), dev(k, bf), dev(v, bf), dev(do, bf)
    o, lse = m.tree_attn_fwd_gateway(tq, tk, tv, dev(bias), dev(ce))
    dq, dk, dv, dkp, dvp = m.tree_attn_bwd_gateway(tq, tk, tv, o, tdo, lse, dev(bias), dev(ce))
    m.tree_check_device_status()
    ro, rl = oracle.gateway_attn_ref_fwd(q, k, v, P, pv, ce)
    rdq, rdk, rdv = oracle.gateway_attn_ref_bwd(q, k, v, do, P, pv, ce)
    assert_close("O", o, ro, BF16_TOL)
    assert_close("LSE", lse, rl, F32_TOL)
    assert_close("dQ", dq, rdq, BF16_TOL)
    assert_close("dK", dk, rdk[P:], BF16_TOL)
    assert_close("dV", dv, rdv[P:], BF16_TOL)
    assert_close("dK past", dkp, rdk[:P], BF16_TOL)
    assert_close("dV past", dvp, rdv[:P], BF16_TOL)
    if not pv.any():
        assert float(dkp.abs().max()) == 0.0 and float(dvp.abs().max()) == 0.0


def test_gateway_bad_bias_sets_device_flag():
    """A bias other than 0 or -inf is reported through the device error word and read as
    -inf (eq. 16 allows only those two values)."""
    need_cuda()
    m = tma()
    P, T = 4, 130
    k = torch.zeros((P + T, Hkv, D), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((T, Hq, D), dtype=torch.bfloat16, device="cuda")
    bias = torch.tensor([0.0, -1.0, 0.0, float("-inf")], device="cuda")
    end = torch.arange(T, dtype=torch.int32, device="cuda")
    m.tree_attn_fwd_gateway(q, k, k, bias, end)
    with pytest.raises(m.TreeError) as ei:
        m.tree_check_device_status()
    assert ei.value.status == 7
    m.tree_check_device_status()


def test_gateway_full_size_one_kv_group():
    """The bench's gateway configuration at full size: the long-prompt agentic tree
    (16,640 rows, 32 / 8 heads) cut below its 1024-token prompt, three of its six child
    partitions (2048 rows each) run with all heads, the prompt's dK / dV summed over them
    in fp32; every row of KV group 2 (its four query heads) against the oracle run on that
    group alone."""
    need_cuda()
    m = tma()
    tree = synth.agentic_long()
    pk = m.tree_pack(tree.seqs)
    end, par = pk["subtree_end"], pk["parent_row"]
    P = int(pk["node_end"][0]) + 1
    kids = [int(r) for r in range(P, pk["T"]) if par[r] == P - 1][:3]
    q, k, v, do = synth.attention_config("agentic_long", pk["T"])
    g, G = 2, 4
    hs = slice(G * g, G * (g + 1))
    bf = torch.bfloat16
    pv = np.ones(P, dtype=bool)
    bias = dev(np.zeros(P, dtype=np.float32))
    dkp = torch.zeros((P, 8, 128), dtype=torch.float32, device="cuda")
    dvp = torch.zeros_like(dkp)
    sum_dk = np.zeros((P, 1, 128))
    sum_dv = np.zeros((P, 1, 128))
    for r in kids:
        rows = slice(r, int(end[r]) + 1)
        ce = (end[rows] - r).astype(np.int32)
        kk, vv = np.concatenate([k[:P], k[rows]]), np.concatenate([v[:P], v[rows]])
        tq, tk, tv, tdo = dev(q[rows], bf), dev(kk, bf), dev(vv, bf), dev(do[rows], bf)
        o, lse = m.tree_attn_fwd_gateway(tq, tk, tv, bias, dev(ce))
        dq, dk, dv, dkp, dvp = m.tree_attn_bwd_gateway(tq, tk, tv, o, tdo, lse, bias, dev(ce),
                                                       dk_past=dkp, dv_past=dvp)
        m.tree_check_device_status()
        gq, gk, gv, gdo = q[rows, hs], kk[:, g:g + 1], vv[:, g:g + 1], do[rows, hs]
        ro, rl = oracle.gateway_attn_ref_fwd(gq, gk, gv, P, pv, ce)
        rdq, rdk, rdv = oracle.gateway_attn_ref_bwd(gq, gk, gv, gdo, P, pv, ce)
        assert_close("O", host(o)[:, hs], ro, BF16_TOL)
        assert_close("LSE", host(lse)[hs], rl, F32_TOL)
        assert_close("dQ", host(dq)[:, hs], rdq, BF16_TOL)
        assert_close("dK own", host(dk)[:, g:g + 1], rdk[P:], BF16_TOL)
        assert_close("dV own", host(dv)[:, g:g + 1], rdv[P:], BF16_TOL)
        sum_dk += rdk[:P]
        sum_dv += rdv[:P]
    assert_close("dK past (sum over children)", host(dkp)[:, g:g + 1], sum_dk, BF16_TOL)
    assert_close("dV past (sum over children)", host(dvp)[:, g:g + 1], sum_dv, BF16_TOL)
