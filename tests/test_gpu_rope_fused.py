"""GPU parity of tree_attn_bwd_rope: the attention backward with the inverse depth
rotation fused into the kernel that writes dq and dk, against the oracle's chain
(rotate q0, k0 by depth; attention backward; rotate dq, dk back)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_common import BF16_TOL, F32_TOL, assert_close, dev, host, need_cuda, tma, torch

pytestmark = pytest.mark.gpu


def _case(seqs, Hq, Hkv, d, dtype, seed):
    need_cuda()
    m = tma()
    pk = m.tree_pack(seqs)
    T = pk["T"]
    bf = dtype == "bf16"
    td = torch.bfloat16 if bf else torch.float32
    q0 = synth.normal(10 * seed + 1, (T, Hq, d), bf16=bf)
    k0 = synth.normal(10 * seed + 2, (T, Hkv, d), bf16=bf)
    v = synth.normal(10 * seed + 3, (T, Hkv, d), bf16=bf)
    do = synth.normal(10 * seed + 4, (T, Hq, d), bf16=bf)
    tq, tk, tv, tdo = (dev(x, td) for x in (q0, k0, v, do))
    pos, end = dev(pk["position_ids"]), dev(pk["subtree_end"])
    m.tree_rope(tq, tk, pos)
    o, lse = m.tree_attn_fwd(tq, tk, tv, end)
    dq0, dk0, dv = m.tree_attn_bwd_rope(tq, tk, tv, o, tdo, lse, end, pos)
    # the unfused chain on the GPU: backward, then tree_rope's inverse
    dq, dk, dv2 = m.tree_attn_bwd(tq, tk, tv, o, tdo, lse, end)
    m.tree_rope(dq, dk, pos, inverse=True)
    m.tree_check_device_status()

    paths = oracle.pack_ref(seqs)["paths"]
    q, k = oracle.rope_ref(q0, paths), oracle.rope_ref(k0, paths)
    rdq, rdk, rdv = oracle.attn_ref_bwd(q, k, v, do, paths)
    tol = BF16_TOL if bf else F32_TOL
    assert_close("dq0", dq0, oracle.rope_ref(rdq, paths, inverse=True), tol)
    assert_close("dk0", dk0, oracle.rope_ref(rdk, paths, inverse=True), tol)
    assert_close("dv", dv, rdv, tol)
    # dv is the same computation in both calls (up to the order of its fp32 sums across
    # work units, which the default mode does not fix)
    assert_close("dv of both calls", dv, host(dv2), tol)
    # fused (one rounding) and unfused (two roundings) agree to a couple of bf16 ulps
    assert_close("fused vs unfused dq", dq0, host(dq), tol)
    assert_close("fused vs unfused dk", dk0, host(dk), tol)


@pytest.mark.parametrize("seed", [0, 1])
def test_fused_rope_random_trees_bf16(seed):
    """Galton-Watson trees of a few hundred rows on the tensor-core path."""
    t = synth.galton_watson(seed=seed, budget=[333, 517][seed], seg=(5, 90), vocab=1000)
    _case(t.seqs, 8, 2, 128, "bf16", seed)


def test_fused_rope_fp32_head_64():
    """fp32 and d = 64 take the tf32-split tensor-core backward, then the rotation as its
    own pass."""
    t = synth.galton_watson(seed=2, budget=300, seg=(5, 60), vocab=1000)
    _case(t.seqs, 4, 2, 64, "f32", 2)


def test_fused_rope_short_prompt_agentic_full_size():
    """The short-prompt agentic tree at full size (T = 2304, 32/8 heads, d = 128, bf16)."""
    _case(synth.agentic_short().seqs, 32, 8, 128, "bf16", 0)


def test_fused_rope_rejects_bad_arguments():
    need_cuda()
    m = tma()
    t = synth.tiny_tree()
    pk = m.tree_pack(t.seqs)
    T = pk["T"]
    x = dev(synth.normal(1, (T, 2, 128), bf16=True), torch.bfloat16)
    lse = torch.zeros(2, T, dtype=torch.float32, device="cuda")
    end, pos = dev(pk["subtree_end"]), dev(pk["position_ids"])
    with pytest.raises(m.TreeError):
        m.tree_attn_bwd_rope(x, x, x, x, x, lse, end, pos, theta_base=1.0)
