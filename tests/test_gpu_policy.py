"""GPU parity of tree_policy_loss (per-occurrence clipped policy objective) with the
oracle, and the whole policy step: log-probs, objective, backward into the LM head."""
import numpy as np
import pytest

import oracle
import synth
from gpu_common import F32_TOL, assert_close, dev, host, need_cuda, tma, torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,eps_low,eps_high", [(1, 0.2, 0.2), (1000, 0.2, 0.2), (70001, 0.1, 0.28)])
def test_policy_loss_matches_oracle(n, eps_low, eps_high):
    need_cuda()
    m = tma()
    rng = np.random.default_rng(n)
    logp = (-rng.uniform(0.0, 8.0, n)).astype(np.float32)
    old = (logp + rng.normal(0.0, 0.5, n)).astype(np.float32)
    adv = rng.normal(0.0, 1.0, n).astype(np.float32)
    w = rng.uniform(0.0, 1.0, n).astype(np.float32)
    mask = (rng.random(n) > 0.1).astype(np.uint8)
    loss, g, total = m.tree_policy_loss(dev(logp), dev(old), dev(adv), dev(w), dev(mask), eps_low, eps_high)
    rl, rt, rg = oracle.policy_loss_ref(logp, old, adv, w, mask, eps_low, eps_high)
    # away from the clip kinks the fp32 ratio picks the same branch as the fp64 one
    r = np.exp(logp.astype(np.float64) - old)
    far = (np.abs(r - (1 - eps_low)) > 1e-5) & (np.abs(r - (1 + eps_high)) > 1e-5)
    assert_close("loss", host(loss)[far], rl[far], F32_TOL)
    assert_close("grad_logp", host(g)[far], rg[far], F32_TOL)
    # at a kink the objective is continuous, so the loss still matches; its gradient is one
    # of the two one-sided values, the unclipped -w m A r or 0 (the clipped side), depending
    # on which side the kernel's fp32 ratio falls: either is a valid result
    near = ~far
    if near.any():
        assert_close("loss at the kinks", host(loss)[near], rl[near], F32_TOL)
        gk = host(g)[near]
        unclipped = -(w.astype(np.float64) * mask * adv * r)[near]
        assert np.all((np.abs(gk - unclipped) <= F32_TOL + 1e-5 * np.abs(unclipped)) | (np.abs(gk) <= F32_TOL))
    assert float(host(total)[0]) == pytest.approx(float(host(loss).astype(np.float64).sum()), rel=1e-6, abs=1e-4)
    assert float(host(total)[0]) == pytest.approx(rt, rel=1e-5, abs=1e-3)


def test_policy_loss_optional_inputs_and_empty():
    need_cuda()
    m = tma()
    logp = dev(np.array([-1.0, -2.0], dtype=np.float32))
    loss, g, total = m.tree_policy_loss(logp, logp, dev(np.array([0.5, -2.0], dtype=np.float32)))
    assert np.allclose(host(g), [-0.5, 2.0]) and np.allclose(host(loss), [-0.5, 2.0])
    e = torch.empty(0, dtype=torch.float32, device="cuda")
    _, _, t0 = m.tree_policy_loss(e, e, e)
    assert float(host(t0)[0]) == 0.0


def test_policy_step_through_lm_head():
    """logprob forward -> clipped objective -> logprob backward, against the oracle chain."""
    need_cuda()
    m = tma()
    t = synth.tiny_tree()
    pk = m.tree_pack(t.seqs)
    T, n_occ = pk["T"], pk["n_occ"]
    h, w, _, _ = synth.lm_head_config(T, 64, 512, n_occ, bf16=False)
    ref = oracle.pack_ref(t.seqs)
    i32 = lambda a: torch.from_numpy(a).cuda()
    th, tw = dev(h), dev(w)
    lse, lp = m.tree_logprob_fwd(th, tw, i32(pk["occ_row_ptr"]), i32(pk["occ_perm"]), i32(pk["occ_targets"]))
    # old log-probs from the oracle's log-probs, with ratios 0.5, 1 or 1.5: away from the
    # clip edges 0.8 / 1.2, so both sides take the same branch
    rlp, _ = oracle.logprob_ref_fwd(h, w, ref["occ_source_rows"], ref["occ_targets"])
    rng = np.random.default_rng(5)
    ratio = rng.choice([0.5, 1.0, 1.5], n_occ)
    old = (rlp - np.log(ratio)).astype(np.float32)
    adv = rng.normal(0.0, 1.0, n_occ).astype(np.float32)
    _, g, _ = m.tree_policy_loss(lp, dev(old), dev(adv), eps_low=0.2)
    dh, dw = m.tree_logprob_bwd(th, tw, lse, i32(pk["occ_row_ptr"]), i32(pk["occ_perm"]), i32(pk["occ_targets"]), g)
    m.tree_check_device_status()
    _, _, rg = oracle.policy_loss_ref(rlp, old, adv, eps_low=0.2)
    rdh, rdw = oracle.logprob_ref_bwd(h, w, ref["occ_source_rows"], ref["occ_targets"], rg)
    assert_close("dH", dh, rdh, F32_TOL)
    assert_close("dW", dw, rdw, F32_TOL)
