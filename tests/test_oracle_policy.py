"""Pins of the per-occurrence clipped policy objective (oracle/policy.py).

Trie packing, "The training-loop change is small": each occurrence carries its own
advantage, old log-probability, clipping rule, mask and weight. Tree Training
§3.1 eq. 1: the policy-gradient per-token objective is -A_t log p.
"""
import numpy as np
import pytest

import oracle

rng = np.random.default_rng(11)


def _case(n=400, spread=0.6):
    logp = -rng.uniform(0.0, 6.0, n)
    old = logp + rng.normal(0.0, spread, n)
    adv = rng.normal(0.0, 1.0, n)
    w = rng.uniform(0.0, 1.0, n)
    m = (rng.random(n) > 0.2).astype(np.float64)
    return logp, old, adv, w, m


def test_on_policy_gradient_is_eq1():
    """At logp = old_logp the gradient is that of -w A log p (Tree Training eq. 1)."""
    logp, _, adv, w, m = _case()
    _, _, g = oracle.policy_loss_ref(logp, logp, adv, w, m, eps_low=0.2)
    assert np.allclose(g, -w * m * adv, rtol=0, atol=1e-15)


def test_loss_at_ratio_one_is_minus_weighted_advantage():
    logp, _, adv, w, m = _case()
    loss, total, _ = oracle.policy_loss_ref(logp, logp, adv, w, m)
    assert np.allclose(loss, -w * m * adv)
    assert total == pytest.approx(float((-w * m * adv).sum()))


def test_clipped_region_has_no_gradient():
    """A > 0 with r > 1 + eps, and A < 0 with r < 1 - eps: the clipped term is the minimum
    and constant in logp."""
    eps = 0.2
    logp = np.array([0.0, 0.0, 0.0, 0.0])
    old = np.array([-np.log(1.5), np.log(1.5), -np.log(1.1), np.log(1.1)])  # r = 1.5, 1/1.5, 1.1, 1/1.1
    adv = np.array([2.0, -3.0, 2.0, -3.0])
    loss, _, g = oracle.policy_loss_ref(logp, old, adv, eps_low=eps)
    assert g[0] == 0.0 and g[1] == 0.0
    assert loss[0] == pytest.approx(-(1 + eps) * 2.0)
    assert loss[1] == pytest.approx(-(1 - eps) * -3.0)
    # inside the clip range the gradient is -A r
    assert g[2] == pytest.approx(-2.0 * 1.1)
    assert g[3] == pytest.approx(3.0 / 1.1)


def test_pessimistic_side_keeps_gradient():
    """A > 0 with r < 1 - eps (and A < 0 with r > 1 + eps): min picks the unclipped term."""
    logp = np.zeros(2)
    old = np.array([np.log(2.0), -np.log(2.0)])  # r = 0.5, 2
    adv = np.array([1.5, -0.5])
    loss, _, g = oracle.policy_loss_ref(logp, old, adv, eps_low=0.2)
    assert loss[0] == pytest.approx(-0.5 * 1.5) and g[0] == pytest.approx(-0.5 * 1.5)
    assert loss[1] == pytest.approx(-2.0 * -0.5) and g[1] == pytest.approx(-2.0 * -0.5)


def test_no_clipping_limit_is_plain_importance_weighting():
    """eps -> infinity: L = -sum w m r A, dL/dlogp = -w m r A."""
    logp, old, adv, w, m = _case()
    r = np.exp(logp - old)
    loss, _, g = oracle.policy_loss_ref(logp, old, adv, w, m, eps_low=1e9, eps_high=1e9)
    assert np.allclose(loss, -w * m * r * adv)
    assert np.allclose(g, -w * m * r * adv)


def test_gradient_matches_finite_differences():
    logp, old, adv, w, m = _case(200)
    _, _, g = oracle.policy_loss_ref(logp, old, adv, w, m, eps_low=0.1, eps_high=0.3)
    h = 1e-6
    for o in range(200):
        r = np.exp(logp[o] - old[o])
        # skip points within h of a clip kink (the derivative jumps there)
        if min(abs(r - 0.9), abs(r - 1.3)) < 1e-4:
            continue
        lp, lm = logp.copy(), logp.copy()
        lp[o] += h
        lm[o] -= h
        fd = (oracle.policy_loss_ref(lp, old, adv, w, m, 0.1, 0.3)[1] -
              oracle.policy_loss_ref(lm, old, adv, w, m, 0.1, 0.3)[1]) / (2 * h)
        assert fd == pytest.approx(g[o], abs=1e-7, rel=1e-6)


def test_mask_and_weight_zero_drop_the_occurrence():
    logp, old, adv, w, m = _case(50)
    w[:10] = 0.0
    m[10:20] = 0.0
    loss, _, g = oracle.policy_loss_ref(logp, old, adv, w, m)
    assert not loss[:20].any() and not g[:20].any()


def test_per_occurrence_not_averaged_advantages():
    """Two occurrences of the same row with advantages +a and -a: averaging first would
    give zero loss and gradient; the per-occurrence objective does not (Trie packing)."""
    logp = np.array([-1.0, -1.0])
    old = np.array([-1.5, -1.5])  # r = e^0.5 > 1 + eps
    adv = np.array([1.0, -1.0])
    _, total, g = oracle.policy_loss_ref(logp, old, adv, eps_low=0.2)
    r = np.exp(0.5)
    assert g[0] == 0.0 and g[1] == pytest.approx(-r * -1.0)
    assert total == pytest.approx(-(1.2 * 1.0) + r * 1.0)
