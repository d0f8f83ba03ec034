"""Oracle per-occurrence clipped policy objective (PPO / GRPO style).

Test infrastructure only (see the package docstring).

Trie packing (agillm.io), "The training-loop change is small": for PPO/GRPO the
per-occurrence log-probabilities are gathered as for the SFT loss, and then each
occurrence gets its own advantage, old log-probability, clipping rule, mask and
weight; advantages are not averaged before the nonlinear clipped loss.
Tree Training (arXiv 2511.00413) §3.1 eq. 1: the per-token objective of policy
gradient is l_t = -A_t log p_theta(y_t | x_<=t).

Reading taken (the pages name a clipping rule but print no formula): the PPO clip
with ratio r_o = exp(logp_o - old_logp_o),
    l_o = -min(r_o A_o, clip(r_o, 1 - eps_low, 1 + eps_high) A_o),
    L   = sum_o w_o m_o l_o,
and the gradient dL/dlogp_o that tree_logprob_bwd takes as its incoming gradient.
At r_o = 1 (logp equal to old_logp) it is -w_o m_o A_o, the gradient of eq. 1.
Where the clipped term is the minimum and the ratio lies outside the clip range,
the occurrence contributes no gradient.
"""
from __future__ import annotations

import numpy as np


def policy_loss_ref(logp, old_logp, adv, weight=None, mask=None, eps_low: float = 0.2,
                    eps_high: float | None = None):
    """Per-occurrence loss w m l_o, its sum, and dL/dlogp_o (all float64)."""
    logp = np.asarray(logp, dtype=np.float64)
    old = np.asarray(old_logp, dtype=np.float64)
    a = np.asarray(adv, dtype=np.float64)
    n = logp.shape[0]
    w = np.ones(n) if weight is None else np.asarray(weight, dtype=np.float64)
    m = np.ones(n) if mask is None else np.asarray(mask, dtype=np.float64)
    eps_high = eps_low if eps_high is None else eps_high
    r = np.exp(logp - old)
    unclipped = r * a
    rc = np.clip(r, 1.0 - eps_low, 1.0 + eps_high)
    clipped = rc * a
    # the unclipped term is the minimum (ties included: there both terms agree)
    take_unclipped = unclipped <= clipped
    l = -np.where(take_unclipped, unclipped, clipped)
    loss = w * m * l
    # d(-r A)/dlogp = -r A where the unclipped term is taken; the clipped term has a
    # zero derivative outside the clip range and equals the unclipped one inside it
    grad = np.where(take_unclipped, -w * m * a * r, 0.0)
    return loss, float(loss.sum()), grad
