"""Option distribution and the fidelity measures, float64.

Test infrastructure only.

* Flide, section 3.1, Eq. 1: p_i(o) = exp(w_o^T h_i) / sum_{o'} exp(w_{o'}^T h_i)
  over the options O_i, h_i the final hidden state at the last token of q_i.
* Flide, section 4.1 (metrics) and Appendix B: total variation against a
  reference distribution, top-1 agreement, and the decision at threshold 0.5
  ("acts when the probability of the top option reaches it").
"""
from __future__ import annotations

import numpy as np


def option_logprobs(h, W):
    """h [n, hidden]; W [n_opt, hidden] -> log p [n, n_opt] (max-subtracted)."""
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    z = h @ W.T
    m = z.max(axis=-1, keepdims=True)
    return z - m - np.log(np.exp(z - m).sum(axis=-1, keepdims=True))


def total_variation(p, q):
    return 0.5 * np.abs(np.asarray(p, np.float64) - np.asarray(q, np.float64)).sum(axis=-1)


def top1(p):
    """Index of the largest probability; ties go to the lowest index."""
    return np.argmax(np.asarray(p), axis=-1)      # argmax returns the first maximum


def decision(p, threshold: float = 0.5):
    """The option acted on at the threshold, or -1 when no option reaches it."""
    p = np.asarray(p, dtype=np.float64)
    t = top1(p)
    pt = np.take_along_axis(p, t[..., None], axis=-1)[..., 0]
    return np.where(pt >= threshold, t, -1)


def flips(p, ref, threshold: float = 0.5):
    return decision(p, threshold) != decision(ref, threshold)
