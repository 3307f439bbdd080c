"""The gated delta rule stepped token by token, float64.

Test infrastructure only.

Definition (Flide, section 3.2.2, Eq. 4, the Gated DeltaNet rule of Yang et
al.; the pages write the write strength as eta_t, the configurations as
beta_t):

    S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
    o_t = S_t q_t

S is d_v x d_k (the outer product v k^T fixes the orientation), one state
per head, zero before the first token of a fresh sequence.  alpha_t and
beta_t are one scalar per (token, head).

The product S (I - beta k k^T) is evaluated as S - beta (S k) k^T: the same
matrix by associativity, O(d^2) instead of O(d^3) per token.
"""
from __future__ import annotations

import numpy as np


def gated_delta_rule(q, k, v, alpha, beta, S0=None):
    """q, k [n, H, dk]; v [n, H, dv]; alpha, beta [n, H].

    Returns (o [n, H, dv], S_n [H, dv, dk]), all float64.  ``S0`` is the state
    before the first token (zeros if None).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    a = np.asarray(alpha, dtype=np.float64)
    b = np.asarray(beta, dtype=np.float64)
    n, H, dk = k.shape
    dv = v.shape[2]
    S = np.zeros((H, dv, dk)) if S0 is None else np.array(S0, dtype=np.float64, copy=True)
    o = np.empty((n, H, dv))
    for t in range(n):
        kt, vt, qt = k[t], v[t], q[t]
        Sk = np.einsum("hvk,hk->hv", S, kt)                       # S_{t-1} k_t
        S = a[t][:, None, None] * (S - b[t][:, None, None] * Sk[:, :, None] * kt[:, None, :]) \
            + b[t][:, None, None] * vt[:, :, None] * kt[:, None, :]
        o[t] = np.einsum("hvk,hk->hv", S, qt)
    return o, S
