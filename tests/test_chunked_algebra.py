"""The chunked (WY) form that the CUDA kernels implement, checked in float64
against the step-by-step oracle before any kernel exists.

Within a chunk of C tokens starting from state S0, with g_t the cumulative
sum of log alpha inside the chunk (gamma_t = exp(g_t)):

    u_t  = beta_t (v_t - alpha_t S_{t-1} k_t)          (so S_t = alpha_t S_{t-1} + u_t k_t^T)
    (I + A) U = diag(beta) V - diag(beta gamma) K S0^T,  A_ts = beta_t e^{g_t-g_s} k_t.k_s (s<t)
    => U = Utilde - W S0^T,  Utilde = T diag(beta) V,  W = T diag(beta gamma) K,  T = (I+A)^{-1}
    O    = diag(gamma) Q S0^T + P U,                  P_ts = e^{g_t-g_s} q_t.k_s   (s<=t)
    S_C  = gamma_C S0 + U^T diag(e^{g_C-g}) K

This is the algebra of the gated delta rule (Flide section 3.2.2, Eq. 4)
regrouped by chunk; each segment starts its own chunk (Flide section 3.5).
This test holds its own numpy code; it is not part of the oracle.
"""
import numpy as np
import pytest

from oracle import gdn


def chunked(q, k, v, a, b, C, S0=None):
    n, H, dk = k.shape
    dv = v.shape[2]
    S = np.zeros((H, dv, dk)) if S0 is None else S0.copy()
    o = np.zeros((n, H, dv))
    for c0 in range(0, n, C):
        c1 = min(n, c0 + C)
        for h in range(H):
            Q, K, V = q[c0:c1, h], k[c0:c1, h], v[c0:c1, h]
            g = np.cumsum(np.log(a[c0:c1, h]))
            bb = b[c0:c1, h]
            L = len(g)
            D = np.exp(g[:, None] - g[None, :])
            A = np.tril(bb[:, None] * D * (K @ K.T), -1)
            Tm = np.linalg.inv(np.eye(L) + A)
            W = Tm @ ((bb * np.exp(g))[:, None] * K)
            Ut = Tm @ (bb[:, None] * V)
            U = Ut - W @ S[h].T
            P = np.tril(D * (Q @ K.T))
            o[c0:c1, h] = np.exp(g)[:, None] * (Q @ S[h].T) + P @ U
            S[h] = np.exp(g[-1]) * S[h] + U.T @ (np.exp(g[-1] - g)[:, None] * K)
    return o, S


@pytest.mark.parametrize("n,C", [(1, 4), (7, 4), (16, 4), (37, 8), (64, 64), (130, 64)])
def test_chunked_form_matches_recurrence(n, C):
    rng = np.random.default_rng(n * 100 + C)
    H, dk, dv = 2, 8, 6
    q = rng.standard_normal((n, H, dk)) / 8
    k = rng.standard_normal((n, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((n, H, dv)) / 8
    a = np.exp(-0.1 * np.log1p(np.exp(rng.standard_normal((n, H)))))
    b = 1 / (1 + np.exp(-rng.standard_normal((n, H))))
    S0 = rng.standard_normal((H, dv, dk)) * 0.1
    o1, S1 = gdn.gated_delta_rule(q, k, v, a, b, S0=S0)
    o2, S2 = chunked(q, k, v, a, b, C, S0=S0)
    np.testing.assert_allclose(o2, o1, atol=1e-13)
    np.testing.assert_allclose(S2, S1, atol=1e-13)
