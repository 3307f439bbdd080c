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


def chunk_map(k, v, a, b, C, h, c0):
    """The affine map of chunk [c0, c0+C) on the state of head h (S [d_v, d_k]):
    S_C = S0 M + N, with M = gamma_C I - W^T K'' and N = Utilde^T K'',
    K'' = diag(e^{g_C - g}) K (from U = Utilde - W S0^T)."""
    n, _, dk = k.shape
    c1 = min(n, c0 + C)
    K, V = k[c0:c1, h], v[c0:c1, h]
    g = np.cumsum(np.log(a[c0:c1, h]))
    bb = b[c0:c1, h]
    L = len(g)
    D = np.exp(g[:, None] - g[None, :])
    A = np.tril(bb[:, None] * D * (K @ K.T), -1)
    Tm = np.linalg.inv(np.eye(L) + A)
    W = Tm @ ((bb * np.exp(g))[:, None] * K)
    Ut = Tm @ (bb[:, None] * V)
    Kpp = np.exp(g[-1] - g)[:, None] * K
    return np.exp(g[-1]) * np.eye(dk) - W.T @ Kpp, Ut.T @ Kpp


@pytest.mark.parametrize("G", [1, 2, 3, 5, 9])
def test_two_level_scan_matches_recurrence(G):
    """The state passes' two-level scan: a node's chunks split into G groups
    [g n / G, (g+1) n / G) (in chunks); each later group's zero-start end
    state N_g and transition M_g (identity start, Utilde = 0) composed
    chunk by chunk; the start states S_1 = end of group 0 and
    S_{g+1} = S_g M_g + N_g; every group replayed from its start state.
    Outputs and the end state equal the step-by-step recurrence."""
    rng = np.random.default_rng(4000 + G)
    C, n_ch, H, dk, dv = 4, 27, 2, 8, 6
    n = n_ch * C - 3  # the last chunk ragged
    q = rng.standard_normal((n, H, dk)) / 8
    k = rng.standard_normal((n, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((n, H, dv)) / 8
    a = np.exp(-0.1 * np.log1p(np.exp(rng.standard_normal((n, H)))))
    b = 1 / (1 + np.exp(-rng.standard_normal((n, H))))
    S0 = rng.standard_normal((H, dv, dk)) * 0.1
    o_ref, S_ref = gdn.gated_delta_rule(q, k, v, a, b, S0=S0)
    bounds = [g * n_ch // G for g in range(G + 1)]  # in chunks
    o = np.zeros_like(o_ref)
    S_end = np.zeros_like(S0)
    for h in range(H):
        # first pass: N_g and M_g of every later group, chunk by chunk (M from the identity, N from zero)
        Ms, Ns = [], []
        for g in range(1, G):
            Mg, Ng = np.eye(dk), np.zeros((dv, dk))
            for c in range(bounds[g], bounds[g + 1]):
                Mc, Nc = chunk_map(k, v, a, b, C, h, c * C)
                Mg, Ng = Mg @ Mc, Ng @ Mc + Nc
            Ms.append(Mg)
            Ns.append(Ng)
        # start states: S_1 = end of group 0, then S_{g+1} = S_g M_g + N_g
        t0, t1 = bounds[0] * C, min(n, bounds[1] * C)
        _, S1 = chunked(q[t0:t1, h:h + 1], k[t0:t1, h:h + 1], v[t0:t1, h:h + 1], a[t0:t1, h:h + 1],
                        b[t0:t1, h:h + 1], C, S0=S0[h:h + 1])
        starts = [S0[h], S1[0]]
        for g in range(1, G - 1):
            starts.append(starts[-1] @ Ms[g - 1] + Ns[g - 1])
        # second pass: every group from its start state, with outputs
        for g in range(G):
            t0, t1 = bounds[g] * C, min(n, bounds[g + 1] * C)
            og, Sg = chunked(q[t0:t1, h:h + 1], k[t0:t1, h:h + 1], v[t0:t1, h:h + 1], a[t0:t1, h:h + 1],
                             b[t0:t1, h:h + 1], C, S0=starts[g][None])
            o[t0:t1, h] = og[:, 0]
            if g == G - 1:
                S_end[h] = Sg[0]
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(S_end, S_ref, atol=1e-12)


def test_log_depth_combine_of_group_maps():
    """The groups' affine maps (M_g, N_g) compose associatively:
    (M_a, N_a) then (M_b, N_b) = (M_a M_b, N_a M_b + N_b).  An inclusive
    prefix scan in ceil(log2 G) rounds (every entry combines with the one
    2^r before it) gives the same start states as the sequential chain
    S_{g+1} = S_g M_g + N_g, and both equal the recurrence's state at the
    group boundaries."""
    rng = np.random.default_rng(4100)
    C, n_ch, dk, dv, G = 4, 40, 8, 6, 9
    n = n_ch * C
    q = rng.standard_normal((n, 1, dk)) / 8
    k = rng.standard_normal((n, 1, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((n, 1, dv)) / 8
    a = np.exp(-0.1 * np.log1p(np.exp(rng.standard_normal((n, 1)))))
    b = 1 / (1 + np.exp(-rng.standard_normal((n, 1))))
    S0 = rng.standard_normal((1, dv, dk)) * 0.1
    bounds = [g * n_ch // G for g in range(G + 1)]
    maps = []
    for g in range(G):
        Mg, Ng = np.eye(dk), np.zeros((dv, dk))
        for c in range(bounds[g], bounds[g + 1]):
            Mc, Nc = chunk_map(k, v, a, b, C, 0, c * C)
            Mg, Ng = Mg @ Mc, Ng @ Mc + Nc
        maps.append((Mg, Ng))
    # sequential: S_{g+1} = S_g M_g + N_g from the node's start state
    seq = [S0[0]]
    for Mg, Ng in maps:
        seq.append(seq[-1] @ Mg + Ng)
    # log depth: after round r, entry g holds the composition of groups max(0, g - 2^(r+1) + 1) .. g
    pre = list(maps)
    r = 1
    while r < G:
        pre = [pre[g] if g < r else (pre[g - r][0] @ pre[g][0], pre[g - r][1] @ pre[g][0] + pre[g][1])
               for g in range(G)]
        r *= 2
    for g in range(G):
        np.testing.assert_allclose(S0[0] @ pre[g][0] + pre[g][1], seq[g + 1], atol=1e-12)
    # both equal the step-by-step recurrence at the group boundaries
    for g in range(1, G + 1):
        t1 = bounds[g] * C
        _, S_ref = gdn.gated_delta_rule(q[:t1], k[:t1], v[:t1], a[:t1], b[:t1], S0=S0)
        np.testing.assert_allclose(seq[g], S_ref[0], atol=1e-12)
