"""Pins of the gated-delta-rule oracle (Flide section 3.2.2, Eq. 4).

* brute force: the unrolled product expansion with explicit d x d factors;
* closed form with orthonormal keys; the overwrite property of the delta
  rule; alpha = 1, beta = 0 gives S = 0;
* the hand-worked d = 1 fork;
* resume from a saved state equals the full recompute (section 3.4);
* sibling independence of the tree-level oracle.
"""
import os

import numpy as np

import synth
from oracle import forward, gdn

GOLD = os.path.join(os.path.dirname(__file__), "golden", "hand_fork_example.txt")


def _gold(kind, name):
    for line in open(GOLD):
        f = line.split()
        if f and not f[0].startswith("#") and f[0] == kind and f[1] == name:
            return [float(x) for x in f[2:]]
    raise KeyError(name)


def test_product_expansion_bruteforce():
    """S_t = sum_{i<=t} beta_i v_i k_i^T B_{i+1} ... B_t with the d x d factors
    B_j = alpha_j (I - beta_j k_j k_j^T) multiplied on the right in increasing
    j (unrolling Eq. 4 from S_0 = 0)."""
    rng = np.random.default_rng(0)
    for T in range(1, 7):
        H, dk, dv = 2, 3, 2
        q = rng.standard_normal((T, H, dk))
        k = rng.standard_normal((T, H, dk))
        v = rng.standard_normal((T, H, dv))
        a = rng.uniform(0.5, 1.0, (T, H))
        b = rng.uniform(0.0, 1.0, (T, H))
        o, S = gdn.gated_delta_rule(q, k, v, a, b)
        for h in range(H):
            B = [a[j, h] * (np.eye(dk) - b[j, h] * np.outer(k[j, h], k[j, h])) for j in range(T)]
            for t in range(T):
                St = np.zeros((dv, dk))
                for i in range(t + 1):
                    term = b[i, h] * np.outer(v[i, h], k[i, h])
                    for j in range(i + 1, t + 1):
                        term = term @ B[j]
                    St += term
                np.testing.assert_allclose(o[t, h], St @ q[t, h], atol=1e-14)
            np.testing.assert_allclose(S[h], St, atol=1e-14)


def test_orthonormal_keys_closed_form():
    """k_t = e_t: S_t = sum_i beta_i (prod_{j=i+1..t} alpha_j) v_i e_i^T, and
    q = e_i reads column i exactly."""
    rng = np.random.default_rng(1)
    T, dk, dv = 5, 6, 3
    k = np.eye(dk)[:T][:, None, :]
    v = rng.standard_normal((T, 1, dv))
    a = rng.uniform(0.6, 1.0, (T, 1))
    b = rng.uniform(0.1, 1.0, (T, 1))
    for i in range(T):
        q = np.zeros((T, 1, dk))
        q[:, 0, i] = 1.0
        o, _ = gdn.gated_delta_rule(q, k, v, a, b)
        for t in range(T):
            want = np.zeros(dv) if t < i else b[i, 0] * np.prod(a[i + 1:t + 1, 0]) * v[i, 0]
            np.testing.assert_allclose(o[t, 0], want, atol=1e-15)


def test_delta_rule_overwrites_same_key():
    """beta = 1, alpha = 1, the same unit key twice: the second write replaces
    the first value (S k = v2), which fixes the sign of the delta term."""
    e = np.array([0.6, 0.8, 0.0])
    k = np.stack([e, e])[:, None, :]
    v = np.array([[1.0, 2.0], [-3.0, 5.0]])[:, None, :]
    q = k.copy()
    o, S = gdn.gated_delta_rule(q, k, v, np.ones((2, 1)), np.ones((2, 1)))
    np.testing.assert_allclose(o[0, 0], v[0, 0], atol=1e-15)
    np.testing.assert_allclose(o[1, 0], v[1, 0], atol=1e-15)


def test_no_write_keeps_zero_state():
    rng = np.random.default_rng(2)
    T, H, d = 4, 2, 3
    o, S = gdn.gated_delta_rule(rng.standard_normal((T, H, d)), rng.standard_normal((T, H, d)),
                                rng.standard_normal((T, H, d)), np.ones((T, H)), np.zeros((T, H)))
    assert not o.any() and not S.any()


def test_hand_worked_fork():
    def seq(rows):
        rows = np.array(rows, float)
        n = len(rows)
        return dict(q=np.ones((n, 1, 1)), k=np.ones((n, 1, 1)), v=rows[:, 2].reshape(n, 1, 1),
                    alpha=rows[:, 0].reshape(n, 1), beta=rows[:, 1].reshape(n, 1))
    trunk = seq([(0.5, 0.5, 2), (0.5, 0.5, 4)])
    A = seq([(1, 0.5, 0)])
    B = seq([(0.8, 0.25, 8)])
    tree = synth.Tree([synth.fork_tree(2, [1, 1])])
    nodes = {(0, 0): trunk, (0, 1): A, (0, 2): B}
    hist = {0: {k: v[:0] for k, v in trunk.items()}}
    inp = synth.GdnInputs(1, 1, 1, False, nodes, hist)
    out = forward.gdn_tree(tree, inp)
    np.testing.assert_allclose(out[(0, 0)].ravel(), _gold("gdn", "trunk_out"), atol=1e-15)
    np.testing.assert_allclose(out[(0, 1)].ravel(), _gold("gdn", "branchA_out"), atol=1e-15)
    np.testing.assert_allclose(out[(0, 2)].ravel(), _gold("gdn", "branchB_out"), atol=1e-15)
    cat = {k: np.concatenate([trunk[k], A[k], B[k]]) for k in trunk}
    o, _ = gdn.gated_delta_rule(cat["q"], cat["k"], cat["v"], cat["alpha"], cat["beta"])
    np.testing.assert_allclose(o[-1].ravel(), _gold("gdn", "branchB_if_after_A"), atol=1e-15)


def test_resume_from_state_equals_recompute():
    """Section 3.4: restoring the state at m and continuing is the same
    sequence of operations as the full pass, so the results are identical."""
    rng = np.random.default_rng(4)
    T, H, d, m = 20, 2, 5, 13
    q, k, v = (rng.standard_normal((T, H, d)) for _ in range(3))
    a = rng.uniform(0.8, 1.0, (T, H))
    b = rng.uniform(0.1, 0.9, (T, H))
    o_full, S_full = gdn.gated_delta_rule(q, k, v, a, b)
    _, S_m = gdn.gated_delta_rule(q[:m], k[:m], v[:m], a[:m], b[:m])
    o_res, S_res = gdn.gated_delta_rule(q[m:], k[m:], v[m:], a[m:], b[m:], S0=S_m)
    assert np.array_equal(o_res, o_full[m:]) and np.array_equal(S_res, S_full)


def test_tree_oracle_is_isolated_and_sibling_independent():
    tree = synth.Tree([synth.Request(parents=[-1, 0, 0, 1], n_tok=[7, 3, 4, 2])])
    inp = synth.gdn_inputs(tree, 2, 4, 3, seed=8, bf16=False)
    out = forward.gdn_tree(tree, inp)
    # node 3's isolated pass is root -> 1 -> 3
    seq = {k: np.concatenate([inp.nodes[(0, i)][k] for i in (0, 1, 3)]) for k in inp.nodes[(0, 0)]}
    o, _ = gdn.gated_delta_rule(seq["q"], seq["k"], seq["v"], seq["alpha"], seq["beta"])
    assert np.array_equal(out[(0, 3)], o[-2:])
    inp.nodes[(0, 2)]["v"] = inp.nodes[(0, 2)]["v"] * 5
    out2 = forward.gdn_tree(tree, inp)
    assert np.array_equal(out[(0, 3)], out2[(0, 3)]) and np.array_equal(out[(0, 1)], out2[(0, 1)])
