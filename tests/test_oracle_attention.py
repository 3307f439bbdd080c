"""Pins of the attention oracle against values the definitions fix.

Each check is chosen so that a plausible slip in the oracle (a dropped
scale, a wrong GQA mapping, a sibling leaking in, an off-by-one in the
causal bound, a wrong position for a resumed root) fails one of them.
"""
import math
import os

import numpy as np
import pytest

import synth
from oracle import attention, forward, layout

GOLD = os.path.join(os.path.dirname(__file__), "golden", "hand_fork_example.txt")


def _gold(kind, name):
    for line in open(GOLD):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        if f[0] == kind and f[1] == name:
            return [float(x) for x in f[2:]]
    raise KeyError(name)


def _inp(tree, per_node, hq=1, hkv=1, d=1, hist=None):
    nodes = {}
    for (r, i), (q, k, v) in per_node.items():
        nodes[(r, i)] = {"q": np.array(q, float).reshape(-1, hq, d),
                         "k": np.array(k, float).reshape(-1, hkv, d),
                         "v": np.array(v, float).reshape(-1, hkv, d)}
    hist = hist or {r: {"q": np.zeros((0, hq, d)), "k": np.zeros((0, hkv, d)), "v": np.zeros((0, hkv, d))}
                    for r in range(len(tree.requests))}
    return synth.AttnInputs(hq, hkv, d, False, nodes, hist)


def test_hand_worked_fork():
    """Flide Eq. 3 on the hand example: trunk (0,3), branch A 4, branch B -1/2."""
    tree = synth.Tree([synth.fork_tree(2, [1, 1])])
    inp = _inp(tree, {(0, 0): ([1, 1], [0, math.log(3)], [0, 4]),
                      (0, 1): ([1], [0], [8]),
                      (0, 2): ([1], [math.log(4)], [-4])})
    out = forward.attention_tree(tree, inp, scale=1.0)
    np.testing.assert_allclose(out[(0, 0)].ravel(), _gold("attn", "trunk_out"), atol=1e-14)
    np.testing.assert_allclose(out[(0, 1)].ravel(), _gold("attn", "branchA_out"), atol=1e-14)
    np.testing.assert_allclose(out[(0, 2)].ravel(), _gold("attn", "branchB_out"), atol=1e-14)
    # the leak a fork must avoid: B in one sequence after A
    leak = attention.causal_attention(np.ones((4, 1, 1)),
                                      np.array([0, math.log(3), 0, math.log(4)]).reshape(4, 1, 1),
                                      np.array([0, 4, 8, -4.0]).reshape(4, 1, 1), 1.0, rows=[3])
    np.testing.assert_allclose(leak.ravel(), _gold("attn", "branchB_if_it_saw_A"), atol=1e-14)
    assert abs(leak.ravel()[0] - out[(0, 2)].ravel()[0]) > 0.5


def test_zero_query_is_mean_of_visible_values():
    """q = 0 makes every softmax uniform, so o = mean of v over EXACTLY the
    keys Eq. 3 lets the row see: enumerated literally by layout.visible_keys
    over every token of the request (multi-level tree, resumed root)."""
    rng = np.random.default_rng(7)
    req = synth.Request(parents=[-1, 0, 0, 1, 1, 2], n_tok=[5, 3, 4, 2, 3, 1], hist_len=6)
    req2 = synth.fork_tree(3, [2, 2])
    tree = synth.Tree([req, req2])
    hq, hkv, d = 4, 2, 3
    inp = synth.attn_inputs(tree, hq, hkv, d, seed=11, bf16=False)
    for key in inp.nodes:
        inp.nodes[key]["q"] = np.zeros_like(inp.nodes[key]["q"])
    out = forward.attention_tree(tree, inp, scale=0.5)
    for (r, i), o in out.items():
        R = tree.requests[r]
        for u in range(R.n_tok[i]):
            vis = layout.visible_keys(tree, r, i, u)
            vals = [inp.hist[r]["v"][x] if nd < 0 else inp.nodes[(r, nd)]["v"][x] for nd, x in vis]
            mean = np.mean(np.asarray(vals, np.float64), axis=0)        # [Hkv, d]
            for h in range(hq):
                np.testing.assert_allclose(o[u, h], mean[h // (hq // hkv)], atol=1e-14)
    assert rng is not None


def test_first_row_sees_only_itself():
    rng = np.random.default_rng(1)
    q, k, v = (rng.standard_normal((5, 2, 4)) for _ in range(3))
    o = attention.causal_attention(q, k, v, 0.5, rows=[0])
    np.testing.assert_allclose(o[0], v[0], atol=1e-15)


def test_scale_is_inverse_sqrt_d():
    """d = 4, q = a*1, k1 = b*1 with a*b = ln(3)/2: q.k1 / sqrt(4) = ln 3, so the
    weights of (k0 = 0, k1) are 1:3 exactly; without the scale they would be 1:9."""
    d = 4
    a = 1.0
    b = math.log(3) / 2
    q = np.full((2, 1, d), a)
    k = np.stack([np.zeros(d), np.full(d, b)]).reshape(2, 1, d)
    v = np.stack([np.full(d, 1.0), np.full(d, 5.0)]).reshape(2, 1, d)
    o = attention.causal_attention(q, k, v, 1 / math.sqrt(d), rows=[1])
    np.testing.assert_allclose(o[0, 0], np.full(d, (1 + 3 * 5) / 4), atol=1e-14)


def test_gqa_mapping_consecutive_heads():
    """Hq = 4 over Hkv = 2: heads 0,1 read kv head 0, heads 2,3 kv head 1."""
    n, d = 3, 2
    q = np.zeros((n, 4, d))
    k = np.zeros((n, 2, d))
    v = np.zeros((n, 2, d))
    v[:, 0] = 1.0
    v[:, 1] = -2.0
    o = attention.causal_attention(q, k, v, 1.0)
    np.testing.assert_allclose(o[:, :2], 1.0)
    np.testing.assert_allclose(o[:, 2:], -2.0)


def test_flat_stream_mask_equals_isolated_passes():
    """Brute force on the flat stream: the full T x T score matrix with a -inf
    mask built from Eq. 3 on the stream metadata (request j, node c,
    position t), softmax per row.  Must equal the oracle's isolated passes."""
    req = synth.Request(parents=[-1, 0, 0, 1, 1], n_tok=[4, 3, 2, 2, 1])
    tree = synth.Tree([req, synth.fork_tree(5, [2, 3, 1])])
    hq, hkv, d = 2, 1, 4
    inp = synth.attn_inputs(tree, hq, hkv, d, seed=5, bf16=False)
    lay = layout.stream_layout(tree)
    T = layout.stream_length(tree)
    j, c, t, _ = layout.token_metadata(tree)
    Q = np.zeros((T, hq, d)); K = np.zeros((T, hkv, d)); V = np.zeros((T, hkv, d))
    for (r, i), off in lay.items():
        n = tree.requests[r].n_tok[i]
        Q[off:off + n] = inp.nodes[(r, i)]["q"]
        K[off:off + n] = inp.nodes[(r, i)]["k"]
        V[off:off + n] = inp.nodes[(r, i)]["v"]
    anc = {(r, i): set(layout.ancestors(tree.requests[r], i))
           for r, R in enumerate(tree.requests) for i in range(R.n_nodes)}
    mask = np.zeros((T, T), bool)
    for x in range(T):
        for y in range(T):
            mask[x, y] = j[x] == j[y] and c[y] in anc[(j[x], c[x])] and t[y] <= t[x]
    scale = 1 / math.sqrt(d)
    ref = forward.attention_tree(tree, inp, scale)
    for h in range(hq):
        S = Q[:, h] @ K[:, h * hkv // hq].T * scale
        S = np.where(mask, S, -np.inf)
        P = np.exp(S - S.max(1, keepdims=True))
        O = (P / P.sum(1, keepdims=True)) @ V[:, h * hkv // hq]
        for (r, i), off in lay.items():
            n = tree.requests[r].n_tok[i]
            np.testing.assert_allclose(O[off:off + n], ref[(r, i)][:, h], atol=1e-13)


def test_sibling_perturbation_leaves_branch_unchanged():
    tree = synth.Tree([synth.fork_tree(6, [3, 4, 2])])
    inp = synth.attn_inputs(tree, 2, 2, 4, seed=3, bf16=False)
    a = forward.attention_tree(tree, inp, 0.5)
    inp.nodes[(0, 2)]["k"] = inp.nodes[(0, 2)]["k"] + 7.0
    inp.nodes[(0, 2)]["v"] = inp.nodes[(0, 2)]["v"] - 3.0
    b = forward.attention_tree(tree, inp, 0.5)
    assert np.array_equal(a[(0, 1)], b[(0, 1)]) and np.array_equal(a[(0, 3)], b[(0, 3)])
    assert not np.array_equal(a[(0, 2)], b[(0, 2)])


def test_resumed_root_equals_fresh_pass():
    """Flide section 3.4: a resumed request computes the same function as a
    fresh one.  History + tail + branch vs the unsplit trunk."""
    full = synth.Tree([synth.fork_tree(12, [3])])
    inp = synth.attn_inputs(full, 2, 1, 4, seed=9, bf16=False)
    res = synth.Tree([synth.fork_tree(5, [3], hist_len=7)])
    inp_r = synth.remap_inputs(full, inp, res)
    a = forward.attention_tree(full, inp, 0.5)
    b = forward.attention_tree(res, inp_r, 0.5)
    np.testing.assert_array_equal(a[(0, 1)], b[(0, 1)])
    np.testing.assert_array_equal(a[(0, 0)][7:], b[(0, 0)])


def test_stream_permutation_leaves_results_unchanged():
    """Eq. 3 depends only on each token's (request, node, position), not on
    where the token sits in the flat stream: the masked brute force over a
    randomly permuted stream, un-permuted, equals it over the Eq. 2 order."""
    req = synth.Request(parents=[-1, 0, 0, 2], n_tok=[5, 2, 3, 2])
    tree = synth.Tree([req, synth.fork_tree(4, [3, 1])])
    hq, hkv, d = 2, 1, 4
    inp = synth.attn_inputs(tree, hq, hkv, d, seed=9, bf16=False)
    lay = layout.stream_layout(tree)
    T = layout.stream_length(tree)
    j, c, t, _ = layout.token_metadata(tree)
    Q = np.zeros((T, hq, d)); K = np.zeros((T, hkv, d)); V = np.zeros((T, hkv, d))
    for (r, i), off in lay.items():
        n = tree.requests[r].n_tok[i]
        Q[off:off + n] = inp.nodes[(r, i)]["q"]
        K[off:off + n] = inp.nodes[(r, i)]["k"]
        V[off:off + n] = inp.nodes[(r, i)]["v"]
    anc = {(r, i): set(layout.ancestors(tree.requests[r], i))
           for r, R in enumerate(tree.requests) for i in range(R.n_nodes)}

    def brute(order):
        jj, cc, tt = (np.asarray(z)[order] for z in (j, c, t))
        mask = np.array([[jj[x] == jj[y] and cc[y] in anc[(int(jj[x]), int(cc[x]))] and tt[y] <= tt[x]
                          for y in range(T)] for x in range(T)])
        out = np.zeros((T, hq, d))
        for h in range(hq):
            S = np.where(mask, Q[order, h] @ K[order, h * hkv // hq].T / math.sqrt(d), -np.inf)
            P = np.exp(S - S.max(1, keepdims=True))
            out[:, h] = (P / P.sum(1, keepdims=True)) @ V[order, h * hkv // hq]
        return out

    base = brute(np.arange(T))
    perm = np.random.default_rng(10).permutation(T)
    moved = np.zeros_like(base)
    moved[perm] = brute(perm)
    np.testing.assert_allclose(moved, base, atol=1e-13)
    ref = forward.attention_tree(tree, inp, 1 / math.sqrt(d))
    for (r, i), off in lay.items():
        np.testing.assert_allclose(base[off:off + tree.requests[r].n_tok[i]], ref[(r, i)], atol=1e-13)


@pytest.mark.parametrize("window", [None, 5])
def test_matrix_form_equals_row_loop(window):
    """causal_attention_rows (a masked score matrix per head) reproduces the
    per-row definition on a ragged GQA case, all rows and a subset, with and
    without a sliding window."""
    rng = np.random.default_rng(41)
    n, hq, hkv, d = 37, 6, 2, 16
    q, k, v = (rng.standard_normal((n, h, d)) for h in (hq, hkv, hkv))
    for rows in (None, [0, 1, 17, 36]):
        a = attention.causal_attention(q, k, v, 0.3, rows=rows, window=window)
        b = attention.causal_attention_rows(q, k, v, 0.3, rows=rows, window=window)
        np.testing.assert_allclose(b, a, rtol=0, atol=1e-13)


def test_matrix_form_tree_equals_row_loop():
    tree = synth.Tree([synth.fork_tree(50, [7, 1, 12]), synth.fanout_tree(20, 5, 2, 2)])
    inp = synth.attn_inputs(tree, 4, 2, 32, seed=42, bf16=False)
    a = forward.attention_tree(tree, inp, 0.2)
    b = forward.attention_tree(tree, inp, 0.2, matrix=True)
    for key in a:
        np.testing.assert_allclose(b[key], a[key], rtol=0, atol=1e-13)


def _positions(req):
    """Position of each node's first token along its path (history first, then every ancestor)."""
    pos0 = [req.hist_len] * req.n_nodes
    for i in range(1, req.n_nodes):
        pos0[i] = pos0[req.parents[i]] + req.n_tok[req.parents[i]]
    return pos0


def _zero_query_case(seed):
    req = synth.Request(parents=[-1, 0, 0, 1, 1, 2], n_tok=[5, 3, 4, 2, 3, 1], hist_len=6)
    tree = synth.Tree([req, synth.fork_tree(3, [2, 2])])
    inp = synth.attn_inputs(tree, 4, 2, 3, seed=seed, bf16=False)
    for key in inp.nodes:
        inp.nodes[key]["q"] = np.zeros_like(inp.nodes[key]["q"])
    return tree, inp


def _value(inp, r, nd, x):
    return inp.hist[r]["v"][x] if nd < 0 else inp.nodes[(r, nd)]["v"][x]


@pytest.mark.parametrize("W", [1, 2, 5, 9])
def test_zero_query_window_is_mean_over_window(W):
    """Sliding window (Flide section 3.2.1, t_x - t_y < W): with q = 0 a row's output is the mean of v
    over the keys Eq. 3 lets it see (enumerated by layout.visible_keys) whose position is within W."""
    tree, inp = _zero_query_case(12)
    out = forward.attention_tree(tree, inp, scale=0.5, window=W)
    for (r, i), o in out.items():
        req = tree.requests[r]
        pos0 = _positions(req)
        for u in range(req.n_tok[i]):
            t = pos0[i] + u
            keep = [(nd, x) for nd, x in layout.visible_keys(tree, r, i, u)
                    if t - (x if nd < 0 else pos0[nd] + x) < W]
            mean = np.mean(np.asarray([_value(inp, r, nd, x) for nd, x in keep], np.float64), axis=0)
            for h in range(4):
                np.testing.assert_allclose(o[u, h], mean[h // 2], atol=1e-14)


def test_zero_query_bidirectional_root():
    """Bidirectional state block (Flide Appendix H): a root row sees every token of the history and of
    the root, later and earlier alike; every other row keeps Eq. 3's causal set."""
    tree, inp = _zero_query_case(13)
    out = forward.attention_tree(tree, inp, scale=0.5, bidir_root=True)
    for (r, i), o in out.items():
        req = tree.requests[r]
        for u in range(req.n_tok[i]):
            if i == 0:
                keys = [(-1, x) for x in range(req.hist_len)] + [(0, x) for x in range(req.n_tok[0])]
            else:
                keys = layout.visible_keys(tree, r, i, u)
            mean = np.mean(np.asarray([_value(inp, r, nd, x) for nd, x in keys], np.float64), axis=0)
            for h in range(4):
                np.testing.assert_allclose(o[u, h], mean[h // 2], atol=1e-14)


def test_matrix_form_equals_row_loop_with_bidirectional_block():
    rng = np.random.default_rng(43)
    n, d = 29, 16
    q, k, v = (rng.standard_normal((n, 2, d)) for _ in range(3))
    for bidir, window in ((11, None), (11, 4), (0, 3)):
        a = attention.causal_attention(q, k, v, 0.3, window=window, bidir=bidir)
        b = attention.causal_attention_rows(q, k, v, 0.3, window=window, bidir=bidir)
        np.testing.assert_allclose(b, a, rtol=0, atol=1e-13)
