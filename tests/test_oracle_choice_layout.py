"""Pins of the choice oracle (Flide Eq. 1) and of the layout / accounting
oracle (Flide Eq. 2, Eq. 3; ForkServe cost model)."""
import math
import os

import numpy as np

import synth
from oracle import choice, layout

G = os.path.join(os.path.dirname(__file__), "golden")


def _kv(path):
    d = {}
    for line in open(path):
        f = line.split()
        if f and not f[0].startswith("#"):
            d[f[0]] = [float(x) if "." in x else int(x) for x in f[1:]]
    return d


def test_choice_hand_example():
    gold = None
    for line in open(os.path.join(G, "hand_fork_example.txt")):
        f = line.split()
        if f[:2] == ["choice", "p"]:
            gold = [float(x) for x in f[2:]]
    W = np.eye(4)
    h = np.array([[0.0, math.log(3), 0.0, 0.0]])
    lp = choice.option_logprobs(h, W)
    np.testing.assert_allclose(np.exp(lp[0]), gold, atol=1e-15)


def test_choice_shift_invariance_and_measures():
    rng = np.random.default_rng(0)
    W = rng.standard_normal((4, 6))
    h = rng.standard_normal((3, 6))
    lp = choice.option_logprobs(h, W)
    np.testing.assert_allclose(np.exp(lp).sum(-1), 1.0, atol=1e-15)
    z = h @ W.T
    np.testing.assert_allclose(lp[:, 1] - lp[:, 0], z[:, 1] - z[:, 0], atol=1e-13)
    p = np.array([[0.5, 0.5, 0, 0], [0.1, 0.2, 0.3, 0.4]])
    assert choice.top1(p)[0] == 0 and choice.top1(p)[1] == 3
    np.testing.assert_allclose(choice.total_variation(p, p), 0.0)
    np.testing.assert_allclose(choice.total_variation([1, 0], [0, 1]), 1.0)
    assert list(choice.decision(p)) == [0, -1]


def test_stream_layout_eq2():
    """Trunks of all requests first, then request 1's branches, then request
    2's; deeper levels after (hand-listed)."""
    t = synth.Tree([synth.fork_tree(5, [2, 3]),
                    synth.Request(parents=[-1, 0, 1], n_tok=[4, 1, 2])])
    lay = layout.stream_layout(t)
    assert lay == {(0, 0): 0, (1, 0): 5, (0, 1): 9, (0, 2): 11, (1, 1): 14, (1, 2): 15}
    j, c, tt, ix = layout.token_metadata(t)
    # request 0 branch 2 continues from P = 5
    assert tt[11:14] == [5, 6, 7] and c[11:14] == [2, 2, 2] and ix[11:14] == [0, 1, 2]
    # request 1's level-2 node continues from 4 + 1
    assert tt[15:17] == [5, 6] and j[15] == 1


def test_visible_keys_eq3():
    t = synth.Tree([synth.Request(parents=[-1, 0, 0, 1], n_tok=[3, 2, 2, 1], hist_len=2)])
    vis = layout.visible_keys(t, 0, 3, 0)
    assert vis == sorted([(-1, 0), (-1, 1), (0, 0), (0, 1), (0, 2), (1, 0), (1, 1), (3, 0)])
    vis = layout.visible_keys(t, 0, 2, 0)        # sibling of node 1: no (1, *)
    assert (1, 0) not in vis and (2, 0) in vis and len(vis) == 6


def test_forkserve_cost_model_counts():
    g = _kv(os.path.join(G, "forkserve_cost_model.txt"))
    n, k, L, l, P = (g[x][0] for x in ("sessions", "fanout", "trunk", "residual", "page"))
    tree = synth.Tree([synth.fork_tree(L, [l] * k) for _ in range(n)])
    assert layout.isolated_tokens(tree) == g["isolated_prefill_tokens"][0]
    assert layout.forked_tokens(tree) == g["forked_prefill_tokens"][0]
    assert layout.live_pages(tree, P) * P == g["peak_kv_tokens_forked"][0]
    spine = sum(layout.spine_pages(r, 1, P) for r in tree.requests) * P
    assert spine == g["spine_kv_tokens"][0]


def test_flide_table2_single_question_rows():
    for line in open(os.path.join(G, "flide_table2_single_question.txt")):
        f = line.split()
        if not f or f[0].startswith("#"):
            continue
        n, P, stream, seqs = (int(x) for x in f[1:])
        q = stream - P
        tree = synth.Tree([synth.fork_tree(P, [q] * n)])
        assert layout.forked_tokens(tree) == stream
        assert layout.isolated_tokens(tree) == seqs


def test_deep_tree_counts():
    """Depth-3 fan-out of 4 over trunk 256 with 32-token residuals: forked
    = 256 + 84*32 = 2944 tokens; isolated = 64 leaves x (256 + 3*32) = 22528;
    16 + 84*2 = 184 pages live."""
    req = synth.fanout_tree(256, 32, 4, 3)
    t = synth.Tree([req])
    assert layout.forked_tokens(t) == 256 + 84 * 32 == 2944
    assert layout.isolated_tokens(t) == 64 * (256 + 96) == 22528
    assert layout.live_pages(t, 16) == 184
