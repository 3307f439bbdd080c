"""Tree-level oracle: every node's rows from its own ISOLATED pass.

Test infrastructure only.

Flide, Proposition 3.1 (section 3.2.3, proof in Appendix A): the hidden
state at any token of question q_i equals the one the model computes on
s (+) q_i alone, whatever else is in the round.  So the oracle never forks:
for a node it concatenates the history (a resumed root's earlier tokens,
section 3.4), the root and every ancestor down to the node, runs the plain
layer over that sequence from scratch, and keeps the node's own rows.  A
trunk's rows come from the trunk run alone; a resumed request is a full
recompute, never a restored checkpoint.
"""
from __future__ import annotations

from typing import Dict, Iterable, Optional, Tuple

import numpy as np

from . import attention as _attn
from . import gdn as _gdn
from .layout import ancestors


def _path_seq(inp, r: int, req, node: int, key: str):
    parts = [inp.hist[r][key]] + [inp.nodes[(r, a)][key] for a in ancestors(req, node)]
    return np.concatenate([np.asarray(p, dtype=np.float64) for p in parts], axis=0)


def attention_tree(tree, inp, scale: float, nodes: Optional[Iterable[Tuple[int, int]]] = None,
                   rows: Optional[Dict[Tuple[int, int], Iterable[int]]] = None,
                   window: Optional[int] = None, matrix: bool = False, bidir_root: bool = False):
    """Returns {(r, node): o [n_rows, Hq, d]} for the requested nodes.

    ``rows`` optionally restricts a node to some of its row indices (a
    sampled check); each row is still its isolated-sequence output.
    ``matrix`` evaluates each isolated sequence with the matrix form of the
    same definition (attention.causal_attention_rows) -- for thousands of rows.
    ``window``: sliding width; ``bidir_root``: the root's tokens (with any
    resumed history) form a block seen both ways (attention.visible_range).
    """
    out = {}
    if nodes is None:
        nodes = [(r, i) for r, req in enumerate(tree.requests) for i in range(req.n_nodes)]
    for (r, i) in nodes:
        req = tree.requests[r]
        k = _path_seq(inp, r, req, i, "k")
        v = _path_seq(inp, r, req, i, "v")
        n_before = k.shape[0] - req.n_tok[i]
        sel = list(range(req.n_tok[i])) if rows is None or (r, i) not in rows else list(rows[(r, i)])
        q = np.zeros((k.shape[0], inp.hq, inp.d))
        q[n_before:] = inp.nodes[(r, i)]["q"]
        f = _attn.causal_attention_rows if matrix else _attn.causal_attention
        bidir = inp.hist[r]["k"].shape[0] + req.n_tok[0] if bidir_root else 0
        out[(r, i)] = f(q, k, v, scale, rows=[n_before + u for u in sel], window=window, bidir=bidir)
    return out


def gdn_tree(tree, inp, nodes: Optional[Iterable[Tuple[int, int]]] = None, want_state: bool = False):
    """Returns {(r, node): o [n_tok, H, dv]} (and end states if asked)."""
    out, states = {}, {}
    if nodes is None:
        nodes = [(r, i) for r, req in enumerate(tree.requests) for i in range(req.n_nodes)]
    for (r, i) in nodes:
        req = tree.requests[r]
        seq = {k: _path_seq(inp, r, req, i, k) for k in ("q", "k", "v", "alpha", "beta")}
        o, S = _gdn.gated_delta_rule(seq["q"], seq["k"], seq["v"], seq["alpha"], seq["beta"])
        out[(r, i)] = o[o.shape[0] - req.n_tok[i]:]
        states[(r, i)] = S
    return (out, states) if want_state else out
