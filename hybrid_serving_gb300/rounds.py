"""Host helpers around hs_round: build a round from a tree description and
move per-node arrays into / out of stream order using the library's layout.

A tree description is any object with ``requests``, each request having
``parents`` (node 0 is the root, parents precede children), ``n_tok``,
``readout`` (bools), ``hist_len`` and ``save`` ({node: state slot}).
"""
from __future__ import annotations

from typing import Dict, Optional, Tuple

import numpy as np

from . import _lib
from .api import PagePool, Round, round_caps_for


def build_round(tree, pool: Optional[PagePool] = None, caps=None, temp_slot0: int = 0,
                n_temp_slots: Optional[int] = None, resume: Optional[Dict[int, tuple]] = None):
    """Returns (Round, {(request, node): segment id}).

    ``resume``: {request: (ckpt_slot, [(ntok, [pages...]), ...][, window_row0])}
    for roots resumed at ``hist_len`` (the span list may be empty for
    GDN-only rounds; window_row0 = the root's conv window in the caller's
    window buffer).
    """
    resume = resume or {}
    n_seg = sum(r.n_nodes for r in tree.requests)
    T = sum(sum(r.n_tok) for r in tree.requests)
    depth = 1
    for req in tree.requests:
        d = [0] * req.n_nodes
        for i in range(1, req.n_nodes):
            d[i] = d[req.parents[i]] + 1
        depth = max(depth, max(d) + 1)
    n_hs = sum(len(v[1]) for v in resume.values())
    n_hp = sum(len(p) for v in resume.values() for _, p in v[1])
    if caps is None:
        caps = round_caps_for(T, n_seg, depth, n_hs, n_hp)
    R = Round(caps)
    seg_of = {}
    parents, n_tok, flags, saves = [], [], [], []
    for r, req in enumerate(tree.requests):  # node ids in add order: requests in turn, nodes in order
        for i in range(req.n_nodes):
            seg_of[(r, i)] = len(parents)
            parents.append(-1 if i == 0 else seg_of[(r, req.parents[i])])
            n_tok.append(req.n_tok[i])
            flags.append(_lib.HS_SEG_READOUT if req.readout[i] else _lib.HS_SEG_NO_READOUT)
            saves.append(req.save.get(i, -1))
    R.add_segments(parents, n_tok, flags, saves)
    for r, req in enumerate(tree.requests):
        if req.hist_len:
            res = resume.get(r, (None, []))
            slot, spans = res[0], res[1]
            if len(res) > 2 and res[2] is not None:
                R.set_conv_window(seg_of[(r, 0)], res[2])
            if slot is not None:
                R.gdn_state_resume(seg_of[(r, 0)], slot, req.hist_len)
            if spans:
                R.attach_history(seg_of[(r, 0)], [n for n, _ in spans], [p for _, ps in spans for p in ps])
    R.finalize(pool, temp_slot0, n_seg if n_temp_slots is None else n_temp_slots)
    return R, seg_of


def to_stream(R: Round, seg_of: Dict[Tuple[int, int], int], per_node, key: Optional[str] = None) -> np.ndarray:
    """Scatter {(r, node): array [n, ...]} (or {(r,node): {key: array}}) into stream order."""
    first = next(iter(per_node.values()))
    first = first[key] if key is not None else first
    T = R.info().n_tokens
    out = np.zeros((T,) + tuple(first.shape[1:]), dtype=first.dtype)
    for node, s in seg_of.items():
        a = per_node[node][key] if key is not None else per_node[node]
        info = R.segment(s)
        out[info.stream_off:info.stream_off + info.n_tokens] = a
    return out


def from_stream(R: Round, seg_of: Dict[Tuple[int, int], int], arr) -> Dict[Tuple[int, int], np.ndarray]:
    out = {}
    for node, s in seg_of.items():
        info = R.segment(s)
        out[node] = arr[info.stream_off:info.stream_off + info.n_tokens]
    return out


def split_at_requests(tree, caps, resume: Optional[Dict[int, tuple]] = None):
    """Split a batch of requests into rounds that each fit the capacity bucket ``caps``, at request
    boundaries and in request order (Flide section 3.3.2: rounds are cut between requests, so every
    request's result is the one it has alone -- section 3.5).  Requests are packed greedily: a run of
    whole requests goes into one round while the capacities ``hs_round_caps_for`` derives from the
    run's totals (tokens, nodes, depth, history spans and pages) are within ``caps`` in every field;
    those capacities suffice for any round of those totals, so every group builds.  ``resume`` as for
    build_round.  Returns a list of lists of request indices; a request that does not fit alone
    raises HsError(HS_ECAPACITY)."""
    resume = resume or {}
    bucket = caps.as_dict()

    def totals(r):
        req = tree.requests[r]
        d = [0] * len(req.parents)
        for i in range(1, len(req.parents)):
            d[i] = d[req.parents[i]] + 1
        spans = resume.get(r, (None, []))[1]
        return (sum(req.n_tok), len(req.parents), max(d) + 1, len(spans), sum(len(p) for _, p in spans))

    def fits(t):
        need = round_caps_for(t[0], t[1], t[2], t[3], t[4]).as_dict()
        return all(need[k] <= bucket[k] for k in need)

    groups, cur, acc = [], [], None
    for r in range(len(tree.requests)):
        t = totals(r)
        if not fits(t):
            raise _lib.HsError(_lib.HS_ECAPACITY, f"request {r} alone exceeds the bucket's capacities")
        nxt = t if acc is None else (acc[0] + t[0], acc[1] + t[1], max(acc[2], t[2]), acc[3] + t[3], acc[4] + t[4])
        if cur and not fits(nxt):
            groups.append(cur)
            cur, nxt = [], t
        cur.append(r)
        acc = nxt
    if cur:
        groups.append(cur)
    return groups
