"""Scaled dot-product causal attention over ONE isolated sequence, float64.

Test infrastructure only.

Definition (Flex, "Request-Adaptive Execution for Efficient Hybrid LLM
Inference", section 2, Eq. 1: softmax(Q K^T / sqrt(d_h)) V; Flide, section
3.2.1: in the isolated sequence s (+) q_i a token sees every token at or
before its position): for query row t and head h,

    o[t, h] = sum_{u <= t} softmax_u( scale * q[t, h] . k[u, g] ) v[u, g]

with g = floor(h / (Hq / Hkv)) (grouped-query heads share a key/value head;
the pages name grouped heads but no mapping -- consecutive query heads share
one key/value head).  The softmax subtracts the row maximum before exp.
"""
from __future__ import annotations

import numpy as np


def visible_range(t: int, window: int | None = None, bidir: int = 0):
    """Keys [lo, hi) row t sees: u <= t (causal), t - u < W with a window (Flide, section 3.2.1), and,
    with a bidirectional block of the first ``bidir`` tokens (Flide, Appendix H: the state of a model
    that reads it both ways), every token of that block for a row inside it."""
    hi = t + 1
    if t < bidir:
        hi = bidir
    lo = 0 if window is None else max(0, t - window + 1)
    return lo, hi


def causal_attention(q, k, v, scale: float, rows=None, window: int | None = None, bidir: int = 0):
    """q [n, Hq, d]; k, v [n, Hkv, d]; returns o [len(rows), Hq, d] float64.

    ``rows``: indices t of the query rows to produce (default: all).  A query
    row t only reads q[t]; keys/values in visible_range(t) are read.
    ``window``: optional sliding width W (Flide, section 3.2.1: adds
    t_x - t_y < W).  ``bidir``: the first ``bidir`` tokens form a block seen
    both ways (their rows see the whole block; later rows are causal).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, hq, d = q.shape
    hkv = k.shape[1]
    assert hq % hkv == 0
    g = hq // hkv
    if rows is None:
        rows = range(n)
    rows = list(rows)
    out = np.empty((len(rows), hq, d), dtype=np.float64)
    for o_i, t in enumerate(rows):
        lo, hi = visible_range(t, window, bidir)
        kk = k[lo:hi]                            # [u, Hkv, d]
        vv = v[lo:hi]
        qt = q[t].reshape(hkv, g, d)             # [Hkv, G, d]
        s = np.einsum("hgd,uhd->hgu", qt, kk) * scale
        m = s.max(axis=-1, keepdims=True)
        p = np.exp(s - m)
        l = p.sum(axis=-1, keepdims=True)
        o = np.einsum("hgu,uhd->hgd", p, vv) / l
        out[o_i] = o.reshape(hq, d)
    return out


def causal_attention_rows(q, k, v, scale: float, rows=None, window: int | None = None, bidir: int = 0):
    """The same quantity as causal_attention, evaluated one query head at a
    time as a matrix: the scores of the requested rows against every key,
    the keys after a row (and, with ``window``, those W or more positions
    before it) set to -inf, then the row-max-subtracted softmax and its
    product with V, all in float64.  Same arguments and result layout.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, hq, d = q.shape
    hkv = k.shape[1]
    assert hq % hkv == 0
    g = hq // hkv
    rows = np.arange(n) if rows is None else np.asarray(list(rows), dtype=np.int64)
    u = np.arange(n)
    hi = np.where(rows < bidir, bidir, rows + 1)
    visible = u[None, :] < hi[:, None]
    if window is not None:
        visible &= u[None, :] > rows[:, None] - window
    out = np.empty((len(rows), hq, d), dtype=np.float64)
    for h in range(hq):
        kv = h // g
        s = np.where(visible, (q[rows, h] @ k[:, kv].T) * scale, -np.inf)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        out[:, h] = (p @ v[:, kv]) / p.sum(axis=1, keepdims=True)
    return out
