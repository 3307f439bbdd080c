"""Flat-stream layout, token metadata, visibility and page accounting.

Test infrastructure only (see the package docstring).

Sources:
* Flide, section 3.2, Eq. 2: the round is one stream without padding, state
  trunks of all requests first, then the question branches of request 1,
  request 2, ...; every token carries (request j, branch c, position t) and
  a question's positions continue from the end of its state.
* Flide, section 3.2.1, Eq. 3: x sees y iff j_y = j_x, c_y in {0, c_x} and
  t_y <= t_x.  For trees deeper than trunk + questions (ForkServe README,
  "Copy-on-write context tree": a deeper fan-out is a chain of aliases) the
  branch condition reads "y's node is x's node or one of its ancestors".
* Flide, section 3.4: a resumed request starts its stream at the checkpoint
  position m; its first ``hist_len`` positions live in cached pages.
* ForkServe README, "Copy-on-write context tree": fork copies the parent
  page table and alias length and allocates nothing; writes allocate pages
  for the node's own tokens only.  Live KV is b (L + sum_i l_i); after the
  other residuals are aborted it is b (L + l_star).
"""
from __future__ import annotations

from math import ceil
from typing import Dict, List, Tuple


def depth(req) -> List[int]:
    d = [0] * req.n_nodes
    for i in range(1, req.n_nodes):
        d[i] = d[req.parents[i]] + 1
    return d


def ancestors(req, node: int) -> List[int]:
    """Root-to-node path, node included."""
    p = [node]
    while req.parents[p[-1]] >= 0:
        p.append(req.parents[p[-1]])
    return p[::-1]


def positions(req) -> List[int]:
    """First position of every node (Eq. 2 metadata t): the root starts at the
    history length, a child continues from its parent's last position + 1."""
    pos = [0] * req.n_nodes
    pos[0] = req.hist_len
    for i in range(1, req.n_nodes):
        p = req.parents[i]
        pos[i] = pos[p] + req.n_tok[p]
    return pos


def stream_layout(tree) -> Dict[Tuple[int, int], int]:
    """Offset of every (request, node) in the flat stream of Eq. 2.

    Level by level (trunks, then first-level branches, then deeper levels);
    within a level, request by request; within a request, node order.
    """
    deps = [depth(r) for r in tree.requests]
    max_d = max(max(d) for d in deps)
    off, out = 0, {}
    for lev in range(max_d + 1):
        for r, req in enumerate(tree.requests):
            for i in range(req.n_nodes):
                if deps[r][i] == lev:
                    out[(r, i)] = off
                    off += req.n_tok[i]
    return out


def stream_length(tree) -> int:
    return sum(sum(r.n_tok) for r in tree.requests)


def token_metadata(tree):
    """Per stream token (request j, node c, position t, index within node)."""
    lay = stream_layout(tree)
    T = stream_length(tree)
    j = [0] * T
    c = [0] * T
    t = [0] * T
    ix = [0] * T
    for r, req in enumerate(tree.requests):
        pos = positions(req)
        for i in range(req.n_nodes):
            o = lay[(r, i)]
            for u in range(req.n_tok[i]):
                j[o + u], c[o + u], t[o + u], ix[o + u] = r, i, pos[i] + u, u
    return j, c, t, ix


def visible_keys(tree, r: int, node: int, i: int):
    """Eq. 3 applied literally over every token of request r.

    Returns the visible keys as a sorted list of (node, index) with
    node = -1 for history tokens (positions before the resumed root).
    """
    req = tree.requests[r]
    anc = set(ancestors(req, node))
    pos = positions(req)
    tx = pos[node] + i
    out = []
    for u in range(req.hist_len):                 # history belongs to the root chain
        if u <= tx:
            out.append((-1, u))
    for y in range(req.n_nodes):
        if y not in anc:
            continue
        for u in range(req.n_tok[y]):
            if pos[y] + u <= tx:
                out.append((y, u))
    return sorted(out)


# --------------------------------------------------------------------------
# page / token accounting
# --------------------------------------------------------------------------
def own_pages(n_tok: int, page: int) -> int:
    return ceil(n_tok / page)


def live_pages(tree, page: int) -> int:
    """Pages live after a forked prefill: each node owns ceil(n/page) pages,
    children alias their ancestors' pages (no copies)."""
    return sum(own_pages(n, page) for r in tree.requests for n in r.n_tok)


def isolated_tokens(tree) -> int:
    """Tokens a per-question (isolated) prefill computes: n P + sum |q_i|,
    generalised to trees as the sum over leaves of their path lengths
    (Flide, section 3.1)."""
    tot = 0
    for req in tree.requests:
        kids = [0] * req.n_nodes
        for p in req.parents[1:]:
            kids[p] += 1
        for leaf in range(req.n_nodes):
            if kids[leaf] == 0:
                tot += sum(req.n_tok[a] for a in ancestors(req, leaf))
    return tot


def forked_tokens(tree) -> int:
    """Tokens the forked prefill computes: P + sum |q_i| (each once)."""
    return stream_length(tree)


def spine_pages(req, spine_leaf: int, page: int) -> int:
    return sum(own_pages(req.n_tok[a], page) for a in ancestors(req, spine_leaf))
