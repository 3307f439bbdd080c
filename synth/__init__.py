"""Seeded synthetic inputs for tree-structured (forked) prefill.

This module is the ONE thing the oracle and the CUDA path share: it draws
tree shapes and per-token layer inputs from seeded generators.  It holds none
of the method's arithmetic (no attention, no recurrence, no layout): every
array is keyed by (request, node) so that each side places tokens itself --
the oracle along isolated root-to-node paths, the GPU path into its flat
stream.

Tree model (Flide, "Accelerating Decision Inference with Exact State
Forking", section 3.1 and Figure 2(a); ForkServe README, "Copy-on-write
context tree"): a request is a tree whose node 0 is the shared state (trunk)
and whose other nodes are question branches or deeper residuals.  A resumed
root carries ``hist_len`` tokens of history that earlier passes computed.

Workload recipes (shapes and value laws) follow the benchmark configurations:

* ``tiny``   -- 1 request, trunk 64 + 3 branches of 8; attention 2 heads,
  d=64; GDN 2 heads, d=64; q,k,v ~ N(0,1)/8, GDN k L2-normalised,
  alpha ~ U(0.90, 0.999), beta ~ U(0.1, 0.9); fp32.
* ``attn``   -- trunk 4096 + 8 branches of U[16,64] tokens, GQA 32/8, d=128,
  q,k,v ~ N(0,1) rounded to bf16, 4 option rows ~ N(0,1) fp32 over the
  concatenated head outputs.
* ``gdn``    -- trunk 8192 + 16 branches of U[8,128] tokens, 16 heads,
  d=128; q,v ~ N(0,1)/8, k ~ N(0,1) then L2-normalised (all rounded to bf16);
  alpha = exp(-0.1 softplus(N(0,1))), beta = sigmoid(N(0,1)) in fp32; the
  trunk is drawn 1024 tokens longer so that a resumed round can append them.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import numpy as np

PAGE = 16


# --------------------------------------------------------------------------
# tree shapes
# --------------------------------------------------------------------------
@dataclass
class Request:
    """One request: ``parents[i]`` is node i's parent (-1 for node 0)."""

    parents: List[int]
    n_tok: List[int]
    readout: Optional[List[bool]] = None   # default: leaves
    hist_len: int = 0                      # resumed root: tokens already computed
    save: Optional[Dict[int, int]] = None  # node -> persistent state slot to save

    def __post_init__(self):
        assert len(self.parents) == len(self.n_tok)
        assert self.parents[0] == -1
        if self.readout is None:
            has_child = [False] * len(self.parents)
            for p in self.parents[1:]:
                has_child[p] = True
            self.readout = [not c for c in has_child]
        if self.save is None:
            self.save = {}

    @property
    def n_nodes(self) -> int:
        return len(self.parents)


@dataclass
class Tree:
    requests: List[Request] = field(default_factory=list)

    def useful_tokens(self) -> int:
        """P + sum |q_i| per request: every stream token counted once."""
        return int(sum(sum(r.n_tok) for r in self.requests))


def fork_tree(trunk: int, branches: List[int], hist_len: int = 0) -> Request:
    return Request(parents=[-1] + [0] * len(branches), n_tok=[trunk] + list(branches),
                   hist_len=hist_len)


def fanout_tree(trunk: int, residual: int, fanout: int, depth: int) -> Request:
    """Trunk plus ``depth`` levels of ``fanout`` residuals per node (BFS order)."""
    parents, n_tok = [-1], [trunk]
    frontier = [0]
    for _ in range(depth):
        nxt = []
        for p in frontier:
            for _c in range(fanout):
                parents.append(p)
                n_tok.append(residual)
                nxt.append(len(parents) - 1)
        frontier = nxt
    return Request(parents=parents, n_tok=n_tok)


# --------------------------------------------------------------------------
# value helpers (input preparation only)
# --------------------------------------------------------------------------
def to_bf16_values(x: np.ndarray) -> np.ndarray:
    """float32 array whose values are the round-to-nearest-even bf16 of x."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _l2n(x: np.ndarray) -> np.ndarray:
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _softplus(x):
    return np.log1p(np.exp(-np.abs(x))) + np.maximum(x, 0.0)


# --------------------------------------------------------------------------
# per-node layer inputs
# --------------------------------------------------------------------------
NodeArrays = Dict[Tuple[int, int], Dict[str, np.ndarray]]


@dataclass
class AttnInputs:
    hq: int
    hkv: int
    d: int
    bf16: bool
    nodes: NodeArrays                    # (r, node) -> {"q","k","v"}
    hist: Dict[int, Dict[str, np.ndarray]]  # r -> {"k","v"} history before the root


@dataclass
class GdnInputs:
    h: int
    dk: int
    dv: int
    bf16: bool
    nodes: NodeArrays                    # (r, node) -> {"q","k","v","alpha","beta"}
    hist: Dict[int, Dict[str, np.ndarray]]  # r -> history inputs (oracle recompute)


def _split_nodes(req: Request, arr: np.ndarray, start: int = 0) -> List[np.ndarray]:
    out, off = [], start
    for n in req.n_tok:
        out.append(arr[off:off + n])
        off += n
    return out


def attn_inputs(tree: Tree, hq: int, hkv: int, d: int, seed: int, bf16: bool,
                sigma: float = 1.0) -> AttnInputs:
    nodes, hist = {}, {}
    for r, req in enumerate(tree.requests):
        rng = np.random.default_rng(seed + r)
        n = req.hist_len + sum(req.n_tok)
        q = rng.standard_normal((n, hq, d), dtype=np.float32) * sigma
        k = rng.standard_normal((n, hkv, d), dtype=np.float32) * sigma
        v = rng.standard_normal((n, hkv, d), dtype=np.float32) * sigma
        if bf16:
            q, k, v = to_bf16_values(q), to_bf16_values(k), to_bf16_values(v)
        h = req.hist_len
        hist[r] = {"k": k[:h], "v": v[:h], "q": q[:h]}
        for i, (qq, kk, vv) in enumerate(zip(_split_nodes(req, q, h), _split_nodes(req, k, h),
                                             _split_nodes(req, v, h))):
            nodes[(r, i)] = {"q": qq, "k": kk, "v": vv}
    return AttnInputs(hq, hkv, d, bf16, nodes, hist)


def gdn_inputs(tree: Tree, h: int, dk: int, dv: int, seed: int, bf16: bool,
               law: str = "uniform") -> GdnInputs:
    """``law='uniform'``: alpha~U(.90,.999), beta~U(.1,.9) (tiny workload);
    ``law='softplus'``: alpha=exp(-0.1 softplus(N)), beta=sigmoid(N)."""
    nodes, hist = {}, {}
    for r, req in enumerate(tree.requests):
        rng = np.random.default_rng(seed + r)
        n = req.hist_len + sum(req.n_tok)
        q = rng.standard_normal((n, h, dk), dtype=np.float32) / 8
        k = _l2n(rng.standard_normal((n, h, dk), dtype=np.float32).astype(np.float64)).astype(np.float32)
        v = rng.standard_normal((n, h, dv), dtype=np.float32) / 8
        if law == "uniform":
            alpha = rng.uniform(0.90, 0.999, (n, h)).astype(np.float32)
            beta = rng.uniform(0.1, 0.9, (n, h)).astype(np.float32)
        else:
            a = rng.standard_normal((n, h))
            b = rng.standard_normal((n, h))
            alpha = np.exp(-0.1 * _softplus(a)).astype(np.float32)
            beta = (1.0 / (1.0 + np.exp(-b))).astype(np.float32)
        if bf16:
            q, k, v = to_bf16_values(q), to_bf16_values(k), to_bf16_values(v)
        hl = req.hist_len
        hist[r] = {"q": q[:hl], "k": k[:hl], "v": v[:hl], "alpha": alpha[:hl], "beta": beta[:hl]}
        parts = [_split_nodes(req, a, hl) for a in (q, k, v, alpha, beta)]
        for i in range(req.n_nodes):
            nodes[(r, i)] = {"q": parts[0][i], "k": parts[1][i], "v": parts[2][i],
                             "alpha": parts[3][i], "beta": parts[4][i]}
    return GdnInputs(h, dk, dv, bf16, nodes, hist)


def option_rows(n_opt: int, hidden: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.standard_normal((n_opt, hidden), dtype=np.float32)


# --------------------------------------------------------------------------
# the named workloads
# --------------------------------------------------------------------------
def tiny_tree() -> Tree:
    return Tree([fork_tree(64, [8, 8, 8])])


def attn_tree(seed: int = 2000, trunk: int = 4096, k: int = 8, lo: int = 16, hi: int = 64) -> Tree:
    rng = np.random.default_rng(seed)
    br = [int(x) for x in rng.integers(lo, hi + 1, size=k)]
    return Tree([fork_tree(trunk, br)])


def gdn_tree(seed: int = 3000, trunk: int = 8192, k: int = 16, lo: int = 8, hi: int = 128) -> Tree:
    rng = np.random.default_rng(seed)
    br = [int(x) for x in rng.integers(lo, hi + 1, size=k)]
    return Tree([fork_tree(trunk, br)])


def gdn_checkpoint_trees(m: int, seed: int = 3000, trunk: int = 8192, extra: int = 1024,
                         k: int = 16, ckpt_slot: int = 0):
    """The two rounds of a resumed agent step.

    Round A: the trunk split at ``m`` into a head (saving its end state into
    ``ckpt_slot``) and a tail, then the branches.  Round B: a root resumed at
    position ``m`` whose stream holds trunk tokens [m, trunk+extra), then the
    same branches.  Returns (tree_a, tree_b, full_tree) where ``full_tree`` is
    the unsplit trunk of length trunk+extra that the inputs are drawn from.
    """
    base = gdn_tree(seed, trunk, k)
    br = base.requests[0].n_tok[1:]
    full = Tree([fork_tree(trunk + extra, br)])
    if m < trunk:
        a = Request(parents=[-1, 0] + [1] * k, n_tok=[m, trunk - m] + br, save={0: ckpt_slot})
    else:
        a = Request(parents=[-1] + [0] * k, n_tok=[trunk] + br, save={0: ckpt_slot})
    b = Request(parents=[-1] + [0] * k, n_tok=[trunk + extra - m] + br, hist_len=m)
    return Tree([a]), Tree([b]), full


def remap_inputs(src_tree: Tree, src: "GdnInputs | AttnInputs", dst_tree: Tree):
    """Re-key inputs drawn for ``src_tree`` onto ``dst_tree`` (same token
    sequence along each root-to-leaf path, different node boundaries).

    Both trees must describe the same tokens: the source's root sequence
    (history + root) must cover the destination's history + root chain, and
    branches map to branches in order.  Used to express a checkpointed or
    resumed round over one drawn token sequence.
    """
    out_nodes, out_hist = {}, {}
    for r, (sreq, dreq) in enumerate(zip(src_tree.requests, dst_tree.requests)):
        root = {key: np.concatenate([src.hist[r][key], src.nodes[(r, 0)][key]])
                for key in src.nodes[(r, 0)]}
        # destination trunk chain: nodes whose every child has further children
        # or which are on the path to the branches (chain nodes before the fork)
        chain = [0]
        while True:
            kids = [i for i, p in enumerate(dreq.parents) if p == chain[-1]]
            if len(kids) == 1 and any(p == kids[0] for p in dreq.parents):
                chain.append(kids[0])
            else:
                break
        off = dreq.hist_len
        out_hist[r] = {key: a[:off] for key, a in root.items()}
        for node in chain:
            n = dreq.n_tok[node]
            out_nodes[(r, node)] = {key: a[off:off + n] for key, a in root.items()}
            off += n
        branches_d = [i for i in range(dreq.n_nodes) if i not in chain]
        branches_s = list(range(1, sreq.n_nodes))
        assert len(branches_d) == len(branches_s)
        for bd, bs in zip(branches_d, branches_s):
            out_nodes[(r, bd)] = src.nodes[(r, bs)]
    kw = {k: v for k, v in src.__dict__.items() if k not in ("nodes", "hist")}
    return type(src)(nodes=out_nodes, hist=out_hist, **kw)


# --------------------------------------------------------------------------
# hybrid stack workloads (random-init weights, token ids)
# --------------------------------------------------------------------------
def _bf16n(rng, shape, std=0.02):
    return to_bf16_values(rng.standard_normal(shape, dtype=np.float32) * std)


def stack_weights(hidden: int, pattern: str, hq: int, hkv: int, d: int, gh: int, gd: int, ffn: int, vocab: int,
                  taps: int = 4, seed: int = 4100, pad: int = 128) -> Dict[str, np.ndarray]:
    """All weights N(0, 0.02), rounded to bf16; [out, in] layout.  The fused
    GDN projection (q | k | v | a | b) is padded with zero rows to a multiple
    of ``pad``."""
    rng = np.random.default_rng(seed)
    W = {"embed": _bf16n(rng, (vocab, hidden))}
    for li, kind in enumerate(pattern):
        p = f"l{li}."
        if kind == "A":
            W[p + "wq"] = _bf16n(rng, (hq * d, hidden))
            W[p + "wk"] = _bf16n(rng, (hkv * d, hidden))
            W[p + "wv"] = _bf16n(rng, (hkv * d, hidden))
            W[p + "wo"] = _bf16n(rng, (hidden, hq * d))
        else:
            n = 3 * gh * gd + 2 * gh
            npad = -(-n // pad) * pad
            wp = np.zeros((npad, hidden), np.float32)
            wp[:n] = _bf16n(rng, (n, hidden))
            W[p + "wp"] = wp
            W[p + "conv"] = _bf16n(rng, (3 * gh * gd, taps))
            W[p + "wo"] = _bf16n(rng, (hidden, gh * gd))
        W[p + "wgu"] = _bf16n(rng, (2 * ffn, hidden))
        W[p + "wd"] = _bf16n(rng, (hidden, ffn))
    return W


def token_ids(tree: Tree, vocab: int, seed: int):
    """Uniform token ids per (request, node) and for each request's history."""
    nodes, hist = {}, {}
    for r, req in enumerate(tree.requests):
        rng = np.random.default_rng(seed + r)
        n = req.hist_len + sum(req.n_tok)
        ids = rng.integers(0, vocab, size=n).astype(np.int32)
        hist[r] = ids[:req.hist_len]
        for i, part in enumerate(_split_nodes(req, ids, req.hist_len)):
            nodes[(r, i)] = part
    return nodes, hist


def mixed_tree(seed: int = 4000, n_req: int = 64, lo: int = 512, hi: int = 16384, bmin: int = 2, bmax: int = 12,
               lmin: int = 8, lmax: int = 128) -> Tree:
    """Requests with log-uniform trunks in [lo, hi], bmin..bmax branches of U[lmin, lmax] tokens."""
    rng = np.random.default_rng(seed)
    reqs = []
    for _ in range(n_req):
        P = int(round(np.exp(rng.uniform(np.log(lo), np.log(hi)))))
        k = int(rng.integers(bmin, bmax + 1))
        reqs.append(fork_tree(P, [int(x) for x in rng.integers(lmin, lmax + 1, size=k)]))
    return Tree(reqs)


def agent_tree(n_sessions: int = 10, trunk: int = 256, residual: int = 32, fanout: int = 4, depth: int = 3,
               spine_slot: int = 0) -> Tree:
    """Sessions of a trunk plus ``depth`` levels of ``fanout`` residuals; the
    committed spine follows child 0 at every level, and its leaf saves its
    end state into ``spine_slot + session``."""
    reqs = []
    for s in range(n_sessions):
        r = fanout_tree(trunk, residual, fanout, depth)
        leaf = spine_leaf(r)
        r.save = {leaf: spine_slot + s}
        reqs.append(r)
    return Tree(reqs)


def spine_path(req: Request) -> List[int]:
    """Root-to-leaf path through child 0 at every level (the committed spine)."""
    path = [0]
    while True:
        kids = [i for i, p in enumerate(req.parents) if p == path[-1]]
        if not kids:
            return path
        path.append(kids[0])


def spine_leaf(req: Request) -> int:
    return spine_path(req)[-1]
