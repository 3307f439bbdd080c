"""Flat CUDA graphs over a capacity bucket (Flide section 3.3.2): the step's
device work captured once replays to the same bits as eager launches, and
keeps doing so for a different round of the same capacities uploaded into
the same buffers (the launches depend on the capacities only)."""
import math

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from hybrid_serving_gb300 import api, rounds  # noqa: E402
from hybrid_serving_gb300.graphs import StepGraph  # noqa: E402

HQ, HKV, D, H = 8, 2, 128, 4


class Bucket:
    """Capacity-sized buffers for an attention round and a GDN round."""

    def __init__(self, a_caps, g_caps, n_pages):
        self.a_caps, self.g_caps = a_caps, g_caps
        Ta, Tg = a_caps.max_tokens, g_caps.max_tokens
        bf, dev = torch.bfloat16, "cuda"
        self.a_meta = torch.empty(api.Round(a_caps).meta_bytes() // 4, dtype=torch.int32, device=dev)
        self.g_meta = torch.empty(api.Round(g_caps).meta_bytes() // 4, dtype=torch.int32, device=dev)
        self.q = torch.zeros((Ta, HQ, D), dtype=bf, device=dev)
        self.k = torch.zeros((Ta, HKV, D), dtype=bf, device=dev)
        self.v = torch.zeros_like(self.k)
        self.kp = torch.zeros((HKV, n_pages, 16, D), dtype=bf, device=dev)
        self.vp = torch.zeros_like(self.kp)
        self.out = torch.zeros_like(self.q)
        self.W = torch.from_numpy(synth.option_rows(4, HQ * D, seed=61)).to(dev)
        self.lp = torch.zeros((a_caps.max_readouts, 4), dtype=torch.float32, device=dev)
        self.gq = torch.zeros((Tg, H, D), dtype=bf, device=dev)
        self.gk, self.gv = torch.zeros_like(self.gq), torch.zeros_like(self.gq)
        self.ga = torch.ones((Tg, H), dtype=torch.float32, device=dev)
        self.gb = torch.zeros((Tg, H), dtype=torch.float32, device=dev)
        self.state = torch.zeros((16, H, D, D), dtype=torch.float32, device=dev)
        self.gout = torch.zeros_like(self.gq)
        self.ws = torch.empty(api.gdn_workspace_bytes(g_caps, H, D, D), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def load(self, a_tree, g_tree, seed):
        """Build both rounds (host), upload their metadata and inputs into the bucket's buffers."""
        pool = api.PagePool(self.kp.shape[1])
        Ra, sa = rounds.build_round(a_tree, pool, caps=self.a_caps)
        Rg, sg = rounds.build_round(g_tree, None, caps=self.g_caps, temp_slot0=2, n_temp_slots=14)
        Ra.upload(self.a_meta)
        Rg.upload(self.g_meta)
        ai = synth.attn_inputs(a_tree, HQ, HKV, D, seed=seed, bf16=True)
        gi = synth.gdn_inputs(g_tree, H, D, D, seed=seed + 1, bf16=True, law="softplus")
        for t, key in ((self.q, "q"), (self.k, "k"), (self.v, "v")):
            x = torch.from_numpy(rounds.to_stream(Ra, sa, ai.nodes, key))
            t[:x.shape[0]].copy_(x.to(t.dtype))
        for t, key in ((self.gq, "q"), (self.gk, "k"), (self.gv, "v"), (self.ga, "alpha"), (self.gb, "beta")):
            x = torch.from_numpy(rounds.to_stream(Rg, sg, gi.nodes, key))
            t[:x.shape[0]].copy_(x.to(t.dtype))
        torch.cuda.synchronize()
        return (Ra, sa, pool), (Rg, sg)

    def step(self):
        api.kv_page_write(self.a_caps, self.a_meta, self.k, self.v, self.kp, self.vp, self.status)
        api.fork_attn(self.a_caps, self.a_meta, self.q, self.kp, self.vp, self.out, self.status,
                      scale=1 / math.sqrt(D))
        api.choice_logprobs(self.a_caps, self.a_meta, self.out.view(self.out.shape[0], -1), self.W, self.lp,
                            self.status)
        api.gdn_fork_prefill(self.g_caps, self.g_meta, self.gq, self.gk, self.gv, self.ga, self.gb, self.state,
                             self.gout, self.ws, self.status)

    def results(self, n_a, n_g, n_ro):
        return self.out[:n_a].clone(), self.lp[:n_ro].clone(), self.gout[:n_g].clone()


def _same(a, b):
    return all(torch.equal(x, y) for x, y in zip(a, b))


def test_graph_replay_matches_eager_across_rounds():
    rounds_in = [
        (synth.Tree([synth.fork_tree(700, [20, 45, 3])]), synth.Tree([synth.fork_tree(1600, [30, 70, 5])]), 71),
        (synth.Tree([synth.fork_tree(300, [9, 60]), synth.fork_tree(200, [11])]),
         synth.Tree([synth.fork_tree(1200, [128, 2]), synth.fork_tree(90, [40])]), 72),
    ]
    Ta = max(t.useful_tokens() for t, _, _ in rounds_in)
    Tg = max(t.useful_tokens() for _, t, _ in rounds_in)
    a_caps = api.round_caps_for(Ta, 8, 2)
    g_caps = api.round_caps_for(Tg, 8, 2)
    b = Bucket(a_caps, g_caps, n_pages=Ta // 16 + 32)
    graph = None
    for a_tree, g_tree, seed in rounds_in:
        (Ra, _, pool), (Rg, _) = b.load(a_tree, g_tree, seed)
        n = (Ra.info().n_tokens, Rg.info().n_tokens, Ra.info().n_readouts)
        b.step()                                   # eager
        torch.cuda.synchronize()
        api.check_status(b.status)
        eager = b.results(*n)
        if graph is None:
            graph = StepGraph(b.step)              # captured on the first round's buffers
        for _ in range(2):                         # replays, twice in a row
            graph.replay()
            torch.cuda.synchronize()
            api.check_status(b.status)
            assert _same(b.results(*n), eager)
        Ra.release(pool)
    # the first round again, after the second: still its own bits
    a_tree, g_tree, seed = rounds_in[0]
    (Ra, _, pool), (Rg, _) = b.load(a_tree, g_tree, seed)
    n = (Ra.info().n_tokens, Rg.info().n_tokens, Ra.info().n_readouts)
    b.step()
    torch.cuda.synchronize()
    eager = b.results(*n)
    graph.replay()
    torch.cuda.synchronize()
    assert _same(b.results(*n), eager)


def _subset(inp, group, reqs):
    """The inputs of the requests in ``group``, renumbered 0, 1, ..."""
    import dataclasses
    nodes = {(j, i): inp.nodes[(r, i)] for j, r in enumerate(group) for i in range(reqs[r].n_nodes)}
    hist = {j: inp.hist[r] for j, r in enumerate(group) if r in inp.hist}
    return dataclasses.replace(inp, nodes=nodes, hist=hist)


def test_rounds_split_at_request_boundaries_bitwise():
    """A batch split into rounds of one capacity bucket at request boundaries gives every request the
    same output bits as the batch in one round (attention and GDN): rounds cut between requests change
    nothing a request computes (Flide sections 3.3.2 and 3.5)."""
    from harness import AttnRun, GdnRun
    reqs = [synth.fork_tree(n, br) for n, br in [(300, [20, 7]), (90, [40]), (700, [9, 9, 60]), (150, [3]),
                                                  (1100, [17, 80]), (64, [64])]]
    tree = synth.Tree(reqs)
    ainp = synth.attn_inputs(tree, HQ, HKV, D, seed=71, bf16=True)
    ginp = synth.gdn_inputs(tree, H, D, D, seed=72, bf16=True, law="softplus")
    a_all = AttnRun(tree, ainp, torch.bfloat16).run()
    g_all = GdnRun(tree, ginp, torch.bfloat16).run()
    api.check_status(a_all.status)
    api.check_status(g_all.status)
    ra, rg = a_all.raw_outputs(), g_all.raw_outputs()
    bucket = api.round_caps_for(1300, 8, 2)
    groups = rounds.split_at_requests(tree, bucket)
    assert len(groups) >= 3
    for g in groups:
        sub = synth.Tree([reqs[r] for r in g])
        a = AttnRun(sub, _subset(ainp, g, reqs), torch.bfloat16).run()
        gg = GdnRun(sub, _subset(ginp, g, reqs), torch.bfloat16).run()
        api.check_status(a.status)
        api.check_status(gg.status)
        sa, sg = a.raw_outputs(), gg.raw_outputs()
        for j, r in enumerate(g):
            for i in range(reqs[r].n_nodes):
                assert torch.equal(sa[(j, i)], ra[(r, i)]), ("attention", r, i)
                assert torch.equal(sg[(j, i)], rg[(r, i)]), ("gdn", r, i)
