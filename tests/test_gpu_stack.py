"""Hybrid attention / Gated DeltaNet stack over forked rounds vs the fp64
stack oracle (every branch an isolated pass through all layers).

The stack architecture is not defined by the pages; its parity is pinned by
the oracle's own definition and its component tests.  The model keeps its
residual stream and final norm in fp32 (bf16 between the other operations).
Bars (Flide's Appendix G forward test): the final hidden rows within twice
the distance between the oracle's fp32-projection forward and its fp64
forward (the rounding level of the stack), the option distributions within
TV 1e-3 plus twice that forward's TV, the plain 2e-2 / 1e-3 margins printed
beside them; bit-identical results for a request alone and in a mixed
round; a resumed spine against the full recompute.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import choice as ochoice
from oracle import layout
from oracle import stack as ostack

pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from hybrid_serving_gb300 import api, rounds  # noqa: E402
from hybrid_serving_gb300.stack import HybridStack, StackShape  # noqa: E402

TOL, TV = 2e-2, 1e-3
SMALL = dict(hidden=256, pattern="GGGAGGGA", attn_hq=2, attn_hkv=1, head_d=128, gdn_h=2, gdn_d=128, ffn=512,
             vocab=512)


def _cfgs(dims):
    sh = StackShape(**dims)
    oc = ostack.StackConfig(**dims)
    W = synth.stack_weights(dims["hidden"], dims["pattern"], dims["attn_hq"], dims["attn_hkv"], dims["head_d"],
                            dims["gdn_h"], dims["gdn_d"], dims["ffn"], dims["vocab"], seed=4100)
    return sh, oc, W


def _run(stk, tree, ids_nodes, resume=None, pool=None, n_slots=64, save_windows=None, temp0=32):
    R, seg_of = rounds.build_round(tree, pool, temp_slot0=temp0, n_temp_slots=n_slots - temp0, resume=resume)
    meta = torch.empty(R.meta_bytes() // 4, dtype=torch.int32, device="cuda")
    R.upload(meta)
    ids = torch.zeros(stk.Tcap, dtype=torch.int32, device="cuda")
    T = R.info().n_tokens
    ids[:T] = torch.from_numpy(rounds.to_stream(R, seg_of, ids_nodes)).cuda()
    hid, lp = stk.forward(R, meta, ids, R.info().n_readouts, save_windows=save_windows)
    torch.cuda.synchronize()
    api.check_status(stk.status)
    return R, seg_of, hid.float().cpu().numpy(), lp.cpu().numpy()


def _oracle_node(oc, W, tree, ids_nodes, hist, r, node, both=False):
    req = tree.requests[r]
    seq = np.concatenate([hist[r]] + [ids_nodes[(r, a)] for a in layout.ancestors(req, node)])
    ref = ostack.forward(oc, W, seq)[-req.n_tok[node]:]
    if not both:
        return ref
    return ref, ostack.forward(oc, W, seq, gemm_dtype=np.float32)[-req.n_tok[node]:]


def _assert_tv(lp_gpu, oc, W, h64, h32, what):
    """Option distributions within 1e-3 plus twice the fp32 forward's TV over
    the same rows (Flide App. G's rounding-level bar; the plain 1e-3 bar is
    printed beside it)."""
    p64 = np.exp(ostack.option_logprobs(oc, W, h64))
    p32 = np.exp(ostack.option_logprobs(oc, W, h32))
    tv_ref = float(ochoice.total_variation(p32, p64).max())
    tv = float(ochoice.total_variation(np.exp(lp_gpu), p64).max())
    print(f"[margin] stack {what}: option TV {tv:.3e}, fp32-forward TV {tv_ref:.3e} (bar 1e-3)")
    assert tv <= TV + 2 * tv_ref, (what, tv, tv_ref)


def _assert_rounding_level(got, ref, ref32, what):
    """GPU error within twice the fp32-vs-fp64 oracle distance plus 2e-3
    (Flide App. G: the GPU's and the fp32 forward's departures from fp64 are
    the same kind of perturbation, amplified alike by the stack's rounding
    points; the plain 2e-2 bar is printed beside it)."""
    e_ref = float(np.abs(ref32 - ref).max())
    e_gpu = float(np.abs(got - ref).max())
    print(f"[margin] stack {what}: max-abs {e_gpu:.3e}, fp32-forward distance {e_ref:.3e} (bar 2e-2)")
    assert e_gpu <= 2 * e_ref + 2e-3, (what, e_gpu, e_ref)
    assert e_ref <= 0.25, (what, e_ref)


def test_small_stack_fork_parity_and_choices():
    sh, oc, W = _cfgs(SMALL)
    tree = synth.Tree([synth.fork_tree(150, [17, 1, 40]), synth.fork_tree(70, [9, 33])])
    ids, hist = synth.token_ids(tree, SMALL["vocab"], seed=4200)
    stk = HybridStack(sh, W, max_pos=1024)
    stk.alloc(Tcap=sum(sum(r.n_tok) for r in tree.requests), n_pages=64, n_slots=64)
    R, seg_of, hid, lp = _run(stk, tree, ids, pool=api.PagePool(64))
    got = rounds.from_stream(R, seg_of, hid)
    for r, req in enumerate(tree.requests):
        for i in range(req.n_nodes):
            ref, ref32 = _oracle_node(oc, W, tree, ids, hist, r, i, both=True)
            _assert_rounding_level(got[(r, i)], ref, ref32, (r, i))
    ro = [(r, i) for r, req in enumerate(tree.requests) for i in range(req.n_nodes) if req.readout[i]]
    both = [_oracle_node(oc, W, tree, ids, hist, r, i, both=True) for r, i in ro]
    _assert_tv(lp, oc, W, np.stack([b[0][-1] for b in both]), np.stack([b[1][-1] for b in both]), "fork")


def test_small_stack_batch_invariance_bitwise():
    sh, oc, W = _cfgs(SMALL)
    base = synth.fork_tree(130, [20, 50, 13])
    tree = synth.Tree([synth.fork_tree(90, [30, 7]), base])
    ids, hist = synth.token_ids(tree, SMALL["vocab"], seed=4300)
    stk = HybridStack(sh, W, max_pos=1024)
    stk.alloc(Tcap=sum(sum(r.n_tok) for r in tree.requests), n_pages=64, n_slots=64)
    R, seg_of, hid, _ = _run(stk, tree, ids, pool=api.PagePool(64))
    mixed = rounds.from_stream(R, seg_of, hid)
    for b in range(1, 4):
        t1 = synth.Tree([synth.fork_tree(130, [base.n_tok[b]])])
        ids1 = {(0, 0): ids[(1, 0)], (0, 1): ids[(1, b)]}
        R1, s1, h1, _ = _run(stk, t1, ids1, pool=api.PagePool(64))
        alone = rounds.from_stream(R1, s1, h1)
        assert np.array_equal(alone[(0, 1)], mixed[(1, b)])
        assert np.array_equal(alone[(0, 0)], mixed[(1, 0)])


def test_selective_readout_bitwise():
    """Selective readout (Flide section 3.3.3): the last layer's MLP, the final norm and the option head
    on the readout rows alone give the same bits at those rows, and the same option log-probs, as the
    full forward."""
    sh, oc, W = _cfgs(SMALL)
    tree = synth.Tree([synth.fork_tree(150, [17, 1, 40]), synth.fork_tree(70, [9, 33]),
                       synth.fanout_tree(30, 6, 3, 2)])
    ids, _ = synth.token_ids(tree, SMALL["vocab"], seed=4250)
    stk = HybridStack(sh, W, max_pos=1024)
    stk.alloc(Tcap=tree.useful_tokens(), n_pages=96, n_slots=64)
    R, seg_of = rounds.build_round(tree, api.PagePool(96), temp_slot0=32, n_temp_slots=32)
    meta = torch.empty(R.meta_bytes() // 4, dtype=torch.int32, device="cuda")
    R.upload(meta)
    idd = torch.from_numpy(rounds.to_stream(R, seg_of, ids)).cuda()
    n_ro = R.info().n_readouts
    h_full, lp_full = stk.forward(R, meta, idd, n_ro)
    h_full, lp_full = h_full.clone(), lp_full.clone()
    h_sel, lp_sel = stk.forward(R, meta, idd, n_ro, selective=True)
    torch.cuda.synchronize()
    api.check_status(stk.status)
    rows = torch.tensor(R.readout_rows(), dtype=torch.long, device="cuda")
    assert n_ro == len(rows) > 0
    assert torch.equal(h_sel[rows], h_full[rows])
    assert torch.equal(lp_sel, lp_full)


def _agent_round_trip(dims, n_sessions, trunk, residual, depth, extra, check_leaves, seed):
    """Round A: depth-level fan-out of 4 per session, spine leaf saves its GDN
    state and conv window; commit keeps the spine pages.  Round B: each
    spine resumed with `extra` new tokens.  Both against the oracle."""
    sh, oc, W = _cfgs(dims)
    tree = synth.agent_tree(n_sessions, trunk, residual, 4, depth, spine_slot=0)
    ids, hist = synth.token_ids(tree, dims["vocab"], seed=seed)
    T = tree.useful_tokens()
    n_pages = layout.live_pages(tree, 16) + n_sessions * (-(-extra // 16)) + 16
    n_slots = 32 + sum(r.n_nodes for r in tree.requests) + 8
    stk = HybridStack(sh, W, max_pos=4096)
    stk.alloc(Tcap=max(T, n_sessions * extra), n_pages=n_pages, n_slots=n_slots, n_windows=3 * n_sessions)
    pool = api.PagePool(n_pages)
    # conv windows: the spine leaf's last 3 stream rows -> window rows 3s..3s+2
    R0, seg0 = rounds.build_round(tree, pool, temp_slot0=32, n_temp_slots=n_slots - 32)
    src, dst = [], []
    for s, req in enumerate(tree.requests):
        leaf = synth.spine_leaf(req)
        info = R0.segment(seg0[(s, leaf)])
        src += [info.stream_off + info.n_tokens - 3 + j for j in range(3)]
        dst += [3 * s + j for j in range(3)]
    del R0
    pool = api.PagePool(n_pages)
    sw = [(torch.tensor(src, dtype=torch.int32, device="cuda"), torch.tensor(dst, dtype=torch.int32, device="cuda"),
           len(src))]
    RA, segA, hidA, lpA = _run(stk, tree, ids, pool=pool, n_slots=n_slots, save_windows=sw)
    gotA = rounds.from_stream(RA, segA, hidA)
    for (s, leaf) in check_leaves:
        ref, ref32 = _oracle_node(oc, W, tree, ids, hist, s, leaf, both=True)
        _assert_rounding_level(gotA[(s, leaf)], ref, ref32, ("A", s, leaf))
    # commit: keep each session's spine
    keep, spans = [], {}
    for s, req in enumerate(tree.requests):
        path = synth.spine_path(req)
        keep += [segA[(s, n)] for n in path]
        spans[s] = [(req.n_tok[n], RA.segment_pages(segA[(s, n)])) for n in path]
    RA.release(pool, keep=keep)
    # round B: resume each spine with `extra` new tokens and one readout at the end
    spine_len = trunk + depth * residual
    treeB = synth.Tree([synth.Request(parents=[-1], n_tok=[extra], hist_len=spine_len) for _ in range(n_sessions)])
    idsB = {}
    rng = np.random.default_rng(seed + 99)
    for s in range(n_sessions):
        idsB[(s, 0)] = rng.integers(0, dims["vocab"], size=extra).astype(np.int32)
    resume = {s: (s, spans[s], 3 * s) for s in range(n_sessions)}
    RB, segB, hidB, lpB = _run(stk, treeB, idsB, pool=pool, n_slots=n_slots, resume=resume)
    gotB = rounds.from_stream(RB, segB, hidB)
    last64, last32 = [], []
    n_chk = min(n_sessions, 2)
    for s in range(n_chk):
        req = tree.requests[s]
        seq = np.concatenate([ids[(s, n)] for n in synth.spine_path(req)] + [idsB[(s, 0)]])
        ref = ostack.forward(oc, W, seq)[-extra:]
        ref32 = ostack.forward(oc, W, seq, gemm_dtype=np.float32)[-extra:]
        _assert_rounding_level(gotB[(s, 0)], ref, ref32, ("B", s))
        last64.append(ref[-1])
        last32.append(ref32[-1])
    _assert_tv(lpB[:n_chk], oc, W, np.stack(last64), np.stack(last32), "B")


def test_small_agent_tree_commit_and_resume():
    _agent_round_trip(SMALL, n_sessions=3, trunk=64, residual=8, depth=3, extra=48,
                      check_leaves=[(0, 21), (1, 40), (2, 84)], seed=4400)


FULL = dict(hidden=2048, pattern="GGGAGGGA", attn_hq=16, attn_hkv=4, head_d=128, gdn_h=16, gdn_d=128, ffn=4096,
            vocab=32768)


def test_agent_tree_full_width_commit_and_resume():
    """The deep agent tree at full width: 10 sessions, trunk 256, three
    levels of fan-out 4 of 32-token residuals (multi-level page aliasing),
    then every committed spine extended by 512 resumed tokens."""
    _agent_round_trip(FULL, n_sessions=10, trunk=256, residual=32, depth=3, extra=512,
                      check_leaves=[(0, 21), (7, 84)], seed=5000)


def test_mixed_batch_full_width_invariance_and_sampled_parity():
    """64 requests, trunks log-uniform in [512, 16384], 2-12 branches of
    U[8,128], 8 layers at width 2048.  Every sampled request re-run alone
    gives bit-identical rows; the shortest request's trunk and two branches
    match the oracle at the rounding level."""
    sh, oc, W = _cfgs(FULL)
    tree = synth.mixed_tree(seed=4000)
    ids, hist = synth.token_ids(tree, FULL["vocab"], seed=4500)
    T = tree.useful_tokens()
    n_pages = layout.live_pages(tree, 16) + 64
    n_seg = sum(r.n_nodes for r in tree.requests)
    stk = HybridStack(sh, W, max_pos=20000)
    stk.alloc(Tcap=T, n_pages=n_pages, n_slots=n_seg + 8)
    R, seg_of = rounds.build_round(tree, api.PagePool(n_pages), temp_slot0=0, n_temp_slots=n_seg + 8)
    meta = torch.empty(R.meta_bytes() // 4, dtype=torch.int32, device="cuda")
    R.upload(meta)
    idd = torch.from_numpy(rounds.to_stream(R, seg_of, ids)).cuda()
    hid, lp = stk.forward(R, meta, idd, R.info().n_readouts)
    torch.cuda.synchronize()
    api.check_status(stk.status)
    mixed = hid.clone()
    rows = {k: (R.segment(s).stream_off, R.segment(s).n_tokens) for k, s in seg_of.items()}
    lens = [sum(r.n_tok) for r in tree.requests]
    order = sorted(range(len(lens)), key=lambda r: lens[r])
    sample = sorted(set(order[:4] + order[-2:] + [7, 31]))
    for r in sample:
        req = tree.requests[r]
        t1 = synth.Tree([synth.Request(parents=req.parents, n_tok=req.n_tok)])
        ids1 = {(0, i): ids[(r, i)] for i in range(req.n_nodes)}
        R1, s1 = rounds.build_round(t1, api.PagePool(n_pages), temp_slot0=0, n_temp_slots=8)
        m1 = torch.empty(R1.meta_bytes() // 4, dtype=torch.int32, device="cuda")
        R1.upload(m1)
        i1 = torch.zeros(T, dtype=torch.int32, device="cuda")
        i1[:R1.info().n_tokens] = torch.from_numpy(rounds.to_stream(R1, s1, ids1)).cuda()
        h1, _ = stk.forward(R1, m1, i1, R1.info().n_readouts)
        torch.cuda.synchronize()
        for i in range(req.n_nodes):
            a0, n = rows[(r, i)]
            b0 = R1.segment(s1[(0, i)]).stream_off
            assert torch.equal(h1[b0:b0 + n], mixed[a0:a0 + n]), ("request", r, "node", i)
    # the shortest request, every node, and the option distributions at its readouts (the fp64 stack
    # oracle takes ~25 ms per token per isolated pass, so a 16k-token request is out of a test's reach)
    r = order[0]
    ro_index = {s: k for k, s in enumerate(sorted(s for s in seg_of.values() if R.segment(s).readout_row >= 0))}
    l64, l32, lpg = [], [], []
    lp_h = lp.cpu().numpy()
    for i in range(tree.requests[r].n_nodes):
        a0, n = rows[(r, i)]
        ref, ref32 = _oracle_node(oc, W, tree, ids, hist, r, i, both=True)
        _assert_rounding_level(mixed[a0:a0 + n].float().cpu().numpy(), ref, ref32, ("mixed", r, i))
        if tree.requests[r].readout[i]:
            l64.append(ref[-1])
            l32.append(ref32[-1])
            lpg.append(lp_h[ro_index[seg_of[(r, i)]]])
    _assert_tv(np.stack(lpg), oc, W, np.stack(l64), np.stack(l32), ("mixed", r))
