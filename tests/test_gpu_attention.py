"""ForkAttention parity: the CUDA path through the C ABI vs the fp64 oracle.

Tolerances (max-abs over every compared element): 1e-4 for fp32 inputs,
2e-2 for bf16 inputs with fp32 accumulation; choice distributions within
1e-3 total variation.  Batch invariance is checked bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import choice as ochoice
from oracle import forward, numerics

pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from harness import AttnRun, max_abs  # noqa: E402
from hybrid_serving_gb300 import _lib, api  # noqa: E402

TOL_F32, TOL_BF16, TOL_TV = 1e-4, 2e-2, 1e-3


def _check(tree, inp, dtype, tol, **kw):
    run = AttnRun(tree, inp, dtype, **kw).run()
    api.check_status(run.status)
    got = run.outputs()
    ref = forward.attention_tree(tree, inp, 1 / math.sqrt(inp.d))
    err = max_abs(got, ref)
    print(f"[margin] attention {dtype} max-abs {err:.3e} (bar {tol:.0e})")
    assert err <= tol, f"max abs err {err}"
    return run, got, ref


def test_tiny_fp32():
    tree = synth.tiny_tree()
    inp = synth.attn_inputs(tree, 2, 2, 64, seed=1000, bf16=False, sigma=1 / 8)
    _check(tree, inp, torch.float32, TOL_F32)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_ragged_multi_request(d, dtype):
    tree = synth.Tree([synth.fork_tree(300, [17, 1, 128, 129]), synth.fork_tree(5, [40, 3]),
                       synth.fork_tree(129, [64, 65, 1])])
    inp = synth.attn_inputs(tree, 8, 2, d, seed=1100 + d, bf16=dtype == torch.bfloat16)
    _check(tree, inp, dtype, TOL_BF16 if dtype == torch.bfloat16 else TOL_F32)


def test_deep_tree_bf16():
    tree = synth.Tree([synth.fanout_tree(70, 9, 3, 3), synth.Request(parents=[-1, 0, 1, 1, 0, 4],
                                                                     n_tok=[33, 20, 5, 100, 9, 2])])
    inp = synth.attn_inputs(tree, 4, 4, 128, seed=1200, bf16=True)
    _check(tree, inp, torch.bfloat16, TOL_BF16)


def test_resumed_history_bf16():
    """Round A computes a 200-token trunk; round B resumes at 200 with the
    trunk's pages as history, 37 new trunk tokens and two branches.  The
    oracle recomputes every path from position 0."""
    full = synth.Tree([synth.fork_tree(237, [11, 30])])
    inp = synth.attn_inputs(full, 8, 2, 128, seed=1300, bf16=True)
    a_tree = synth.Tree([synth.fork_tree(200, [4])])
    a_inp = synth.remap_inputs(full, inp, synth.Tree([synth.fork_tree(200, [11, 30])]))
    a_inp.nodes = {(0, 0): a_inp.nodes[(0, 0)], (0, 1): {k: v[:4] for k, v in a_inp.nodes[(0, 1)].items()}}
    A = AttnRun(a_tree, a_inp, torch.bfloat16, n_pages=64).run()
    pages = A.R.segment_pages(A.seg_of[(0, 0)])
    A.R.release(A.pool, keep=[A.seg_of[(0, 0)]])
    b_tree = synth.Tree([synth.fork_tree(37, [11, 30], hist_len=200)])
    b_inp = synth.remap_inputs(full, inp, b_tree)
    B = AttnRun(b_tree, b_inp, torch.bfloat16, pool=A.pool, k_pages=A.k_pages, v_pages=A.v_pages,
                resume={0: (None, [(200, pages)])}).run()
    api.check_status(B.status)
    got = B.outputs()
    ref = forward.attention_tree(b_tree, b_inp, 1 / math.sqrt(128))
    assert max_abs(got, ref) <= TOL_BF16


def test_fragmented_pool_pages():
    """A round whose pages are scattered over the pool (every other page held by an earlier round), so no
    128-key block has consecutive pages and the kernel copies each page on its own: every row against its
    isolated pass, and bit for bit equal to the same round on consecutive pages."""
    from hybrid_serving_gb300 import rounds
    tree = synth.Tree([synth.fork_tree(1024, [40, 64, 17])])
    inp = synth.attn_inputs(tree, 8, 2, 128, seed=1500, bf16=True)
    n_pages = 512
    pool = api.PagePool(n_pages)
    filler = synth.Tree([synth.fork_tree(16, [16] * 150)])  # one page per node
    Rf, seg_f = rounds.build_round(filler, pool)
    Rf.release(pool, keep=list(range(0, Rf.info().n_segments, 2)))  # every other page stays held
    kp = torch.zeros((2, n_pages, 16, 128), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    run = AttnRun(tree, inp, torch.bfloat16, pool=pool, k_pages=kp, v_pages=vp).run()
    api.check_status(run.status)
    trunk_pages = run.R.segment_pages(run.seg_of[(0, 0)])
    assert all(b != a + 1 for a, b in zip(trunk_pages, trunk_pages[1:]))  # no two consecutive
    got = run.outputs()
    ref = forward.attention_tree(tree, inp, 1 / math.sqrt(128))
    err = max_abs(got, ref)
    print(f"[margin] attention on scattered pages max-abs {err:.3e} (bar 2e-2)")
    assert err <= TOL_BF16
    dense = AttnRun(tree, inp, torch.bfloat16).run()  # fresh pool: consecutive pages
    api.check_status(dense.status)
    assert torch.equal(run.out, dense.out)


def test_full_size_all_rows_and_choices():
    """The attention workload at full size (trunk 4096, 8 branches of
    U[16,64], GQA 32/8, d=128, bf16): every trunk row and every row of every
    branch against its isolated pass -- so every work item of the persistent
    kernel is checked -- and the 4-option distribution of every branch."""
    tree = synth.attn_tree()
    inp = synth.attn_inputs(tree, 32, 8, 128, seed=2000, bf16=True)
    run = AttnRun(tree, inp, torch.bfloat16).run()
    api.check_status(run.status)
    got = run.outputs()
    req = tree.requests[0]
    ref = forward.attention_tree(tree, inp, 1 / math.sqrt(128), matrix=True)
    e_tr = float(np.abs(got[(0, 0)] - ref[(0, 0)]).max())
    e_br = max_abs(got, ref, keys=[(0, b) for b in range(1, req.n_nodes)])
    print(f"[margin] attention full size: trunk rows max-abs {e_tr:.3e}, branch rows {e_br:.3e} (bar 2e-2)")
    assert e_tr <= TOL_BF16 and e_br <= TOL_BF16
    # choices: logits over the concatenated head outputs of each branch's last token
    W = synth.option_rows(4, 32 * 128, seed=2001)
    Wd = torch.from_numpy(W).cuda()
    lp = torch.empty((run.R.info().n_readouts, 4), dtype=torch.float32, device="cuda")
    api.choice_logprobs(run.R.caps, run.meta, run.out.view(run.out.shape[0], -1), Wd, lp, run.status)
    torch.cuda.synchronize()
    api.check_status(run.status)
    last = {(0, b): [req.n_tok[b] - 1] for b in range(1, req.n_nodes)}
    ref_last = forward.attention_tree(tree, inp, 1 / math.sqrt(128), nodes=list(last), rows=last)
    h = np.stack([numerics.round_bf16(ref_last[(0, b)][0].reshape(-1)) for b in range(1, req.n_nodes)])
    p_ref = np.exp(ochoice.option_logprobs(h, W))
    p_gpu = np.exp(lp.cpu().numpy().astype(np.float64))
    tv = ochoice.total_variation(p_gpu, p_ref)
    print(f"[margin] attention full size: option TV max {tv.max():.3e} (bar 1e-3)")
    assert tv.max() <= TOL_TV, tv
    assert (ochoice.top1(p_gpu) == ochoice.top1(p_ref)).all()
    # the kernel alone, on the GPU's own hidden rows
    hg = np.stack([got[(0, b)][-1].reshape(-1) for b in range(1, req.n_nodes)])
    assert ochoice.total_variation(p_gpu, np.exp(ochoice.option_logprobs(hg, W))).max() <= 1e-5


def test_batch_invariance_bitwise():
    """A branch's bits do not depend on its siblings or on other requests
    in the round (Flide section 3.5)."""
    base = synth.fork_tree(777, [20, 50, 13, 100])
    other = synth.fork_tree(300, [9, 9])
    tree = synth.Tree([other, base])
    inp = synth.attn_inputs(tree, 8, 2, 128, seed=1400, bf16=True)
    mixed = AttnRun(tree, inp, torch.bfloat16).run().raw_outputs()
    for b in range(1, 5):
        alone_tree = synth.Tree([synth.fork_tree(777, [base.n_tok[b]])])
        alone_inp = synth.AttnInputs(8, 2, 128, True, {(0, 0): inp.nodes[(1, 0)], (0, 1): inp.nodes[(1, b)]},
                                     {0: inp.hist[1]})
        alone = AttnRun(alone_tree, alone_inp, torch.bfloat16).run().raw_outputs()
        assert torch.equal(alone[(0, 1)], mixed[(1, b)]), f"branch {b} differs"
        assert torch.equal(alone[(0, 0)], mixed[(1, 0)])


def test_bad_page_sets_status_without_fault():
    tree = synth.Tree([synth.fork_tree(64, [8])])
    inp = synth.attn_inputs(tree, 2, 2, 64, seed=1500, bf16=True)
    run = AttnRun(tree, inp, torch.bfloat16, n_pages=32, n_pages_kernel=2).run()
    assert int(run.status.item()) == 1  # HS_DEV_BAD_PAGE
    with pytest.raises(_lib.HsError):
        api.check_status(run.status)


MASK_PATHS = [("paired tensor-core", torch.bfloat16, 8, 2, 128), ("CUDA cores fp32", torch.float32, 4, 2, 64),
              ("odd group (CUDA cores)", torch.bfloat16, 6, 2, 128)]
MASKS = [(37, False), (300, False), (0, True), (50, True)]


@pytest.mark.parametrize("path", range(len(MASK_PATHS)))
@pytest.mark.parametrize("mask", range(len(MASKS)))
def test_masks_match_oracle(path, mask):
    """Mask variants (Flide section 3.2.1 sliding window t_x - t_y < W; Appendix H bidirectional state):
    every row of a ragged multi-level round against the oracle's isolated pass with the same mask."""
    name, dt, hq, hkv, d = MASK_PATHS[path]
    W, bidir = MASKS[mask]
    tree = synth.Tree([synth.fork_tree(333, [17, 1, 64, 130]), synth.fanout_tree(60, 20, 2, 2)])
    inp = synth.attn_inputs(tree, hq, hkv, d, seed=1700 + path, bf16=dt == torch.bfloat16)
    run = AttnRun(tree, inp, dt).run_masked(window=W, bidirectional_root=bidir)
    api.check_status(run.status)
    ref = forward.attention_tree(tree, inp, 1 / math.sqrt(d), window=W or None, bidir_root=bidir, matrix=True)
    err = max_abs(run.outputs(), ref)
    tol = TOL_BF16 if dt == torch.bfloat16 else TOL_F32
    print(f"[margin] attention mask W={W} bidir={bidir} {name}: max-abs {err:.3e} (bar {tol:.0e})")
    assert err <= tol


def test_window_batch_invariance_bitwise():
    base = synth.fork_tree(777, [20, 50, 13, 100])
    tree = synth.Tree([synth.fork_tree(300, [9, 9]), base])
    inp = synth.attn_inputs(tree, 8, 2, 128, seed=1800, bf16=True)
    mixed = AttnRun(tree, inp, torch.bfloat16).run_masked(window=200).raw_outputs()
    for b in range(1, 5):
        alone_tree = synth.Tree([synth.fork_tree(777, [base.n_tok[b]])])
        alone_inp = synth.AttnInputs(8, 2, 128, True, {(0, 0): inp.nodes[(1, 0)], (0, 1): inp.nodes[(1, b)]},
                                     {0: inp.hist[1]})
        alone = AttnRun(alone_tree, alone_inp, torch.bfloat16).run_masked(window=200).raw_outputs()
        assert torch.equal(alone[(0, 1)], mixed[(1, b)]), f"branch {b} differs"
        assert torch.equal(alone[(0, 0)], mixed[(1, 0)])


@pytest.mark.parametrize("W, bidir", [(50, False), (0, True), (30, True), (260, False)])
def test_masks_with_resumed_history(W, bidir):
    """Mask variants on a resumed root: round B resumes a 200-token trunk from its cached pages with 37 new
    trunk tokens and two branches, under a sliding window (positions continue through the history, so a
    row's window reaches back into the cached pages) and/or a bidirectional root (the root's rows see the
    whole root and its history); every row against the oracle's masked isolated pass from position 0."""
    full = synth.Tree([synth.fork_tree(237, [11, 30])])
    inp = synth.attn_inputs(full, 8, 2, 128, seed=1310, bf16=True)
    a_tree = synth.Tree([synth.fork_tree(200, [4])])
    a_inp = synth.remap_inputs(full, inp, synth.Tree([synth.fork_tree(200, [11, 30])]))
    a_inp.nodes = {(0, 0): a_inp.nodes[(0, 0)], (0, 1): {k: v[:4] for k, v in a_inp.nodes[(0, 1)].items()}}
    A = AttnRun(a_tree, a_inp, torch.bfloat16, n_pages=64).run()
    pages = A.R.segment_pages(A.seg_of[(0, 0)])
    A.R.release(A.pool, keep=[A.seg_of[(0, 0)]])
    b_tree = synth.Tree([synth.fork_tree(37, [11, 30], hist_len=200)])
    b_inp = synth.remap_inputs(full, inp, b_tree)
    B = AttnRun(b_tree, b_inp, torch.bfloat16, pool=A.pool, k_pages=A.k_pages, v_pages=A.v_pages,
                resume={0: (None, [(200, pages)])}).run_masked(window=W, bidirectional_root=bidir)
    api.check_status(B.status)
    ref = forward.attention_tree(b_tree, b_inp, 1 / math.sqrt(128), window=W or None, bidir_root=bidir, matrix=True)
    err = max_abs(B.outputs(), ref)
    print(f"[margin] attention mask W={W} bidir={bidir} resumed history: max-abs {err:.3e} (bar 2e-02)")
    assert err <= TOL_BF16
