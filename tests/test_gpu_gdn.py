"""Gated DeltaNet fork-prefill parity: the CUDA path through the C ABI vs
the fp64 step-by-step oracle (every branch an isolated pass), plus
checkpoint/resume and batch invariance.

Tolerances: 1e-4 max-abs for fp32 inputs, 2e-2 for bf16 inputs (fp32 state
and accumulation).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import forward
from oracle import gdn as ogdn

pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from harness import GdnRun, max_abs  # noqa: E402
from hybrid_serving_gb300 import _lib, api  # noqa: E402

TOL_F32, TOL_BF16 = 1e-4, 2e-2


def _check(tree, inp, dtype, tol, **kw):
    run = GdnRun(tree, inp, dtype, **kw).run()
    api.check_status(run.status)
    got = run.outputs()
    ref = forward.gdn_tree(tree, inp)
    err = max_abs(got, ref)
    print(f"[margin] gdn {dtype} max-abs {err:.3e} (bar {tol:.0e})")
    assert err <= tol, f"max abs err {err}"
    return run


def test_tiny_fp32():
    tree = synth.tiny_tree()
    inp = synth.gdn_inputs(tree, 2, 64, 64, seed=1000, bf16=False, law="uniform")
    _check(tree, inp, torch.float32, TOL_F32)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_ragged_multi_request(d, dtype):
    tree = synth.Tree([synth.fork_tree(300, [17, 1, 64, 65, 129]), synth.fork_tree(63, [40, 3])])
    inp = synth.gdn_inputs(tree, 4, d, d, seed=1100 + d, bf16=dtype == torch.bfloat16, law="softplus")
    _check(tree, inp, dtype, TOL_BF16 if dtype == torch.bfloat16 else TOL_F32)


def test_deep_tree_bf16():
    tree = synth.Tree([synth.fanout_tree(100, 33, 3, 3)])
    inp = synth.gdn_inputs(tree, 2, 128, 128, seed=1200, bf16=True, law="softplus")
    _check(tree, inp, torch.bfloat16, TOL_BF16)


@pytest.mark.parametrize("m", [448, 463])
def test_checkpoint_then_resume(m):
    """Round A splits the 500-token trunk at m and saves the state at m into
    slot 0; round B resumes there with trunk tokens [m, 600) and the same
    branches.  Outputs match the oracle's full recompute; with m on a chunk
    boundary they match a fresh round over the whole trunk bit for bit."""
    a_tree, b_tree, full = synth.gdn_checkpoint_trees(m, trunk=500, extra=100, k=3)
    inp = synth.gdn_inputs(full, 4, 128, 128, seed=1300, bf16=True, law="softplus")
    a_inp = synth.remap_inputs(full, inp, a_tree)
    state = torch.zeros((16, 4, 128, 128), dtype=torch.float32, device="cuda")
    A = GdnRun(a_tree, a_inp, torch.bfloat16, state_pool=state, temp_slot0=4).run()
    api.check_status(A.status)
    assert max_abs(A.outputs(), forward.gdn_tree(a_tree, a_inp)) <= TOL_BF16
    # the saved checkpoint equals the oracle's state after the first m trunk tokens
    tr = inp.nodes[(0, 0)]
    _, S_m = ogdn.gated_delta_rule(tr["q"][:m], tr["k"][:m], tr["v"][:m], tr["alpha"][:m], tr["beta"][:m])
    np.testing.assert_allclose(state[0].cpu().numpy(), S_m, atol=1e-3)
    snap = state[0].clone()
    b_inp = synth.remap_inputs(full, inp, b_tree)
    B = GdnRun(b_tree, b_inp, torch.bfloat16, state_pool=state, temp_slot0=4, resume={0: (0, [])}).run()
    api.check_status(B.status)
    got = B.outputs()
    assert max_abs(got, forward.gdn_tree(b_tree, b_inp)) <= TOL_BF16
    assert torch.equal(state[0], snap)          # resuming reads the checkpoint, never writes it
    if m % 64 == 0:
        F = GdnRun(full, inp, torch.bfloat16, state_pool=torch.zeros_like(state), temp_slot0=4).run()
        fresh = F.raw_outputs()
        raw = B.raw_outputs()
        assert torch.equal(raw[(0, 0)], fresh[(0, 0)][m:])
        for b in range(1, 4):
            assert torch.equal(raw[(0, b)], fresh[(0, b)])


def test_full_size_sampled():
    """Trunk 8192 + 16 branches of U[8,128], 16 heads, d=128, bf16: the
    trunk and the first and last branch against their isolated passes."""
    tree = synth.gdn_tree()
    inp = synth.gdn_inputs(tree, 16, 128, 128, seed=3000, bf16=True, law="softplus")
    run = GdnRun(tree, inp, torch.bfloat16).run()
    api.check_status(run.status)
    got = run.outputs()
    nodes = [(0, 1), (0, tree.requests[0].n_nodes - 1)]
    ref = forward.gdn_tree(tree, inp, nodes=nodes)
    e_br = max_abs(got, ref, keys=nodes)
    # trunk rows: the trunk's own pass
    tr = inp.nodes[(0, 0)]
    o_tr, _ = ogdn.gated_delta_rule(tr["q"], tr["k"], tr["v"], tr["alpha"], tr["beta"])
    e_tr = float(np.abs(got[(0, 0)] - o_tr).max())
    print(f"[margin] gdn full size: trunk rows max-abs {e_tr:.3e}, branches {e_br:.3e} (bar 2e-2)")
    assert e_br <= TOL_BF16
    assert e_tr <= TOL_BF16


_RESUME_REF = {}


def _resume_reference(full, inp):
    """The oracle over the whole extended trunk (9216 tokens) and every branch after it.  A branch's
    isolated pass is the trunk's recurrence continued over the branch's tokens, so each branch
    continues from the fp64 state the trunk pass ends in: the same operations in the same order as
    a pass over trunk + branch, computed once for the two checkpoint positions."""
    if not _RESUME_REF:
        tr = inp.nodes[(0, 0)]
        o_tr, S = ogdn.gated_delta_rule(tr["q"], tr["k"], tr["v"], tr["alpha"], tr["beta"])
        _RESUME_REF[(0, 0)] = o_tr
        for b in range(1, full.requests[0].n_nodes):
            x = inp.nodes[(0, b)]
            _RESUME_REF[(0, b)], _ = ogdn.gated_delta_rule(x["q"], x["k"], x["v"], x["alpha"], x["beta"], S0=S)
    return _RESUME_REF


@pytest.mark.parametrize("m", [8192, 8155])
def test_full_size_resume(m):
    """Resume after appending 1024 trunk tokens, at full size: round A runs the 8192-token trunk (split
    at m, its state saved there) and the 16 branches; round B resumes at m with trunk tokens
    [m, 9216) and the same 16 branches.  Every row of round B -- each trunk row past m and every
    row of every branch -- against the oracle's full recompute of the 9216-token trunk.  (A fresh
    pass over 9216 tokens groups its 144 chunks for the state scan differently from the resumed
    round, so the two agree to rounding, not bit for bit, even at the aligned m.)"""
    a_tree, b_tree, full = synth.gdn_checkpoint_trees(m)
    inp = synth.gdn_inputs(full, 16, 128, 128, seed=3000, bf16=True, law="softplus")
    state = torch.zeros((24, 16, 128, 128), dtype=torch.float32, device="cuda")
    A = GdnRun(a_tree, synth.remap_inputs(full, inp, a_tree), torch.bfloat16, state_pool=state,
               temp_slot0=4).run()
    api.check_status(A.status)
    snap = state[0].clone()
    B = GdnRun(b_tree, synth.remap_inputs(full, inp, b_tree), torch.bfloat16, state_pool=state, temp_slot0=4,
               resume={0: (0, [])}).run()
    api.check_status(B.status)
    assert torch.equal(state[0], snap)          # resuming reads the checkpoint, never writes it
    got = B.outputs()
    ref = _resume_reference(full, inp)
    e_tr = float(np.abs(got[(0, 0)] - ref[(0, 0)][m:]).max())
    e_br = max(float(np.abs(got[(0, b)] - ref[(0, b)]).max()) for b in range(1, b_tree.requests[0].n_nodes))
    print(f"[margin] gdn resume m={m}: trunk tail max-abs {e_tr:.3e}, branches {e_br:.3e} (bar 2e-2)")
    assert got[(0, 0)].shape[0] == 9216 - m
    assert e_tr <= TOL_BF16 and e_br <= TOL_BF16


def test_batch_invariance_bitwise():
    base = synth.fork_tree(333, [20, 50, 13, 100])
    other = synth.fork_tree(200, [9, 70])
    tree = synth.Tree([other, base])
    inp = synth.gdn_inputs(tree, 4, 128, 128, seed=1400, bf16=True, law="softplus")
    mixed = GdnRun(tree, inp, torch.bfloat16).run().raw_outputs()
    for b in range(1, 5):
        alone_tree = synth.Tree([synth.fork_tree(333, [base.n_tok[b]])])
        alone_inp = synth.GdnInputs(4, 128, 128, True, {(0, 0): inp.nodes[(1, 0)], (0, 1): inp.nodes[(1, b)]},
                                    {0: inp.hist[1]})
        alone = GdnRun(alone_tree, alone_inp, torch.bfloat16).run().raw_outputs()
        assert torch.equal(alone[(0, 1)], mixed[(1, b)]), f"branch {b} differs"
        assert torch.equal(alone[(0, 0)], mixed[(1, 0)])


def test_state_checkpoint_copy_and_bad_slot():
    state = torch.randn((4, 2, 64, 64), device="cuda")
    api.gdn_state_checkpoint(state, 1, 3)
    torch.cuda.synchronize()
    assert torch.equal(state[1], state[3])
    with pytest.raises(_lib.HsError):
        api.gdn_state_checkpoint(state, 1, 4)
    # a tree whose temporary slots lie beyond the pool: the kernel reports it
    tree = synth.Tree([synth.fork_tree(70, [8, 9])])
    inp = synth.gdn_inputs(tree, 2, 64, 64, seed=1500, bf16=True, law="softplus")
    run = GdnRun(tree, inp, torch.bfloat16, state_pool=torch.zeros((2, 2, 64, 64), device="cuda"),
                 temp_slot0=5, n_temp=4)            # the trunk's end state goes to slot 5 of a 2-slot pool
    api.gdn_fork_prefill(run.R.caps, run.meta, run.q, run.k, run.v, run.alpha, run.beta, run.state, run.out,
                         run.ws, run.status)
    torch.cuda.synchronize()
    assert int(run.status.item()) == 2  # HS_DEV_BAD_SLOT


def test_scan_group_counts():
    """Long nodes split into 2, 3, 4, 5, 7 and 8 scan groups (24 .. 100 chunks of 64; the last one
    ragged) in one round: the first pass (group 0's end, each later group's N and M as two chains
    in one CTA), the start states combined from them and the replay with outputs, against the
    step-by-step recurrence; a branch after each trunk continues from the trunk's end state."""
    lens = [24 * 64, 36 * 64 - 5, 48 * 64, 60 * 64 + 17, 84 * 64, 100 * 64 - 33]
    tree = synth.Tree([synth.fork_tree(n, [37]) for n in lens])
    inp = synth.gdn_inputs(tree, 2, 128, 128, seed=3100, bf16=True, law="softplus")
    _check(tree, inp, torch.bfloat16, TOL_BF16)
