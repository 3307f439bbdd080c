"""The workspace-free GDN entry point (hs_gdn_fork_prefill_noalloc).

Some callers cannot allocate device memory -- a plug-in that may only touch
the buffers handed to it, or a host framework that owns every device
allocation -- so they cannot supply the scratch workspace that
hs_gdn_fork_prefill needs.  The no-alloc entry point uses a scratch array
built into the library instead.  This test calls it through the C ABI twice
in a row, on two different rounds, and checks each output (and each written
state) against the regular entry point on the same inputs, within the bf16
tolerance of the other GDN tests.  It also checks that a round too large for
the built-in scratch is refused before anything runs.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from hybrid_serving_gb300 import _lib, api, rounds  # noqa: E402

TOL_BF16 = 2e-2


def _round(tree, inp, n_slots=16):
    R, seg = rounds.build_round(tree, None, temp_slot0=2, n_temp_slots=n_slots - 2)
    meta = torch.empty(R.meta_bytes() // 4, dtype=torch.int32, device="cuda")
    R.upload(meta)
    dev = lambda key, dt: torch.from_numpy(rounds.to_stream(R, seg, inp.nodes, key)).cuda().to(dt)  # noqa: E731
    return R, meta, [dev(k, torch.bfloat16) for k in "qkv"] + [dev(k, torch.float32) for k in ("alpha", "beta")]


def _run(noalloc: bool, R, meta, x, h, d, n_slots=16):
    q, k, v, a, b = x
    state = torch.zeros((n_slots, h, d, d), dtype=torch.float32, device="cuda")
    out = torch.full_like(v, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    if noalloc:
        code = _lib.lib.hs_gdn_fork_prefill_noalloc(ctypes.byref(R.caps), meta.data_ptr(), _lib.HS_BF16, h, d, d, 64,
                                                    q.data_ptr(), k.data_ptr(), v.data_ptr(), a.data_ptr(),
                                                    b.data_ptr(), state.data_ptr(), n_slots, out.data_ptr(),
                                                    status.data_ptr(), stream)
        _lib.check(code)
    else:
        ws = torch.empty(api.gdn_workspace_bytes(R.caps, h, d, d), dtype=torch.uint8, device="cuda")
        api.gdn_fork_prefill(R.caps, meta, q, k, v, a, b, state, out, ws, status)
    torch.cuda.synchronize()
    api.check_status(status)
    return out.float().cpu().numpy(), state.cpu().numpy()


def test_noalloc_matches_workspace_entry_point_twice():
    cases = [
        (synth.Tree([synth.fork_tree(300, [17, 1, 64, 65, 129])]), 4, 128, 91),
        (synth.Tree([synth.fork_tree(63, [40, 3]), synth.fanout_tree(70, 20, 2, 2)]), 2, 64, 92),
    ]
    for tree, h, d, seed in cases:                      # two calls in a row, different rounds
        inp = synth.gdn_inputs(tree, h, d, d, seed=seed, bf16=True, law="softplus")
        R, meta, x = _round(tree, inp)
        assert api.gdn_workspace_bytes(R.caps, h, d, d) <= _lib_scratch_bytes()
        ref_o, ref_s = _run(False, R, meta, x, h, d)
        got_o, got_s = _run(True, R, meta, x, h, d)
        assert np.isfinite(got_o).all()
        assert float(np.abs(got_o - ref_o).max()) <= TOL_BF16
        assert float(np.abs(got_s - ref_s).max()) <= TOL_BF16


def test_noalloc_refuses_rounds_beyond_the_scratch():
    tree = synth.Tree([synth.fork_tree(8192, [64] * 4)])
    inp = synth.gdn_inputs(tree, 16, 128, 128, seed=93, bf16=True, law="softplus")
    R, meta, x = _round(tree, inp)
    assert api.gdn_workspace_bytes(R.caps, 16, 128, 128) > _lib_scratch_bytes()
    q, k, v, a, b = x
    state = torch.zeros((16, 16, 128, 128), dtype=torch.float32, device="cuda")
    out = torch.zeros_like(v)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    code = _lib.lib.hs_gdn_fork_prefill_noalloc(ctypes.byref(R.caps), meta.data_ptr(), _lib.HS_BF16, 16, 128, 128,
                                                64, q.data_ptr(), k.data_ptr(), v.data_ptr(), a.data_ptr(),
                                                b.data_ptr(), state.data_ptr(), 16, out.data_ptr(), status.data_ptr(),
                                                torch.cuda.current_stream().cuda_stream)
    assert code == _lib.HS_ECAPACITY
    assert "scratch" in _lib.last_error()


def _lib_scratch_bytes() -> int:
    return 32 << 20          # HS_GDN_NOALLOC_SCRATCH_BYTES in include/hs.h
