"""The workspace-free GDN entry point (hs_gdn_fork_prefill_noalloc).

Some callers cannot allocate device memory -- a plug-in that may only touch
the buffers handed to it, or a host framework that owns every device
allocation -- so they cannot supply the scratch workspace that
hs_gdn_fork_prefill needs.  The no-alloc entry point uses a scratch array
built into the library instead.

It runs the same kernels as the regular entry point with only the scratch
address changed, so its outputs and written states must be bit-identical to
the regular entry point's on the same inputs.  The test runs three no-alloc
calls in a row through the C ABI: a large d=128 round (several scan groups),
then a smaller d=128 round with fewer chunks and groups -- so the scratch
still holds the large round's entries when the small one reads its own --
then a d=64 round; each is compared bit for bit with the regular entry point.
It also checks that a round too large for the built-in scratch is refused
before anything runs.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from hybrid_serving_gb300 import _lib, api, rounds  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _scratch_bytes() -> int:
    """HS_GDN_NOALLOC_SCRATCH_BYTES as include/hs.h defines it."""
    src = open(os.path.join(ROOT, "include", "hs.h")).read()
    m = re.search(r"#define\s+HS_GDN_NOALLOC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", src)
    assert m, "HS_GDN_NOALLOC_SCRATCH_BYTES not found in include/hs.h"
    return int(m.group(1)) << int(m.group(2))


def _round(tree, inp, n_slots=16):
    R, seg = rounds.build_round(tree, None, temp_slot0=2, n_temp_slots=n_slots - 2)
    meta = torch.empty(R.meta_bytes() // 4, dtype=torch.int32, device="cuda")
    R.upload(meta)
    dev = lambda key, dt: torch.from_numpy(rounds.to_stream(R, seg, inp.nodes, key)).cuda().to(dt)  # noqa: E731
    return R, meta, [dev(k, torch.bfloat16) for k in "qkv"] + [dev(k, torch.float32) for k in ("alpha", "beta")]


def _noalloc(R, meta, x, h, d, state, out, status):
    q, k, v, a, b = x
    return _lib.lib.hs_gdn_fork_prefill_noalloc(ctypes.byref(R.caps), meta.data_ptr(), _lib.HS_BF16, h, d, d, 64,
                                                q.data_ptr(), k.data_ptr(), v.data_ptr(), a.data_ptr(), b.data_ptr(),
                                                state.data_ptr(), state.shape[0], out.data_ptr(), status.data_ptr(),
                                                torch.cuda.current_stream().cuda_stream)


def _run(noalloc: bool, R, meta, x, h, d, n_slots=16):
    q, k, v, a, b = x
    state = torch.zeros((n_slots, h, d, d), dtype=torch.float32, device="cuda")
    out = torch.full_like(v, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if noalloc:
        _lib.check(_noalloc(R, meta, x, h, d, state, out, status))
    else:
        ws = torch.empty(api.gdn_workspace_bytes(R.caps, h, d, d), dtype=torch.uint8, device="cuda")
        api.gdn_fork_prefill(R.caps, meta, q, k, v, a, b, state, out, ws, status)
    torch.cuda.synchronize()
    api.check_status(status)
    return out.float().cpu().numpy(), state.cpu().numpy()


def test_noalloc_bit_identical_to_workspace_entry_point_in_a_row():
    cases = [
        # 3000-token trunk: 47 chunks, three scan groups; five branches
        (synth.Tree([synth.fork_tree(3000, [17, 1, 64, 65, 129])]), 4, 128, 90),
        # fewer chunks and no scan group, reading scratch the previous call filled
        (synth.Tree([synth.fork_tree(300, [40, 3, 70])]), 4, 128, 91),
        (synth.Tree([synth.fork_tree(63, [40, 3]), synth.fanout_tree(70, 20, 2, 2)]), 2, 64, 92),
    ]
    prepared = []
    for tree, h, d, seed in cases:
        inp = synth.gdn_inputs(tree, h, d, d, seed=seed, bf16=True, law="softplus")
        R, meta, x = _round(tree, inp)
        assert api.gdn_workspace_bytes(R.caps, h, d, d) <= _scratch_bytes()
        prepared.append((R, meta, x, h, d, _run(False, R, meta, x, h, d)))
    got = [_run(True, R, meta, x, h, d) for R, meta, x, h, d, _ in prepared]   # the no-alloc calls, back to back
    for (R, meta, x, h, d, (ref_o, ref_s)), (got_o, got_s) in zip(prepared, got):
        assert np.isfinite(got_o).all()
        assert np.array_equal(got_o, ref_o), float(np.abs(got_o - ref_o).max())
        assert np.array_equal(got_s, ref_s), float(np.abs(got_s - ref_s).max())


def test_noalloc_refuses_rounds_beyond_the_scratch():
    tree = synth.Tree([synth.fork_tree(8192, [64] * 4)])
    inp = synth.gdn_inputs(tree, 16, 128, 128, seed=93, bf16=True, law="softplus")
    R, meta, x = _round(tree, inp)
    assert api.gdn_workspace_bytes(R.caps, 16, 128, 128) > _scratch_bytes()
    state = torch.zeros((16, 16, 128, 128), dtype=torch.float32, device="cuda")
    out = torch.zeros_like(x[2])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _noalloc(R, meta, x, 16, 128, state, out, status) == _lib.HS_ECAPACITY
    assert "scratch" in _lib.last_error()


def test_noalloc_reports_shape_errors_like_the_workspace_entry_point():
    tree = synth.Tree([synth.fork_tree(8192, [64] * 4)])          # also too large for the scratch
    inp = synth.gdn_inputs(tree, 16, 128, 128, seed=94, bf16=True, law="softplus")
    R, meta, x = _round(tree, inp)
    state = torch.zeros((16, 16, 128, 128), dtype=torch.float32, device="cuda")
    out = torch.zeros_like(x[2])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # an unsupported head size is a shape error, not a capacity error, from both entry points
    assert _noalloc(R, meta, x, 16, 96, state, out, status) == _lib.HS_EUNSUPPORTED
