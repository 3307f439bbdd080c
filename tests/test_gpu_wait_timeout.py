"""Failure detection of the bounded device waits, without a GPU fault: one CTA
holds tensor memory and a bulk copy in flight while two warps wait on barriers
that nothing completes (the suspending and the spinning poll of the tcgen05
kernels).  The waits give up after their limit, the status word reads
HS_DEV_TIMEOUT, the host maps it to HS_EDEVICE, and the context stays usable:
a ForkAttention round right after matches the oracle."""
import math

import pytest
import torch

import synth
from oracle import forward

pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from harness import AttnRun, max_abs  # noqa: E402
from hybrid_serving_gb300 import _lib, api  # noqa: E402


@pytest.mark.parametrize("limit", [20_000, 2_000_000])
def test_wait_runs_out_and_the_context_stays_usable(limit):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(2, dtype=torch.int64, device="cuda")
    api.debug_wait_timeout(limit, status, elapsed)
    torch.cuda.synchronize()  # the kernel returned: no fault, no hang
    assert int(status.item()) == _lib.HS_DEV_TIMEOUT
    with pytest.raises(_lib.HsError) as e:
        api.check_status(status)
    assert e.value.code == _lib.HS_EDEVICE
    el = elapsed.cpu().tolist()
    print(f"[wait] limit {limit} clocks: waited {el[0]} (try_wait), {el[1]} (test_wait)")
    for x in el:  # each wait lasted its limit and gave up after it (a suspended try_wait may overshoot by
        assert limit < x < 4 * limit + 2_000_000  # its own time slice, about a microsecond)
    # the context still runs the hot path correctly
    tree = synth.Tree([synth.fork_tree(150, [20, 7])])
    inp = synth.attn_inputs(tree, 8, 2, 128, seed=1900, bf16=True)
    run = AttnRun(tree, inp, torch.bfloat16).run()
    api.check_status(run.status)
    assert max_abs(run.outputs(), forward.attention_tree(tree, inp, 1 / math.sqrt(128))) <= 2e-2


def test_wait_timeout_refuses_bad_arguments():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for bad in (0, -5, (1 << 31) + 1):
        with pytest.raises(_lib.HsError) as e:
            api.debug_wait_timeout(bad, status)
        assert e.value.code == _lib.HS_EINVAL
    assert int(status.item()) == 0
