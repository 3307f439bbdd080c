"""The GDN chunk list built on the GPU (hs_round_build_chunks) from the
segment table equals the host round build's metadata word for word: the
host-built blob is uploaded with every chunk word, each node's chunk fields
and the header's chunk counts zeroed, the kernel rebuilds them, and the
whole blob comes back equal to the host's."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from hybrid_serving_gb300 import api, rounds  # noqa: E402

# metadata words (include/hs.h record layouts; meta.h indices)
H_N_SEG, H_N_CHUNK, H_OFF_SEG, H_OFF_CHUNK, H_MAX_SEG_CHUNKS = 2, 6, 10, 15, 30
SEGW, CHUNKW, S_CHUNK_OFF, S_N_CHUNK = 16, 4, 9, 10

TREES = [
    synth.Tree([synth.fork_tree(64, [8, 8, 8])]),
    synth.Tree([synth.fork_tree(300, [17, 1, 128, 129]), synth.fork_tree(5, [40, 3])]),
    synth.Tree([synth.fanout_tree(40, 7, 3, 3)]),
    synth.gdn_tree(),
    synth.mixed_tree(seed=4000),
]


@pytest.mark.parametrize("ti", range(len(TREES)))
def test_device_chunk_list_equals_host(ti):
    tree = TREES[ti]
    R, _ = rounds.build_round(tree, None, temp_slot0=0, n_temp_slots=sum(r.n_nodes for r in tree.requests) + 4)
    host = R.pack().numpy().copy()
    blanked = host.copy()
    n_seg, n_chunk = int(host[H_N_SEG]), int(host[H_N_CHUNK])
    oc, os_ = int(host[H_OFF_CHUNK]), int(host[H_OFF_SEG])
    blanked[oc:oc + n_chunk * CHUNKW] = 0
    for i in range(n_seg):
        blanked[os_ + i * SEGW + S_CHUNK_OFF] = 0
        blanked[os_ + i * SEGW + S_N_CHUNK] = 0
    blanked[H_N_CHUNK] = 0
    blanked[H_MAX_SEG_CHUNKS] = 0
    assert not np.array_equal(blanked, host)
    meta = torch.from_numpy(blanked).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.round_build_chunks(R.caps, meta, status)
    torch.cuda.synchronize()
    api.check_status(status)
    np.testing.assert_array_equal(meta.cpu().numpy(), host)
