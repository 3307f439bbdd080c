"""The GDN chunk list (hs_round_build_chunks) and the attention tile table
(hs_round_build_tiles) built on the GPU from the segment table equal the
host round build's metadata word for word: the host-built blob is uploaded
with the rebuilt parts zeroed (chunk words, each node's chunk fields and the
chunk counts; tile records, tile span lists and the tile counts), the
kernel rebuilds them, and the whole blob comes back equal to the host's."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

from hybrid_serving_gb300 import api, rounds  # noqa: E402

# metadata words (include/hs.h record layouts; meta.h indices)
H_N_SEG, H_N_TILE, H_N_TILE_SPAN, H_N_CHUNK = 2, 4, 5, 6
H_OFF_SEG, H_OFF_TILE, H_OFF_TILE_SPAN, H_OFF_CHUNK, H_MAX_SEG_CHUNKS = 10, 13, 14, 15, 30
SEGW, CHUNKW, TILEW, S_CHUNK_OFF, S_N_CHUNK = 16, 4, 8, 9, 10

TREES = [
    synth.Tree([synth.fork_tree(64, [8, 8, 8])]),
    synth.Tree([synth.fork_tree(300, [17, 1, 128, 129]), synth.fork_tree(5, [40, 3])]),
    synth.Tree([synth.fanout_tree(40, 7, 3, 3)]),
    synth.gdn_tree(),
    synth.mixed_tree(seed=4000),
    synth.attn_tree(),
    synth.agent_tree(),
]


@pytest.mark.parametrize("ti", range(len(TREES)))
def test_device_chunk_list_equals_host(ti):
    tree = TREES[ti]
    R, _ = rounds.build_round(tree, None, temp_slot0=1000, n_temp_slots=sum(r.n_nodes for r in tree.requests) + 4)
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


def _resumed_round():
    """Two resumed roots with 2 and 1 history spans (the live pages of an earlier round), branches behind
    them, and a fresh request."""
    pool = api.PagePool(4096)
    R0, s0 = rounds.build_round(synth.Tree([synth.fork_tree(300, [4]), synth.fork_tree(40, [4])]), pool)
    p0, p1 = R0.segment_pages(s0[(0, 0)]), R0.segment_pages(s0[(1, 0)])
    R0.release(pool, keep=[s0[(0, 0)], s0[(1, 0)]])
    tree = synth.Tree([synth.fork_tree(70, [30, 200, 5], hist_len=300), synth.fork_tree(129, [1], hist_len=40),
                       synth.fork_tree(50, [60, 60, 60])])
    resume = {0: (None, [(256, p0[:16]), (44, p0[16:])]), 1: (None, [(40, p1)])}
    return rounds.build_round(tree, pool, resume=resume)


@pytest.mark.parametrize("ti", range(len(TREES) + 1))
def test_device_tile_table_equals_host(ti):
    if ti < len(TREES):
        tree = TREES[ti]
        n_pages = tree.useful_tokens() // 16 + 64 * sum(r.n_nodes for r in tree.requests)
        R, _ = rounds.build_round(tree, api.PagePool(n_pages), temp_slot0=1000)
    else:
        R, _ = _resumed_round()
    host = R.pack().numpy().copy()
    blanked = host.copy()
    n_tile, n_ts = int(host[H_N_TILE]), int(host[H_N_TILE_SPAN])
    ot, ots = int(host[H_OFF_TILE]), int(host[H_OFF_TILE_SPAN])
    blanked[ot:ot + n_tile * TILEW] = 0
    blanked[ots:ots + n_ts] = 0
    blanked[H_N_TILE] = 0
    blanked[H_N_TILE_SPAN] = 0
    assert not np.array_equal(blanked, host)
    meta = torch.from_numpy(blanked).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.round_build_tiles(R.caps, meta, status)
    torch.cuda.synchronize()
    api.check_status(status)
    np.testing.assert_array_equal(meta.cpu().numpy(), host)
