"""Host-side tests of the round builder and page pool (no GPU).

The packed metadata is decoded here from its documented record layout and
compared, bit for bit, with the oracle's layout (Flide Eq. 2), positions,
token metadata and -- for every query row -- the key set of Eq. 3, after
mapping each physical page row the attention kernel would read back to
the token written there.
"""
import re
import subprocess

import numpy as np
import pytest

import synth
from oracle import layout

api = pytest.importorskip("hybrid_serving_gb300.api")
from hybrid_serving_gb300 import _lib, rounds  # noqa: E402

PAGE = 16
# record layouts (words) of the metadata blob
H = dict(N_TOK=1, N_SEG=2, N_SPAN=3, N_TILE=4, N_TILE_SPAN=5, N_CHUNK=6, N_READOUT=7, N_LEVEL=8, N_PAGE_REF=9,
         OFF_SEG=10, OFF_TOK=11, OFF_SPAN=12, OFF_TILE=13, OFF_TILE_SPAN=14, OFF_CHUNK=15, OFF_READOUT=16,
         OFF_LEVEL=17, OFF_LEVEL_SEG=18, OFF_PAGE_REF=19)
SEGW, TOKW, SPANW, TILEW, CHUNKW = 16, 2, 4, 8, 4


class Blob:
    def __init__(self, words):
        self.w = np.asarray(words, dtype=np.int64)

    def h(self, k):
        return int(self.w[H[k]])

    def arr(self, off, n, width):
        o = self.h(off)
        return self.w[o:o + n * width].reshape(n, width) if width > 1 else self.w[o:o + n]

    @property
    def segs(self):
        return self.arr("OFF_SEG", self.h("N_SEG"), SEGW)

    @property
    def toks(self):
        return self.arr("OFF_TOK", self.h("N_TOK"), TOKW)

    @property
    def spans(self):
        return self.arr("OFF_SPAN", self.h("N_SPAN"), SPANW)

    @property
    def tiles(self):
        return self.arr("OFF_TILE", self.h("N_TILE"), TILEW)

    @property
    def tile_spans(self):
        return self.arr("OFF_TILE_SPAN", self.h("N_TILE_SPAN"), 1)

    @property
    def chunks(self):
        return self.arr("OFF_CHUNK", self.h("N_CHUNK"), CHUNKW)

    @property
    def page_ref(self):
        return self.arr("OFF_PAGE_REF", self.h("N_PAGE_REF"), 1)

    @property
    def readouts(self):
        return self.arr("OFF_READOUT", self.h("N_READOUT"), 1)


def make(tree, n_pages=4096, resume=None, pool=None):
    pool = pool or api.PagePool(n_pages)
    R, seg_of = rounds.build_round(tree, pool, resume=resume)
    return R, seg_of, pool, Blob(R.pack().numpy())


def _random_tree(seed):
    """Seeded random forest: 1-3 requests of 1-7 nodes, each node's parent
    drawn among the earlier nodes, lengths around the page (16), tile (128)
    and chunk (64) edges."""
    rng = np.random.default_rng(seed)
    edge = [1, 2, 15, 16, 17, 63, 64, 65, 127, 128, 129]
    reqs = []
    for _ in range(int(rng.integers(1, 4))):
        n = int(rng.integers(1, 8))
        parents = [-1] + [int(rng.integers(0, i)) for i in range(1, n)]
        n_tok = [int(rng.choice(edge)) if rng.random() < 0.6 else int(rng.integers(1, 200)) for _ in range(n)]
        reqs.append(synth.Request(parents=parents, n_tok=n_tok))
    return synth.Tree(reqs)


TREES = [
    synth.Tree([synth.fork_tree(64, [8, 8, 8])]),
    synth.Tree([synth.fork_tree(300, [17, 1, 128, 129]), synth.fork_tree(5, [40, 3])]),
    synth.Tree([synth.fanout_tree(40, 7, 3, 3)]),
    synth.Tree([synth.Request(parents=[-1, 0, 1, 1, 0, 4], n_tok=[33, 20, 5, 100, 9, 2]),
                synth.fork_tree(129, [64, 65, 1])]),
] + [_random_tree(7100 + i) for i in range(16)]


def test_abi_exports_every_declared_symbol():
    hdr = open(__import__("os").path.join(__import__("os").path.dirname(__file__), "..", "include", "hs.h")).read()
    declared = set(re.findall(r"\b(hs_[a-z0-9_]+)\s*\(", hdr))
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (hs_[a-z0-9_]+)$", out, re.M))
    assert declared, "no declarations parsed"
    assert declared <= exported, f"not exported: {sorted(declared - exported)}"
    assert declared <= set(_lib.EXPORTED), f"not bound: {sorted(declared - set(_lib.EXPORTED))}"


@pytest.mark.parametrize("ti", range(len(TREES)))
def test_layout_positions_tokens_match_oracle(ti):
    tree = TREES[ti]
    R, seg_of, pool, B = make(tree)
    lay = layout.stream_layout(tree)
    for (r, i), s in seg_of.items():
        info = R.segment(s)
        assert info.stream_off == lay[(r, i)]
        assert info.pos0 == layout.positions(tree.requests[r])[i]
        assert info.request == r and info.n_tokens == tree.requests[r].n_tok[i]
        assert info.level == layout.depth(tree.requests[r])[i]
    j, c, t, ix = layout.token_metadata(tree)
    node_of = {s: rn for rn, s in seg_of.items()}
    toks = B.toks
    assert B.h("N_TOK") == layout.stream_length(tree)
    for row in range(B.h("N_TOK")):
        r, i = node_of[int(toks[row, 0])]
        assert (r, i, int(toks[row, 1])) == (j[row], c[row], ix[row])


def _phys_of_tokens(R, seg_of, B):
    """(page, row) -> (node, index) for every token the KV write puts in a page."""
    where = {}
    segs = B.segs
    pref = B.page_ref
    for (r, i), s in seg_of.items():
        n = int(segs[s, 1])
        for u in range(n):
            where[(int(pref[int(segs[s, 12]) + u // PAGE]), u % PAGE)] = ((r, i), u)
    return where


@pytest.mark.parametrize("ti", range(len(TREES)))
def test_visible_keys_match_eq3(ti):
    """For every query row: the keys the tiles make visible (shared spans in
    full, own spans up to the row's index for the row's own node) map back
    to exactly the oracle's Eq. 3 set."""
    tree = TREES[ti]
    R, seg_of, pool, B = make(tree)
    where = _phys_of_tokens(R, seg_of, B)
    node_of = {s: rn for rn, s in seg_of.items()}
    toks, spans, tiles, ts, pref = B.toks, B.spans, B.tiles, B.tile_spans, B.page_ref
    covered = np.zeros(B.h("N_TOK"), int)
    for tl in tiles:
        row0, n_rows, soff, n_sh, n_own = (int(x) for x in tl[:5])
        for row in range(row0, row0 + n_rows):
            covered[row] += 1
            seg, idx = int(toks[row, 0]), int(toks[row, 1])
            got = []
            for k in range(n_sh + n_own):
                sp = spans[int(ts[soff + k])]
                off, ntok, owner = int(sp[0]), int(sp[1]), int(sp[2])
                if k < n_sh:
                    nvis = ntok
                else:
                    nvis = idx + 1 if owner == seg else 0
                for key in range(nvis):
                    (rn, u) = where[(int(pref[off + key // PAGE]), key % PAGE)]
                    got.append((rn[1], u))
            r, i = node_of[seg]
            assert sorted(got) == layout.visible_keys(tree, r, i, idx), (row, seg, idx)
    assert (covered == 1).all()


def test_history_spans_and_resume():
    full = synth.Tree([synth.fork_tree(70, [5, 9])])
    pool = api.PagePool(256)
    R0, s0, _, B0 = make(full, pool=pool)
    pages = R0.segment_pages(s0[(0, 0)])
    R0.release(pool, keep=[s0[(0, 0)]])
    assert pool.stats()[1] == len(pages) == 5
    res = synth.Tree([synth.fork_tree(11, [5, 9], hist_len=70)])
    R1, s1, _, B1 = make(res, pool=pool, resume={0: (3, [(70, pages)])})
    assert R1.segment(s1[(0, 0)]).pos0 == 70 and R1.segment(s1[(0, 0)]).init_slot == 3
    assert R1.segment(s1[(0, 1)]).pos0 == 81
    # history pages gained the round's reference
    assert all(pool.refcount(p) == 2 for p in pages)
    # visible keys of the first branch token: history 0..69, root tail 0..10, itself
    toks, spans, tiles, ts = B1.toks, B1.spans, B1.tiles, B1.tile_spans
    row = R1.segment(s1[(0, 1)]).stream_off
    tl = [t for t in tiles if t[0] <= row < t[0] + t[1]][0]
    n_keys = sum(int(spans[int(ts[int(tl[2]) + k])][1]) for k in range(int(tl[3])))
    assert n_keys == 70 + 11
    R1.release(pool)
    assert all(pool.refcount(p) == 1 for p in pages)


@pytest.mark.parametrize("ti", range(len(TREES)))
def test_chunks_slots_readouts(ti):
    """Each node's chunks start at its first token and tile it in 64-token
    steps (Flide section 3.5); a child starts from its parent's end slot;
    inner nodes get distinct temporary slots, leaves none; readout rows are
    the last token of each leaf."""
    tree = TREES[ti]
    R, seg_of, pool, B = make(tree)
    ch = B.chunks
    inner_slots = []
    for (r, i), s in seg_of.items():
        info = R.segment(s)
        mine = [c for c in ch if c[0] == s]
        assert [int(c[3]) for c in mine] == list(range(len(mine)))
        assert [int(c[1]) for c in mine] == [info.stream_off + 64 * k for k in range(len(mine))]
        assert sum(int(c[2]) for c in mine) == info.n_tokens
        assert all(1 <= int(c[2]) <= 64 for c in mine)
        has_child = i in tree.requests[r].parents
        assert (info.end_slot >= 0) == has_child
        if has_child:
            inner_slots.append(info.end_slot)
        p = tree.requests[r].parents[i]
        if p >= 0:
            assert info.init_slot == R.segment(seg_of[(r, p)]).end_slot >= 0
        else:
            assert info.init_slot == -1
        if tree.requests[r].readout[i]:
            assert info.readout_row == info.stream_off + info.n_tokens - 1
    assert list(B.readouts) == [R.segment(s).readout_row for s in sorted(seg_of.values())
                                if R.segment(s).readout_row >= 0]
    assert len(set(inner_slots)) == len(inner_slots)
    assert B.h("N_CHUNK") == sum(-(-n // 64) for req in tree.requests for n in req.n_tok)


def test_scan_group_table():
    """The two-level scan of the GDN state chain: a node of n >= 24 chunks is
    split into G = min(9, n // 12) groups (fixed examples below), listed per
    level as (node, group) pairs for groups 1 .. G-1 in node order, with each
    long node pointing at its group-1 entry; short nodes have one group."""
    expect_groups = {1: 1, 23: 1, 24: 2, 35: 2, 36: 3, 47: 3, 48: 4, 72: 6, 107: 8, 108: 9, 200: 9}
    lens = [47 * 64, 48 * 64 - 10, 72 * 64, 200 * 64, 5]          # the second is 48 chunks (last one short)
    tree = synth.Tree([synth.fork_tree(lens[0], [lens[1], 60]), synth.fork_tree(lens[2], [lens[3]]),
                       synth.fork_tree(lens[4], [7])])
    R, seg_of, pool, B = make(tree, n_pages=8192)
    n_scan, o_scan, o_lev = int(B.w[32]), int(B.w[33]), int(B.w[34])
    table = [tuple(int(v) for v in B.w[o_scan + 2 * k:o_scan + 2 * k + 2]) for k in range(n_scan)]
    segs = B.segs
    expected = []
    levels = int(B.w[8])
    for lev in range(levels):
        assert int(B.w[o_lev + lev]) == len(expected)           # prefix offset of this level
        for s in range(len(segs)):
            if int(segs[s][5]) != lev:
                continue
            n_ch = int(segs[s][10])
            G = expect_groups.get(n_ch, 1 if n_ch < 24 else min(9, n_ch // 12))
            assert int(segs[s][14]) == (len(expected) if G > 1 else -1)
            expected += [(s, g) for g in range(1, G)]
    assert int(B.w[o_lev + levels]) == len(expected)
    assert table == expected
    # the fixed examples are all present
    got = {int(segs[s][10]) for s in range(len(segs))}
    assert {47, 48, 72, 200} <= got
    # group chunk ranges [g n / G, (g+1) n / G) tile each long node exactly, each >= 12 chunks
    for s in range(len(segs)):
        n_ch = int(segs[s][10])
        G = expect_groups.get(n_ch, 1 if n_ch < 24 else min(9, n_ch // 12))
        bounds = [g * n_ch // G for g in range(G + 1)]
        assert bounds[0] == 0 and bounds[-1] == n_ch
        assert all(b - a >= (12 if G > 1 else 1) for a, b in zip(bounds, bounds[1:]))


def test_forkserve_pages_fork_and_commit():
    """ForkServe cost model: 10 sessions x (trunk 256 + 4 x 32), page 16:
    240 pages live at fork; keeping each session's winner (index 0) leaves
    the spine, 10 x (16 + 2) = 180 pages."""
    pool = api.PagePool(1024)
    tree = synth.Tree([synth.fork_tree(256, [32] * 4) for _ in range(10)])
    R, seg_of = rounds.build_round(tree, pool)
    assert pool.stats()[1] == 240
    keep = [seg_of[(r, i)] for r in range(10) for i in (0, 1)]
    R.release(pool, keep=keep)
    assert pool.stats()[1] == 180


def test_deep_tree_pages():
    pool = api.PagePool(4096)
    tree = synth.Tree([synth.fanout_tree(256, 32, 4, 3) for _ in range(10)])
    R, seg_of = rounds.build_round(tree, pool)
    assert pool.stats()[1] == 1840 == layout.live_pages(tree, 16)
    assert R.info().n_tokens == 29440


def test_errors_leave_state_unchanged():
    caps = api.round_caps_for(100, 4, 2)
    R = api.Round(caps)
    with pytest.raises(_lib.HsError) as e:
        R.add_segment(-1, 0)
    assert e.value.code == _lib.HS_EINVAL
    with pytest.raises(_lib.HsError):
        R.add_segment(5, 3)                          # unknown parent
    root = R.add_segment(-1, 60)
    R.add_segment(root, 50)
    pool = api.PagePool(64)
    with pytest.raises(_lib.HsError) as e:
        R.finalize(pool)                             # 110 tokens > 100
    assert e.value.code == _lib.HS_ECAPACITY
    assert pool.stats() == (64, 0)
    # pool exhaustion: nothing allocated
    small = api.PagePool(3)
    R2, _ = None, None
    tree = synth.Tree([synth.fork_tree(40, [8])])
    with pytest.raises(_lib.HsError) as e:
        rounds.build_round(tree, small)
    assert e.value.code == _lib.HS_ENOPAGES and small.stats() == (3, 0)
    # two nodes saving into one slot
    R3 = api.Round(api.round_caps_for(100, 4, 2))
    a = R3.add_segment(-1, 10, save_slot=2)
    R3.add_segment(a, 5, save_slot=2)
    with pytest.raises(_lib.HsError):
        R3.finalize(None, 0, 4)
    # depth above max_levels
    R4 = api.Round(api.round_caps_for(100, 4, 1))
    a = R4.add_segment(-1, 10)
    R4.add_segment(a, 5)
    with pytest.raises(_lib.HsError) as e:
        R4.finalize(None)
    assert e.value.code == _lib.HS_ECAPACITY


def test_device_calls_fail_without_gpu():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    caps = api.round_caps_for(10, 1, 1)
    st = _lib.lib.hs_gdn_state_checkpoint(None, 1, 0, 0, 1, 4, 4, None)
    assert st == _lib.HS_EINVAL
    import ctypes
    buf = (ctypes.c_float * 64)()
    st = _lib.lib.hs_gdn_state_checkpoint(ctypes.cast(buf, ctypes.c_void_p), 2, 0, 1, 1, 4, 4, None)
    assert st == _lib.HS_ECUDA


def test_device_status_codes_map_to_edevice():
    """Every nonzero status word is HS_EDEVICE with a message naming the
    code; zero is HS_OK."""
    import ctypes as C
    assert _lib.lib.hs_check_status(C.byref(C.c_int32(0))) == _lib.HS_OK
    for code, words in [(1, "page"), (2, "slot"), (3, "metadata"), (4, "wait"), (99, "unknown")]:
        assert _lib.lib.hs_check_status(C.byref(C.c_int32(code))) == _lib.HS_EDEVICE
        assert words in _lib.last_error(), (code, _lib.last_error())



def _held_pages(pool, n_tok):
    """Pages of one committed node (n_tok tokens) that stay live in `pool`."""
    R = api.Round(api.round_caps_for(n_tok, 1, 1))
    root = R.add_segment(-1, n_tok)
    R.finalize(pool)
    pages = R.segment_pages(root)
    R.release(pool, keep=[root])
    return pages


def test_finalize_retry_and_release_checks():
    """A finalize that failed (too few temporary slots) and is retried builds
    the same metadata as a first finalize; decref rejects a page listed more
    often than it is referenced; release wants the round's own pool."""
    def make(hist_pages):
        R = api.Round(api.round_caps_for(200, 6, 3, n_hist_spans=2, n_hist_pages=4))
        root = R.add_segment(-1, 40)
        R.attach_history(root, [20, 12], hist_pages)
        R.gdn_state_resume(root, 3, 32)
        mid = R.add_segment(root, 30)
        R.add_segment(mid, 9)
        R.add_segment(mid, 17)
        R.add_segment(root, 5)
        return R
    pool, other = api.PagePool(64), api.PagePool(64)
    held = _held_pages(pool, 40)
    assert held == _held_pages(other, 40) and pool.stats() == (61, 3)
    R0 = make(held)
    R0.finalize(other, 8, 4)
    want = R0.pack().clone()
    R = make(held)
    with pytest.raises(_lib.HsError) as e:
        R.finalize(pool, 8, 1)                       # two inner nodes, one temporary slot
    assert e.value.code == _lib.HS_ECAPACITY
    assert pool.stats() == (61, 3)
    R.finalize(pool, 8, 4)
    assert np.array_equal(R.pack().numpy(), want.numpy())
    with pytest.raises(_lib.HsError):
        R.release(other)                             # not the round's pool
    with pytest.raises(_lib.HsError):
        pool.decref([held[0], held[0], held[0]])     # two references, listed three times
    assert [pool.refcount(p) for p in held] == [2, 2, 2]
    R.release(pool)
    assert [pool.refcount(p) for p in held] == [1, 1, 1] and pool.stats() == (61, 3)
    pool.decref(held)
    assert pool.stats() == (64, 0)
    Rn = api.Round(api.round_caps_for(10, 1, 1))
    Rn.add_segment(-1, 4)
    Rn.finalize(None)
    Rn.release(None)


@pytest.mark.parametrize("seed", range(6))
def test_resumed_rounds_visible_keys_match_eq3(seed):
    """Round A: a random forest; each request keeps one random root-to-leaf
    path (commit).  Round B resumes every request from that path -- its
    pages as history spans, one per kept node -- with a random subtree on
    top.  Every row of round B reaches exactly the Eq. 3 key set of the
    oracle, history included, and the history pages gain and lose the round's
    reference."""
    rng = np.random.default_rng(8000 + seed)
    tree_a = _random_tree(8100 + seed)
    pool = api.PagePool(4096)
    Ra, seg_a, _, _ = make(tree_a, pool=pool)
    keep, hist = [], {}
    for r, req in enumerate(tree_a.requests):
        path = [int(rng.integers(0, req.n_nodes))]
        while req.parents[path[-1]] >= 0:
            path.append(req.parents[path[-1]])
        path.reverse()
        keep += [seg_a[(r, n)] for n in path]
        hist[r] = [(req.n_tok[n], Ra.segment_pages(seg_a[(r, n)])) for n in path]
    Ra.release(pool, keep=keep)
    live = pool.stats()[1]
    reqs_b = []
    for r in range(len(tree_a.requests)):
        sub = _random_tree(8200 + 10 * seed + r).requests[0]
        reqs_b.append(synth.Request(parents=sub.parents, n_tok=sub.n_tok, hist_len=sum(n for n, _ in hist[r])))
    tree_b = synth.Tree(reqs_b)
    Rb, seg_b, _, B = make(tree_b, pool=pool, resume={r: (None, hist[r]) for r in hist})
    assert pool.stats()[1] == live + sum(-(-n // PAGE) for req in reqs_b for n in req.n_tok)
    where = _phys_of_tokens(Rb, seg_b, B)
    for r, spans in hist.items():  # history rows: position u of the kept path
        u = 0
        for n, pages in spans:
            for k in range(n):
                where[(pages[k // PAGE], k % PAGE)] = ((r, -1), u + k)
            u += n
    node_of = {s: rn for rn, s in seg_b.items()}
    toks, sp, ts, pref = B.toks, B.spans, B.tile_spans, B.page_ref
    for tl in B.tiles:
        row0, n_rows, soff, n_sh, n_own = (int(x) for x in tl[:5])
        for row in range(row0, row0 + n_rows):
            seg, idx = int(toks[row, 0]), int(toks[row, 1])
            got = []
            for k in range(n_sh + n_own):
                off, ntok, owner = (int(x) for x in sp[int(ts[soff + k])][:3])
                nvis = ntok if k < n_sh else (idx + 1 if owner == seg else 0)
                for key in range(nvis):
                    (rn, u) = where[(int(pref[off + key // PAGE]), key % PAGE)]
                    got.append((rn[1], u))
            r, i = node_of[seg]
            assert sorted(got) == layout.visible_keys(tree_b, r, i, idx), (seed, row)
    Rb.release(pool)
    assert pool.stats()[1] == live


OFF_PRED, KPRED = 31, 3


@pytest.mark.parametrize("ti", range(len(TREES)))
def test_conv_predecessor_rows(ti):
    """Per token, the stream rows of the kConvTaps - 1 = 3 tokens before it in
    its standalone sequence (Flide section 3.2.2: a node's first tokens read
    their ancestors' last ones); before the sequence start -1, or, for a root
    resumed with a saved conv window w0 (section 3.4), the window row encoded
    as -2 - (w0 + 3 + offset) for the offsets -3..-1 before the root."""
    tree = TREES[ti]
    windows = {}
    if ti % 2:  # resumed roots with a conv window on every other tree
        tree = synth.Tree([synth.Request(parents=q.parents, n_tok=q.n_tok, hist_len=5 + 3 * r)
                           for r, q in enumerate(tree.requests)])
        windows = {r: 7 * r for r in range(len(tree.requests))}
    pool = api.PagePool(4096)
    R, seg_of = rounds.build_round(tree, pool, resume={r: (None, [], w) for r, w in windows.items()})
    words = R.pack().numpy().astype(np.int64)
    pred = words[int(words[OFF_PRED]):][:R.info().n_tokens * KPRED].reshape(-1, KPRED)
    for (r, i), s in seg_of.items():
        req = tree.requests[r]
        pos = layout.positions(req)
        chain = layout.ancestors(req, i) + [i]
        info = R.segment(s)
        for u in range(req.n_tok[i]):
            for k in range(1, KPRED + 1):
                p = pos[i] + u - k
                want = -1
                if p >= req.hist_len:
                    a = [c for c in chain if pos[c] <= p < pos[c] + req.n_tok[c]][0]
                    want = R.segment(seg_of[(r, a)]).stream_off + p - pos[a]
                elif r in windows and p >= req.hist_len - KPRED:
                    want = -2 - (windows[r] + KPRED + (p - req.hist_len))
                assert pred[info.stream_off + u, k - 1] == want, (ti, r, i, u, k)


@pytest.mark.parametrize("ti", range(len(TREES)))
def test_bulk_add_equals_one_by_one(ti):
    """hs_round_add_segments builds, bit for bit, the round that one
    hs_round_add_segment call per node builds."""
    tree = TREES[ti]
    _, _, _, bulk = make(tree)
    n_seg = sum(r.n_nodes for r in tree.requests)
    depth = max(max(layout.depth(r)) for r in tree.requests) + 1
    R = api.Round(api.round_caps_for(sum(sum(r.n_tok) for r in tree.requests), n_seg, depth))
    for req in tree.requests:
        ids = []
        for i in range(req.n_nodes):
            flags = _lib.HS_SEG_READOUT if req.readout[i] else _lib.HS_SEG_NO_READOUT
            ids.append(R.add_segment(-1 if i == 0 else ids[req.parents[i]], req.n_tok[i], flags))
    R.finalize(api.PagePool(4096), 0, n_seg)
    assert np.array_equal(R.pack().numpy(), bulk.w.astype(np.int32))


def test_bulk_add_checks_everything_first():
    R = api.Round(api.round_caps_for(100, 6, 3))
    assert R.add_segments([-1, 0], [10, 5], [0, 0], [-1, -1]) == 0
    for parents, n_tok, flags, saves, code in [
            ([-1, 0, 4], [4, 4, 4], [0, 0, 0], [-1, -1, -1], _lib.HS_EINVAL),   # node 4 its own parent
            ([5, 0], [4, 4], [0, 0], [-1, -1], _lib.HS_EINVAL),                # parent added after it
            ([1, 0], [4, 0], [0, 0], [-1, -1], _lib.HS_EINVAL),                # empty node
            ([0, 0], [4, 4], [0, 8], [-1, -1], _lib.HS_EINVAL),                # unknown flag
            ([0, 0], [4, 4], [0, 0], [-1, -7], _lib.HS_EINVAL),                # bad save slot
            ([-1, 0, 1, 2, 3], [1] * 5, [0] * 5, [-1] * 5, _lib.HS_ECAPACITY)]:  # 7 nodes > 6
        with pytest.raises(_lib.HsError) as e:
            R.add_segments(parents, n_tok, flags, saves)
        assert e.value.code == code
    # nothing of the refused calls was added: the next id is still 2
    assert R.add_segments([1], [3], [0], [-1]) == 2


@pytest.mark.parametrize("ti", range(len(TREES)))
def test_tile_readout_flag(ti):
    """Word 7 of a tile record is 1 exactly when one of the tile's rows is a
    readout row (the attention kernel keeps ~16 bits of P there), and every
    row of the stream lies in exactly one tile."""
    tree = TREES[ti]
    R, seg_of, pool, B = make(tree)
    ro = set(int(x) for x in B.readouts)
    covered = []
    for tl in B.tiles:
        rows = range(int(tl[0]), int(tl[0]) + int(tl[1]))
        covered.extend(rows)
        assert int(tl[7]) == int(any(r in ro for r in rows)), tl
    assert sorted(covered) == list(range(B.h("N_TOK")))


def test_split_at_requests():
    """Rounds cut at request boundaries (Flide section 3.3.2): every group is a run of whole requests in
    order, builds under the bucket's capacities, and the groups cover the batch; a request larger than
    the bucket is refused."""
    tree = synth.mixed_tree(seed=4000)                          # 64 requests, trunks 512 .. 16384
    bucket = api.round_caps_for(40000, 120, 2)
    groups = rounds.split_at_requests(tree, bucket)
    assert [r for g in groups for r in g] == list(range(len(tree.requests)))
    assert len(groups) > 1
    for g in groups:
        sub = synth.Tree([tree.requests[r] for r in g])
        R, _ = rounds.build_round(sub, api.PagePool(sub.useful_tokens() // 16 + 64 * len(g)), caps=bucket)
        assert R.info().n_tokens == sub.useful_tokens()
    # greedy: the next request did not fit into the group before it
    for a, b in zip(groups, groups[1:]):
        sub = synth.Tree([tree.requests[r] for r in a + b[:1]])
        need = api.round_caps_for(sub.useful_tokens(), sum(r.n_nodes for r in sub.requests), 2).as_dict()
        assert any(need[k] > v for k, v in bucket.as_dict().items())
    with pytest.raises(_lib.HsError) as e:
        rounds.split_at_requests(tree, api.round_caps_for(1000, 120, 2))
    assert e.value.code == _lib.HS_ECAPACITY


def test_pool_allocates_lowest_free_pages_ascending():
    """Whatever order rounds release their pages in, the next allocation takes the lowest free ids in
    ascending order, so a node's pages stay consecutive across rounds (ForkServe README, "Copy-on-write
    context tree": pages are reused once nothing references them)."""
    pool = api.PagePool(300)
    tree = synth.Tree([synth.fork_tree(1000, [40, 17, 64])])
    first = None
    for step in range(4):
        R, seg_of = rounds.build_round(tree, pool)
        pages = [list(R.segment_pages(s)) for s in range(R.info().n_segments)]
        flat = [p for ps in pages for p in ps]
        assert flat == sorted(flat) and flat == list(range(len(flat)))  # consecutive from page 0
        if first is None:
            first = pages
        assert pages == first
        R.release(pool)
        assert pool.stats() == (300, 0)
    # interleaved lifetimes: pages freed out of order are handed out lowest first
    R1, _ = rounds.build_round(tree, pool)
    R2, _ = rounds.build_round(tree, pool)
    n1 = pool.stats()[1] // 2
    R1.release(pool)
    R3, _ = rounds.build_round(tree, pool)
    flat3 = [p for s in range(R3.info().n_segments) for p in R3.segment_pages(s)]
    assert flat3 == list(range(n1))
    R2.release(pool)
    R3.release(pool)
    assert pool.stats() == (300, 0)


def test_gate_up_interleave_and_swiglu_gemm_argument_checks():
    """The gate/up weight layout of hs_gemm_bf16_swiglu (per 128 outputs: their gate rows, then their up rows),
    and the entry point's refusals, which it decides before touching a device."""
    import ctypes as C
    from hybrid_serving_gb300.stack import interleave_gate_up
    F, K = 384, 3
    w = np.arange(2 * F * K, dtype=np.float64).reshape(2 * F, K)
    il = interleave_gate_up(w)
    for j in range(F // 128):
        assert np.array_equal(il[256 * j:256 * j + 128], w[128 * j:128 * j + 128])          # gate rows
        assert np.array_equal(il[256 * j + 128:256 * j + 256], w[F + 128 * j:F + 128 * j + 128])  # up rows
    assert sorted(map(tuple, il)) == sorted(map(tuple, w))
    buf = (C.c_uint8 * 4096)()
    p = C.cast(buf, C.c_void_p)
    lib = _lib.lib
    assert lib.hs_gemm_bf16_swiglu(8, 384, 64, p, 64, p, 64, p, 192, None, None) == _lib.HS_EUNSUPPORTED  # N2 % 256
    assert lib.hs_gemm_bf16_swiglu(8, 512, 48, p, 64, p, 64, p, 256, None, None) == _lib.HS_EUNSUPPORTED  # K % 64
    assert lib.hs_gemm_bf16_swiglu(8, 512, 64, None, 64, p, 64, p, 256, None, None) == _lib.HS_EINVAL    # null A
    assert lib.hs_gemm_bf16_swiglu(8, 512, 64, p, 64, p, 64, p, 128, None, None) == _lib.HS_EINVAL       # ldc < N2/2


@pytest.mark.parametrize("seed", range(6))
def test_level_lists_longest_first(seed):
    """Each level's node list (the GDN state pass's task order) holds exactly that level's nodes, by chunk
    count, most first, in stream order among equals."""
    tree = _random_tree(4000 + seed)
    R, seg_of, pool, b = make(tree)
    segs = b.segs
    n_lev = b.h("N_LEVEL")
    lev_off = b.arr("OFF_LEVEL", n_lev + 1, 1)
    lst = b.w[b.h("OFF_LEVEL_SEG"):b.h("OFF_LEVEL_SEG") + b.h("N_SEG")]
    S_STREAM_OFF, S_LEVEL, S_N_CHUNK = 0, 5, 10
    for lev in range(n_lev):
        ids = [int(x) for x in lst[lev_off[lev]:lev_off[lev + 1]]]
        assert sorted(ids) == [i for i in range(b.h("N_SEG")) if segs[i][S_LEVEL] == lev]
        key = [(-int(segs[i][S_N_CHUNK]), int(segs[i][S_STREAM_OFF])) for i in ids]
        assert key == sorted(key), (lev, key)
