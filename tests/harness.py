"""GPU test harness: runs a tree through the C ABI and returns per-node
outputs as float64 numpy arrays (no oracle code here)."""
from __future__ import annotations

import numpy as np
import torch

from hybrid_serving_gb300 import api, rounds

DEV = "cuda:0"


def _dev(a: np.ndarray, dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(DEV).to(dtype)


def _zeros_status():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


class AttnRun:
    """Upload a tree, run hs_fork_attn_prefill, keep the pools for reuse."""

    def __init__(self, tree, inp, dtype=torch.bfloat16, n_pages=None, pool=None, k_pages=None, v_pages=None,
                 resume=None, n_pages_kernel=None):
        self.tree, self.inp, self.dtype = tree, inp, dtype
        T = sum(sum(r.n_tok) for r in tree.requests)
        if pool is None:
            n_pages = n_pages or (T // 16 + sum(r.n_nodes for r in tree.requests) + 16)
            pool = api.PagePool(n_pages)
            k_pages = torch.zeros((inp.hkv, n_pages, 16, inp.d), dtype=dtype, device=DEV)
            v_pages = torch.zeros_like(k_pages)
        self.pool, self.k_pages, self.v_pages = pool, k_pages, v_pages
        self.R, self.seg_of = rounds.build_round(tree, pool, resume=resume)
        self.meta = torch.empty(self.R.meta_bytes() // 4, dtype=torch.int32, device=DEV)
        self.R.upload(self.meta)
        self.q = _dev(rounds.to_stream(self.R, self.seg_of, inp.nodes, "q"), dtype)
        self.k = _dev(rounds.to_stream(self.R, self.seg_of, inp.nodes, "k"), dtype)
        self.v = _dev(rounds.to_stream(self.R, self.seg_of, inp.nodes, "v"), dtype)
        self.out = torch.full_like(self.q, float("nan"))
        self.status = _zeros_status()
        self.n_pages_kernel = n_pages_kernel

    def run(self, scale=None):
        kp, vp = self.k_pages, self.v_pages
        if self.n_pages_kernel is not None:  # a smaller pool than the pages the round allocated
            kp = self.k_pages[:, : self.n_pages_kernel].contiguous()
            vp = self.v_pages[:, : self.n_pages_kernel].contiguous()
        api.fork_attn_prefill(self.R.caps, self.meta, self.q, self.k, self.v, kp, vp, self.out,
                              self.status, scale=scale)
        torch.cuda.synchronize()
        return self

    def run_masked(self, window=0, bidirectional_root=False):
        """Page write, then the attention with a mask (hs_fork_attn_masked)."""
        api.kv_page_write(self.R.caps, self.meta, self.k, self.v, self.k_pages, self.v_pages, self.status)
        api.fork_attn(self.R.caps, self.meta, self.q, self.k_pages, self.v_pages, self.out, self.status,
                      window=window, bidirectional_root=bidirectional_root)
        torch.cuda.synchronize()
        return self

    def outputs(self):
        o = self.out.float().cpu().numpy().astype(np.float64)
        return rounds.from_stream(self.R, self.seg_of, o)

    def raw_outputs(self):
        o = self.out.cpu()
        return rounds.from_stream(self.R, self.seg_of, o)


class GdnRun:
    def __init__(self, tree, inp, dtype=torch.bfloat16, state_pool=None, n_slots=None, temp_slot0=None,
                 resume=None, n_temp=None):
        self.tree, self.inp, self.dtype = tree, inp, dtype
        n_seg = sum(r.n_nodes for r in tree.requests)
        if state_pool is None:
            n_slots = n_slots or (n_seg + 8)
            state_pool = torch.zeros((n_slots, inp.h, inp.dv, inp.dk), dtype=torch.float32, device=DEV)
        self.state = state_pool
        t0 = temp_slot0 if temp_slot0 is not None else 8
        n_temp = n_temp if n_temp is not None else max(0, state_pool.shape[0] - t0)
        self.R, self.seg_of = rounds.build_round(tree, None, temp_slot0=t0, n_temp_slots=n_temp, resume=resume)
        self.meta = torch.empty(self.R.meta_bytes() // 4, dtype=torch.int32, device=DEV)
        self.R.upload(self.meta)
        st = lambda key, dt: _dev(rounds.to_stream(self.R, self.seg_of, inp.nodes, key), dt)  # noqa: E731
        self.q, self.k, self.v = st("q", dtype), st("k", dtype), st("v", dtype)
        self.alpha, self.beta = st("alpha", torch.float32), st("beta", torch.float32)
        self.out = torch.full((self.q.shape[0], inp.h, inp.dv), float("nan"), dtype=dtype, device=DEV)
        nb = api.gdn_workspace_bytes(self.R.caps, inp.h, inp.dk, inp.dv)
        self.ws = torch.empty(max(nb, 256), dtype=torch.uint8, device=DEV)
        self.status = _zeros_status()

    def run(self):
        api.gdn_fork_prefill(self.R.caps, self.meta, self.q, self.k, self.v, self.alpha, self.beta, self.state,
                             self.out, self.ws, self.status)
        torch.cuda.synchronize()
        return self

    def outputs(self):
        o = self.out.float().cpu().numpy().astype(np.float64)
        return rounds.from_stream(self.R, self.seg_of, o)

    def raw_outputs(self):
        return rounds.from_stream(self.R, self.seg_of, self.out.cpu())


def max_abs(a: dict, b: dict, keys=None) -> float:
    keys = keys or a.keys()
    return max(float(np.max(np.abs(np.asarray(a[k], np.float64) - np.asarray(b[k], np.float64)))) for k in keys)
