"""Hybrid attention / Gated DeltaNet stack over a forked round, on the C ABI.

Sequencing and argument marshalling only: every operation is a kernel of
libhsfork.so (tcgen05 GEMMs with the residual fused into the epilogue,
RMSNorm, rotary embedding at standalone positions, the GDN front end with
predecessors across the fork, ForkAttention, Gated DeltaNet fork prefill,
the gate/up GEMM with SwiGLU in its epilogue, option log-probs).  PyTorch
only allocates device memory.

Layer definition (the pages give none; see the oracle for the same text):
pre-norm residual blocks of a token mixer ('A' attention, 'G' Gated
DeltaNet) and a SwiGLU MLP; final RMSNorm; option logits against embedding
rows of the option tokens (Flide section 3.1, Eq. 1).  The residual stream
and the final norm's output are kept in fp32; every other tensor between
operations is stored in bf16 (gates fp32), but the gate/up products enter
SwiGLU straight from the GEMM's fp32 accumulators.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np
import torch

from . import _lib, api
from ._lib import check, lib

DEV = "cuda"


@dataclass
class StackShape:
    hidden: int = 2048
    pattern: str = "GGGAGGGA"
    attn_hq: int = 16
    attn_hkv: int = 4
    head_d: int = 128
    gdn_h: int = 16
    gdn_d: int = 128
    ffn: int = 4096
    vocab: int = 32768
    rope_theta: float = 1e4
    eps: float = 1e-6
    option_ids: List[int] = field(default_factory=lambda: [11, 12, 13, 14])


def _s(stream=None) -> int:
    return (stream or torch.cuda.current_stream()).cuda_stream


def _dt(t) -> int:
    return _lib.HS_F32 if t.dtype == torch.float32 else _lib.HS_BF16


def gemm(A, B, Cout, M: int, R=None, status=None, stream=None):
    """Cout[:M] = A[:M] @ B^T (+ R[:M]) through hs_gemm_bf16 (Cout and R bf16 or fp32)."""
    N, K = B.shape
    check(lib.hs_gemm_bf16(M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), Cout.data_ptr(),
                           Cout.stride(0), R.data_ptr() if R is not None else None,
                           R.stride(0) if R is not None else 0, _dt(Cout), status.data_ptr(), _s(stream)))


def gemm_swiglu(A, B_il, Cout, M: int, status=None, stream=None):
    """Cout[:M] = silu(A[:M] @ Bg^T) * (A[:M] @ Bu^T) through hs_gemm_bf16_swiglu (B_il: the gate and up
    weights interleaved in blocks of 128 rows, see interleave_gate_up)."""
    N2, K = B_il.shape
    check(lib.hs_gemm_bf16_swiglu(M, N2, K, A.data_ptr(), A.stride(0), B_il.data_ptr(), B_il.stride(0),
                                  Cout.data_ptr(), Cout.stride(0), status.data_ptr(), _s(stream)))


def interleave_gate_up(w: np.ndarray) -> np.ndarray:
    """[gate rows; up rows] ([2F, K]) in the row order hs_gemm_bf16_swiglu takes: per block of 128 outputs,
    its 128 gate rows, then its 128 up rows (a weight layout chosen at load time)."""
    F2, K = w.shape
    F = F2 // 2
    assert F2 % 2 == 0 and F % 128 == 0, "ffn must be a multiple of 128"
    return np.ascontiguousarray(w.reshape(2, F // 128, 128, K).transpose(1, 0, 2, 3).reshape(F2, K))


def rmsnorm(x, T: int, dim: int, eps: float, out, stream=None):
    """out[:T] = RMSNorm(x[:T]) with unit weight (x and out bf16 or fp32)."""
    check(lib.hs_rmsnorm(x.data_ptr(), x.stride(0), _dt(x), T, dim, None, eps, out.data_ptr(), out.stride(0),
                         _dt(out), _s(stream)))


class HybridStack:
    def __init__(self, shape: StackShape, weights: Dict[str, np.ndarray], max_pos: int):
        self.sh = shape
        self.W = {k: torch.from_numpy(interleave_gate_up(np.asarray(v)) if k.endswith("wgu")
                                      else np.ascontiguousarray(v)).to(DEV).to(torch.bfloat16)
                  for k, v in weights.items()}
        opt = np.asarray(weights["embed"], np.float32)[list(shape.option_ids)]
        self.opt = torch.from_numpy(np.ascontiguousarray(opt)).to(DEV)
        tab = np.empty((max_pos, shape.head_d // 2, 2), np.float32)
        check(lib.hs_rope_table(tab.ctypes.data, max_pos, shape.head_d, shape.rope_theta))
        self.rope = torch.from_numpy(tab).to(DEV)
        self.max_pos = max_pos
        self.n_attn = shape.pattern.count("A")
        self.n_gdn = shape.pattern.count("G")
        self.status = torch.zeros(1, dtype=torch.int32, device=DEV)

    # ------------------------------------------------------------------ pools
    def alloc(self, Tcap: int, n_pages: int, n_slots: int, n_windows: int = 0, caps=None):
        sh = self.sh
        bf = torch.bfloat16
        self.Tcap = Tcap
        self.h = torch.zeros((Tcap, sh.hidden), dtype=torch.float32, device=DEV)  # residual stream
        self.a = torch.zeros((Tcap, sh.hidden), dtype=bf, device=DEV)             # normed GEMM input
        self.hf = torch.zeros((Tcap, sh.hidden), dtype=torch.float32, device=DEV)  # final norm
        wp_n = max(v.shape[0] for k, v in self.W.items() if k.endswith("wp")) if self.n_gdn else 0
        self.proj = torch.zeros((Tcap, max(wp_n, 8)), dtype=bf, device=DEV)  # the GDN projection
        self.q = torch.zeros((Tcap, sh.attn_hq, sh.head_d), dtype=bf, device=DEV)
        self.k = torch.zeros((Tcap, sh.attn_hkv, sh.head_d), dtype=bf, device=DEV)
        self.v = torch.zeros_like(self.k)
        # token-mixer outputs: one buffer, a contiguous [Tcap, heads * d] view per mixer kind
        wa, wg = sh.attn_hq * sh.head_d, sh.gdn_h * sh.gdn_d
        self.o = torch.zeros(Tcap * max(wa, wg), dtype=bf, device=DEV)
        self.o_attn = self.o[:Tcap * wa].view(Tcap, wa)
        self.o_gdn = self.o[:Tcap * wg].view(Tcap, wg)
        self.gq = torch.zeros((Tcap, sh.gdn_h, sh.gdn_d), dtype=bf, device=DEV)
        self.gk = torch.zeros_like(self.gq)
        self.gv = torch.zeros_like(self.gq)
        self.ga = torch.zeros((Tcap, sh.gdn_h), dtype=torch.float32, device=DEV)
        self.gb = torch.zeros_like(self.ga)
        self.m = torch.zeros((Tcap, sh.ffn), dtype=bf, device=DEV)
        self.kp = [torch.zeros((sh.attn_hkv, n_pages, 16, sh.head_d), dtype=bf, device=DEV) for _ in range(self.n_attn)]
        self.vp = [torch.zeros_like(t) for t in self.kp]
        self.state = [torch.zeros((n_slots, sh.gdn_h, sh.gdn_d, sh.gdn_d), dtype=torch.float32, device=DEV)
                      for _ in range(self.n_gdn)]
        self.win = [torch.zeros((max(n_windows, 1), wp_n), dtype=bf, device=DEV) for _ in range(self.n_gdn)]
        self.n_windows = n_windows
        self.ws = None

    def _ws(self, caps):
        nb = api.gdn_workspace_bytes(caps, self.sh.gdn_h, self.sh.gdn_d, self.sh.gdn_d)
        if self.ws is None or self.ws.numel() < nb:
            self.ws = torch.empty(max(nb, 256), dtype=torch.uint8, device=DEV)
        return self.ws

    # ---------------------------------------------------------------- forward
    def forward(self, R: api.Round, meta: torch.Tensor, ids: torch.Tensor, n_readout: int,
                save_windows: Optional[List[tuple]] = None, stream=None, selective: bool = False):
        """One forked prefill round.  ``ids`` device int32 [Tcap] in stream
        order.  ``save_windows``: [(device src rows int32, device dst rows
        int32, n)] -- after each GDN layer's projection, copy those stream rows
        into the layer's conv-window buffer (a checkpoint's window).
        ``selective`` (Flide section 3.3.3, selective readout): after the last
        layer's token mixer only the readout rows go on -- its MLP, the final
        norm and the option head run on those rows alone (row for row the same
        bits: every step after the mixer works on each row by itself and the
        GEMM's rows do not depend on M); the returned hidden rows are then
        final at the readout rows only.
        Returns (final hidden [T, hidden] fp32 view, option logprobs [n_readout, n_opt])."""
        sh, st = self.sh, self.status
        caps = R.caps
        T = R.info().n_tokens
        s = _s(stream)
        if selective and n_readout > 0:
            ro_rows = torch.tensor(R.readout_rows(), dtype=torch.int32).to(DEV, non_blocking=True)
            ro_idx = torch.arange(n_readout, dtype=torch.int32, device=DEV)
            hr = torch.empty((n_readout, sh.hidden), dtype=torch.float32, device=DEV)
            ar = torch.empty((n_readout, sh.hidden), dtype=torch.bfloat16, device=DEV)
            fr = torch.empty_like(hr)
            mr = torch.empty((n_readout, sh.ffn), dtype=torch.bfloat16, device=DEV)
        last = len(sh.pattern) - 1
        row_bytes = sh.hidden * 4  # (fp32 rows)
        check(lib.hs_embed(ids.data_ptr(), T, self.W["embed"].data_ptr(), sh.vocab, sh.hidden, self.h.data_ptr(),
                           _lib.HS_F32, st.data_ptr(), s))
        ai = gi = 0
        for li, kind in enumerate(sh.pattern):
            p = f"l{li}."
            rmsnorm(self.h, T, sh.hidden, sh.eps, self.a, stream)
            if kind == "A":
                qv = self.q.view(self.Tcap, -1)
                kv = self.k.view(self.Tcap, -1)
                vv = self.v.view(self.Tcap, -1)
                gemm(self.a, self.W[p + "wq"], qv, T, status=st, stream=stream)
                gemm(self.a, self.W[p + "wk"], kv, T, status=st, stream=stream)
                gemm(self.a, self.W[p + "wv"], vv, T, status=st, stream=stream)
                check(lib.hs_rope_apply(C.byref(caps), meta.data_ptr(), qv.data_ptr(), qv.stride(0), 0, sh.attn_hq,
                                        sh.head_d, self.rope.data_ptr(), self.max_pos, st.data_ptr(), s))
                check(lib.hs_rope_apply(C.byref(caps), meta.data_ptr(), kv.data_ptr(), kv.stride(0), 0, sh.attn_hkv,
                                        sh.head_d, self.rope.data_ptr(), self.max_pos, st.data_ptr(), s))
                ov = self.o_attn.view(self.Tcap, sh.attn_hq, sh.head_d)
                api.fork_attn_prefill(caps, meta, self.q, self.k, self.v, self.kp[ai], self.vp[ai], ov, st,
                                      stream=stream)
                gemm(self.o_attn, self.W[p + "wo"], self.h, T, R=self.h, status=st,
                     stream=stream)
                ai += 1
            else:
                wp = self.W[p + "wp"]
                pv = self.proj[:, :wp.shape[0]]
                gemm(self.a, wp, pv, T, status=st, stream=stream)
                if save_windows:
                    for src_rows, dst_rows, n in save_windows:
                        check(lib.hs_copy_rows(pv.data_ptr(), pv.stride(0) * 2, src_rows.data_ptr(),
                                               self.win[gi].data_ptr(), self.win[gi].stride(0) * 2,
                                               dst_rows.data_ptr(), n, wp.shape[0] * 2, s))
                win = self.win[gi] if self.n_windows else None
                check(lib.hs_gdn_prep(C.byref(caps), meta.data_ptr(), pv.data_ptr(), pv.stride(0),
                                      win.data_ptr() if win is not None else None,
                                      win.stride(0) if win is not None else 0, self.n_windows,
                                      self.W[p + "conv"].data_ptr(), sh.gdn_h, sh.gdn_d, self.gq.data_ptr(),
                                      self.gk.data_ptr(), self.gv.data_ptr(), self.ga.data_ptr(), self.gb.data_ptr(),
                                      st.data_ptr(), s))
                ov = self.o_gdn.view(self.Tcap, sh.gdn_h, sh.gdn_d)
                api.gdn_fork_prefill(caps, meta, self.gq, self.gk, self.gv, self.ga, self.gb, self.state[gi], ov,
                                     self._ws(caps), st, stream=stream)
                gemm(self.o_gdn, self.W[p + "wo"], self.h, T, R=self.h, status=st,
                     stream=stream)
                gi += 1
            if selective and li == last and n_readout > 0:
                # the readout rows alone from here on: gather, MLP + final norm, scatter back for the head
                check(lib.hs_copy_rows(self.h.data_ptr(), row_bytes, ro_rows.data_ptr(), hr.data_ptr(), row_bytes,
                                       ro_idx.data_ptr(), n_readout, row_bytes, s))
                rmsnorm(hr, n_readout, sh.hidden, sh.eps, ar, stream)
                gemm_swiglu(ar, self.W[p + "wgu"], mr, n_readout, status=st, stream=stream)
                gemm(mr, self.W[p + "wd"], hr, n_readout, R=hr, status=st, stream=stream)
                rmsnorm(hr, n_readout, sh.hidden, sh.eps, fr, stream)
                check(lib.hs_copy_rows(fr.data_ptr(), row_bytes, ro_idx.data_ptr(), self.hf.data_ptr(), row_bytes,
                                       ro_rows.data_ptr(), n_readout, row_bytes, s))
                break
            rmsnorm(self.h, T, sh.hidden, sh.eps, self.a, stream)
            gemm_swiglu(self.a, self.W[p + "wgu"], self.m, T, status=st, stream=stream)
            gemm(self.m, self.W[p + "wd"], self.h, T, R=self.h, status=st, stream=stream)
        else:
            rmsnorm(self.h, T, sh.hidden, sh.eps, self.hf, stream)
        lp = torch.empty((max(n_readout, 1), len(sh.option_ids)), dtype=torch.float32, device=DEV)
        api.choice_logprobs(caps, meta, self.hf, self.opt, lp, st, stream=stream)
        return self.hf[:T], lp[:n_readout]
