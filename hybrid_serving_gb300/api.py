"""Python face of the C ABI (include/hs.h), same names without the ``hs_``
prefix.  Argument marshalling only: tensors are passed as device pointers,
shapes are read off the tensors, every step runs in libhsfork.so.

Device memory and streams come from PyTorch; nothing here computes.
"""
from __future__ import annotations

import ctypes as C
import math
from typing import Optional, Sequence

import torch

from . import _lib
from ._lib import Caps, HsError, RoundInfo, SegmentInfo, check, lib

PAGE = 16
CHUNK = 64


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return _lib.HS_BF16
    if t.dtype == torch.float32:
        return _lib.HS_F32
    raise HsError(_lib.HS_EUNSUPPORTED, f"dtype {t.dtype}")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need(cond: bool, msg: str, *args):
    # the message is formatted only on failure: these checks run on every call of the hot path
    if not cond:
        raise HsError(_lib.HS_EINVAL, msg.format(*args))


def _cur_dev() -> int:
    try:
        return torch.cuda.current_device()
    except (RuntimeError, AssertionError):  # no usable CUDA: every device tensor check then fails
        return -1


def _device_ok(name: str, t: torch.Tensor, dev: int):
    if not t.is_cuda:
        _need(False, "{} must be a CUDA tensor", name)
    if t.get_device() != dev:
        _need(False, "{} is on {}, not the current device cuda:{}", name, t.device, dev)


def _on_device(name: str, t, dev: int, dtype=None, dim: Optional[int] = None, contiguous: bool = True):
    """The C ABI takes raw device pointers with the layouts hs.h documents, so a
    host tensor, another dtype or a strided view would be misread: refuse them."""
    if not isinstance(t, torch.Tensor):
        _need(False, "{} must be a tensor", name)
    _device_ok(name, t, dev)
    if dtype is not None and t.dtype != dtype:
        _need(False, "{} must be {} (got {})", name, dtype, t.dtype)
    if dim is not None and t.dim() != dim:
        _need(False, "{} must have {} dimensions (got shape {})", name, dim, tuple(t.shape))
    if contiguous and not t.is_contiguous():
        _need(False, "{} must be contiguous", name)


def _meta_status(caps: Caps, dev_meta, dev_status, dev: int):
    _on_device("dev_meta", dev_meta, dev, torch.int32)
    _need(dev_meta.numel() * 4 >= lib.hs_round_meta_bytes(C.byref(caps)), "dev_meta is smaller than the caps' metadata")
    _on_device("dev_status", dev_status, dev, torch.int32)
    _need(dev_status.numel() >= 1, "dev_status needs one int32")


def _rows(name: str, t, caps: Caps):
    if t.shape[0] < caps.max_tokens:
        _need(False, "{} has {} rows < caps.max_tokens = {}", name, t.shape[0], caps.max_tokens)


def _check_pages(caps, dev_meta, dev_status, dt, k_new, v_new, k_pages, v_pages, dev):
    _meta_status(caps, dev_meta, dev_status, dev)
    _on_device("k_pages", k_pages, dev, dt, 4)
    _on_device("v_pages", v_pages, dev, dt, 4)
    if k_pages.shape != v_pages.shape or k_pages.shape[2] != PAGE:
        _need(False, "k_pages {} and v_pages {} must both be [hkv, n_pages, 16, d]", tuple(k_pages.shape),
              tuple(v_pages.shape))
    if k_new is not None:
        _on_device("k_new", k_new, dev, dt, 3)
        _on_device("v_new", v_new, dev, dt, 3)
        _rows("k_new", k_new, caps)
        ks = k_new.shape
        if ks != v_new.shape or ks[1] != k_pages.shape[0] or ks[2] != k_pages.shape[3]:
            _need(False, "k_new/v_new {} do not match the pools' [hkv, ., ., d]", tuple(ks))


def _check_attn(caps, q, out, k_pages, dt, dev):
    _on_device("q", q, dev, dt, 3)
    _on_device("out", out, dev, dt, 3)
    _rows("q", q, caps)
    if out.shape != q.shape:
        _need(False, "out {} must match q {}", tuple(out.shape), tuple(q.shape))
    _need(q.shape[2] == k_pages.shape[3], "q and the pools differ in head size")


def _i32arr(xs: Sequence[int]):
    return (C.c_int32 * max(1, len(xs)))(*xs)


def round_caps_for(n_tokens: int, n_segments: int, n_levels: int, n_hist_spans: int = 0,
                   n_hist_pages: int = 0, page_size: int = PAGE) -> Caps:
    c = Caps()
    check(lib.hs_round_caps_for(n_tokens, n_segments, n_levels, n_hist_spans, n_hist_pages, page_size,
                                C.byref(c)))
    return c


class PagePool:
    """Host bookkeeping of a caller-owned KV page pool (refcounted pages)."""

    def __init__(self, n_pages: int, page_size: int = PAGE):
        self._h = C.c_void_p()
        check(lib.hs_page_pool_create(n_pages, page_size, C.byref(self._h)))
        self.n_pages = n_pages
        self.page_size = page_size

    def __del__(self):
        if getattr(self, "_h", None):
            lib.hs_page_pool_destroy(self._h)
            self._h = None

    def stats(self):
        f, l = C.c_int32(), C.c_int32()
        check(lib.hs_page_pool_stats(self._h, C.byref(f), C.byref(l)))
        return f.value, l.value

    def refcount(self, page: int) -> int:
        r = C.c_int32()
        check(lib.hs_page_pool_refcount(self._h, page, C.byref(r)))
        return r.value

    def decref(self, pages: Sequence[int]):
        check(lib.hs_page_pool_decref(self._h, _i32arr(pages), len(pages)))


class Round:
    """A round of request trees flattened into one stream (hs_round)."""

    def __init__(self, caps: Caps):
        self.caps = caps
        self._h = C.c_void_p()
        check(lib.hs_round_create(C.byref(caps), C.byref(self._h)))

    def __del__(self):
        if getattr(self, "_h", None):
            lib.hs_round_destroy(self._h)
            self._h = None

    def add_segment(self, parent: int, n_tokens: int, flags: int = 0, save_slot: int = -1) -> int:
        s = C.c_int32()
        check(lib.hs_round_add_segment(self._h, parent, n_tokens, flags, save_slot, C.byref(s)))
        return s.value

    def add_segments(self, parents: Sequence[int], n_tokens: Sequence[int], flags: Sequence[int],
                     save_slots: Sequence[int]) -> int:
        """Adds len(parents) nodes in one call; returns the first new node id."""
        first = C.c_int32()
        n = len(parents)
        check(lib.hs_round_add_segments(self._h, n, _i32arr(parents), _i32arr(n_tokens), _i32arr(flags),
                                        _i32arr(save_slots), C.byref(first)))
        return first.value

    def gdn_state_resume(self, seg: int, ckpt_slot: int, ckpt_pos: int):
        check(lib.hs_gdn_state_resume(self._h, seg, ckpt_slot, ckpt_pos))

    def set_conv_window(self, seg: int, window_row0: int):
        check(lib.hs_round_set_conv_window(self._h, seg, window_row0))

    def attach_history(self, seg: int, ntok: Sequence[int], pages: Sequence[int]):
        check(lib.hs_round_attach_history(self._h, seg, len(ntok), _i32arr(ntok), _i32arr(pages)))

    def finalize(self, pool: Optional[PagePool], temp_slot0: int = 0, n_temp_slots: int = 0):
        check(lib.hs_round_finalize(self._h, pool._h if pool is not None else None, temp_slot0, n_temp_slots))

    def meta_bytes(self) -> int:
        return int(lib.hs_round_meta_bytes(C.byref(self.caps)))

    def pack(self, out: "torch.Tensor" = None) -> "torch.Tensor":
        """The metadata blob in host memory; `out` (int32, contiguous, e.g. a
        pinned buffer for an asynchronous upload) receives it if given."""
        n = self.meta_bytes()
        if out is None:
            out = torch.empty(n // 4, dtype=torch.int32)
        if out.device.type != "cpu" or not out.is_contiguous() or out.numel() * 4 < n:
            raise ValueError("pack needs a contiguous host int32 tensor of at least meta_bytes()/4 words")
        check(lib.hs_round_pack(self._h, out.data_ptr(), n))
        return out

    def upload(self, dev_meta: torch.Tensor, stream=None):
        check(lib.hs_round_upload(self._h, dev_meta.data_ptr(), dev_meta.numel() * dev_meta.element_size(),
                                  _stream(stream)))

    def info(self) -> RoundInfo:
        i = RoundInfo()
        check(lib.hs_round_get_info(self._h, C.byref(i)))
        return i

    def segment(self, seg: int) -> SegmentInfo:
        s = SegmentInfo()
        check(lib.hs_round_segment(self._h, seg, C.byref(s)))
        return s

    def segment_pages(self, seg: int):
        n = C.c_int32()
        check(lib.hs_round_segment_pages(self._h, seg, None, 0, C.byref(n)))
        buf = (C.c_int32 * max(1, n.value))()
        check(lib.hs_round_segment_pages(self._h, seg, buf, n.value, C.byref(n)))
        return list(buf[:n.value])

    def readout_rows(self):
        n = C.c_int32()
        check(lib.hs_round_readout_rows(self._h, None, 0, C.byref(n)))
        buf = (C.c_int32 * max(1, n.value))()
        check(lib.hs_round_readout_rows(self._h, buf, n.value, C.byref(n)))
        return list(buf[:n.value])

    def release(self, pool: Optional[PagePool], keep: Sequence[int] = ()):
        check(lib.hs_round_release(self._h, pool._h if pool is not None else None, _i32arr(keep), len(keep)))


# ---------------------------------------------------------------------------
# hot path
# ---------------------------------------------------------------------------
def fork_attn_prefill(caps: Caps, dev_meta: torch.Tensor, q, k_new, v_new, k_pages, v_pages, out,
                      dev_status: torch.Tensor, scale: Optional[float] = None, stream=None):
    """q [T,hq,d], k_new/v_new [T,hkv,d], k_pages/v_pages [hkv,n_pages,16,d], out [T,hq,d]."""
    dt = _dt(q)
    dev = _cur_dev()
    _check_pages(caps, dev_meta, dev_status, q.dtype, k_new, v_new, k_pages, v_pages, dev)
    _check_attn(caps, q, out, k_pages, q.dtype, dev)
    T, hq, d = q.shape
    hkv = k_new.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    check(lib.hs_fork_attn_prefill(C.byref(caps), dev_meta.data_ptr(), dt, hq, hkv, d, scale, q.data_ptr(),
                                   k_new.data_ptr(), v_new.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
                                   k_pages.shape[1], out.data_ptr(), dev_status.data_ptr(), _stream(stream)))


def round_build_chunks(caps: Caps, dev_meta: torch.Tensor, dev_status: torch.Tensor, stream=None):
    """Rebuild the GDN chunk list of the round in dev_meta on the GPU (hs_round_build_chunks)."""
    dev = _cur_dev()
    _meta_status(caps, dev_meta, dev_status, dev)
    check(lib.hs_round_build_chunks(C.byref(caps), dev_meta.data_ptr(), dev_status.data_ptr(), _stream(stream)))


def round_build_tiles(caps: Caps, dev_meta: torch.Tensor, dev_status: torch.Tensor, stream=None):
    """Rebuild the attention tile table of the round in dev_meta on the GPU (hs_round_build_tiles)."""
    dev = _cur_dev()
    _meta_status(caps, dev_meta, dev_status, dev)
    check(lib.hs_round_build_tiles(C.byref(caps), dev_meta.data_ptr(), dev_status.data_ptr(), _stream(stream)))


def kv_page_write(caps: Caps, dev_meta: torch.Tensor, k_new, v_new, k_pages, v_pages, dev_status: torch.Tensor,
                  stream=None):
    _dt(k_new)
    _check_pages(caps, dev_meta, dev_status, k_new.dtype, k_new, v_new, k_pages, v_pages,
                 _cur_dev())
    T, hkv, d = k_new.shape
    check(lib.hs_kv_page_write(C.byref(caps), dev_meta.data_ptr(), _dt(k_new), hkv, d, k_new.data_ptr(),
                               v_new.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), k_pages.shape[1],
                               dev_status.data_ptr(), _stream(stream)))


def fork_attn(caps: Caps, dev_meta: torch.Tensor, q, k_pages, v_pages, out, dev_status: torch.Tensor,
              scale: Optional[float] = None, stream=None, window: int = 0, bidirectional_root: bool = False):
    """hs_fork_attn; a sliding ``window`` or ``bidirectional_root`` goes through hs_fork_attn_masked."""
    _dt(q)
    dev = _cur_dev()
    _check_pages(caps, dev_meta, dev_status, q.dtype, None, None, k_pages, v_pages, dev)
    _check_attn(caps, q, out, k_pages, q.dtype, dev)
    T, hq, d = q.shape
    hkv = k_pages.shape[0]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if window or bidirectional_root:
        mask = _lib.AttnMask(int(window), int(bool(bidirectional_root)))
        check(lib.hs_fork_attn_masked(C.byref(caps), dev_meta.data_ptr(), _dt(q), hq, hkv, d, scale, C.byref(mask),
                                      q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), k_pages.shape[1],
                                      out.data_ptr(), dev_status.data_ptr(), _stream(stream)))
        return
    check(lib.hs_fork_attn(C.byref(caps), dev_meta.data_ptr(), _dt(q), hq, hkv, d, scale, q.data_ptr(),
                           k_pages.data_ptr(), v_pages.data_ptr(), k_pages.shape[1], out.data_ptr(),
                           dev_status.data_ptr(), _stream(stream)))


def gdn_workspace_bytes(caps: Caps, h: int, dk: int, dv: int) -> int:
    return int(lib.hs_gdn_workspace_bytes(C.byref(caps), h, dk, dv))


def _check_gdn(caps, dev_meta, dev_status, q, k, v, alpha, beta, state_pool, out, dev):
    dt = q.dtype
    _dt(q)
    _meta_status(caps, dev_meta, dev_status, dev)
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        _on_device(name, t, dev, dt, 3)
        _rows(name, t, caps)
    if k.shape != q.shape:
        _need(False, "k {} must match q {}", tuple(k.shape), tuple(q.shape))
    _need(v.shape[1] == q.shape[1] and out.shape[1:] == v.shape[1:], "v and out must be [Tcap, h, dv]")
    for name, t in (("alpha", alpha), ("beta", beta)):
        _on_device(name, t, dev, torch.float32, 2)
        _rows(name, t, caps)
        _need(t.shape[1] == q.shape[1], "{} must be [Tcap, h]", name)
    _on_device("state_pool", state_pool, dev, torch.float32, 4)
    ss = state_pool.shape
    if ss[1] != q.shape[1] or ss[2] != v.shape[2] or ss[3] != q.shape[2]:
        _need(False, "state_pool {} must be [n_slots, h, dv, dk]", tuple(ss))


def gdn_fork_prefill(caps: Caps, dev_meta: torch.Tensor, q, k, v, alpha, beta, state_pool, out, ws,
                     dev_status: torch.Tensor, chunk: int = CHUNK, stream=None):
    """q,k [T,h,dk], v [T,h,dv], alpha,beta [T,h] fp32, state_pool [slots,h,dv,dk] fp32, out [T,h,dv]."""
    dev = _cur_dev()
    _check_gdn(caps, dev_meta, dev_status, q, k, v, alpha, beta, state_pool, out, dev)
    _on_device("ws", ws, dev)
    T, h, dk = q.shape
    dv = v.shape[2]
    check(lib.hs_gdn_fork_prefill(C.byref(caps), dev_meta.data_ptr(), _dt(q), h, dk, dv, chunk, q.data_ptr(),
                                  k.data_ptr(), v.data_ptr(), alpha.data_ptr(), beta.data_ptr(),
                                  state_pool.data_ptr(), state_pool.shape[0], out.data_ptr(), ws.data_ptr(),
                                  ws.numel() * ws.element_size(), dev_status.data_ptr(), _stream(stream)))


def gdn_fork_prefill_noalloc(caps: Caps, dev_meta: torch.Tensor, q, k, v, alpha, beta, state_pool, out,
                             dev_status: torch.Tensor, chunk: int = CHUNK, stream=None):
    """hs_gdn_fork_prefill without a workspace argument: for callers that
    cannot allocate device memory (the library's built-in scratch is used)."""
    _check_gdn(caps, dev_meta, dev_status, q, k, v, alpha, beta, state_pool, out, _cur_dev())
    T, h, dk = q.shape
    dv = v.shape[2]
    check(lib.hs_gdn_fork_prefill_noalloc(C.byref(caps), dev_meta.data_ptr(), _dt(q), h, dk, dv, chunk,
                                          q.data_ptr(), k.data_ptr(), v.data_ptr(), alpha.data_ptr(),
                                          beta.data_ptr(), state_pool.data_ptr(), state_pool.shape[0],
                                          out.data_ptr(), dev_status.data_ptr(), _stream(stream)))


def gdn_state_checkpoint(state_pool, src_slot: int, dst_slot: int, stream=None):
    _on_device("state_pool", state_pool, _cur_dev(), torch.float32, 4)
    n, h, dv, dk = state_pool.shape
    check(lib.hs_gdn_state_checkpoint(state_pool.data_ptr(), n, src_slot, dst_slot, h, dk, dv, _stream(stream)))


def choice_logprobs(caps: Caps, dev_meta: torch.Tensor, hidden, option_rows, logprobs,
                    dev_status: torch.Tensor, stream=None):
    """hidden [T, dim] (a strided 2-D view is fine), option_rows [n_opt, dim] fp32, logprobs [n_ro, n_opt]."""
    _dt(hidden)
    dev = _cur_dev()
    _meta_status(caps, dev_meta, dev_status, dev)
    _on_device("hidden", hidden, dev, hidden.dtype, 2, contiguous=False)
    _need(hidden.stride(1) == 1, "hidden rows must be contiguous")
    _rows("hidden", hidden, caps)
    _on_device("option_rows", option_rows, dev, torch.float32, 2)
    _need(option_rows.shape[1] == hidden.shape[1], "option_rows must be [n_opt, hidden_dim]")
    _on_device("logprobs", logprobs, dev, torch.float32, 2)
    _need(logprobs.shape[1] == option_rows.shape[0], "logprobs must be [n_readouts, n_opt]")
    dim = hidden.shape[1]
    check(lib.hs_choice_logprobs(C.byref(caps), dev_meta.data_ptr(), _dt(hidden), hidden.data_ptr(),
                                 hidden.stride(0), dim, option_rows.data_ptr(), option_rows.shape[0],
                                 logprobs.data_ptr(), dev_status.data_ptr(), _stream(stream)))


def check_status(dev_status: torch.Tensor):
    w = C.c_int32(int(dev_status.item()))
    check(lib.hs_check_status(C.byref(w)))


def debug_wait_timeout(wait_cycles: int, dev_status: torch.Tensor, dev_elapsed: Optional[torch.Tensor] = None,
                       stream=None):
    """Run the bounded-wait failure path on purpose (hs_debug_wait_timeout): the status word receives
    HS_DEV_TIMEOUT and dev_elapsed (int64[2]) the clocks each of the two waits lasted."""
    dev = _cur_dev()
    _on_device("dev_status", dev_status, dev, torch.int32)
    _need(dev_status.numel() >= 1, "dev_status needs one int32")
    if dev_elapsed is not None:
        _on_device("dev_elapsed", dev_elapsed, dev, torch.int64)
        _need(dev_elapsed.numel() >= 2, "dev_elapsed needs two int64")
    check(lib.hs_debug_wait_timeout(int(wait_cycles), dev_status.data_ptr(), _ptr(dev_elapsed), _stream(stream)))
