"""ctypes binding of libhsfork.so (include/hs.h): argument marshalling only.

Every device call goes to the CUDA library; there is no Python or CPU
fallback.  If the library is not built, importing this module raises.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libhsfork.so")

HS_OK, HS_EINVAL, HS_ECAPACITY, HS_EUNSUPPORTED, HS_ECUDA, HS_EDEVICE, HS_ENOPAGES = 0, -1, -2, -3, -4, -5, -6
# device status codes (values of the int32 status word)
HS_DEV_OK, HS_DEV_BAD_PAGE, HS_DEV_BAD_SLOT, HS_DEV_BAD_META, HS_DEV_TIMEOUT = 0, 1, 2, 3, 4
HS_F32, HS_BF16 = 0, 1
HS_SEG_READOUT, HS_SEG_NO_READOUT = 1, 2
_NAMES = {HS_EINVAL: "HS_EINVAL", HS_ECAPACITY: "HS_ECAPACITY", HS_EUNSUPPORTED: "HS_EUNSUPPORTED",
          HS_ECUDA: "HS_ECUDA", HS_EDEVICE: "HS_EDEVICE", HS_ENOPAGES: "HS_ENOPAGES"}


class HsError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_NAMES.get(code, code)}: {msg}")
        self.code = code


class Caps(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("max_tokens", "max_segments", "max_hist_spans", "max_tiles",
                                          "max_tile_spans", "max_chunks", "max_readouts", "max_page_refs",
                                          "max_levels")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class RoundInfo(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("n_tokens", "n_segments", "n_tiles", "n_chunks", "n_readouts",
                                          "n_levels", "n_pages_allocated", "n_spans", "n_tile_spans",
                                          "n_page_refs")]


class SegmentInfo(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("stream_off", "n_tokens", "pos0", "request", "parent", "level",
                                          "init_slot", "end_slot", "readout_row", "n_pages")]


class AttnMask(C.Structure):
    _fields_ = [("window", C.c_int32), ("bidirectional_root", C.c_int32)]


P = C.c_void_p
I32 = C.c_int32
I32P = C.POINTER(C.c_int32)
CAPSP = C.POINTER(Caps)

_SIGS = {
    "hs_round_caps_for": (I32, [I32, I32, I32, I32, I32, I32, CAPSP]),
    "hs_page_pool_create": (I32, [I32, I32, C.POINTER(P)]),
    "hs_page_pool_destroy": (None, [P]),
    "hs_page_pool_stats": (I32, [P, I32P, I32P]),
    "hs_page_pool_refcount": (I32, [P, I32, I32P]),
    "hs_page_pool_decref": (I32, [P, I32P, I32]),
    "hs_round_create": (I32, [CAPSP, C.POINTER(P)]),
    "hs_round_destroy": (None, [P]),
    "hs_round_add_segment": (I32, [P, I32, I32, I32, I32, I32P]),
    "hs_round_add_segments": (I32, [P, I32, I32P, I32P, I32P, I32P, I32P]),
    "hs_gdn_state_resume": (I32, [P, I32, I32, I32]),
    "hs_round_attach_history": (I32, [P, I32, I32, I32P, I32P]),
    "hs_round_finalize": (I32, [P, P, I32, I32]),
    "hs_round_meta_bytes": (C.c_size_t, [CAPSP]),
    "hs_round_pack": (I32, [P, P, C.c_size_t]),
    "hs_round_upload": (I32, [P, P, C.c_size_t, P]),
    "hs_round_get_info": (I32, [P, C.POINTER(RoundInfo)]),
    "hs_round_segment": (I32, [P, I32, C.POINTER(SegmentInfo)]),
    "hs_round_segment_pages": (I32, [P, I32, I32P, I32, I32P]),
    "hs_round_readout_rows": (I32, [P, I32P, I32, I32P]),
    "hs_round_release": (I32, [P, P, I32P, I32]),
    "hs_round_build_chunks": (I32, [CAPSP, P, P, P]),
    "hs_round_build_tiles": (I32, [CAPSP, P, P, P]),
    "hs_fork_attn_masked": (I32, [CAPSP, P, I32, I32, I32, I32, C.c_float, C.POINTER(AttnMask), P, P, P, I32, P,
                                  P, P]),
    "hs_fork_attn_prefill": (I32, [CAPSP, P, I32, I32, I32, I32, C.c_float, P, P, P, P, P, I32, P, P, P]),
    "hs_kv_page_write": (I32, [CAPSP, P, I32, I32, I32, P, P, P, P, I32, P, P]),
    "hs_fork_attn": (I32, [CAPSP, P, I32, I32, I32, I32, C.c_float, P, P, P, I32, P, P, P]),
    "hs_gdn_workspace_bytes": (C.c_size_t, [CAPSP, I32, I32, I32]),
    "hs_gdn_fork_prefill": (I32, [CAPSP, P, I32, I32, I32, I32, I32, P, P, P, P, P, P, I32, P, P, C.c_size_t,
                                  P, P]),
    "hs_gdn_fork_prefill_noalloc": (I32, [CAPSP, P, I32, I32, I32, I32, I32, P, P, P, P, P, P, I32, P, P, P]),
    "hs_gdn_state_checkpoint": (I32, [P, I32, I32, I32, I32, I32, I32, P]),
    "hs_choice_logprobs": (I32, [CAPSP, P, I32, P, C.c_int64, I32, P, I32, P, P, P]),
    "hs_round_set_conv_window": (I32, [P, I32, I32]),
    "hs_gemm_bf16": (I32, [I32, I32, I32, P, C.c_int64, P, C.c_int64, P, C.c_int64, P, C.c_int64, I32, P, P]),
    "hs_gemm_bf16_swiglu": (I32, [I32, I32, I32, P, C.c_int64, P, C.c_int64, P, C.c_int64, P, P]),
    "hs_embed": (I32, [P, I32, P, I32, I32, P, I32, P, P]),
    "hs_rmsnorm": (I32, [P, C.c_int64, I32, I32, I32, P, C.c_float, P, C.c_int64, I32, P]),
    "hs_rope_table": (I32, [P, I32, I32, C.c_double]),
    "hs_rope_apply": (I32, [CAPSP, P, P, C.c_int64, I32, I32, I32, P, I32, P, P]),
    "hs_gdn_prep": (I32, [CAPSP, P, P, C.c_int64, P, C.c_int64, I32, P, I32, I32, P, P, P, P, P, P, P]),
    "hs_swiglu": (I32, [P, C.c_int64, I32, I32, P, C.c_int64, P]),
    "hs_copy_rows": (I32, [P, C.c_int64, P, P, C.c_int64, P, I32, I32, P]),
    "hs_check_status": (I32, [I32P]),
    "hs_debug_wait_timeout": (I32, [C.c_int64, P, P, P]),
    "hs_last_error": (C.c_char_p, []),
    "hs_launch_count": (C.c_int64, []),
    "hs_version": (C.c_char_p, []),
}

EXPORTED = tuple(_SIGS)


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built (build it with hybrid_serving_gb300._build.build())")
    lib = C.CDLL(LIB_PATH)
    for name, (res, args) in _SIGS.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


lib = _load()


def check(code: int):
    if code != HS_OK:
        raise HsError(code, lib.hs_last_error().decode())
    return code


def last_error() -> str:
    return lib.hs_last_error().decode()


def launch_count() -> int:
    return int(lib.hs_launch_count())


def version() -> str:
    return lib.hs_version().decode()
