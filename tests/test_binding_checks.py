"""The Python binding's tensor checks, on the CPU.

The C ABI takes raw device pointers, so the binding refuses tensors whose
placement, dtype, shape or layout the kernels would misread.  Here the
library's device entry points are replaced by a recorder (the host entry
points stay real) and the device-placement test is bypassed, so that:

  * the test harness's attention and GDN runs and the hybrid stack's whole
    forward pass, driven through their real code, pass every check and
    reach the library with the arguments they always sent;
  * tensors on the host, of another dtype, strided, or short of the round's
    capacity are refused with HS_EINVAL before any library call.
"""
import numpy as np
import pytest
import torch

import synth

api = pytest.importorskip("hybrid_serving_gb300.api")
from hybrid_serving_gb300 import _lib, rounds  # noqa: E402
from hybrid_serving_gb300 import stack as hstack  # noqa: E402

import harness  # noqa: E402

DEVICE_CALLS = {"hs_fork_attn_prefill", "hs_kv_page_write", "hs_fork_attn", "hs_gdn_fork_prefill",
                "hs_gdn_fork_prefill_noalloc", "hs_gdn_state_checkpoint", "hs_choice_logprobs",
                "hs_round_upload", "hs_embed", "hs_rmsnorm", "hs_gemm_bf16", "hs_rope_apply", "hs_gdn_prep",
                "hs_swiglu", "hs_copy_rows", "hs_gemm_bf16_swiglu"}


class Recorder:
    """Stands in for the loaded library: device calls are recorded and succeed,
    everything else goes to the real library."""

    def __init__(self, real):
        self.real = real
        self.calls = []

    def __getattr__(self, name):
        if name in DEVICE_CALLS:
            def call(*args):
                self.calls.append(name)
                return 0
            return call
        return getattr(self.real, name)


@pytest.fixture
def host_run(monkeypatch):
    rec = Recorder(_lib.lib)
    monkeypatch.setattr(api, "lib", rec)
    monkeypatch.setattr(hstack, "lib", rec)
    monkeypatch.setattr(api, "_device_ok", lambda *a: None)
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    monkeypatch.setattr(api, "_stream", lambda stream=None: 0)
    monkeypatch.setattr(hstack, "_s", lambda stream=None: 0)
    monkeypatch.setattr(torch.cuda, "synchronize", lambda *a, **k: None)
    monkeypatch.setattr(harness, "DEV", "cpu")
    monkeypatch.setattr(hstack, "DEV", "cpu")
    return rec


def test_harness_runs_pass_the_checks(host_run):
    tree = synth.Tree([synth.fork_tree(200, [17, 40, 5]), synth.fork_tree(33, [1])])
    for d, dt in ((128, torch.bfloat16), (64, torch.float32)):
        inp = synth.attn_inputs(tree, 8, 2, d, seed=7, bf16=dt == torch.bfloat16)
        harness.AttnRun(tree, inp, dt).run()
        harness.AttnRun(tree, inp, dt, n_pages=64, n_pages_kernel=2).run()
        g = synth.gdn_inputs(tree, 2, d, d, seed=9, bf16=dt == torch.bfloat16, law="softplus")
        harness.GdnRun(tree, g, dt).run()
    assert host_run.calls.count("hs_fork_attn_prefill") == 4
    assert host_run.calls.count("hs_gdn_fork_prefill") == 2


def test_stack_forward_passes_the_checks(host_run):
    dims = dict(hidden=256, pattern="GA", attn_hq=2, attn_hkv=1, head_d=128, gdn_h=2, gdn_d=128, ffn=512,
                vocab=512)
    for wide in (False, True):
        if wide:  # a token mixer output narrower than the other's: its own contiguous view
            dims = dict(dims, attn_hq=4)
        W = synth.stack_weights(dims["hidden"], dims["pattern"], dims["attn_hq"], dims["attn_hkv"],
                                dims["head_d"], dims["gdn_h"], dims["gdn_d"], dims["ffn"], dims["vocab"], seed=1)
        stk = hstack.HybridStack(hstack.StackShape(**dims), W, max_pos=512)
        tree = synth.Tree([synth.fork_tree(40, [5, 7])])
        pool = api.PagePool(64)
        R, seg_of = rounds.build_round(tree, pool, temp_slot0=4, n_temp_slots=4)
        stk.alloc(Tcap=R.info().n_tokens, n_pages=64, n_slots=8)
        meta = torch.empty(R.meta_bytes() // 4, dtype=torch.int32)
        ids = torch.zeros(stk.Tcap, dtype=torch.int32)
        host_run.calls.clear()
        stk.forward(R, meta, ids, R.info().n_readouts)
        assert host_run.calls.count("hs_fork_attn_prefill") == 1
        assert host_run.calls.count("hs_gdn_fork_prefill") == 1
        assert host_run.calls.count("hs_choice_logprobs") == 1
        assert stk.o_attn.is_contiguous() and stk.o_gdn.is_contiguous()
        assert stk.o_attn.shape[1] == dims["attn_hq"] * 128 and stk.o_gdn.shape[1] == dims["gdn_h"] * 128


def _attn_case():
    tree = synth.Tree([synth.fork_tree(40, [5, 7])])
    pool = api.PagePool(16)
    R, _ = rounds.build_round(tree, pool)
    T = R.info().n_tokens
    bf = torch.bfloat16
    t = dict(meta=torch.empty(R.meta_bytes() // 4, dtype=torch.int32), q=torch.zeros((T, 4, 64), dtype=bf),
             k=torch.zeros((T, 2, 64), dtype=bf), v=torch.zeros((T, 2, 64), dtype=bf),
             kp=torch.zeros((2, 16, 16, 64), dtype=bf), vp=torch.zeros((2, 16, 16, 64), dtype=bf),
             out=torch.zeros((T, 4, 64), dtype=bf), st=torch.zeros(1, dtype=torch.int32))
    return R, t


def _call(R, t):
    api.fork_attn_prefill(R.caps, t["meta"], t["q"], t["k"], t["v"], t["kp"], t["vp"], t["out"], t["st"])


@pytest.mark.parametrize("bad", ["float_k", "strided_q", "short_q", "pool_shapes", "short_meta", "head_size"])
def test_misread_tensors_are_refused(host_run, bad):
    R, t = _attn_case()
    _call(R, t)  # the good case goes through
    assert host_run.calls == ["hs_fork_attn_prefill"]
    if bad == "float_k":
        t["k"] = t["k"].float()
    elif bad == "strided_q":
        t["q"] = torch.zeros((t["q"].shape[0], 8, 64), dtype=torch.bfloat16)[:, ::2]
    elif bad == "short_q":
        t["q"], t["out"] = t["q"][:-1], t["out"][:-1]
    elif bad == "pool_shapes":
        t["vp"] = torch.zeros((2, 8, 16, 64), dtype=torch.bfloat16)
    elif bad == "short_meta":
        t["meta"] = t["meta"][:-1]
    elif bad == "head_size":
        t["q"] = torch.zeros((t["q"].shape[0], 4, 128), dtype=torch.bfloat16)
        t["out"] = torch.zeros_like(t["q"])
    with pytest.raises(_lib.HsError) as e:
        _call(R, t)
    assert e.value.code == _lib.HS_EINVAL
    assert host_run.calls == ["hs_fork_attn_prefill"]  # nothing more reached the library


def test_host_tensors_are_refused_without_a_call(monkeypatch):
    rec = Recorder(_lib.lib)
    monkeypatch.setattr(api, "lib", rec)
    R, t = _attn_case()
    with pytest.raises(_lib.HsError) as e:
        _call(R, t)
    assert e.value.code == _lib.HS_EINVAL and "CUDA" in str(e.value)
    assert rec.calls == []
