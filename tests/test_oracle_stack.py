"""Pins of the stack oracle's components against mathematical facts.

The pages define no layer, so the stack as a whole is "parity unpinned":
only its parts are pinned here (closed forms and invariants a slip would
break), and its composition is the oracle's own definition.
"""
import math

import numpy as np

import synth
from oracle import stack as ostack


def test_rmsnorm_closed_form_and_scale_invariance():
    x = np.full((2, 8), 3.0)
    np.testing.assert_allclose(ostack.rmsnorm(x, 0.0), 1.0, atol=1e-15)
    rng = np.random.default_rng(0)
    y = rng.standard_normal((3, 16))
    np.testing.assert_allclose(ostack.rmsnorm(7.5 * y, 0.0), ostack.rmsnorm(y, 0.0), atol=1e-14)
    np.testing.assert_allclose(np.mean(ostack.rmsnorm(y, 0.0) ** 2, axis=-1), 1.0, atol=1e-14)


def test_rope_identity_at_zero_rotation_and_relative_position():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, 2, 8))
    np.testing.assert_allclose(ostack.rope(q, [0], 1e4), q, atol=1e-15)
    # d = 2: a plain rotation by the angle p (theta^0 = 1)
    x = np.array([[[1.0, 2.0]]])
    p = 0.7
    want = np.array([math.cos(p) * 1 - math.sin(p) * 2, math.sin(p) * 1 + math.cos(p) * 2])
    np.testing.assert_allclose(ostack.rope(x, [p], 1e4)[0, 0], want, atol=1e-15)
    # norm preserved; <rope(q,m), rope(k,n)> depends on m - n only
    k = rng.standard_normal((1, 2, 8))
    for m, n, s in [(3, 1, 5), (10, 10, 7), (0, 4, 100)]:
        a = (ostack.rope(q, [m], 1e4) * ostack.rope(k, [n], 1e4)).sum(-1)
        b = (ostack.rope(q, [m + s], 1e4) * ostack.rope(k, [n + s], 1e4)).sum(-1)
        np.testing.assert_allclose(a, b, atol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(ostack.rope(q, [37], 1e4), axis=-1), np.linalg.norm(q, axis=-1),
                               atol=1e-13)


def test_causal_conv_delta_kernels_shift():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((6, 3))
    for j in range(4):
        w = np.zeros((3, 4))
        w[:, j] = 1.0
        y = ostack.causal_conv(x, w)
        want = np.zeros_like(x)
        want[j:] = x[:6 - j]
        np.testing.assert_allclose(y, want, atol=0)


def test_silu_softplus_identities():
    x = np.linspace(-6, 6, 25)
    np.testing.assert_allclose(ostack.silu(x) - ostack.silu(-x), x, atol=1e-14)
    np.testing.assert_allclose(ostack.softplus(x) - ostack.softplus(-x), x, atol=1e-14)
    assert ostack.silu(np.array(0.0)) == 0.0


def test_stack_is_causal():
    """A prefix's rows do not depend on later tokens (every mixer is causal)."""
    dims = dict(hidden=128, pattern="GA", attn_hq=1, attn_hkv=1, head_d=128, gdn_h=1, gdn_d=128, ffn=128,
                vocab=64)
    cfg = ostack.StackConfig(**dims)
    W = synth.stack_weights(128, "GA", 1, 1, 128, 1, 128, 128, 64, seed=5)
    ids = np.random.default_rng(3).integers(0, 64, 12)
    full = ostack.forward(cfg, W, ids)
    pre = ostack.forward(cfg, W, ids[:7])
    # identical operations on the prefix rows, up to BLAS blocking of the projections
    assert np.mean(np.abs(full[:7] - pre) <= 1e-2 * np.maximum(1, np.abs(pre))) > 0.99
