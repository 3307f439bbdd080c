"""A hybrid attention / Gated DeltaNet stack over ONE isolated sequence, fp64.

Test infrastructure only.

PARITY UNPINNED as a whole: the pages never define the layer of their
hybrid models, so the composition below is this oracle's own definition;
only its components are pinned (tests/test_oracle_stack.py) and the
mixers it calls (attention, gdn) are pinned on their own.  The definition taken here: pre-norm residual blocks, each a token
mixer followed by a SwiGLU MLP.

* RMSNorm: x / sqrt(mean(x^2) + eps), weight one.
* Attention mixer: q, k, v = x Wq^T, x Wk^T, x Wv^T; rotate-half rotary
  embedding of q and k at the token's position in its standalone sequence
  (Flide section 3.2: positions of a question continue from its state);
  causal attention with scale 1/sqrt(d) (Flex, section 2, Eq. 1), grouped
  query heads; output projection; residual.
* Gated DeltaNet mixer: p = x Wp^T holds q | k | v | a | b; q, k, v go
  through a depthwise causal convolution of 4 taps (y_t = sum_k w[ch][k]
  x_{t-k}, zero before the sequence; Flide section 3.2.2: a short causal
  convolution in front of the rule), SiLU, L2 normalisation of each q and k
  head; alpha = exp(-0.1 softplus(a)), beta = sigmoid(b); the gated delta
  rule (Eq. 4); output projection; residual.
* MLP: silu(x Wg^T) * (x Wu^T), down projection, residual.
* Readout: final RMSNorm; option log-probabilities against the embedding
  rows of the option tokens (Flide section 3.1, Eq. 1).

The model keeps its residual stream and the final norm's output in fp32 and
stores every other tensor between operations in bf16 (the gates in fp32);
the gate and up projections go into SwiGLU unrounded (the library applies
SwiGLU to the fp32 accumulators of the projection that forms them):
the oracle computes each operation in fp64 and rounds its stored result to
the same precision at the same points, so that it defines the model itself.

``forward(..., gemm_dtype=np.float32)`` runs the projections in fp32 instead:
the "reference library in lower precision" of Flide's Appendix G forward
test (an fp32 forward against fp64), which measures how far rounding alone
moves a bf16 stack; a port must stay within twice that distance.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List

import numpy as np

from . import attention as _attn
from . import gdn as _gdn
from .numerics import round_bf16, round_f32


@dataclass
class StackConfig:
    hidden: int = 2048
    pattern: str = "GGGAGGGA"
    attn_hq: int = 16
    attn_hkv: int = 4
    head_d: int = 128
    gdn_h: int = 16
    gdn_d: int = 128
    ffn: int = 4096
    vocab: int = 32768
    taps: int = 4
    rope_theta: float = 1e4
    eps: float = 1e-6
    option_ids: List[int] = field(default_factory=lambda: [11, 12, 13, 14])


def rmsnorm(x, eps):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def rope(x, pos, theta):
    """x [n, heads, d]; rotate-half at positions pos [n]."""
    d = x.shape[-1]
    half = d // 2
    inv = theta ** (-2.0 * np.arange(half) / d)
    ang = np.asarray(pos, np.float64)[:, None] * inv[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def silu(x):
    return x / (1.0 + np.exp(-x))


def softplus(x):
    return np.log1p(np.exp(-np.abs(x))) + np.maximum(x, 0.0)


def causal_conv(x, w):
    """x [n, C]; w [C, taps]: y_t = sum_k w[:, k] x_{t-k} (zero before the start)."""
    n = x.shape[0]
    y = np.zeros_like(x, dtype=np.float64)
    for k in range(w.shape[1]):
        if k < n:
            y[k:] += w[:, k][None, :] * x[:n - k]
    return y


def forward(cfg: StackConfig, W: Dict[str, np.ndarray], ids, rows=None, gemm_dtype=np.float64):
    """Run the stack over one isolated token sequence (positions 0..n-1).

    Returns the final-norm hidden rows (fp32 values, fp64 dtype) for
    ``rows`` (default all).
    """
    def mm(a, w):
        return (np.asarray(a, gemm_dtype) @ np.asarray(w, gemm_dtype).T).astype(np.float64)

    ids = np.asarray(ids)
    n = len(ids)
    pos = np.arange(n)
    E = np.asarray(W["embed"], np.float64)
    h = E[ids]
    for li, kind in enumerate(cfg.pattern):
        p = f"l{li}."
        a = round_bf16(rmsnorm(h, cfg.eps))
        if kind == "A":
            hq, hkv, d = cfg.attn_hq, cfg.attn_hkv, cfg.head_d
            q = round_bf16(mm(a, W[p + "wq"])).reshape(n, hq, d)
            k = round_bf16(mm(a, W[p + "wk"])).reshape(n, hkv, d)
            v = round_bf16(mm(a, W[p + "wv"])).reshape(n, hkv, d)
            q = round_bf16(rope(q, pos, cfg.rope_theta))
            k = round_bf16(rope(k, pos, cfg.rope_theta))
            o = round_bf16(_attn.causal_attention(q, k, v, 1.0 / np.sqrt(d)))
            h = round_f32(h + mm(o.reshape(n, hq * d), W[p + "wo"]))
        else:
            H, d = cfg.gdn_h, cfg.gdn_d
            C = 3 * H * d
            pr = round_bf16(mm(a, W[p + "wp"]))
            y = silu(causal_conv(pr[:, :C], np.asarray(W[p + "conv"], np.float64)))
            q = y[:, :H * d].reshape(n, H, d)
            kk = y[:, H * d:2 * H * d].reshape(n, H, d)
            v = round_bf16(y[:, 2 * H * d:].reshape(n, H, d))
            q = round_bf16(q / np.sqrt((q * q).sum(-1, keepdims=True) + 1e-6))
            kk = round_bf16(kk / np.sqrt((kk * kk).sum(-1, keepdims=True) + 1e-6))
            al = round_f32(np.exp(-0.1 * softplus(pr[:, C:C + H])))
            be = round_f32(1.0 / (1.0 + np.exp(-pr[:, C + H:C + 2 * H])))
            o, _ = _gdn.gated_delta_rule(q, kk, v, al, be)
            o = round_bf16(o)
            h = round_f32(h + mm(o.reshape(n, H * d), W[p + "wo"]))
        b = round_bf16(rmsnorm(h, cfg.eps))
        gu = mm(b, W[p + "wgu"])
        F = cfg.ffn
        m = round_bf16(silu(gu[:, :F]) * gu[:, F:])
        h = round_f32(h + mm(m, W[p + "wd"]))
    out = round_f32(rmsnorm(h, cfg.eps))
    return out if rows is None else out[list(rows)]


def option_logprobs(cfg: StackConfig, W, hidden_rows):
    from .choice import option_logprobs as _olp
    opt = np.asarray(W["embed"], np.float64)[list(cfg.option_ids)]
    return _olp(hidden_rows, opt)
