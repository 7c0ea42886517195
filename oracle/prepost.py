"""Oracle of the passes around the KDA operator -- TEST INFRASTRUCTURE ONLY.

Plain fp64 numpy, one token at a time.  Only ``tests/``, the smoke check and
the benchmark's CPU-baseline leg may use it; the CUDA library shares no code
with it.

Sources ("Kimi K3：从三条信息流到完整系统", wineandchord.com):

* §从投影到 Chunkwise 的完整接口, eq. (2):
  ``q, k = L2Norm(Swish(ShortConv(W x)))``, ``v = Swish(ShortConv(W_v x))``,
  ``beta = Sigmoid(W_beta x)``.
* §下界 log-decay 是一个 kernel 设计, eq. (6):
  ``y = W_o [Sigmoid(W_g x) * RMSNorm(o)]`` -- the bracket is computed here.
* The model's config values quoted in §模型账本与公开边界: short_conv_kernel_size
  = 4, rms_norm_eps = 1e-5.

Readings where the pages give no formula (the CUDA library takes the same):
ShortConv is the causal depthwise convolution ``y_t = sum_i w[i] x_{t-3+i}``
per channel, no bias, zero (or the caller's saved state) before a
sequence's first token; Swish(x) = x * Sigmoid(x); L2Norm divides a head's
d channels by ``sqrt(sum x^2 + l2_eps)`` with l2_eps = 1e-6; RMSNorm divides
a head's d channels by ``sqrt(mean x^2 + eps)`` and multiplies by a
per-channel weight shared by the heads.

Parity status: pinned by ``tests/test_oracle_prepost.py`` (the convolution
against numpy's convolve, closed forms of Swish, Sigmoid, the norms, and
the conv-state split invariant).
"""
from __future__ import annotations

import numpy as np

CONV_TAPS = 4


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu")
        if x.dtype == torch.bfloat16:
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def swish(x):
    return x * sigmoid(x)


def qkv_prep(x_qkv, conv_w, beta_logit=None, cu_seqlens=None, conv_state_in=None,
             l2_eps: float = 1e-6):
    """eq. (2) after the projections.

    x_qkv [B, T, 3, H, d]; conv_w [3, H, d, 4] (tap 3 multiplies x_t);
    beta_logit [B, T, H] or None; cu_seqlens [N+1] (then B == 1) or None;
    conv_state_in [N, 3, 3, H, d] (the three x rows before each sequence,
    oldest first) or None (zeros).
    Returns (q, k, v [B, T, H, d], beta [B, T, H] or None,
    conv_state_out [N, 3, 3, H, d]) in fp64.
    """
    x = _f64(x_qkv)
    w = _f64(conv_w)
    B, T, _, H, d = x.shape
    flat = x.reshape(B * T, 3, H, d)
    if cu_seqlens is None:
        cu = np.arange(B + 1) * T
    else:
        cu = np.asarray(_f64(cu_seqlens), dtype=np.int64)
        assert B == 1
    N = len(cu) - 1
    st_in = np.zeros((N, 3, 3, H, d)) if conv_state_in is None else _f64(conv_state_in)
    y = np.zeros((B * T, 3, H, d))
    st_out = np.zeros((N, 3, 3, H, d))
    for n in range(N):
        bos, eos = int(cu[n]), int(cu[n + 1])
        hist = [st_in[n, j] for j in range(3)]          # x_{bos-3}, x_{bos-2}, x_{bos-1}
        for t in range(bos, eos):
            window = hist[-3:] + [flat[t]]
            acc = np.zeros((3, H, d))
            for i in range(CONV_TAPS):
                acc += w[..., i] * window[i]
            y[t] = swish(acc)
            hist.append(flat[t])
        for j in range(3):
            st_out[n, j] = hist[-3 + j]
    y = y.reshape(B, T, 3, H, d)
    q, k, v = y[:, :, 0], y[:, :, 1], y[:, :, 2]
    q = q / np.sqrt((q * q).sum(-1, keepdims=True) + l2_eps)
    k = k / np.sqrt((k * k).sum(-1, keepdims=True) + l2_eps)
    beta = None if beta_logit is None else sigmoid(_f64(beta_logit))
    return q, k, v, beta, st_out


def output_gate(o, gate, norm_w=None, eps: float = 1e-5):
    """eq. (6)'s bracket, row-wise over the last axis: Sigmoid(gate) *
    o / sqrt(mean(o^2) + eps) * norm_w."""
    o = _f64(o)
    g = _f64(gate)
    w = np.ones(o.shape[-1]) if norm_w is None else _f64(norm_w)
    rms = np.sqrt((o * o).mean(-1, keepdims=True) + eps)
    return sigmoid(g) * (o / rms * w)
