"""Pins of the pre/post oracle (oracle/prepost.py) against what the pages
and the mathematics fix: numpy's convolution for ShortConv, closed forms of
Swish / Sigmoid and of both norms, and the conv-state split invariant."""
import math

import numpy as np
import pytest

from oracle import prepost


def _rand(seed, B=1, T=23, H=2, d=8):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, T, 3, H, d))
    w = rng.standard_normal((3, H, d, 4)) * 0.5
    bl = rng.standard_normal((B, T, H))
    return rng, x, w, bl


def test_short_conv_is_causal_convolution():
    """ShortConv of one channel is numpy's full convolution with the taps
    reversed, truncated to the sequence (zero history): v (Swish, no norm)
    equals Swish of that convolution."""
    rng, x, w, _ = _rand(1)
    _, _, v, _, _ = prepost.qkv_prep(x, w)
    for h in range(2):
        for c in range(8):
            xs = x[0, :, 2, h, c]
            ref = np.convolve(xs, w[2, h, c, ::-1])[: len(xs)]
            np.testing.assert_allclose(v[0, :, h, c], ref * (1 / (1 + np.exp(-ref))), rtol=1e-13,
                                       atol=1e-15)


def test_swish_sigmoid_closed_forms():
    assert prepost.swish(np.array(0.0)) == 0.0
    np.testing.assert_allclose(prepost.swish(np.array(1.0)), 1 / (1 + math.exp(-1)), rtol=1e-15)
    np.testing.assert_allclose(prepost.swish(np.array(40.0)), 40.0, rtol=1e-15)
    np.testing.assert_allclose(prepost.swish(np.array(-40.0)), -40.0 * math.exp(-40.0), rtol=1e-12)
    _, x, w, bl = _rand(2)
    bl[0, 0, 0] = 0.0
    _, _, _, beta, _ = prepost.qkv_prep(x, w, bl)
    assert beta[0, 0, 0] == 0.5
    assert np.all((beta > 0) & (beta < 1))


def test_identity_taps_and_l2_norm():
    """Taps (0, 0, 0, 1) make ShortConv the identity: v = Swish(x_v) and
    q = Swish(x_q) / ||Swish(x_q)|| (unit norm up to eps)."""
    _, x, _, _ = _rand(3)
    w = np.zeros((3, 2, 8, 4))
    w[..., 3] = 1.0
    q, k, v, _, _ = prepost.qkv_prep(x, w, l2_eps=0.0)
    np.testing.assert_allclose(v[0], prepost.swish(x[0, :, 2]), rtol=1e-15)
    np.testing.assert_allclose(np.linalg.norm(q, axis=-1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(np.linalg.norm(k, axis=-1), 1.0, rtol=1e-14)
    sq = prepost.swish(x[0, :, 0])
    np.testing.assert_allclose(q[0], sq / np.linalg.norm(sq, axis=-1, keepdims=True), rtol=1e-14)


@pytest.mark.parametrize("cut", [0, 1, 2, 3, 10, 22])
def test_conv_state_split_invariant(cut):
    """Running a sequence in two calls, passing conv_state_out of the first
    as conv_state_in of the second, equals one call."""
    _, x, w, _ = _rand(4)
    full = prepost.qkv_prep(x, w)
    a = prepost.qkv_prep(x[:, :cut], w)
    b = prepost.qkv_prep(x[:, cut:], w, conv_state_in=a[4])
    for i in range(3):
        np.testing.assert_allclose(np.concatenate([a[i], b[i]], axis=1), full[i], rtol=1e-14,
                                   atol=1e-15)
    np.testing.assert_allclose(b[4], full[4], rtol=0, atol=0)


def test_conv_state_out_holds_last_three_rows():
    _, x, w, _ = _rand(5, T=7)
    st_in = np.random.default_rng(9).standard_normal((1, 3, 3, 2, 8))
    *_, st = prepost.qkv_prep(x, w, conv_state_in=st_in)
    np.testing.assert_array_equal(st[0], x[0, -3:])
    *_, st2 = prepost.qkv_prep(x[:, :1], w, conv_state_in=st_in)    # shorter than three
    np.testing.assert_array_equal(st2[0, :2], st_in[0, 1:])
    np.testing.assert_array_equal(st2[0, 2], x[0, 0])


def test_varlen_sequences_are_convolved_separately():
    _, x, w, bl = _rand(6, T=30)
    cu = np.array([0, 5, 5, 18, 30])
    packed = prepost.qkv_prep(x, w, bl, cu_seqlens=cu)
    for n in range(4):
        s, e = cu[n], cu[n + 1]
        one = prepost.qkv_prep(x[:, s:e], w, bl[:, s:e])
        for i in range(4):
            np.testing.assert_allclose(packed[i][:, s:e], one[i], rtol=1e-15, atol=0)
        np.testing.assert_allclose(packed[4][n], one[4][0], rtol=0, atol=0)


def test_output_gate_closed_forms():
    """Gate -> +inf (Sigmoid = 1) and unit weight: the mean square of y is
    ms / (ms + eps); gate = 0 halves it; the weight scales channels."""
    rng = np.random.default_rng(7)
    o = rng.standard_normal((5, 16))
    ms = (o * o).mean(-1)
    y = prepost.output_gate(o, np.full_like(o, 60.0), eps=1e-5)
    np.testing.assert_allclose((y * y).mean(-1), ms / (ms + 1e-5), rtol=1e-12)
    y0 = prepost.output_gate(o, np.zeros_like(o), eps=1e-5)
    np.testing.assert_allclose(y0, 0.5 * y, rtol=1e-12)
    wgt = rng.uniform(0.5, 2.0, 16)
    yw = prepost.output_gate(o, np.full_like(o, 60.0), wgt, eps=1e-5)
    np.testing.assert_allclose(yw, y * wgt, rtol=1e-12)
