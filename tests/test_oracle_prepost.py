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


# ----------------------------------------------------------------- planted mistakes

def _prep_mutant(kind):
    """Plausible wrong restatements of eq. (2)'s tail, to show the pins above
    catch them (same signature as prepost.qkv_prep)."""
    def qkv_prep(x_qkv, conv_w, beta_logit=None, cu_seqlens=None, conv_state_in=None, l2_eps=1e-6):
        x = prepost._f64(x_qkv)
        w = prepost._f64(conv_w)
        B, T, _, H, d = x.shape
        flat = x.reshape(B * T, 3, H, d)
        cu = np.arange(B + 1) * T if cu_seqlens is None else np.asarray(prepost._f64(cu_seqlens), dtype=np.int64)
        N = len(cu) - 1
        st_in = np.zeros((N, 3, 3, H, d)) if conv_state_in is None else prepost._f64(conv_state_in)
        y = np.zeros((B * T, 3, H, d))
        st_out = np.zeros((N, 3, 3, H, d))
        carry = None
        for n in range(N):
            bos, eos = int(cu[n]), int(cu[n + 1])
            hist = [st_in[n, j] for j in range(3)]
            if kind == "history_across_sequences" and carry is not None:
                hist = carry
            for t in range(bos, eos):
                window = hist[-3:] + [flat[t]]
                if kind == "taps_reversed":
                    window = window[::-1]
                acc = sum(w[..., i] * window[i] for i in range(4))
                y[t] = acc if kind == "no_swish" else prepost.swish(acc)
                hist = hist + [flat[t]]
            carry = hist
            for j in range(3):
                st_out[n, j] = hist[-1 - j] if kind == "state_newest_first" else hist[-3 + j]
        y = y.reshape(B, T, 3, H, d)
        q, k, v = y[:, :, 0], y[:, :, 1], y[:, :, 2]
        axis = -2 if kind == "norm_over_heads" else -1
        q = q / np.sqrt((q * q).sum(axis, keepdims=True) + l2_eps)
        k = k / np.sqrt((k * k).sum(axis, keepdims=True) + l2_eps)
        if kind == "norm_v":
            v = v / np.sqrt((v * v).sum(-1, keepdims=True) + l2_eps)
        beta = None if beta_logit is None else prepost.sigmoid(prepost._f64(beta_logit))
        return q, k, v, beta, st_out
    return qkv_prep


def _gate_mutant(kind):
    def output_gate(o, gate, norm_w=None, eps=1e-5):
        o = prepost._f64(o)
        g = prepost._f64(gate)
        w = np.ones(o.shape[-1]) if norm_w is None else prepost._f64(norm_w)
        if kind == "mean_not_rms":
            den = np.abs(o.mean(-1, keepdims=True)) + eps
        else:
            den = np.sqrt((o * o).mean(-1, keepdims=True) + eps)
        act = prepost.swish(g) if kind == "swish_gate" else prepost.sigmoid(g)
        return act * (o / den * w)
    return output_gate


def _prep_pins_pass():
    try:
        test_short_conv_is_causal_convolution()
        test_identity_taps_and_l2_norm()
        for cut in (0, 1, 2, 3, 10, 22):
            test_conv_state_split_invariant(cut)
        test_conv_state_out_holds_last_three_rows()
        test_varlen_sequences_are_convolved_separately()
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("kind", ["taps_reversed", "no_swish", "norm_over_heads", "norm_v",
                                  "state_newest_first", "history_across_sequences"])
def test_prep_pins_catch_planted_mistakes(kind, monkeypatch):
    """Every mutant of the prep oracle fails at least one pin above, while the
    oracle itself passes them all."""
    assert _prep_pins_pass()
    monkeypatch.setattr(prepost, "qkv_prep", _prep_mutant(kind))
    assert not _prep_pins_pass()


def test_prep_mutant_without_mistake_passes(monkeypatch):
    """The mutant factory with no planted mistake is the oracle again (so the
    failures above come from the planted mistakes alone)."""
    monkeypatch.setattr(prepost, "qkv_prep", _prep_mutant("none"))
    assert _prep_pins_pass()


@pytest.mark.parametrize("kind", ["mean_not_rms", "swish_gate"])
def test_gate_pins_catch_planted_mistakes(kind, monkeypatch):
    test_output_gate_closed_forms()
    monkeypatch.setattr(prepost, "output_gate", _gate_mutant(kind))
    with pytest.raises(AssertionError):
        test_output_gate_closed_forms()
