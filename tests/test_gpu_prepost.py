"""Parity of the pre/post passes (kda_qkv_prep, kda_output_gate, through the
C ABI) with the fp64 oracle in oracle/prepost.py.

Bar: per element, |gpu - oracle| <= 2 ulp of the output format at the exact
value (bf16) or 64 fp32 ulp (the fp32 path's fast sigmoid and reciprocal
square root), plus 1e-6 RMS for terms that cancel to near zero.  These
passes are one rounding of a short fp32 computation (no long accumulation),
so the operator's 2e-2 / 1e-4 RMS bound would be far too loose for them.
"""
import numpy as np
import pytest
import torch

from gated_delta_rule_11_gb300 import inputs, kda
from gated_delta_rule_11_gb300 import build as kbuild
from oracle import prepost
from tests._parity import assert_elementwise

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kda.load_library()


def _ulps(t):
    return 2.0 if t.dtype == torch.bfloat16 else 64.0


def _cu(seqlens):
    return torch.tensor(np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32), device="cuda")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("with_state", [False, True])
def test_prep_small_varlen(dtype, d, with_state):
    seqlens = (1, 2, 3, 17, 64, 65, 0, 130)
    T, H = sum(seqlens), 3
    inp = inputs.make_prep_inputs(T, H, d, dtype, device="cuda", seed=d + with_state,
                                  N_state=len(seqlens) if with_state else 0)
    cu = _cu(seqlens)
    q, k, v, beta, st = kda.kda_qkv_prep(inp["x_qkv"], inp["conv_w"], inp["beta_logit"], cu,
                                         inp["conv_state"], output_conv_state=True)
    torch.cuda.synchronize()
    rq, rk, rv, rb, rst = prepost.qkv_prep(inp["x_qkv"], inp["conv_w"], inp["beta_logit"],
                                           cu.cpu().numpy(), inp["conv_state"])
    assert_elementwise("q", q, rq, ulps=_ulps(q))
    assert_elementwise("k", k, rk, ulps=_ulps(k))
    assert_elementwise("v", v, rv, ulps=_ulps(v))
    assert_elementwise("beta", beta, rb, ulps=_ulps(beta))
    assert torch.equal(st.float().cpu(), torch.from_numpy(rst).float())   # states are copies


def test_prep_split_equals_unsplit_bit_for_bit():
    H, d, T = 4, 128, 200
    inp = inputs.make_prep_inputs(T, H, d, "bf16", device="cuda", seed=11)
    x, w = inp["x_qkv"], inp["conv_w"]
    full = kda.kda_qkv_prep(x, w, output_conv_state=True)
    for cut in (1, 3, 64, 137):
        a = kda.kda_qkv_prep(x[:, :cut].contiguous(), w, output_conv_state=True)
        b = kda.kda_qkv_prep(x[:, cut:].contiguous(), w, None, None, a[4], output_conv_state=True)
        for i in range(3):
            assert torch.equal(torch.cat([a[i], b[i]], dim=1), full[i]), (cut, i)
        assert torch.equal(b[4], full[4])


def test_prep_decode_one_token_per_sequence():
    """Decode: each of N sequences brings one token and its conv state."""
    N, H, d = 9, 2, 128
    inp = inputs.make_prep_inputs(N, H, d, "bf16", device="cuda", seed=12, N_state=N)
    cu = torch.arange(N + 1, dtype=torch.int32, device="cuda")
    q, k, v, beta, st = kda.kda_qkv_prep(inp["x_qkv"], inp["conv_w"], inp["beta_logit"], cu,
                                         inp["conv_state"], output_conv_state=True)
    torch.cuda.synchronize()
    rq, rk, rv, rb, rst = prepost.qkv_prep(inp["x_qkv"], inp["conv_w"], inp["beta_logit"],
                                           np.arange(N + 1), inp["conv_state"])
    for name, g, r in (("q", q, rq), ("k", k, rk), ("v", v, rv), ("beta", beta, rb)):
        assert_elementwise(name, g, r, ulps=_ulps(g))
    assert torch.equal(st.float().cpu(), torch.from_numpy(rst).float())


def test_prep_empty_sequences_pass_state_through():
    H, d = 2, 64
    inp = inputs.make_prep_inputs(5, H, d, "f32", device="cuda", seed=13, N_state=3)
    cu = torch.tensor([0, 0, 5, 5], dtype=torch.int32, device="cuda")
    *_, st = kda.kda_qkv_prep(inp["x_qkv"], inp["conv_w"], None, cu, inp["conv_state"],
                              output_conv_state=True)
    torch.cuda.synchronize()
    assert torch.equal(st[0], inp["conv_state"][0]) and torch.equal(st[2], inp["conv_state"][2])
    *_, st0 = kda.kda_qkv_prep(inp["x_qkv"], inp["conv_w"], None, cu, None, output_conv_state=True)
    torch.cuda.synchronize()
    assert torch.count_nonzero(st0[0]) == 0 and torch.count_nonzero(st0[2]) == 0


def test_prep_varlen_workload_sampled():
    """The packed 131072 + 65536 + 32768 + 8192 tokens, H = 96, d = 128 bf16:
    full GPU pass, oracle on windows around sequence starts, ends and middles
    for sampled heads (each window run as its own sequence from the three
    rows before it)."""
    w = inputs.WORKLOADS["varlen_bf16_H96_237568"]
    T, H, d = w.total_tokens, w.H, w.dk
    inp = inputs.make_prep_inputs(T, H, d, "bf16", device="cuda", seed=14)
    cu = _cu(w.seqlens)
    q, k, v, beta, st = kda.kda_qkv_prep(inp["x_qkv"], inp["conv_w"], inp["beta_logit"], cu,
                                         output_conv_state=True)
    torch.cuda.synchronize()
    bounds = cu.cpu().tolist()
    hs = [0, 50, 95]
    x = inp["x_qkv"][:, :, :, hs]
    wt = inp["conv_w"][:, hs]
    for n in range(len(w.seqlens)):
        bos, eos = bounds[n], bounds[n + 1]
        for s in (bos, bos + 61, (bos + eos) // 2, eos - 40):
            e = min(s + 40, eos)
            prev = x[:, max(bos, s - 3):s][0]
            hist = torch.zeros((3, 3, len(hs), d), dtype=x.dtype, device="cuda")
            if prev.shape[0]:
                hist[3 - prev.shape[0]:] = prev
            rq, rk, rv, rb, _ = prepost.qkv_prep(x[:, s:e], wt, inp["beta_logit"][:, s:e][:, :, hs],
                                                 None, hist[None])
            assert_elementwise(f"q[{s}:{e}]", q[:, s:e][:, :, hs], rq, ulps=2.0)
            assert_elementwise(f"k[{s}:{e}]", k[:, s:e][:, :, hs], rk, ulps=2.0)
            assert_elementwise(f"v[{s}:{e}]", v[:, s:e][:, :, hs], rv, ulps=2.0)
            assert_elementwise(f"beta[{s}:{e}]", beta[:, s:e][:, :, hs], rb, ulps=2.0)
        assert torch.equal(st[n], inp["x_qkv"][0, eos - 3:eos])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("rows", [1, 5, 1003])
def test_output_gate(dtype, d, rows):
    inp = inputs.make_post_inputs(rows, d, dtype, device="cuda", seed=rows + d)
    y = kda.kda_output_gate(inp["o"], inp["gate"], inp["norm_w"])
    y1 = kda.kda_output_gate(inp["o"], inp["gate"], None, eps=1e-3)
    torch.cuda.synchronize()
    assert_elementwise("y", y, prepost.output_gate(inp["o"], inp["gate"], inp["norm_w"]), ulps=_ulps(y))
    assert_elementwise("y (unit weight, eps 1e-3)", y1,
                       prepost.output_gate(inp["o"], inp["gate"], None, eps=1e-3), ulps=_ulps(y1))


def test_output_gate_workload_sampled():
    """[237568 tokens x 96 heads, 128] bf16 rows: full pass, oracle on
    sampled rows."""
    rows = inputs.WORKLOADS["varlen_bf16_H96_237568"].total_tokens * 96
    inp = inputs.make_post_inputs(rows, 128, "bf16", device="cuda", seed=15)
    y = kda.kda_output_gate(inp["o"], inp["gate"], inp["norm_w"])
    torch.cuda.synchronize()
    idx = torch.tensor(sorted(set(np.random.default_rng(0).integers(0, rows, 4000).tolist()) | {0, rows - 1}),
                       device="cuda")
    ref = prepost.output_gate(inp["o"][idx], inp["gate"][idx], inp["norm_w"])
    assert_elementwise("y sampled", y[idx], ref, ulps=_ulps(y[idx]))


def test_no_device_wait_gave_up():
    kda.check_device_status()
