"""Parity of the segment-split prefill (kda_chunk_fwd_split, through the C
ABI) with the fp64 oracle on the same seeded inputs.

Each sequence is cut into segments that run at the same time; segments 1..
are corrected with the composed entering state.  Bar as the prefill's:
max|gpu - oracle| <= 2e-2 * RMS(oracle) for out and final_state (bf16
inputs, fp32 state).  Cases span several segments with ragged last
segments, packed sequences that are empty, shorter than one segment or one
tile, every gate map, A_log and scale, and the full 12-head 131,072-token
shape on sampled heads.
"""
import numpy as np
import pytest
import torch

from gated_delta_rule_11_gb300 import inputs, kda
from gated_delta_rule_11_gb300 import build as kbuild
from tests._parity import TOL, assert_close, oracle_heads

pytestmark = pytest.mark.gpu
TOL16 = TOL[torch.bfloat16]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kda.load_library()


def _w(H, B=1, T=0, seqlens=(), s0_std=0.1, seed=0, z_std=2.0):
    return inputs.Workload("split", "prefill", H=H, dk=128, dv=128, dtype="bf16", z_std=z_std,
                           s0_std=s0_std, seed=seed, B=B, T=T, seqlens=tuple(seqlens))


def _split_vs_oracle(w, tau, heads=None, gate_mode="bounded", gate_per_head=False, **kw):
    inp = inputs.make_prefill_inputs(w, device="cuda")
    g = inp["g_raw"]
    if gate_per_head:
        g = g[..., 0].contiguous()
    args = (inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["init_state"], inp["cu_seqlens"])
    out, fin = kda.kda_chunk_fwd_split(*args, segment_tokens=tau, gate_mode=gate_mode,
                                       gate_per_head=gate_per_head, **kw)
    torch.cuda.synchronize()
    hs = list(range(w.H)) if heads is None else list(heads)
    ref_inp = dict(inp)
    ref_inp["g_raw"] = g
    okw = {}
    if gate_mode != "bounded" or gate_per_head:
        okw = {"gate_mode": gate_mode, "gate_scalar": gate_per_head}
    ref_out, ref_fin = oracle_heads(ref_inp, hs, A_log=kw.get("A_log"), scale=kw.get("scale", 1.0),
                                    **okw)
    assert_close(f"split out (tau {tau})", out[:, :, hs], ref_out, TOL16)
    assert_close(f"split final_state (tau {tau})", fin[:, hs], ref_fin, TOL16)
    return inp, out, fin


@pytest.mark.parametrize("B,T,seqlens,tau", [
    (1, 1000, (), 256),        # four segments, the last ragged (232 tokens)
    (2, 300, (), 64),          # five segments per sequence, two sequences
    (1, 0, (0, 17, 300, 1000, 33, 16), 128),   # packed: empty, shorter than a tile / segment
    (1, 512, (), 16),          # one tile per segment: 32 segments
])
def test_split_matches_oracle(B, T, seqlens, tau):
    _split_vs_oracle(_w(2, B=B, T=T, seqlens=seqlens, seed=T + tau + len(seqlens)), tau)


def test_split_with_head_log_scale_and_query_scale():
    w = _w(3, B=1, T=700, seed=21)
    _split_vs_oracle(w, 160, A_log=torch.tensor([0.0, 0.5, -0.7], device="cuda"),
                     scale=128 ** -0.5)


@pytest.mark.parametrize("gate_mode,per_head", [("neg_softplus", False), ("log_decay", False),
                                                ("bounded", True), ("none", False)])
def test_split_every_gate_map(gate_mode, per_head):
    w = _w(2, B=1, T=600, seed=22, z_std=1.0)
    if gate_mode == "log_decay":
        # a log-decay input must be <= 0: use -|z| / 4 drawn from the same seed
        inp = inputs.make_prefill_inputs(w, device="cuda")
        g = -(inp["g_raw"].float().abs() * 0.25).to(torch.bfloat16)
        args = (inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["init_state"])
        out, fin = kda.kda_chunk_fwd_split(*args, segment_tokens=144, gate_mode="log_decay")
        torch.cuda.synchronize()
        ref_inp = dict(inp)
        ref_inp["g_raw"] = g
        ro, rf = oracle_heads(ref_inp, [0, 1], gate_mode="log_decay")
        assert_close("split out (log_decay)", out, ro, TOL16)
        assert_close("split final_state (log_decay)", fin, rf, TOL16)
        return
    _split_vs_oracle(w, 144, gate_mode=gate_mode, gate_per_head=per_head)


def test_split_equals_unsplit_within_tolerance_on_a_layer_slice():
    """12 heads of the 8192-token layer: split (automatic segment length) and
    unsplit runs against the oracle on sampled heads."""
    w = _w(12, B=1, T=8192, s0_std=0.0, seed=2)
    inp = inputs.make_prefill_inputs(w, device="cuda")
    args = (inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], None)
    tau = kda.split_segment_tokens(1, 8192, 12, 1, False,
                                   torch.cuda.get_device_properties(0).multi_processor_count)
    assert tau > 0 and tau % 16 == 0
    o_s, f_s = kda.kda_chunk_fwd_split(*args)
    o_u, f_u = kda.kda_chunk_fwd(*args)
    torch.cuda.synchronize()
    hs = [0, 7, 11]
    ro, rf = oracle_heads(inp, hs)
    assert_close("split out (layer slice)", o_s[:, :, hs], ro, TOL16)
    assert_close("split final (layer slice)", f_s[:, hs], rf, TOL16)
    assert_close("unsplit out (layer slice)", o_u[:, :, hs], ro, TOL16)


@pytest.mark.slow
def test_tp8_workload_sampled_heads():
    """B=1, H=12, T=131072 (the 96-head layer sharded 8 ways by head): the
    split launch the benchmark times, oracle on two heads."""
    w = inputs.WORKLOADS["tp8_bf16_H12_T131072"]
    inp = inputs.make_prefill_inputs(w, device="cuda")
    args = (inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], None)
    out, fin = kda.kda_chunk_fwd_split(*args)
    torch.cuda.synchronize()
    hs = [0, 11]
    ro, rf = oracle_heads(inp, hs)
    assert_close("tp8 split out", out[:, :, hs], ro, TOL16)
    assert_close("tp8 split final_state", fin[:, hs], rf, TOL16)


def test_split_writes_nothing_outside_its_outputs_and_is_deterministic():
    w = _w(2, B=1, T=0, seqlens=(200, 9, 77), seed=23)
    inp = inputs.make_prefill_inputs(w, device="cuda")
    T, H, dv = 286, 2, 128
    canary = -1234.5
    big = torch.full((T * H * dv + 4096,), canary, dtype=torch.bfloat16, device="cuda")
    out = big[:T * H * dv].view(1, T, H, dv)
    bigf = torch.full((3 * H * 128 * 128 + 4096,), canary, device="cuda")
    fin = bigf[:3 * H * 128 * 128].view(3, H, 128, 128)
    args = [inp[n] for n in ("q", "k", "v", "g_raw", "beta")]
    kda.kda_chunk_fwd_split(*args, inp["init_state"], inp["cu_seqlens"], segment_tokens=48,
                            out=out, final_state=fin)
    o2, f2 = kda.kda_chunk_fwd_split(*args, inp["init_state"], inp["cu_seqlens"], segment_tokens=48)
    torch.cuda.synchronize()
    assert torch.all(big[T * H * dv:] == canary)
    assert torch.all(bigf[3 * H * 128 * 128:] == canary)
    assert torch.equal(out, o2) and torch.equal(fin, f2)


def test_split_rejects_bad_arguments_without_launch():
    w = _w(1, B=1, T=64, seed=24)
    inp = inputs.make_prefill_inputs(w, device="cuda")
    args = [inp[n] for n in ("q", "k", "v", "g_raw", "beta")]
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_chunk_fwd_split(*args, segment_tokens=40)
    assert ei.value.status_name == "KDA_ERR_ARG"
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        kda.kda_chunk_fwd_split(*args, segment_tokens=32, workspace=small)
    f32 = [t.float() for t in args]
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_chunk_fwd_split(*f32, segment_tokens=32)
    assert ei.value.status_name == "KDA_ERR_SHAPE"
    kda.check_device_status()
