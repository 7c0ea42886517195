"""Parity of the CUDA prefill (kda_chunk_fwd, through the C ABI) with the
fp64 oracle, element by element on the same seeded inputs.

Bar: max|gpu - oracle| <= tol * RMS(oracle) for out and final_state
separately, tol = 2e-2 (bf16 inputs, fp32 state) and 1e-4 (fp32 path).
Small cases run the oracle on everything (several 16-token tiles, ragged
tails, empty and one-token sequences); the full-size workloads run the GPU
on everything and the oracle on sampled heads.
"""
import os

import numpy as np
import pytest
import torch

from gated_delta_rule_11_gb300 import inputs, kda
from gated_delta_rule_11_gb300 import build as kbuild
from tests._parity import TOL, assert_close, oracle_heads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kda.load_library()


def _w(dtype, H, dk, dv, z_std=2.0, s0_std=0.1, seed=0, B=1, T=0, seqlens=()):
    return inputs.Workload("test", "prefill", H=H, dk=dk, dv=dv, dtype=dtype, z_std=z_std,
                           s0_std=s0_std, seed=seed, B=B, T=T, seqlens=tuple(seqlens))


def _run_and_compare(w, heads=None, **kw):
    inp = inputs.make_prefill_inputs(w, device="cuda")
    out, fin = kda.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"],
                                 inp["init_state"], inp["cu_seqlens"], **kw)
    torch.cuda.synchronize()
    hs = list(range(w.H)) if heads is None else list(heads)
    ref_out, ref_fin = oracle_heads(inp, hs, A_log=kw.get("A_log"), scale=kw.get("scale", 1.0))
    tol = TOL[w.torch_dtype]
    e1 = assert_close("out", out[:, :, hs], ref_out, tol)
    e2 = assert_close("final_state", fin[:, hs], ref_fin, tol)
    return e1, e2


SMALL = [
    # dtype, H, dk, dv, B, T, seqlens
    ("f32", 1, 32, 32, 1, 64, ()),
    ("f32", 3, 64, 128, 2, 37, ()),
    ("f32", 2, 128, 64, 1, 0, (1, 15, 17, 31, 0, 100)),
    ("f32", 2, 128, 128, 1, 200, ()),
    ("f32", 1, 32, 128, 3, 5, ()),
    ("bf16", 2, 128, 128, 2, 100, ()),
    ("bf16", 3, 128, 128, 1, 0, (1, 15, 16, 17, 33, 0, 250)),
    ("bf16", 2, 64, 32, 1, 0, (7, 64, 65)),
    ("bf16", 1, 32, 64, 2, 48, ()),
]


@pytest.mark.parametrize("dtype,H,dk,dv,B,T,seqlens", SMALL)
def test_small_cases(dtype, H, dk, dv, B, T, seqlens):
    _run_and_compare(_w(dtype, H, dk, dv, B=B, T=T, seqlens=seqlens, seed=H * 7 + dk + T))


@pytest.mark.parametrize("dtype,dk", [("bf16", 128), ("f32", 64)])
def test_many_short_sequences(dtype, dk):
    """Two hundred packed sequences, many empty or shorter than a tile: every
    chain's span, the partial last tiles and the states all match."""
    rng = np.random.default_rng(31)
    seqlens = tuple(int(x) for x in rng.choice([0, 1, 5, 15, 16, 17, 33], size=200))
    _run_and_compare(_w(dtype, 2, dk, dk, seqlens=seqlens, seed=31))


def test_zero_initial_state_and_scale_and_head_log_scale():
    w = _w("bf16", 3, 128, 128, B=2, T=80, s0_std=0.0, seed=5)
    A_log = torch.tensor([0.0, 0.5, -0.7], device="cuda")
    _run_and_compare(w, A_log=A_log, scale=128 ** -0.5)
    w32 = _w("f32", 2, 64, 64, B=1, T=70, seed=6)
    _run_and_compare(w32, A_log=torch.tensor([0.3, -0.2], device="cuda"), scale=0.5)


def test_tiny_f32_workload():
    """B=1, H=1, T=64, d=32, fp32, seed 0: every output against the oracle."""
    _run_and_compare(inputs.WORKLOADS["tiny_f32_T64_d32"])


def test_small_bf16_workload():
    """B=2, H=4, T=1024, d=128, bf16 inputs, fp32 state, S_0 ~ N(0, 0.1)."""
    _run_and_compare(inputs.WORKLOADS["small_bf16_B2_H4_T1024"])


def test_layer_workload_sampled_heads():
    """B=1, H=96, T=8192, d=128 bf16: full GPU run, oracle on sampled heads."""
    _run_and_compare(inputs.WORKLOADS["layer_bf16_H96_T8192"], heads=[0, 41, 95])


@pytest.mark.slow
def test_varlen_workload_sampled_heads():
    """Packed 131072 + 65536 + 32768 + 8192 tokens, H=96, d=128, bf16: full GPU
    run (the launch the benchmark times), oracle on two heads of every sequence."""
    _run_and_compare(inputs.WORKLOADS["varlen_bf16_H96_237568"], heads=[3, 90])


def test_empty_sequences_keep_initial_state():
    w = _w("bf16", 2, 128, 128, seqlens=(0, 20, 0), seed=9)
    inp = inputs.make_prefill_inputs(w, device="cuda")
    out, fin = kda.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"],
                                 inp["init_state"], inp["cu_seqlens"])
    torch.cuda.synchronize()
    assert torch.equal(fin[0], inp["init_state"][0])
    assert torch.equal(fin[2], inp["init_state"][2])


def test_all_sequences_empty():
    w = _w("f32", 2, 32, 32, seqlens=(0, 0), seed=10)
    inp = inputs.make_prefill_inputs(w, device="cuda")
    _, fin = kda.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"],
                               inp["init_state"], inp["cu_seqlens"])
    torch.cuda.synchronize()
    assert torch.equal(fin, inp["init_state"])


def test_resume_from_final_state_matches_unsplit():
    """Checkpoint/resume: a prefix, then the suffix from the prefix's final
    state, matches the oracle of the unsplit sequence (split off a 16-token
    tile boundary, so the two runs tile the tokens differently)."""
    w = _w("bf16", 2, 128, 128, B=1, T=300, seed=11)
    inp = inputs.make_prefill_inputs(w, device="cuda")
    f = lambda sl, s0: kda.kda_chunk_fwd(*(inp[n][:, sl].contiguous() for n in
                                           ("q", "k", "v", "g_raw", "beta")), s0)
    o_a, s_a = f(slice(0, 123), inp["init_state"])
    o_b, s_b = f(slice(123, 300), s_a)
    torch.cuda.synchronize()
    ref_out, ref_fin = oracle_heads(inp, [0, 1])
    assert_close("resumed out", torch.cat([o_a, o_b], dim=1), ref_out, TOL[torch.bfloat16])
    assert_close("resumed final state", s_b, ref_fin, TOL[torch.bfloat16])


def test_deterministic_and_no_writes_outside_outputs():
    w = _w("bf16", 2, 128, 128, B=1, T=0, seqlens=(40, 9), seed=12)
    inp = inputs.make_prefill_inputs(w, device="cuda")
    T, H, dv = 49, 2, 128
    canary = -1234.5
    big = torch.full((T * H * dv + 4096,), canary, dtype=torch.bfloat16, device="cuda")
    out = big[:T * H * dv].view(1, T, H, dv)
    bigf = torch.full((2 * H * 128 * 128 + 4096,), canary, device="cuda")
    fin = bigf[:2 * H * 128 * 128].view(2, H, 128, 128)
    args = [inp[n] for n in ("q", "k", "v", "g_raw", "beta")]
    kda.kda_chunk_fwd(*args, inp["init_state"], inp["cu_seqlens"], out=out, final_state=fin)
    o2, f2 = kda.kda_chunk_fwd(*args, inp["init_state"], inp["cu_seqlens"])
    torch.cuda.synchronize()
    assert torch.all(big[T * H * dv:] == canary)
    assert torch.all(bigf[2 * H * 128 * 128:] == canary)
    assert torch.equal(out, o2) and torch.equal(fin, f2)


def test_runs_on_the_callers_stream():
    w = _w("bf16", 2, 128, 128, B=1, T=64, seed=13)
    inp = inputs.make_prefill_inputs(w, device="cuda")
    args = [inp[n] for n in ("q", "k", "v", "g_raw", "beta")]
    ref, _ = kda.kda_chunk_fwd(*args, inp["init_state"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o, _ = kda.kda_chunk_fwd(*args, inp["init_state"])
    s.synchronize()
    assert torch.equal(o, ref)


def test_misaligned_pointer_is_rejected_without_launch():
    w = _w("bf16", 1, 128, 128, B=1, T=32, seed=14)
    inp = inputs.make_prefill_inputs(w, device="cuda")
    raw = torch.zeros(32 * 128 + 1, dtype=torch.bfloat16, device="cuda")
    bad_q = raw[1:].view(1, 32, 1, 128)          # 2-byte offset
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_chunk_fwd(bad_q, inp["k"], inp["v"], inp["g_raw"], inp["beta"], inp["init_state"])
    assert ei.value.status_name == "KDA_ERR_ALIGN"


def test_no_device_wait_gave_up():
    """After every launch above, no bounded device wait timed out."""
    kda.check_device_status()


def test_loaded_library_is_in_tree():
    lib = kda.load_library()
    path = os.path.realpath(kda.library_path())
    assert os.path.exists(path)
    with open("/proc/self/maps") as f:
        assert path in f.read()
