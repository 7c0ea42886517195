"""Gate variants on the GPU (prefill, decode step, speculative replay)
against the fp64 oracle with the same gate map.

Modes: "bounded" (eq. (5)), "log_decay" (the gate input is g), "neg_softplus"
(Kimi Linear's unbounded -softplus), "none" (the plain delta rule); each per
key channel or one per (token, head) (gated delta).  The unbounded inputs
include tiles whose cumulative log-decay falls far below -80, where dividing
by the in-tile decay would overflow: the prefill must take its position-pair
path and stay finite.  Bar: max|gpu - oracle| <= tol * RMS (+ one bf16 ulp of
the reference for bf16 outputs), tol 2e-2 (bf16) / 1e-4 (fp32).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_11_gb300 import inputs, kda
from gated_delta_rule_11_gb300 import build as kbuild
from tests._parity import TOL, assert_close, oracle_heads

pytestmark = pytest.mark.gpu

MODES = ["bounded", "log_decay", "neg_softplus", "none"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kda.load_library()


def gate_input(mode, shape, seed, dtype, device="cuda"):
    """Seeded gate inputs for a mode (None for "none").  log_decay: g <= 0 with
    a heavy tail (10% of values near -30); neg_softplus: z ~ N(0, 2) with 10%
    near +40 (g ~ -40); bounded: z ~ N(0, 2)."""
    if mode == "none":
        return None
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(shape, generator=g) * 2.0
    tail = torch.rand(shape, generator=g) < 0.1
    if mode == "log_decay":
        x = -(x.abs() * 0.5)
        x = torch.where(tail, torch.full_like(x, -30.0), x)
    elif mode == "neg_softplus":
        x = torch.where(tail, torch.full_like(x, 40.0), x)
    return x.to(dtype).to(device)


def _prefill_case(dtype, H, dk, dv, mode, per_head, seqlens, seed):
    w = inputs.Workload("test", "prefill", H=H, dk=dk, dv=dv, dtype=dtype, z_std=2.0,
                        s0_std=0.1, seed=seed, seqlens=tuple(seqlens))
    inp = inputs.make_prefill_inputs(w, device="cuda")
    T = sum(seqlens)
    gshape = (1, T, H) if per_head else (1, T, H, dk)
    inp["g_raw"] = gate_input(mode, gshape, seed + 1, w.torch_dtype)
    A_log = torch.tensor([0.2 * (i % 3) - 0.2 for i in range(H)], device="cuda")
    out, fin = kda.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"],
                                 inp["init_state"], inp["cu_seqlens"], A_log=A_log, scale=0.7,
                                 gate_mode=mode, gate_per_head=per_head)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all() and torch.isfinite(fin).all()
    if mode == "none":
        inp["g_raw"] = torch.zeros(gshape, dtype=w.torch_dtype, device="cuda")
    ro, rf = oracle_heads(inp, range(H), A_log=A_log, scale=0.7,
                          gate_mode=mode, gate_scalar=per_head)
    tol = TOL[w.torch_dtype]
    assert_close(f"{mode} out", out, ro, tol)
    assert_close(f"{mode} final_state", fin, rf, tol)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("per_head", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prefill_gate_variants(mode, per_head, dtype):
    _prefill_case(dtype, 2, 128, 128, mode, per_head, (37, 100, 0, 16), seed=50 + MODES.index(mode))


@pytest.mark.parametrize("mode", ["log_decay", "neg_softplus"])
def test_prefill_unbounded_small_heads(mode):
    _prefill_case("f32", 3, 64, 32, mode, False, (70, 5), seed=60)


def _decode_tok(w, mode, per_head, seed):
    tok = inputs.make_decode_token(w, 0, device="cuda", seed=seed)
    shape = (w.N, w.H) if per_head else (w.N, w.H, w.dk)
    tok["g_raw"] = gate_input(mode, shape, seed + 7, w.torch_dtype)
    return tok


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("per_head", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_step_gate_variants(mode, per_head, dtype):
    w = inputs.Workload("test", "decode", H=3, dk=128, dv=64, dtype=dtype, z_std=2.0,
                        s0_std=0.1, seed=70, N=5, steps=1)
    S = inputs.make_decode_state(w, device="cuda")
    S_ref = S.cpu().double().numpy()
    tok = _decode_tok(w, mode, per_head, 71 + MODES.index(mode))
    out = kda.kda_decode_step(tok["q"], tok["k"], tok["v"], tok["g_raw"], tok["beta"], S,
                              gate_mode=mode, gate_per_head=per_head)
    torch.cuda.synchronize()
    ro, rs = oracle.kda_oracle_decode(tok["q"], tok["k"], tok["v"], tok["g_raw"], tok["beta"],
                                      S_ref, gate_mode=mode, gate_scalar=per_head)
    tol = TOL[w.torch_dtype]
    assert_close(f"{mode} decode out", out, ro, tol)
    assert_close(f"{mode} decode state", S, rs, tol)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("per_head", [False, True])
def test_replay_gate_variants(mode, per_head):
    w = inputs.Workload("test", "spec", H=2, dk=128, dv=128, dtype="bf16", z_std=2.0,
                        s0_std=0.1, seed=80, N=4, steps=1, drafts=5)
    S = inputs.make_decode_state(w, device="cuda")
    S0 = S.cpu().double().numpy()
    d = inputs.make_decode_drafts(w, 0, device="cuda", min_accepted=0)
    shape = (w.N, w.drafts, w.H) if per_head else (w.N, w.drafts, w.H, w.dk)
    d["g_raw"] = gate_input(mode, shape, 81 + MODES.index(mode), w.torch_dtype)
    out = kda.kda_decode_steps(d["q"], d["k"], d["v"], d["g_raw"], d["beta"], S, d["accepted"],
                               gate_mode=mode, gate_per_head=per_head)
    torch.cuda.synchronize()
    acc = d["accepted"].cpu().tolist()
    pick = lambda t: None if t is None else torch.cat([t[n, :acc[n]] for n in range(w.N)])[None].cpu()
    cu = np.concatenate([[0], np.cumsum(acc)]).astype(np.int32)
    ro, rf = oracle.kda_oracle_fwd(pick(d["q"]), pick(d["k"]), pick(d["v"]), pick(d["g_raw"]),
                                   pick(d["beta"]), S0, cu, gate_mode=mode, gate_scalar=per_head)
    tol = TOL[torch.bfloat16]
    if sum(acc):
        got = torch.cat([out[n, :acc[n]] for n in range(w.N)])
        assert_close(f"{mode} replay out", got, ro[0], tol)
    assert_close(f"{mode} replay state", S, rf, tol)


@pytest.mark.parametrize("mode", ["log_decay", "neg_softplus"])
def test_unbounded_gate_mixes_factored_and_pair_tiles(mode):
    """Moderate gates keep most 16-token tiles inside fp32's range for
    e^{-b} (factored form); a few tokens with a huge decay push their tiles
    past it (position-pair form).  Both kinds in one launch on the
    tensor-core prefill, against the oracle."""
    seqlens = (160, 77, 16)
    w = inputs.Workload("test", "prefill", H=2, dk=128, dv=128, dtype="bf16", z_std=1.0,
                        s0_std=0.1, seed=95, seqlens=seqlens)
    inp = inputs.make_prefill_inputs(w, device="cuda")
    T = sum(seqlens)
    g = torch.Generator().manual_seed(96)
    if mode == "log_decay":
        z = -torch.rand((1, T, 2, 128), generator=g) * 2.0                 # |g| < 2 per token
        big = -200.0
    else:
        z = torch.randn((1, T, 2, 128), generator=g) - 1.0                 # softplus ~ 0.3
        big = 200.0
    spikes = torch.tensor([5, 40, 170, 200])                               # a few tiles only
    z[:, spikes] = big
    inp["g_raw"] = z.to(torch.bfloat16).cuda()
    out, fin = kda.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"],
                                 inp["init_state"], inp["cu_seqlens"], gate_mode=mode)
    torch.cuda.synchronize()
    assert kda.chunk_fwd_kernel(torch.bfloat16, 128, 128) == "prefill_tc_kernel"
    ro, rf = oracle_heads(inp, [0, 1], gate_mode=mode)
    tol = TOL[torch.bfloat16]
    assert_close(f"{mode} mixed out", out, ro, tol)
    assert_close(f"{mode} mixed final_state", fin, rf, tol)
    # the spikes really make pair tiles and the rest factored ones
    gl = oracle.kda_oracle_log_decay(inp["g_raw"].float().cpu().numpy()[0, :, 0], mode)
    bc = [gl[t0:t0 + 16].sum(0).min() for t0 in range(0, T, 16)]
    assert min(bc) < -85 and max(bc) > -40


def test_default_gate_still_on_tensor_cores_and_variants_reject_bad_args():
    assert kda.chunk_fwd_kernel(torch.bfloat16, 128, 128) == "prefill_tc_kernel"
    w = inputs.Workload("test", "prefill", H=1, dk=128, dv=128, dtype="bf16", z_std=1.0,
                        s0_std=0.0, seed=90, B=1, T=32)
    inp = inputs.make_prefill_inputs(w, device="cuda")
    with pytest.raises(ValueError):
        kda.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"],
                          gate_mode="softplus")
    with pytest.raises(ValueError):   # per-head gates have no channel axis
        kda.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"],
                          gate_per_head=True)
    out, fin = kda.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], None, inp["beta"], gate_mode="none")
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()


def test_no_device_wait_gave_up():
    kda.check_device_status()
