"""Parity of the CUDA decode step (kda_decode_step, through the C ABI) with
the fp64 oracle run one token at a time.  Same bar as prefill: max-abs
error <= tol * RMS per tensor, tol 2e-2 (bf16) / 1e-4 (fp32)."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_11_gb300 import inputs, kda
from gated_delta_rule_11_gb300 import build as kbuild
from tests._parity import TOL, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kda.load_library()


def _w(dtype, H, dk, dv, N, seed=0):
    return inputs.Workload("test", "decode", H=H, dk=dk, dv=dv, dtype=dtype, z_std=2.0,
                           s0_std=0.1, seed=seed, N=N, steps=3)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64), (128, 128), (32, 128)])
def test_small_decode_steps(dtype, dk, dv):
    w = _w(dtype, 3, dk, dv, N=5, seed=dk + dv)
    S = inputs.make_decode_state(w, device="cuda")
    S_ref = S.cpu().double().numpy()
    A_log = torch.tensor([0.0, 0.4, -0.3], device="cuda")
    for step in range(3):
        tok = inputs.make_decode_token(w, step, device="cuda")
        out = kda.kda_decode_step(tok["q"], tok["k"], tok["v"], tok["g_raw"], tok["beta"], S,
                                  A_log=A_log, scale=0.75)
        torch.cuda.synchronize()
        ref_out, S_ref = oracle.kda_oracle_decode(tok["q"], tok["k"], tok["v"], tok["g_raw"],
                                                  tok["beta"], S_ref, A_log=A_log.cpu(),
                                                  scale=0.75)
        tol = TOL[w.torch_dtype]
        assert_close(f"out step {step}", out, ref_out, tol)
        assert_close(f"state step {step}", S, S_ref, tol)


def test_decode_workload_100_steps_sampled():
    """N=256, H=96, d=128, fp32 state ~N(0, 0.1): 100 consecutive steps on the
    full state (the launch the benchmark times); every step's out and the
    final state are checked on sampled (sequence, head) pairs."""
    w = inputs.WORKLOADS["decode_bf16_N256_H96"]
    S = inputs.make_decode_state(w, device="cuda")
    rng = np.random.default_rng(0)
    pairs = sorted(set((int(n), int(h)) for n, h in
                       zip(rng.integers(0, w.N, 64), rng.integers(0, w.H, 64))))
    ns = torch.tensor([p[0] for p in pairs])
    hs = torch.tensor([p[1] for p in pairs])
    S_ref = S[ns, hs].cpu().double().numpy()[:, None]          # [P, 1, dk, dv]
    tol = TOL[w.torch_dtype]
    worst = 0.0
    for step in range(w.steps):
        tok = inputs.make_decode_token(w, step, device="cuda")
        out = kda.kda_decode_step(tok["q"], tok["k"], tok["v"], tok["g_raw"], tok["beta"], S)
        pick = lambda t: t[ns, hs].cpu()[:, None]
        ref_out, S_ref = oracle.kda_oracle_decode(pick(tok["q"]), pick(tok["k"]), pick(tok["v"]),
                                                  pick(tok["g_raw"]), pick(tok["beta"]), S_ref)
        worst = max(worst, assert_close(f"out step {step}", out[ns, hs][:, None], ref_out, tol))
    torch.cuda.synchronize()
    assert_close("final state", S[ns, hs][:, None], S_ref, tol)


def test_decode_is_deterministic():
    w = _w("bf16", 4, 128, 128, N=7, seed=3)
    S1 = inputs.make_decode_state(w, device="cuda")
    S2 = S1.clone()
    tok = inputs.make_decode_token(w, 0, device="cuda")
    args = [tok[n] for n in ("q", "k", "v", "g_raw", "beta")]
    o1 = kda.kda_decode_step(*args, S1)
    o2 = kda.kda_decode_step(*args, S2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(S1, S2)
