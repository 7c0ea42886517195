"""Degenerate inputs of the method on every kernel, against the oracle:
beta = 0 (no write: the state only decays), beta = 1, gate inputs at
+-1e4 (alpha at its bounds e^{-5} and 1 under eq. (5)), zero keys and zero
queries.  Same bar as the other parity tests."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_11_gb300 import inputs, kda
from gated_delta_rule_11_gb300 import build as kbuild
from tests._parity import TOL, assert_close, oracle_heads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kda.load_library()


def _degenerate(inp, seed):
    """Overwrite blocks of tokens with the degenerate values."""
    T = inp["q"].shape[1]
    g = torch.Generator(device="cpu").manual_seed(seed)
    kinds = torch.randint(0, 6, (T,), generator=g)
    for t in range(T):
        kd = int(kinds[t])
        if kd == 0:
            inp["beta"][:, t] = 0
        elif kd == 1:
            inp["beta"][:, t] = 1
        elif kd == 2:
            inp["g_raw"][:, t] = 1e4        # alpha -> e^{-5}
        elif kd == 3:
            inp["g_raw"][:, t] = -1e4       # alpha -> 1
        elif kd == 4:
            inp["k"][:, t] = 0
        else:
            inp["q"][:, t] = 0
    return inp


@pytest.mark.parametrize("dtype,dk,dv", [("bf16", 128, 128), ("f32", 64, 128), ("bf16", 32, 64)])
def test_prefill_degenerate_inputs(dtype, dk, dv):
    w = inputs.Workload("test", "prefill", H=2, dk=dk, dv=dv, dtype=dtype, z_std=2.0, s0_std=0.1,
                        seed=dk + dv, seqlens=(100, 37, 1))
    inp = _degenerate(inputs.make_prefill_inputs(w, device="cuda"), seed=3)
    out, fin = kda.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"],
                                 inp["init_state"], inp["cu_seqlens"])
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all() and torch.isfinite(fin).all()
    ro, rf = oracle_heads(inp, [0, 1])
    tol = TOL[w.torch_dtype]
    assert_close("out", out, ro, tol)
    assert_close("final_state", fin, rf, tol)


def test_decode_and_replay_degenerate_inputs():
    w = inputs.Workload("test", "spec", H=3, dk=128, dv=128, dtype="bf16", z_std=2.0, s0_std=0.1,
                        seed=5, N=6, steps=1, drafts=6)
    S = inputs.make_decode_state(w, device="cuda")
    S0 = S.cpu().double().numpy()
    d = inputs.make_decode_drafts(w, 0, device="cuda")
    d["beta"][:, 0] = 0
    d["beta"][:, 1] = 1
    d["g_raw"][:, 2] = 1e4
    d["g_raw"][:, 3] = -1e4
    d["k"][:, 4] = 0
    d["q"][:, 5] = 0
    full = torch.full((w.N,), w.drafts, dtype=torch.int32, device="cuda")
    out = kda.kda_decode_steps(d["q"], d["k"], d["v"], d["g_raw"], d["beta"], S, full)
    torch.cuda.synchronize()
    flat = lambda t: t.reshape((1, -1) + tuple(t.shape[2:])).cpu()
    cu = np.arange(w.N + 1, dtype=np.int32) * w.drafts
    ro, rf = oracle.kda_oracle_fwd(flat(d["q"]), flat(d["k"]), flat(d["v"]), flat(d["g_raw"]),
                                   flat(d["beta"]), S0, cu)
    tol = TOL[torch.bfloat16]
    assert_close("replay out", out.reshape((1, -1) + tuple(out.shape[2:])), ro, tol)
    assert_close("replay state", S, rf, tol)
    # the single step on the first degenerate token of each kind
    S1 = torch.from_numpy(S0).float().cuda()
    for i in range(w.drafts):
        t = {x: d[x][:, i].contiguous() for x in ("q", "k", "v", "g_raw", "beta")}
        o = kda.kda_decode_step(t["q"], t["k"], t["v"], t["g_raw"], t["beta"], S1)
        torch.cuda.synchronize()
        r_o = ro[0].reshape(w.N, w.drafts, w.H, w.dv)[:, i]
        assert_close(f"step {i} out", o, r_o, tol)
    assert_close("steps state", S1, rf, tol)


def test_no_device_wait_gave_up():
    kda.check_device_status()
