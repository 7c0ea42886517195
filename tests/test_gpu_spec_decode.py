"""Parity of the speculative-replay decode (kda_decode_steps, through the C
ABI) with the fp64 oracle run over each sequence's accepted prefix.

Each sequence n applies the first accepted[n] of its K verified tokens; the
oracle sees exactly those tokens as a packed sequence starting from the same
state.  Bar as for decode: max|gpu - oracle| <= tol * RMS (+ one bf16 ulp of
the reference for bf16 outputs), tol 2e-2 (bf16) / 1e-4 (fp32).  Rows of
tokens that are not applied must stay untouched and a sequence with nothing
accepted must keep its state bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_11_gb300 import inputs, kda
from gated_delta_rule_11_gb300 import build as kbuild
from tests._parity import TOL, assert_close

pytestmark = pytest.mark.gpu

CANARY = -1234.5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kda.load_library()


def _w(dtype, H, dk, dv, N, K, seed=0):
    return inputs.Workload("test", "spec", H=H, dk=dk, dv=dv, dtype=dtype, z_std=2.0,
                           s0_std=0.1, seed=seed, N=N, steps=1, drafts=K)


def _oracle_replay(tok, S_ref, acc, A_log=None, scale=1.0):
    """Oracle over the accepted prefixes: out rows of the applied tokens
    (packed in sequence order) and the states after them."""
    acc = [int(a) for a in acc]
    N, K, H, dk = tok["q"].shape
    pick = lambda t: torch.cat([t[n, :acc[n]] for n in range(N)], dim=0)[None].cpu()
    cu = np.concatenate([[0], np.cumsum(acc)]).astype(np.int32)
    out, fin = oracle.kda_oracle_fwd(pick(tok["q"]), pick(tok["k"]), pick(tok["v"]),
                                     pick(tok["g_raw"]), pick(tok["beta"]), S_ref, cu,
                                     A_log=None if A_log is None else A_log.cpu(), scale=scale)
    return out[0], fin


def _applied_rows(out, acc):
    return torch.cat([out[n, :int(a)] for n, a in enumerate(acc)], dim=0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv,K", [(32, 32, 3), (64, 128, 5), (128, 64, 2), (128, 128, 8),
                                     (32, 128, 4), (128, 128, 1),
                                     # more drafts than one 8-token block: later blocks
                                     # are prepared after the first one's tokens
                                     (128, 128, 12), (64, 64, 17)])
def test_small_replay_matches_oracle(dtype, dk, dv, K):
    w = _w(dtype, 3, dk, dv, N=6, K=K, seed=dk + dv + K)
    S = inputs.make_decode_state(w, device="cuda")
    S0 = S.clone()
    tok = inputs.make_decode_drafts(w, 0, device="cuda", min_accepted=0)
    acc = tok["accepted"].cpu().tolist()
    A_log = torch.tensor([0.0, 0.4, -0.3], device="cuda")
    out = torch.full((6, K, 3, dv), CANARY, dtype=w.torch_dtype, device="cuda")
    kda.kda_decode_steps(tok["q"], tok["k"], tok["v"], tok["g_raw"], tok["beta"], S,
                         tok["accepted"], out=out, A_log=A_log, scale=0.75)
    torch.cuda.synchronize()
    ref_out, ref_fin = _oracle_replay(tok, S0.cpu().double().numpy(), acc, A_log, 0.75)
    tol = TOL[w.torch_dtype]
    if sum(acc):
        assert_close("applied out rows", _applied_rows(out, acc), ref_out, tol)
    assert_close("state after replay", S, ref_fin, tol)
    for n, a in enumerate(acc):
        assert torch.all(out[n, a:] == CANARY), f"sequence {n}: rows past accepted={a} written"
        if a == 0:
            assert torch.equal(S[n], S0[n])


def test_accepted_zero_and_out_of_range_counts_are_clamped():
    w = _w("bf16", 2, 128, 128, N=4, K=4, seed=21)
    S = inputs.make_decode_state(w, device="cuda")
    tok = inputs.make_decode_drafts(w, 0, device="cuda")
    acc_raw = torch.tensor([0, -3, 9, 4], dtype=torch.int32, device="cuda")
    S_clamped = S.clone()
    S0 = S.clone()
    args = [tok[n] for n in ("q", "k", "v", "g_raw", "beta")]
    o1 = kda.kda_decode_steps(*args, S, acc_raw)
    o2 = kda.kda_decode_steps(*args, S_clamped, torch.tensor([0, 0, 4, 4], dtype=torch.int32,
                                                             device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(S, S_clamped) and torch.equal(o1, o2)
    assert torch.equal(S[0], S0[0]) and torch.equal(S[1], S0[1])


def test_replay_split_is_bit_exact_and_matches_single_steps():
    """Replaying a prefix in two launches (the state carried in fp32 between
    them) is bit-identical to one launch; single-token steps agree to fp32
    rounding (their reduction order over the key channels differs)."""
    w = _w("bf16", 4, 128, 128, N=5, K=6, seed=22)
    S1 = inputs.make_decode_state(w, device="cuda")
    S2, S3 = S1.clone(), S1.clone()
    tok = inputs.make_decode_drafts(w, 0, device="cuda", min_accepted=0)
    acc = tok["accepted"].cpu().tolist()
    names = ("q", "k", "v", "g_raw", "beta")
    out = kda.kda_decode_steps(*(tok[x] for x in names), S1, tok["accepted"])
    first = torch.tensor([min(a, 2) for a in acc], dtype=torch.int32, device="cuda")
    rest = torch.tensor([max(a - 2, 0) for a in acc], dtype=torch.int32, device="cuda")
    o_a = kda.kda_decode_steps(*(tok[x][:, :2].contiguous() for x in names), S2, first)
    o_b = kda.kda_decode_steps(*(tok[x][:, 2:].contiguous() for x in names), S2, rest)
    torch.cuda.synchronize()
    assert torch.equal(S1, S2)
    for n in range(5):
        a = acc[n]
        assert torch.equal(out[n, :min(a, 2)], o_a[n, :min(a, 2)])
        assert torch.equal(out[n, 2:a], o_b[n, :max(a - 2, 0)])
    for n in range(5):
        for i in range(acc[n]):
            t = {x: tok[x][n:n + 1, i] for x in names}
            o = kda.kda_decode_step(t["q"], t["k"], t["v"], t["g_raw"], t["beta"], S3[n:n + 1])
            torch.cuda.synchronize()
            torch.testing.assert_close(o[0].float(), out[n, i].float(), rtol=0, atol=2 ** -7)
    torch.cuda.synchronize()
    torch.testing.assert_close(S3, S1, rtol=1e-5, atol=1e-6)


def test_all_accepted_by_default():
    w = _w("f32", 2, 64, 64, N=3, K=3, seed=23)
    S1 = inputs.make_decode_state(w, device="cuda")
    S2 = S1.clone()
    tok = inputs.make_decode_drafts(w, 0, device="cuda")
    args = [tok[n] for n in ("q", "k", "v", "g_raw", "beta")]
    o1 = kda.kda_decode_steps(*args, S1)
    o2 = kda.kda_decode_steps(*args, S2, torch.full((3,), 3, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(S1, S2) and torch.equal(o1, o2)


def test_spec_workload_sampled():
    """N=256, H=96, d=128, K=8 verified tokens with 1..8 accepted: full GPU
    launch (the one the benchmark times) on the whole state, oracle on
    sampled (sequence, head) pairs, several rounds in a row."""
    w = inputs.WORKLOADS["spec_bf16_N256_H96_K8"]
    S = inputs.make_decode_state(w, device="cuda")
    rng = np.random.default_rng(1)
    pairs = sorted(set((int(n), int(h)) for n, h in
                       zip(rng.integers(0, w.N, 48), rng.integers(0, w.H, 48))))
    ns = torch.tensor([p[0] for p in pairs])
    hs = torch.tensor([p[1] for p in pairs])
    S_ref = S[ns, hs].cpu().double().numpy()[:, None]          # [P, 1, dk, dv]
    tol = TOL[w.torch_dtype]
    for step in range(4):
        tok = inputs.make_decode_drafts(w, step, device="cuda")
        out = kda.kda_decode_steps(tok["q"], tok["k"], tok["v"], tok["g_raw"], tok["beta"], S,
                                   tok["accepted"])
        acc = tok["accepted"].cpu()[ns].tolist()
        sub = {x: tok[x][ns, :, hs][:, :, None] for x in ("q", "k", "v", "g_raw", "beta")}
        ref_out, S_ref = _oracle_replay(sub, S_ref, acc)
        got = _applied_rows(out[ns, :, hs][:, :, None], acc)
        assert_close(f"out round {step}", got, ref_out, tol)
    torch.cuda.synchronize()
    assert_close("final state", S[ns, hs][:, None], S_ref, tol)


def test_rejects_bad_accepted_dtype():
    w = _w("bf16", 1, 32, 32, N=2, K=2, seed=24)
    S = inputs.make_decode_state(w, device="cuda")
    tok = inputs.make_decode_drafts(w, 0, device="cuda")
    with pytest.raises(Exception):
        kda.kda_decode_steps(tok["q"], tok["k"], tok["v"], tok["g_raw"], tok["beta"], S,
                             tok["accepted"].long())


def test_no_device_wait_gave_up():
    kda.check_device_status()
