"""Parity of the state checkpoints emitted by the prefill
(kda_chunk_fwd_checkpointed, through the C ABI).

Checkpoint i of a sequence is the state after its first (i + 1) * E tokens;
the oracle gives it as the final state of that prefix.  Bar as for prefill:
max|gpu - oracle| <= tol * RMS, tol 2e-2 (bf16) / 1e-4 (fp32).  Outputs and
final states must be bit-identical to the plain kda_chunk_fwd (checkpoints
only add stores), and nothing past the buffer's rows is written.
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


def _w(dtype, H, dk, dv, seed, B=1, T=0, seqlens=(), s0_std=0.1):
    return inputs.Workload("test", "prefill", H=H, dk=dk, dv=dv, dtype=dtype, z_std=2.0,
                           s0_std=s0_std, seed=seed, B=B, T=T, seqlens=tuple(seqlens))


def _seq_bounds(inp, w):
    if inp["cu_seqlens"] is not None:
        cu = inp["cu_seqlens"].cpu().tolist()
        return [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
    return [(b, 0, w.T) for b in range(w.B)]


def _oracle_checkpoints(inp, w, every, heads):
    """Oracle states after every E tokens of each sequence, in buffer order."""
    S0 = inp["init_state"]
    rows = []
    for n, (b, s, e) in enumerate(_seq_bounds(inp, w)):
        for i in range((e - s) // every):
            end = s + (i + 1) * every
            sl = lambda t: t[b:b + 1, s:end][:, :, heads].cpu()
            init = None if S0 is None else S0[n:n + 1, heads].cpu()
            _, fin = oracle.kda_oracle_fwd(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]),
                                           sl(inp["g_raw"]), sl(inp["beta"]), init)
            rows.append(fin[0])
    return np.stack(rows) if rows else np.zeros((0, len(heads), w.dk, w.dv))


CASES = [
    # dtype, H, dk, dv, B, T, seqlens, every
    ("bf16", 2, 128, 128, 1, 0, (16, 100, 0, 33, 256, 47), 16),
    ("bf16", 3, 128, 128, 1, 0, (300, 64, 129), 64),
    ("bf16", 2, 128, 128, 2, 200, (), 48),
    ("f32", 2, 64, 128, 1, 0, (40, 96, 15), 32),
    ("f32", 1, 32, 32, 3, 70, (), 16),
    ("bf16", 2, 64, 64, 1, 0, (80, 17), 16),
    # more sequences than a warp: each chain's first checkpoint row is a
    # warp-strided count over all the sequences before it
    ("bf16", 2, 128, 128, 1, 0, tuple((16, 0, 40, 5, 33)[i % 5] for i in range(70)), 16),
]


@pytest.mark.parametrize("dtype,H,dk,dv,B,T,seqlens,every", CASES)
def test_checkpoints_match_oracle_prefix_states(dtype, H, dk, dv, B, T, seqlens, every):
    w = _w(dtype, H, dk, dv, seed=dk + dv + every + len(seqlens), B=B, T=T, seqlens=seqlens)
    inp = inputs.make_prefill_inputs(w, device="cuda")
    args = [inp[n] for n in ("q", "k", "v", "g_raw", "beta")]
    rows, first = kda.checkpoint_layout(inp["cu_seqlens"], args[0].shape[0], args[0].shape[1], every)
    big = torch.full(((rows + 1) * H * dk * dv,), CANARY, device="cuda")
    ck = big[:rows * H * dk * dv].view(rows, H, dk, dv)
    out, fin, ck, first2 = kda.kda_chunk_fwd_checkpointed(
        *args, inp["init_state"], inp["cu_seqlens"], checkpoint_every=every, checkpoints=ck)
    o_ref, f_ref = kda.kda_chunk_fwd(*args, inp["init_state"], inp["cu_seqlens"])
    torch.cuda.synchronize()
    assert first2 == first
    assert torch.equal(out, o_ref) and torch.equal(fin, f_ref)
    assert torch.all(big[rows * H * dk * dv:] == CANARY)
    heads = list(range(H))
    ref = _oracle_checkpoints(inp, w, every, heads)
    assert ref.shape[0] == rows
    if rows:
        assert_close("checkpoints", ck, ref, TOL[w.torch_dtype])
    # the last checkpoint of a sequence whose length E divides is its final state
    for n, (b, s, e) in enumerate(_seq_bounds(inp, w)):
        L = e - s
        if L and L % every == 0:
            assert torch.equal(ck[first[n] + L // every - 1], fin[n])


def test_checkpoint_then_resume_matches_unsplit():
    """A prefix cache hit: resume from a mid-sequence checkpoint with the
    remaining tokens and get the unsplit run's outputs and final state."""
    w = _w("bf16", 2, 128, 128, seed=31, B=1, T=320)
    inp = inputs.make_prefill_inputs(w, device="cuda")
    args = [inp[n] for n in ("q", "k", "v", "g_raw", "beta")]
    out, fin, ck, first = kda.kda_chunk_fwd_checkpointed(*args, inp["init_state"],
                                                         checkpoint_every=128)
    tail = [t[:, 256:].contiguous() for t in args]
    o2, f2 = kda.kda_chunk_fwd(*tail, ck[first[0] + 1:first[0] + 2].contiguous())
    torch.cuda.synchronize()
    from tests._parity import oracle_heads
    ref_out, ref_fin = oracle_heads(inp, [0, 1])
    tol = TOL[torch.bfloat16]
    assert_close("resumed out", o2, ref_out[:, 256:], tol)
    assert_close("resumed final state", f2, ref_fin, tol)


def test_checkpoints_on_layer_workload_sampled():
    """B=1, H=96, T=8192, d=128 bf16 with a checkpoint every 512 tokens (the
    hash-block granularity of the prefix cache): 16 checkpoints, oracle on
    sampled heads at three positions."""
    w = inputs.WORKLOADS["layer_bf16_H96_T8192"]
    inp = inputs.make_prefill_inputs(w, device="cuda")
    args = [inp[n] for n in ("q", "k", "v", "g_raw", "beta")]
    out, fin, ck, first = kda.kda_chunk_fwd_checkpointed(*args, None, checkpoint_every=512)
    torch.cuda.synchronize()
    assert ck.shape[0] == 16
    heads = [5, 77]
    tol = TOL[torch.bfloat16]
    for i in (0, 7, 15):
        end = (i + 1) * 512
        sl = lambda t: t[:, :end][:, :, heads].cpu()
        _, ref = oracle.kda_oracle_fwd(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]),
                                       sl(inp["g_raw"]), sl(inp["beta"]), None)
        assert_close(f"checkpoint {i}", ck[i, heads][None], ref, tol)
    assert torch.equal(ck[15], fin[0])


def test_short_buffer_is_never_overrun():
    """A caller that passes fewer rows than the layout needs through the C
    ABI gets the leading rows only; nothing past the buffer changes."""
    import ctypes
    w = _w("bf16", 2, 128, 128, seed=33, B=1, T=256)
    inp = inputs.make_prefill_inputs(w, device="cuda")
    args = [inp[n] for n in ("q", "k", "v", "g_raw", "beta")]
    _, _, full, _ = kda.kda_chunk_fwd_checkpointed(*args, inp["init_state"], checkpoint_every=64)
    big = torch.full((5 * 2 * 128 * 128,), CANARY, device="cuda")
    lib = kda.load_library()
    out = torch.empty_like(inp["v"])
    prm = kda._params(-5.0, None, 1.0)
    st = lib.kda_chunk_fwd_checkpointed(kda._dtype_code(inp["q"]), 1, 256, 2, 128, 128,
                                        *[kda._ptr(t) for t in args], kda._ptr(inp["init_state"]),
                                        None, 1, kda._ptr(out), None, 64, kda._ptr(big), 2,
                                        ctypes.byref(prm), None)
    torch.cuda.synchronize()
    assert st == 0
    got = big.view(5, 2, 128, 128)
    assert torch.equal(got[:2], full[:2])
    assert torch.all(got[2:] == CANARY)


def test_bad_interval_is_rejected():
    w = _w("bf16", 1, 128, 128, seed=34, B=1, T=64)
    inp = inputs.make_prefill_inputs(w, device="cuda")
    args = [inp[n] for n in ("q", "k", "v", "g_raw", "beta")]
    with pytest.raises(ValueError):
        kda.kda_chunk_fwd_checkpointed(*args, checkpoint_every=24)


def test_no_device_wait_gave_up():
    kda.check_device_status()
