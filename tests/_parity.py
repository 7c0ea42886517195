"""Helpers shared by the GPU parity tests: tolerances, error measure and
head-sliced oracle runs.  The oracle runs on the host in fp64 on exactly the
values the GPU received."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# max|gpu - ref| <= TOL * RMS(ref), per output tensor (out, final state).
TOL = {torch.bfloat16: 2e-2, torch.float32: 1e-4}

# A bf16 output cannot be closer to the exact value than its own rounding:
# on heavy-tailed outputs (max/RMS ~ 13 on the decode workload) rounding the
# exact fp64 answer to bf16 alone reaches 3.5e-2 x RMS.  Where that happens
# (and only there, see assert_close) the representation error -- up to one
# bf16 ulp, 2^-8 |ref|, which also covers a result within rounding distance
# of a boundary landing on either neighbour -- is not counted:
#     |gpu - ref| <= TOL * RMS(ref) + 2^-8 |ref|      (elementwise)
# Everywhere else, and for every fp32 output, the plain bound is asserted.
BF16_ULP_REL = 2.0 ** -8


def _np(x):
    return x.detach().float().cpu().double().numpy() if hasattr(x, "detach") else np.asarray(x)


def rel_err(gpu, ref) -> float:
    """Plain measure: max|gpu - ref| / RMS(ref)."""
    g, r = _np(gpu), np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
    if rms == 0.0:
        return float(np.max(np.abs(g - r))) if g.size else 0.0
    return float(np.max(np.abs(g - r))) / rms


def compute_err(gpu, ref) -> float:
    """max over elements of (|gpu - ref| - representation allowance) / RMS(ref)."""
    g, r = _np(gpu), np.asarray(ref, dtype=np.float64)
    if not r.size:
        return 0.0
    allow = BF16_ULP_REL * np.abs(r) if getattr(gpu, "dtype", None) == torch.bfloat16 else 0.0
    rms = float(np.sqrt(np.mean(r * r)))
    excess = np.maximum(np.abs(g - r) - allow, 0.0)
    if rms == 0.0:
        return float(np.max(excess))
    return float(np.max(excess)) / rms


def rounding_floor(gpu, ref) -> float:
    """max|round_bf16(ref) - ref| / RMS(ref) for a bf16 output (0 otherwise):
    how close any output in this format can come to the exact answer."""
    if getattr(gpu, "dtype", None) != torch.bfloat16:
        return 0.0
    r = np.asarray(ref, dtype=np.float64)
    rb = torch.from_numpy(r).to(torch.bfloat16).double().numpy()
    return rel_err(rb, r)


def assert_close(name, gpu, ref, tol):
    """The literal bound max|gpu - ref| <= tol * RMS(ref) wherever a bf16
    output can meet it with room to spare: rounding the exact answer to bf16
    costs at most half the tolerance, leaving the other half for the
    computation (every state, the large prefill outputs).  Where the
    rounding alone takes more than that (heavy-tailed outputs: decode, and
    small cases whose few elements make max/RMS large), the one-ulp
    allowance above is used instead, which still bounds the error beyond
    the format's own rounding by tol * RMS.  Both numbers are printed."""
    plain = rel_err(gpu, ref)
    floor = rounding_floor(gpu, ref)
    literal = floor <= 0.5 * tol
    e = plain if literal else compute_err(gpu, ref)
    print(f"[parity] {name}: plain max|gpu-ref|/RMS = {plain:.3e}, "
          f"bf16 rounding floor = {floor:.3e}, "
          f"{'literal bound' if literal else 'beyond one-ulp allowance'} {e:.3e} <= {tol:.1e}")
    assert np.isfinite(e) and e <= tol, (
        f"{name}: error {e:.3e} x RMS exceeds {tol:.1e} "
        f"({'plain max-abs/RMS' if literal else 'beyond the bf16 rounding of the exact answer'}; "
        f"plain {plain:.3e}, rounding floor {floor:.3e})")
    return e


def assert_elementwise(name, gpu, ref, ulps=2.0):
    """Per-element bound for the elementwise passes (no long accumulation):
    |gpu - ref| <= ulps * ulp(ref) + 1e-6 * RMS(ref), with ulp the output
    format's spacing at |ref| (bf16: 2^(e-7), fp32: 2^(e-23) for |ref| in
    [2^e, 2^(e+1))); the small absolute term covers fp32 rounding of terms
    that cancel to near zero."""
    g, r = _np(gpu), np.asarray(ref, dtype=np.float64)
    if not r.size:
        return 0.0
    bits = 7 if getattr(gpu, "dtype", None) == torch.bfloat16 else 23
    e2 = np.floor(np.log2(np.maximum(np.abs(r), 1e-300)))
    ulp = np.exp2(e2 - bits)
    rms = float(np.sqrt(np.mean(r * r)))
    bound = ulps * ulp + 1e-6 * rms
    worst = float(np.max(np.abs(g - r) / bound))
    print(f"[parity] {name}: max |gpu-ref| / ({ulps:g} ulp + 1e-6 RMS) = {worst:.3f}, "
          f"plain max|gpu-ref|/RMS = {rel_err(gpu, ref):.3e}")
    assert np.isfinite(worst) and worst <= 1.0, (
        f"{name}: an element is {worst:.2f}x beyond {ulps:g} ulp of the exact value")
    return worst


def oracle_heads(inp, heads, A_log=None, scale=1.0, g_min=-5.0, **gate_kw):
    """Run the oracle on a subset of heads of a prefill input dict (gate_kw:
    gate_mode / gate_scalar of the oracle).
    Returns (out [B, T, len(heads), dv], final [N, len(heads), dk, dv])."""
    hs = list(heads)
    sl = lambda t: None if t is None else t[:, :, hs].contiguous().cpu()
    init = inp.get("init_state")
    init = None if init is None else init[:, hs].contiguous().cpu()
    cu = inp.get("cu_seqlens")
    cu = None if cu is None else cu.cpu().numpy()
    Al = None if A_log is None else A_log[hs].cpu()
    return oracle.kda_oracle_fwd(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["g_raw"]),
                                 inp["beta"][:, :, hs].contiguous().cpu(), init, cu,
                                 A_log=Al, scale=scale, g_min=g_min, **gate_kw)
