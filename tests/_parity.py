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
# exact fp64 answer to bf16 alone reaches 3.5e-2 x RMS.  So for bf16 outputs
# the representation error -- up to one bf16 ulp, 2^-8 |ref|, which also
# covers a result within rounding distance of a boundary landing on either
# neighbour -- is not counted, just as input rounding is not:
#     |gpu - ref| <= TOL * RMS(ref) + 2^-8 |ref|      (elementwise)
# fp32 outputs (the fp32 path and every state) use the plain bound.
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


def assert_close(name, gpu, ref, tol):
    e = compute_err(gpu, ref)
    assert np.isfinite(e) and e <= tol, (
        f"{name}: error {e:.3e} x RMS beyond the output format's rounding exceeds {tol:.1e} "
        f"(plain max-abs/RMS {rel_err(gpu, ref):.3e})")
    return e


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
