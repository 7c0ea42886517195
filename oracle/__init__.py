"""KDA oracle -- TEST INFRASTRUCTURE ONLY.

A plain fp64 CPU implementation of the Kimi Delta Attention recurrence
(``kda_oracle.c`` in this folder, built with gcc).  Only ``tests/``,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import
this package; the CUDA library never does, and the two share no code.

What it computes (from "Kimi K3：从三条信息流到完整系统", wineandchord.com):

* §KDA 是带逐通道遗忘的 delta rule, eq. (1) in its expanded form
  ``S_t = D + beta_t k_t (v_t - D^T k_t)^T`` with ``D = Diag(alpha_t) S_{t-1}``,
  and ``o_t = S_t^T q_t``: per (sequence, head), token by token,
  ``D = Diag(alpha) S``; ``e = v - D^T k``; ``S = D + beta k e^T``;
  ``o = scale * S^T q`` (the read sees this token's write).
* §下界 log-decay 是一个 kernel 设计, eq. (5): ``g = g_min *
  sigmoid(e^A z)``, ``alpha = e^g``, ``g_min = -5``.
* Gate variants ("Kimi K3: Two point eight trillion parameters, open
  weights, and forty-seven pages of how", §What changed between the paper
  and the model, and the four update rules before it): Kimi Linear's
  unbounded ``g = -softplus(e^A z)``, the gate given as ``g`` itself, no gate
  (``alpha = 1``, the plain delta rule), and one scalar gate per (token,
  head) shared by all key channels (gated delta).

Inputs are widened to fp64 exactly (bf16 and fp32 values are representable),
so input rounding never counts as error.  Parity status of each function is
listed in its docstring; all of them are pinned by ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libkda_oracle.so")

_lib = None
_lock = threading.Lock()

G_MIN_DEFAULT = -5.0
GATE_MODES = {"bounded": 0, "log_decay": 1, "neg_softplus": 2, "none": 3}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags only: no -march, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-std=c11",
                           "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            lib.kda_oracle_fwd.restype = ctypes.c_int
            lib.kda_oracle_fwd.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                dp, dp, dp, dp, dp, ip, ctypes.c_int, dp, dp,
                ctypes.c_double, ctypes.c_double, ctypes.c_int, ctypes.c_int, dp, dp, ctypes.c_int]
            lib.kda_oracle_gate.restype = ctypes.c_double
            lib.kda_oracle_gate.argtypes = [ctypes.c_double, ctypes.c_double, ctypes.c_double]
            lib.kda_oracle_log_decay.restype = ctypes.c_double
            lib.kda_oracle_log_decay.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                                 ctypes.c_double]
            _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor (bf16 has no numpy dtype: widen via fp32)
        import torch
        x = x.detach().to("cpu")
        if x.dtype == torch.bfloat16:
            x = x.float()
        x = x.numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def kda_oracle_gate(z, A_log: float = 0.0, g_min: float = G_MIN_DEFAULT):
    """eq. (5) elementwise in fp64: ``g_min * sigmoid(exp(A_log) * z)``."""
    lib = _load()
    z = _f64(z)
    flat = z.reshape(-1)
    out = np.empty_like(flat)
    for i, zi in enumerate(flat):
        out[i] = lib.kda_oracle_gate(float(zi), float(A_log), float(g_min))
    return out.reshape(z.shape)


def kda_oracle_log_decay(z, gate_mode: str = "bounded", A_log: float = 0.0,
                         g_min: float = G_MIN_DEFAULT):
    """The log-decay g of each gate input under ``gate_mode`` (see GATE_MODES)."""
    lib = _load()
    mode = GATE_MODES[gate_mode]
    z = _f64(z)
    flat = z.reshape(-1)
    out = np.empty_like(flat)
    for i, zi in enumerate(flat):
        out[i] = lib.kda_oracle_log_decay(mode, float(zi), float(A_log), float(g_min))
    return out.reshape(z.shape)


def kda_oracle_fwd(q, k, v, g_raw, beta, init_state=None, cu_seqlens=None, *,
                   A_log=None, g_min: float = G_MIN_DEFAULT, scale: float = 1.0,
                   gate_is_log_decay: bool = False, gate_mode: str = "bounded",
                   gate_scalar: bool = False, nthreads: int | None = None):
    """Sequential fp64 KDA forward.

    Shapes: q, k [B, T, H, dk]; g_raw [B, T, H, dk] ([B, T, H] with
    ``gate_scalar``; ignored, may be None, with gate_mode "none"); v [B, T, H,
    dv]; beta [B, T, H]; init_state [N, H, dk, dv] or None (zeros);
    cu_seqlens [N+1] (then B == 1) or None (then N = B, each batch row one
    sequence).  ``gate_mode`` picks the map from gate input to log-decay
    (GATE_MODES; "bounded" is eq. (5)); ``gate_is_log_decay`` is the same as
    gate_mode "log_decay" (the gate input is g = log(alpha) itself).

    Returns (out [B, T, H, dv], final_state [N, H, dk, dv]) in fp64.
    """
    lib = _load()
    mode = GATE_MODES["log_decay" if gate_is_log_decay else gate_mode]
    q, k, v, g_raw, beta = (_f64(x) for x in (q, k, v, g_raw, beta))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == q.shape
    if mode != GATE_MODES["none"]:
        assert g_raw.shape == ((B, T, H) if gate_scalar else q.shape)
    else:
        g_raw = None
    assert v.shape == (B, T, H, dv) and beta.shape == (B, T, H)
    if cu_seqlens is None:
        cu = np.arange(B + 1, dtype=np.int32) * T
    else:
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int32))
        assert B == 1, "packed sequences require B == 1"
    N = len(cu) - 1
    S0 = _f64(init_state)
    if S0 is not None:
        assert S0.shape == (N, H, dk, dv)
    Al = _f64(A_log)
    if Al is not None:
        Al = Al.reshape(H)
    out = np.zeros((B, T, H, dv), dtype=np.float64)
    fin = np.zeros((N, H, dk, dv), dtype=np.float64)
    nt = default_threads() if nthreads is None else nthreads
    rc = lib.kda_oracle_fwd(B * T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw),
                            _ptr(beta), cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                            N, _ptr(S0), _ptr(Al), float(g_min), float(scale),
                            int(mode), int(bool(gate_scalar)), _ptr(out), _ptr(fin), int(nt))
    if rc != 0:
        raise ValueError(f"kda_oracle_fwd rejected its arguments (code {rc})")
    return out, fin


def kda_oracle_decode(q, k, v, g_raw, beta, state, *, A_log=None,
                      g_min: float = G_MIN_DEFAULT, scale: float = 1.0,
                      gate_mode: str = "bounded", gate_scalar: bool = False,
                      nthreads: int | None = None):
    """One decode step: every (sequence, head) advances by exactly one token.

    q, k, g_raw [N, H, dk]; v [N, H, dv]; beta [N, H]; state [N, H, dk, dv].
    This is the sequential forward with N sequences of length 1.
    Returns (out [N, H, dv], new_state [N, H, dk, dv]) in fp64.
    """
    q, k, v, g_raw, beta = (_f64(x) for x in (q, k, v, g_raw, beta))
    N, H, dk = q.shape
    cu = np.arange(N + 1, dtype=np.int32)
    out, fin = kda_oracle_fwd(q[None], k[None], v[None], None if g_raw is None else g_raw[None],
                              beta[None], init_state=state, cu_seqlens=cu, A_log=A_log,
                              g_min=g_min, scale=scale, gate_mode=gate_mode,
                              gate_scalar=gate_scalar, nthreads=nthreads)
    return out[0], fin
