"""Thin Python binding of libkda (include/kda.h) over ctypes.

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, their device pointers and the current CUDA stream are passed to
the C ABI, and a non-OK status raises ``KdaError``.  All arithmetic runs in
the library's CUDA kernels; there is no fallback.  PyTorch provides device
memory and streams.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

from . import build as _build

KDA_F32, KDA_BF16 = 0, 1
_STATUS = {0: "KDA_OK", 1: "KDA_ERR_ARG", 2: "KDA_ERR_DTYPE", 3: "KDA_ERR_SHAPE",
           4: "KDA_ERR_ALIGN", 5: "KDA_ERR_LAUNCH", 6: "KDA_ERR_TIMEOUT", 7: "KDA_ERR_SCRATCH"}

_lib = None
_lock = threading.Lock()

EXPORTED = ("kda_chunk_fwd", "kda_decode_step", "kda_status_str", "kda_last_cuda_error",
            "kda_version", "kda_launch_count", "kda_check_device_status", "kda_chunk_fwd_kernel",
            "kda_decode_steps", "kda_chunk_fwd_checkpointed", "kda_checkpoint_rows",
            "kda_qkv_prep", "kda_output_gate", "kda_selftest_bounded_wait",
            "kda_chunk_fwd_split", "kda_chunk_fwd_split_workspace", "kda_split_segment_tokens",
            "kda_chunk_fwd_split_noalloc", "kda_chunk_fwd_kcp_workspace", "kda_chunk_fwd_kcp_part",
            "kda_chunk_fwd_kcp_finish")


class KdaError(RuntimeError):
    def __init__(self, fn, status, detail=""):
        self.status = status
        self.status_name = _STATUS.get(status, str(status))
        super().__init__(f"{fn} returned {self.status_name}: {detail}")


class KdaParams(ctypes.Structure):
    _fields_ = [("g_min", ctypes.c_float), ("A_log", ctypes.c_void_p), ("scale", ctypes.c_float),
                ("gate_mode", ctypes.c_int), ("gate_per_head", ctypes.c_int)]


# kda_gate_mode: how g_raw becomes the log-decay g (see include/kda.h)
GATE_MODES = {"bounded": 0, "log_decay": 1, "neg_softplus": 2, "none": 3}


def library_path() -> str:
    return _build.LIB_PATH


def load_library(build_if_missing: bool = False):
    """Load libkda.so (raises if it is missing and building is not requested)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(
                    f"libkda.so not found at {path}: build it first "
                    "(python -m gated_delta_rule_11_gb300.build)")
            _build.build()
        lib = ctypes.CDLL(path)
        vp, i = ctypes.c_void_p, ctypes.c_int
        lib.kda_chunk_fwd.restype = i
        lib.kda_chunk_fwd.argtypes = [i, i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp, i, vp, vp,
                                      ctypes.POINTER(KdaParams), vp]
        lib.kda_decode_step.restype = i
        lib.kda_decode_step.argtypes = [i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp,
                                        ctypes.POINTER(KdaParams), vp]
        lib.kda_chunk_fwd_checkpointed.restype = i
        lib.kda_chunk_fwd_checkpointed.argtypes = [i, i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp, i,
                                                   vp, vp, i, vp, ctypes.c_longlong,
                                                   ctypes.POINTER(KdaParams), vp]
        lib.kda_chunk_fwd_split.restype = i
        lib.kda_chunk_fwd_split.argtypes = [i, i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp, i, i,
                                            vp, vp, vp, ctypes.c_ulonglong,
                                            ctypes.POINTER(KdaParams), vp]
        lib.kda_chunk_fwd_kcp_workspace.restype = ctypes.c_ulonglong
        lib.kda_chunk_fwd_kcp_workspace.argtypes = [i, i, i, i, i]
        lib.kda_chunk_fwd_kcp_part.restype = i
        lib.kda_chunk_fwd_kcp_part.argtypes = [i, i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp,
                                               ctypes.c_ulonglong, ctypes.POINTER(KdaParams), vp]
        lib.kda_chunk_fwd_kcp_finish.restype = i
        lib.kda_chunk_fwd_kcp_finish.argtypes = [i, i, i, i, i, i, vp, vp, vp, vp, ctypes.c_ulonglong, vp]
        lib.kda_chunk_fwd_split_noalloc.restype = i
        lib.kda_chunk_fwd_split_noalloc.argtypes = [i, i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp, i,
                                                    i, vp, vp, ctypes.POINTER(KdaParams), vp]
        lib.kda_chunk_fwd_split_workspace.restype = ctypes.c_ulonglong
        lib.kda_chunk_fwd_split_workspace.argtypes = [i, i, i, i, i, i, i]
        lib.kda_split_segment_tokens.restype = i
        lib.kda_split_segment_tokens.argtypes = [i, i, i, i, i, i]
        lib.kda_checkpoint_rows.restype = ctypes.c_longlong
        lib.kda_checkpoint_rows.argtypes = [i, i, vp, i, i]
        lib.kda_qkv_prep.restype = i
        lib.kda_qkv_prep.argtypes = [i, i, i, i, i, vp, vp, vp, vp, i, vp, vp, vp, vp, vp, vp,
                                     ctypes.c_float, vp]
        lib.kda_output_gate.restype = i
        lib.kda_output_gate.argtypes = [i, ctypes.c_longlong, i, vp, vp, vp, ctypes.c_float, vp, vp]
        lib.kda_decode_steps.restype = i
        lib.kda_decode_steps.argtypes = [i, i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp, vp,
                                         ctypes.POINTER(KdaParams), vp]
        lib.kda_status_str.restype = ctypes.c_char_p
        lib.kda_status_str.argtypes = [i]
        lib.kda_last_cuda_error.restype = i
        lib.kda_last_cuda_error.argtypes = []
        lib.kda_version.restype = i
        lib.kda_version.argtypes = []
        lib.kda_launch_count.restype = ctypes.c_ulonglong
        lib.kda_launch_count.argtypes = []
        lib.kda_check_device_status.restype = i
        lib.kda_check_device_status.argtypes = []
        lib.kda_selftest_bounded_wait.restype = i
        lib.kda_selftest_bounded_wait.argtypes = [i, vp]
        lib.kda_chunk_fwd_kernel.restype = ctypes.c_char_p
        lib.kda_chunk_fwd_kernel.argtypes = [i, i, i]
        _lib = lib
        return lib


def launch_count() -> int:
    """Kernels enqueued by libkda in this process so far."""
    return int(load_library().kda_launch_count())


def chunk_fwd_kernel(dtype: torch.dtype, dk: int, dv: int):
    """Name of the kernel kda_chunk_fwd uses for this dtype and head size."""
    code = KDA_F32 if dtype == torch.float32 else KDA_BF16
    r = load_library().kda_chunk_fwd_kernel(code, dk, dv)
    return None if r is None else r.decode()


def check_device_status() -> None:
    """Synchronise and raise KdaError if a kernel gave up a bounded wait."""
    lib = load_library()
    st = lib.kda_check_device_status()
    if st != 0:
        _raise(lib, "kda_check_device_status", st)


def selftest_bounded_wait(limit_us: int = 1000, stream=None) -> None:
    """Enqueue the library's test kernel whose bounded wait gives up after
    ``limit_us``; the next check_device_status() then raises KDA_ERR_TIMEOUT."""
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    st = lib.kda_selftest_bounded_wait(int(limit_us), _stream_handle(dev, stream))
    if st != 0:
        _raise(lib, "kda_selftest_bounded_wait", st)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return KDA_F32
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    raise TypeError(f"KDA inputs must be float32 or bfloat16, got {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t, name, shape, dtype, device):
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _params(g_min, A_log, scale, gate_mode="bounded", gate_per_head=False):
    if gate_mode not in GATE_MODES:
        raise ValueError(f"gate_mode must be one of {sorted(GATE_MODES)}")
    return KdaParams(float(g_min or 0.0), None if A_log is None else A_log.data_ptr(),
                     float(scale or 0.0), GATE_MODES[gate_mode], int(bool(gate_per_head)))


def _check_gate(g_raw, lead, dk, dt, dev, gate_mode, gate_per_head):
    """g_raw is [*lead, dk] per channel, [*lead] per head, unused with no gate."""
    if gate_mode == "none" and g_raw is None:
        return
    _check(g_raw, "g_raw", tuple(lead) if gate_per_head else tuple(lead) + (dk,), dt, dev)


def _stream_handle(device, stream):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _raise(lib, fn, st):
    detail = lib.kda_status_str(st).decode()
    if st == 5:
        detail += f" (cudaError {lib.kda_last_cuda_error()})"
    raise KdaError(fn, st, detail)


def kda_chunk_fwd(q, k, v, g_raw, beta, init_state=None, cu_seqlens=None, *,
                  out=None, final_state=None, output_final_state: bool = True,
                  g_min: float = -5.0, A_log=None, scale: float = 1.0,
                  gate_mode: str = "bounded", gate_per_head: bool = False, stream=None):
    """KDA forward over whole sequences (prefill).

    q, k, g_raw [B, T, H, dk]; v [B, T, H, dv]; beta [B, T, H] (all float32 or
    all bfloat16, on one CUDA device); init_state [N, H, dk, dv] float32 or
    None; cu_seqlens int32 [N+1] on the device (then B == 1) or None.
    gate_mode: "bounded" (eq. (5)), "log_decay", "neg_softplus" or "none";
    gate_per_head: g_raw is [B, T, H] (one gate per token and head).
    Returns (out [B, T, H, dv], final_state [N, H, dk, dv] float32 or None).
    """
    out, final_state, _ = _chunk_fwd(q, k, v, g_raw, beta, init_state, cu_seqlens, out,
                                     final_state, output_final_state, g_min, A_log, scale,
                                     stream, 0, None, 0, "kda_chunk_fwd", gate_mode, gate_per_head)
    return out, final_state


def checkpoint_layout(cu_seqlens, B: int, T: int, every: int):
    """Rows of the checkpoint buffer and each sequence's first row.

    cu_seqlens: int32 [N+1] (any device; read on the host) or None for B
    sequences of length T.  Returns (rows, first_rows list of N ints):
    sequence n's checkpoint i (state after (i + 1) * every tokens) is row
    first_rows[n] + i.
    """
    lib = load_library()
    if cu_seqlens is None:
        cu = np.arange(B + 1, dtype=np.int32) * T
        rows = lib.kda_checkpoint_rows(B, T, None, B, int(every))
    else:
        cu = np.ascontiguousarray(cu_seqlens.detach().cpu().numpy().astype(np.int32))
        rows = lib.kda_checkpoint_rows(1, int(T), cu.ctypes.data, len(cu) - 1, int(every))
    if rows < 0:
        raise ValueError("checkpoint layout: every must be a positive multiple of 16 and "
                         "cu_seqlens non-decreasing within [0, T]")
    per = np.diff(cu.astype(np.int64)) // int(every)
    first = np.concatenate([[0], np.cumsum(per)[:-1]]).astype(np.int64).tolist()
    return int(rows), first


def kda_chunk_fwd_checkpointed(q, k, v, g_raw, beta, init_state=None, cu_seqlens=None, *,
                               checkpoint_every: int, checkpoints=None, out=None,
                               final_state=None, output_final_state: bool = True,
                               g_min: float = -5.0, A_log=None, scale: float = 1.0,
                               gate_mode: str = "bounded", gate_per_head: bool = False,
                               stream=None):
    """kda_chunk_fwd that also saves the state every ``checkpoint_every``
    tokens (a positive multiple of 16) of each sequence.

    Returns (out, final_state, checkpoints [rows, H, dk, dv] float32,
    first_rows): checkpoint i of sequence n (the state after its first
    (i + 1) * checkpoint_every tokens) is checkpoints[first_rows[n] + i].
    """
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    rows, first = checkpoint_layout(cu_seqlens, B, T, checkpoint_every)
    if checkpoints is None:
        checkpoints = torch.empty((rows, H, dk, dv), dtype=torch.float32, device=q.device)
    else:
        _check(checkpoints, "checkpoints", (rows, H, dk, dv), torch.float32, q.device)
    out, final_state, _ = _chunk_fwd(q, k, v, g_raw, beta, init_state, cu_seqlens, out,
                                     final_state, output_final_state, g_min, A_log, scale,
                                     stream, int(checkpoint_every), checkpoints, rows,
                                     "kda_chunk_fwd_checkpointed", gate_mode, gate_per_head)
    return out, final_state, checkpoints, first


def split_segment_tokens(B: int, T: int, H: int, N: int, varlen: bool, sm_count: int) -> int:
    """Segment length for kda_chunk_fwd_split that puts every chain in one
    wave on ``sm_count`` multiprocessors, or 0 when splitting cannot."""
    return int(load_library().kda_split_segment_tokens(int(B), int(T), int(H), int(N),
                                                        int(bool(varlen)), int(sm_count)))


def split_workspace_bytes(B: int, T: int, H: int, dk: int, dv: int, N: int,
                          segment_tokens: int) -> int:
    """Bytes of device workspace kda_chunk_fwd_split needs (0: rejected sizes)."""
    return int(load_library().kda_chunk_fwd_split_workspace(int(B), int(T), int(H), int(dk),
                                                             int(dv), int(N),
                                                             int(segment_tokens)))


def kda_chunk_fwd_split(q, k, v, g_raw, beta, init_state=None, cu_seqlens=None, *,
                        segment_tokens: int | None = None, workspace=None, out=None,
                        final_state=None, output_final_state: bool = True,
                        g_min: float = -5.0, A_log=None, scale: float = 1.0,
                        gate_mode: str = "bounded", gate_per_head: bool = False, stream=None):
    """kda_chunk_fwd with every sequence cut into segments of
    ``segment_tokens`` tokens that run concurrently (bf16, dk = dv = 128).

    segment_tokens None: split_segment_tokens for this device's SM count;
    when that is 0 (enough chains already), the plain kda_chunk_fwd runs.
    workspace: a uint8 CUDA tensor of at least split_workspace_bytes(...)
    bytes (allocated here when None).  Returns (out, final_state).
    """
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("kda_chunk_fwd_split runs on CUDA tensors only")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if segment_tokens is None:
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        segment_tokens = split_segment_tokens(B, T, H, N, cu_seqlens is not None, sms)
        if segment_tokens == 0:
            return kda_chunk_fwd(q, k, v, g_raw, beta, init_state, cu_seqlens, out=out,
                                 final_state=final_state, output_final_state=output_final_state,
                                 g_min=g_min, A_log=A_log, scale=scale, gate_mode=gate_mode,
                                 gate_per_head=gate_per_head, stream=stream)
    need = split_workspace_bytes(B, T, H, dk, dv, max(N, 1), segment_tokens)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    elif (workspace.device != dev or workspace.dtype != torch.uint8 or
          not workspace.is_contiguous() or workspace.numel() < need):
        raise ValueError(f"workspace must be a contiguous uint8 tensor of >= {need} bytes on {dev}")
    out, final_state, _ = _chunk_fwd(q, k, v, g_raw, beta, init_state, cu_seqlens, out,
                                     final_state, output_final_state, g_min, A_log, scale,
                                     stream, 0, None, 0, "kda_chunk_fwd_split", gate_mode,
                                     gate_per_head, split=(int(segment_tokens), workspace))
    return out, final_state


def kcp_workspace_bytes(B: int, T: int, H: int, dk: int, dv: int) -> int:
    """Device workspace one rank needs for kda_chunk_fwd_kcp_part / _finish (0: rejected sizes)."""
    return int(load_library().kda_chunk_fwd_kcp_workspace(int(B), int(T), int(H), int(dk), int(dv)))


def kda_chunk_fwd_kcp_part(q, k, v, g_raw, beta, workspace, *, g_min: float = -5.0, A_log=None,
                           scale: float = 1.0, gate_mode: str = "bounded", gate_per_head: bool = False,
                           stream=None):
    """A rank r >= 1's part of a sequence split across ranks: its tokens
    (q, k, g_raw [B, T, H, 128], v [B, T, H, 128], beta [B, T, H], bf16) run
    from a zero state and as the transition.  Returns the pair tensor
    [B, 2, H, 128, 128] float32 ([:, 0] the zero-state final state, [:, 1]
    the transition) to exchange with the other ranks; the workspace (uint8,
    kcp_workspace_bytes) keeps the rows kda_chunk_fwd_kcp_finish needs."""
    lib = load_library()
    dev, dt = q.device, q.dtype
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    for nm, t, shp in (("q", q, (B, T, H, dk)), ("k", k, (B, T, H, dk)), ("v", v, (B, T, H, dv)),
                       ("beta", beta, (B, T, H))):
        _check(t, nm, shp, dt, dev)
    _check_gate(g_raw, (B, T, H), dk, dt, dev, gate_mode, gate_per_head)
    if A_log is not None:
        _check(A_log, "A_log", (H,), torch.float32, dev)
    need = kcp_workspace_bytes(B, T, H, dk, dv)
    if workspace.device != dev or workspace.dtype != torch.uint8 or workspace.numel() < need:
        raise ValueError(f"workspace must be a uint8 tensor of >= {need} bytes on {dev}")
    pair = torch.empty((B, 2, H, dk, dk), dtype=torch.float32, device=dev)
    prm = _params(g_min, A_log, scale, gate_mode, gate_per_head)
    st = lib.kda_chunk_fwd_kcp_part(_dtype_code(q), B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw),
                                    _ptr(beta), _ptr(pair), _ptr(workspace), workspace.numel(),
                                    ctypes.byref(prm), _stream_handle(dev, stream))
    if st != 0:
        _raise(lib, "kda_chunk_fwd_kcp_part", st)
    return pair


def kda_chunk_fwd_kcp_finish(pairs, rank: int, workspace, B: int, T: int, H: int, *, dk: int = 128,
                             dv: int = 128, out=None, final_state=None, stream=None):
    """A rank r >= 1's outputs after the exchange: pairs [rank + 1, B, 2, H,
    dk, dk] float32 on the device (entry [0][:, 0] is rank 0's final state).
    Returns (out [B, T, H, dv] bf16, final_state [B, H, dk, dv] float32, the
    state after this rank's tokens)."""
    lib = load_library()
    dev = workspace.device
    _check(pairs, "pairs", (rank + 1, B, 2, H, dk, dk), torch.float32, dev)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=torch.bfloat16, device=dev)
    _check(out, "out", (B, T, H, dv), torch.bfloat16, dev)
    if final_state is None:
        final_state = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    _check(final_state, "final_state", (B, H, dk, dv), torch.float32, dev)
    st = lib.kda_chunk_fwd_kcp_finish(B, T, H, dk, dv, int(rank), _ptr(pairs), _ptr(out), _ptr(final_state),
                                      _ptr(workspace), workspace.numel(), _stream_handle(dev, stream))
    if st != 0:
        _raise(lib, "kda_chunk_fwd_kcp_finish", st)
    return out, final_state


# Size of the library's own scratch buffer used by kda_chunk_fwd_split_noalloc.
SPLIT_SCRATCH_BYTES = 64 << 20


def kda_chunk_fwd_split_noalloc(q, k, v, g_raw, beta, init_state=None, cu_seqlens=None, *,
                                segment_tokens: int, out, final_state=None, g_min: float = -5.0,
                                A_log=None, scale: float = 1.0, gate_mode: str = "bounded",
                                gate_per_head: bool = False, stream=None):
    """kda_chunk_fwd_split with the scratch inside the library (no device
    allocation: neither here nor in the library).  For callers that cannot
    allocate device memory, e.g. a process whose memory belongs to its own
    caching pool.  ``out`` (and ``final_state``, if wanted) must be given;
    sizes needing more than SPLIT_SCRATCH_BYTES of scratch raise KdaError
    KDA_ERR_SCRATCH.  Calls on one device share the buffer: keep them ordered
    on one stream.  Returns (out, final_state)."""
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("kda_chunk_fwd_split_noalloc runs on CUDA tensors only")
    dt = q.dtype
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    for nm, t, shp in (("q", q, (B, T, H, dk)), ("k", k, (B, T, H, dk)),
                       ("v", v, (B, T, H, dv)), ("beta", beta, (B, T, H)), ("out", out, (B, T, H, dv))):
        _check(t, nm, shp, dt, dev)
    _check_gate(g_raw, (B, T, H), dk, dt, dev, gate_mode, gate_per_head)
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if cu_seqlens is not None and (cu_seqlens.dtype != torch.int32 or cu_seqlens.device != dev):
        raise ValueError("cu_seqlens must be an int32 tensor on the inputs' device")
    if init_state is not None:
        _check(init_state, "init_state", (N, H, dk, dv), torch.float32, dev)
    if final_state is not None:
        _check(final_state, "final_state", (N, H, dk, dv), torch.float32, dev)
    if A_log is not None:
        _check(A_log, "A_log", (H,), torch.float32, dev)
    prm = _params(g_min, A_log, scale, gate_mode, gate_per_head)
    st = lib.kda_chunk_fwd_split_noalloc(_dtype_code(q), B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v),
                                         _ptr(g_raw), _ptr(beta), _ptr(init_state),
                                         _ptr(cu_seqlens), N, int(segment_tokens), _ptr(out),
                                         _ptr(final_state), ctypes.byref(prm),
                                         _stream_handle(dev, stream))
    if st != 0:
        _raise(lib, "kda_chunk_fwd_split_noalloc", st)
    return out, final_state


def _chunk_fwd(q, k, v, g_raw, beta, init_state, cu_seqlens, out, final_state,
               output_final_state, g_min, A_log, scale, stream, every, ckpt, ckpt_rows, name,
               gate_mode="bounded", gate_per_head=False, split=None):
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise ValueError(f"{name} runs on CUDA tensors only")
    dt = q.dtype
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    for nm, t, shp in (("q", q, (B, T, H, dk)), ("k", k, (B, T, H, dk)),
                       ("v", v, (B, T, H, dv)), ("beta", beta, (B, T, H))):
        _check(t, nm, shp, dt, dev)
    _check_gate(g_raw, (B, T, H), dk, dt, dev, gate_mode, gate_per_head)
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32 or cu_seqlens.device != dev or cu_seqlens.dim() != 1:
            raise ValueError("cu_seqlens must be a 1-D int32 tensor on the inputs' device")
        if B != 1:
            raise ValueError("packed sequences (cu_seqlens) require B == 1")
        N = cu_seqlens.numel() - 1
    else:
        N = B
    if init_state is not None:
        _check(init_state, "init_state", (N, H, dk, dv), torch.float32, dev)
    if A_log is not None:
        _check(A_log, "A_log", (H,), torch.float32, dev)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=dt, device=dev)
    else:
        _check(out, "out", (B, T, H, dv), dt, dev)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    elif final_state is not None:
        _check(final_state, "final_state", (N, H, dk, dv), torch.float32, dev)
    prm = _params(g_min, A_log, scale, gate_mode, gate_per_head)
    common = (_dtype_code(q), B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw),
              _ptr(beta), _ptr(init_state), _ptr(cu_seqlens), N, _ptr(out), _ptr(final_state))
    if split is not None:
        tau, ws = split
        head = common[:14]
        st = lib.kda_chunk_fwd_split(*head, tau, _ptr(out), _ptr(final_state), _ptr(ws),
                                     ws.numel(), ctypes.byref(prm), _stream_handle(dev, stream))
    elif ckpt is None:
        st = lib.kda_chunk_fwd(*common, ctypes.byref(prm), _stream_handle(dev, stream))
    else:
        st = lib.kda_chunk_fwd_checkpointed(*common, int(every), _ptr(ckpt), int(ckpt_rows),
                                            ctypes.byref(prm), _stream_handle(dev, stream))
    if st != 0:
        _raise(lib, name, st)
    return out, final_state, ckpt


def kda_decode_step(q, k, v, g_raw, beta, state, *, out=None, g_min: float = -5.0,
                    A_log=None, scale: float = 1.0, gate_mode: str = "bounded",
                    gate_per_head: bool = False, stream=None):
    """Advance N sequences by one token; ``state`` [N, H, dk, dv] float32 is
    updated in place.  q, k, g_raw [N, H, dk] (g_raw [N, H] with
    gate_per_head); v [N, H, dv]; beta [N, H].  Returns out [N, H, dv]."""
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("kda_decode_step runs on CUDA tensors only")
    dt = q.dtype
    N, H, dk = q.shape
    dv = v.shape[-1]
    for name, t, shp in (("q", q, (N, H, dk)), ("k", k, (N, H, dk)),
                         ("v", v, (N, H, dv)), ("beta", beta, (N, H))):
        _check(t, name, shp, dt, dev)
    _check_gate(g_raw, (N, H), dk, dt, dev, gate_mode, gate_per_head)
    _check(state, "state", (N, H, dk, dv), torch.float32, dev)
    if A_log is not None:
        _check(A_log, "A_log", (H,), torch.float32, dev)
    if out is None:
        out = torch.empty((N, H, dv), dtype=dt, device=dev)
    else:
        _check(out, "out", (N, H, dv), dt, dev)
    prm = _params(g_min, A_log, scale, gate_mode, gate_per_head)
    st = lib.kda_decode_step(_dtype_code(q), N, H, dk, dv, _ptr(q), _ptr(k), _ptr(v),
                             _ptr(g_raw), _ptr(beta), _ptr(state), _ptr(out),
                             ctypes.byref(prm), _stream_handle(dev, stream))
    if st != 0:
        _raise(lib, "kda_decode_step", st)
    return out


def kda_decode_steps(q, k, v, g_raw, beta, state, accepted=None, *, out=None,
                     g_min: float = -5.0, A_log=None, scale: float = 1.0,
                     gate_mode: str = "bounded", gate_per_head: bool = False, stream=None):
    """Speculative replay: sequence n applies its first accepted[n] of K drafted
    tokens to ``state`` [N, H, dk, dv] (float32, in place) in one pass.
    q, k, g_raw [N, K, H, dk]; v [N, K, H, dv]; beta [N, K, H]; accepted int32
    [N] on the device or None (all K).  Returns out [N, K, H, dv] (rows of
    tokens that are not applied are left as they were in ``out``)."""
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("kda_decode_steps runs on CUDA tensors only")
    dt = q.dtype
    N, K, H, dk = q.shape
    dv = v.shape[-1]
    for name, t, shp in (("q", q, (N, K, H, dk)), ("k", k, (N, K, H, dk)),
                         ("v", v, (N, K, H, dv)), ("beta", beta, (N, K, H))):
        _check(t, name, shp, dt, dev)
    _check_gate(g_raw, (N, K, H), dk, dt, dev, gate_mode, gate_per_head)
    _check(state, "state", (N, H, dk, dv), torch.float32, dev)
    if accepted is not None:
        _check(accepted, "accepted", (N,), torch.int32, dev)
    if A_log is not None:
        _check(A_log, "A_log", (H,), torch.float32, dev)
    if out is None:
        out = torch.zeros((N, K, H, dv), dtype=dt, device=dev)
    else:
        _check(out, "out", (N, K, H, dv), dt, dev)
    prm = _params(g_min, A_log, scale, gate_mode, gate_per_head)
    st = lib.kda_decode_steps(_dtype_code(q), N, K, H, dk, dv, _ptr(q), _ptr(k), _ptr(v),
                              _ptr(g_raw), _ptr(beta), _ptr(accepted), _ptr(state), _ptr(out),
                              ctypes.byref(prm), _stream_handle(dev, stream))
    if st != 0:
        _raise(lib, "kda_decode_steps", st)
    return out


def _prep_outputs(out, B, T, H, d, dt, dev, want_beta):
    """The (q, k, v, beta) buffers of kda_qkv_prep: allocated when ``out`` is
    None, else checked like every input (shape, dtype, device, contiguity),
    so a short or misplaced buffer is refused before any kernel writes it."""
    if out is None:
        q, k, v = (torch.empty((B, T, H, d), dtype=dt, device=dev) for _ in range(3))
        beta = torch.empty((B, T, H), dtype=dt, device=dev) if want_beta else None
        return q, k, v, beta
    if not isinstance(out, (tuple, list)) or len(out) != 4:
        raise TypeError("out must be a tuple (q, k, v, beta)")
    q, k, v, beta = out
    for name, t in (("out q", q), ("out k", k), ("out v", v)):
        if t is None:
            raise ValueError(f"{name} is missing")
        _check(t, name, (B, T, H, d), dt, dev)
    if want_beta:
        if beta is None:
            raise ValueError("out beta is missing although beta_logit is given")
        _check(beta, "out beta", (B, T, H), dt, dev)
    elif beta is not None:
        raise ValueError("out beta is given but beta_logit is None")
    return q, k, v, beta


def _gate_output(out, o):
    """The y buffer of kda_output_gate: new, or checked against o."""
    if out is None:
        return torch.empty_like(o)
    _check(out, "out", tuple(o.shape), o.dtype, o.device)
    return out


def kda_qkv_prep(x_qkv, conv_w, beta_logit=None, cu_seqlens=None, conv_state_in=None, *,
                 conv_state_out=None, output_conv_state: bool = False, l2_eps: float = 0.0,
                 out=None, stream=None):
    """q, k = L2Norm(Swish(ShortConv(x_q|k))), v = Swish(ShortConv(x_v)),
    beta = Sigmoid(beta_logit).

    x_qkv [B, T, 3, H, d]; conv_w [3, H, d, 4] float32; beta_logit [B, T, H] or
    None; cu_seqlens int32 [N+1] on the device (then B == 1) or None;
    conv_state_in [N, 3, 3, H, d] or None.  Returns (q, k, v [B, T, H, d],
    beta [B, T, H] or None, conv_state_out [N, 3, 3, H, d] or None).
    """
    lib = load_library()
    dev = x_qkv.device
    if dev.type != "cuda":
        raise ValueError("kda_qkv_prep runs on CUDA tensors only")
    dt = x_qkv.dtype
    B, T, three, H, d = x_qkv.shape
    if three != 3:
        raise ValueError("x_qkv must be [B, T, 3, H, d]")
    _check(x_qkv, "x_qkv", (B, T, 3, H, d), dt, dev)
    _check(conv_w, "conv_w", (3, H, d, 4), torch.float32, dev)
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32 or cu_seqlens.device != dev or cu_seqlens.dim() != 1:
            raise ValueError("cu_seqlens must be a 1-D int32 tensor on the inputs' device")
        if B != 1:
            raise ValueError("packed sequences (cu_seqlens) require B == 1")
        N = cu_seqlens.numel() - 1
    else:
        N = B
    if beta_logit is not None:
        _check(beta_logit, "beta_logit", (B, T, H), dt, dev)
    if conv_state_in is not None:
        _check(conv_state_in, "conv_state_in", (N, 3, 3, H, d), dt, dev)
    if conv_state_out is None and output_conv_state:
        conv_state_out = torch.empty((N, 3, 3, H, d), dtype=dt, device=dev)
    elif conv_state_out is not None:
        _check(conv_state_out, "conv_state_out", (N, 3, 3, H, d), dt, dev)
    q, k, v, beta = _prep_outputs(out, B, T, H, d, dt, dev, beta_logit is not None)
    st = lib.kda_qkv_prep(_dtype_code(x_qkv), B, T, H, d, _ptr(x_qkv), _ptr(conv_w),
                          _ptr(beta_logit), _ptr(cu_seqlens), N, _ptr(conv_state_in),
                          _ptr(conv_state_out), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                          float(l2_eps), _stream_handle(dev, stream))
    if st != 0:
        _raise(lib, "kda_qkv_prep", st)
    return q, k, v, beta, conv_state_out


def kda_output_gate(o, gate, norm_w=None, *, eps: float = 0.0, out=None, stream=None):
    """y = Sigmoid(gate) * RMSNorm(o) over the last axis (one head's dv
    channels); o, gate [..., dv]; norm_w [dv] float32 or None."""
    lib = load_library()
    dev = o.device
    if dev.type != "cuda":
        raise ValueError("kda_output_gate runs on CUDA tensors only")
    d = o.shape[-1]
    _check(gate, "gate", tuple(o.shape), o.dtype, dev)
    _check(o, "o", tuple(o.shape), o.dtype, dev)
    if norm_w is not None:
        _check(norm_w, "norm_w", (d,), torch.float32, dev)
    y = _gate_output(out, o)
    st = lib.kda_output_gate(_dtype_code(o), o.numel() // d, d, _ptr(o), _ptr(gate), _ptr(norm_w),
                             float(eps), _ptr(y), _stream_handle(dev, stream))
    if st != 0:
        _raise(lib, "kda_output_gate", st)
    return y
