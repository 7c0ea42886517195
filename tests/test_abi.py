"""The C-ABI library builds, loads and exports what include/kda.h declares;
host-side validation rejects bad arguments before touching the GPU.
(No compute call here: these run without a GPU.)"""
import ctypes
import os
import re

import pytest

from gated_delta_rule_11_gb300 import build as kbuild
from gated_delta_rule_11_gb300 import kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kda.load_library()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^[ \t]*(?:[A-Za-z_]\w*[ \t*]+)+(kda_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for fn in ("kda_chunk_fwd", "kda_decode_step", "kda_status_str"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib):
    for fn in declared_functions():
        assert hasattr(lib, fn), f"libkda.so does not export {fn}"
    assert set(kda.EXPORTED) <= set(declared_functions())


def test_status_strings(lib):
    for code in range(7):
        s = lib.kda_status_str(code)
        assert s and len(s) > 1
    assert lib.kda_status_str(99) == b"unknown status"
    assert lib.kda_version() >= 10000


def _fwd(lib, dt=1, B=1, T=16, H=1, dk=128, dv=128, ptr=4096, init=None, cu=None, N=1,
         out=4096, fin=None):
    p = ctypes.c_void_p(ptr)
    return lib.kda_chunk_fwd(dt, B, T, H, dk, dv, p, p, p, p, p, init, cu, N,
                             ctypes.c_void_p(out) if out else None, fin, None, None)


def test_validation_rejects_before_launch(lib):
    # Every case fails validation, so no pointer is dereferenced and no CUDA call is made.
    assert _fwd(lib, dt=7) == 2                      # dtype
    assert _fwd(lib, dk=48) == 3                     # head dimension
    assert _fwd(lib, dv=256) == 3
    assert _fwd(lib, B=-1) == 1
    assert _fwd(lib, H=0) == 1
    assert _fwd(lib, N=2) == 1                       # N must equal B without cu_seqlens
    assert _fwd(lib, ptr=4100) == 4                  # misaligned
    assert _fwd(lib, out=0) == 1                     # missing output
    assert _fwd(lib, B=2, cu=ctypes.c_void_p(4096), N=2) == 1   # packed needs B == 1
    assert _fwd(lib, B=0, T=16, N=0) == 0            # empty batch: nothing to do
    p = ctypes.c_void_p(4096)
    assert lib.kda_decode_step(1, 4, 2, 128, 100, p, p, p, p, p, p, p, None, None) == 3
    assert lib.kda_decode_step(1, 4, 2, 128, 128, p, p, p, p, p, None, p, None, None) == 1
    assert lib.kda_decode_step(1, 4, 2, 128, 128, p, p, p, p, ctypes.c_void_p(4097), p, p,
                               None, None) == 4           # bf16 beta needs 2-byte alignment
    assert lib.kda_decode_step(1, 4, 2, 128, 128, p, p, p, p, p, ctypes.c_void_p(4104), p,
                               None, None) == 4           # state needs 16 bytes
    assert lib.kda_decode_step(1, 0, 2, 128, 128, None, None, None, None, None, None, None,
                               None, None) == 0


def test_kernel_selection(lib):
    import torch
    assert kda.chunk_fwd_kernel(torch.bfloat16, 128, 128) == "prefill_tc_kernel"
    assert kda.chunk_fwd_kernel(torch.float32, 128, 128) == "prefill_simt_kernel"
    assert kda.chunk_fwd_kernel(torch.bfloat16, 64, 128) == "prefill_simt_kernel"
    assert lib.kda_chunk_fwd_kernel(1, 48, 128) is None


def test_python_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros(1, 16, 1, 32)
    with pytest.raises(ValueError):
        kda.kda_chunk_fwd(x, x, x, x, torch.zeros(1, 16, 1))


def test_checkpoint_rows_host_helper(lib):
    """Rows of the checkpoint buffer: floor(L_n / E) per sequence; no GPU."""
    cu = (ctypes.c_int32 * 7)(0, 16, 116, 116, 149, 405, 452)
    assert lib.kda_checkpoint_rows(1, 452, cu, 6, 16) == 1 + 6 + 0 + 2 + 16 + 2
    assert lib.kda_checkpoint_rows(1, 452, cu, 6, 64) == 0 + 1 + 0 + 0 + 4 + 0
    assert lib.kda_checkpoint_rows(3, 200, None, 3, 48) == 3 * 4
    assert lib.kda_checkpoint_rows(2, 15, None, 2, 16) == 0
    assert lib.kda_checkpoint_rows(1, 452, cu, 6, 24) == -1          # not a multiple of 16
    assert lib.kda_checkpoint_rows(1, 452, cu, 6, 0) == -1
    assert lib.kda_checkpoint_rows(1, 400, cu, 6, 16) == -1          # past T
    bad = (ctypes.c_int32 * 3)(0, 40, 20)
    assert lib.kda_checkpoint_rows(1, 40, bad, 2, 16) == -1          # decreasing
    rows, first = kda.checkpoint_layout(None, 3, 200, 48)
    assert rows == 12 and first == [0, 4, 8]
    import torch
    rows, first = kda.checkpoint_layout(torch.tensor([0, 16, 116, 116, 149, 405, 452],
                                                     dtype=torch.int32), 1, 452, 16)
    assert rows == 27 and first == [0, 1, 7, 7, 9, 25]


def test_checkpointed_validation_rejects_before_launch(lib):
    p = ctypes.c_void_p(4096)

    def ck(every, buf, rows, dt=1):
        return lib.kda_chunk_fwd_checkpointed(dt, 1, 64, 1, 128, 128, p, p, p, p, p, None, None,
                                              1, p, None, every, buf, rows, None, None)
    assert ck(24, p, 4) == 1                       # interval not a multiple of 16
    assert ck(0, p, 4) == 1
    assert ck(16, p, -1) == 1
    assert ck(16, ctypes.c_void_p(4104), 4) == 4   # buffer needs 16-byte alignment
    assert ck(16, p, 4, dt=9) == 2
    p0 = ctypes.c_void_p(4096)
    assert lib.kda_decode_steps(1, 4, 0, 2, 128, 128, p0, p0, p0, p0, p0, None, p0, p0,
                                None, None) == 1   # K must be >= 1
    assert lib.kda_decode_steps(1, 4, 3, 2, 128, 128, p0, p0, p0, p0, p0, ctypes.c_void_p(4098),
                                p0, p0, None, None) == 4   # accepted needs 4-byte alignment


def test_prep_and_gate_output_buffers_are_checked():
    """Caller-supplied output buffers of the pre/post passes get the same
    shape / dtype / device / contiguity checks as inputs (CPU tensors stand
    in for device ones: only the host-side checks run)."""
    import torch
    B, T, H, d, dt, dev = 1, 8, 2, 32, torch.bfloat16, torch.device("cpu")
    ok = lambda: torch.empty((B, T, H, d), dtype=dt)
    beta = torch.empty((B, T, H), dtype=dt)
    q, k, v, b = kda._prep_outputs((ok(), ok(), ok(), beta), B, T, H, d, dt, dev, True)
    assert b is beta
    with pytest.raises(ValueError):          # too short
        kda._prep_outputs((torch.empty((B, T - 1, H, d), dtype=dt), ok(), ok(), beta),
                          B, T, H, d, dt, dev, True)
    with pytest.raises(TypeError):           # wrong dtype
        kda._prep_outputs((ok(), ok().float(), ok(), beta), B, T, H, d, dt, dev, True)
    with pytest.raises(ValueError):          # not contiguous
        kda._prep_outputs((ok(), ok(), torch.empty((B, T, d, H), dtype=dt).transpose(2, 3), beta),
                          B, T, H, d, dt, dev, True)
    with pytest.raises(ValueError):          # beta buffer missing while beta_logit is given
        kda._prep_outputs((ok(), ok(), ok(), None), B, T, H, d, dt, dev, True)
    with pytest.raises(ValueError):          # beta buffer given without beta_logit
        kda._prep_outputs((ok(), ok(), ok(), beta), B, T, H, d, dt, dev, False)
    with pytest.raises(TypeError):
        kda._prep_outputs((ok(), ok(), ok()), B, T, H, d, dt, dev, False)
    o = torch.empty((5, d), dtype=dt)
    assert kda._gate_output(None, o).shape == o.shape
    with pytest.raises(ValueError):
        kda._gate_output(torch.empty((4, d), dtype=dt), o)
    with pytest.raises(TypeError):
        kda._gate_output(torch.empty((5, d), dtype=torch.float32), o)


def test_selftest_wait_limit_is_validated(lib):
    # out-of-range limits are refused on the host, before any launch
    assert lib.kda_selftest_bounded_wait(0, None) == 1
    assert lib.kda_selftest_bounded_wait(100001, None) == 1


def _split(lib, dt=1, B=1, T=1024, H=2, dk=128, dv=128, ptr=4096, N=1, tau=256, ws=4096,
           ws_bytes=1 << 40, cu=None):
    p = ctypes.c_void_p(ptr)
    return lib.kda_chunk_fwd_split(dt, B, T, H, dk, dv, p, p, p, p, p, None, cu, N, tau, p, None,
                                   ctypes.c_void_p(ws) if ws else None, ws_bytes, None, None)


def test_split_validation_rejects_before_launch(lib):
    # Every case fails validation, so no pointer is dereferenced and no CUDA call is made.
    assert _split(lib, dt=0) == 3                 # fp32: the split runs on the bf16 tensor-core path
    assert _split(lib, dk=64, dv=64) == 3
    assert _split(lib, dt=7) == 2
    assert _split(lib, tau=0) == 1 and _split(lib, tau=40) == 1 and _split(lib, tau=-16) == 1
    assert _split(lib, B=2, N=1) == 1             # N must equal B without cu_seqlens
    assert _split(lib, ws=0) == 1                 # workspace required
    assert _split(lib, ws=4096 + 16) == 4         # workspace 256-byte aligned
    need = lib.kda_chunk_fwd_split_workspace(1, 1024, 2, 128, 128, 1, 256)
    assert need > 0
    assert _split(lib, ws_bytes=need - 1) == 1    # too small
    assert _split(lib, ptr=4096 + 2) == 4         # misaligned tensors


def test_split_workspace_and_segment_helpers(lib):
    ws = lib.kda_chunk_fwd_split_workspace
    # rejected sizes give 0
    assert ws(1, 1024, 2, 64, 64, 1, 256) == 0 and ws(1, 1024, 2, 128, 128, 1, 24) == 0
    assert ws(1, 1024, 2, 128, 128, 0, 256) == 0
    # grows with the tokens (second output) and the virtual chains (states)
    a, b = ws(1, 1024, 2, 128, 128, 1, 256), ws(1, 2048, 2, 128, 128, 1, 256)
    c = ws(1, 1024, 2, 128, 128, 1, 128)
    assert 0 < a < b and a < c
    assert a >= 1024 * 2 * 128 * 2 + 2 * 2 * 128 * 128 * 4   # out2 plus two state sets
    seg = lib.kda_split_segment_tokens
    # 12 chains on 152 SMs: 6 segments (11 chains each) for equal lengths, 5 for packed
    assert seg(1, 131072, 12, 1, 0, 152) == 131072 // 6 // 16 * 16 + 16 * (131072 // 6 % 16 != 0)
    t5 = seg(1, 131072, 12, 1, 1, 152)
    assert t5 % 16 == 0 and -(-131072 // t5) == 5
    # 96 chains (the layer shape): no split fits one wave
    assert seg(1, 8192, 96, 1, 0, 152) == 0
    assert seg(1, 8192, 0, 1, 0, 152) == 0 and seg(1, 8192, 12, 1, 0, 0) == 0
    for tau, n in ((seg(1, 8192, 12, 1, 0, 152), 6), (seg(1, 100000, 4, 1, 0, 152), 19)):
        assert tau % 16 == 0 and -(-(8192 if n == 6 else 100000) // tau) <= n
