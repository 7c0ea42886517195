"""kda_chunk_fwd_split_noalloc: the segment-split prefill for callers that
cannot allocate device memory (a process whose device memory all belongs to
its own caching pool, or a C caller without a device allocator), with its
scratch in a fixed 64 MiB buffer inside the library.

Through the C ABI, two calls in a row on different inputs each match the
workspace entry point (kda_chunk_fwd_split) within the prefill tolerance, so
nothing left in the shared buffer by the first call leaks into the second;
sizes beyond the buffer are refused without touching the GPU.  This file is
collected last on purpose.
"""
import pytest
import torch

from gated_delta_rule_11_gb300 import inputs, kda
from gated_delta_rule_11_gb300 import build as kbuild
from tests._parity import TOL, assert_close


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kda.load_library()


def test_sizes_beyond_the_static_buffer_are_refused():
    # 96 heads x 8192 tokens need far more scratch than the buffer holds:
    # refused before any CUDA call (fake, aligned device pointers).
    lib = kda.load_library()
    assert lib.kda_chunk_fwd_split_workspace(1, 8192, 96, 128, 128, 1, 1024) > kda.SPLIT_SCRATCH_BYTES
    p = __import__("ctypes").c_void_p(4096)
    st = lib.kda_chunk_fwd_split_noalloc(1, 1, 8192, 96, 128, 128, p, p, p, p, p, None, None, 1,
                                         1024, p, None, None, None)
    assert kda._STATUS[st] == "KDA_ERR_SCRATCH"
    assert b"scratch" in lib.kda_status_str(st)


@pytest.mark.gpu
def test_two_calls_in_a_row_match_the_workspace_entry_point():
    cases = [
        (inputs.Workload("noalloc", "prefill", H=2, dk=128, dv=128, dtype="bf16", z_std=2.0,
                         s0_std=0.1, seed=41, B=1, T=3000), 512),
        (inputs.Workload("noalloc", "prefill", H=3, dk=128, dv=128, dtype="bf16", z_std=1.0,
                         s0_std=0.1, seed=42, seqlens=(700, 0, 33, 1500)), 256),
    ]
    for w, tau in cases:
        inp = inputs.make_prefill_inputs(w, device="cuda")
        args = [inp[n] for n in ("q", "k", "v", "g_raw", "beta")]
        need = kda.split_workspace_bytes(1, inp["q"].shape[1], w.H, 128, 128, w.n_seqs, tau)
        assert 0 < need <= kda.SPLIT_SCRATCH_BYTES
        ref_out, ref_fin = kda.kda_chunk_fwd_split(*args, inp["init_state"], inp["cu_seqlens"],
                                                   segment_tokens=tau)
        out = torch.empty_like(inp["v"])
        fin = torch.empty_like(ref_fin)
        kda.kda_chunk_fwd_split_noalloc(*args, inp["init_state"], inp["cu_seqlens"],
                                        segment_tokens=tau, out=out, final_state=fin)
        torch.cuda.synchronize()
        assert_close("no-alloc split out", out, ref_out.float().double().cpu().numpy(),
                     TOL[torch.bfloat16])
        assert_close("no-alloc split final_state", fin, ref_fin.double().cpu().numpy(),
                     TOL[torch.bfloat16])
    kda.check_device_status()
