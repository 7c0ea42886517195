"""Failure detection without a fault: a bounded device wait that gives up is
reported on the host, and the context stays usable.

The library's self-test kernel waits on a barrier that nothing arrives at,
with the same bounded wait its prefill and prep kernels use (no copy or
tensor-core work is in flight), so the wait runs out by construction, not
by hanging anything."""
import pytest
import torch

from gated_delta_rule_11_gb300 import build as kbuild
from gated_delta_rule_11_gb300 import inputs, kda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kda.load_library()


def test_timed_out_wait_is_reported_then_cleared():
    kda.check_device_status()                       # nothing pending before
    kda.selftest_bounded_wait(1000)                 # 1 ms
    with pytest.raises(kda.KdaError) as ei:
        kda.check_device_status()
    assert ei.value.status_name == "KDA_ERR_TIMEOUT"
    kda.check_device_status()                       # the report is cleared


def test_context_usable_after_a_timeout():
    kda.selftest_bounded_wait(500)
    with pytest.raises(kda.KdaError):
        kda.check_device_status()
    w = inputs.Workload("after_timeout", "prefill", H=2, dk=128, dv=128, dtype="bf16", z_std=1.0,
                        s0_std=0.0, seed=3, seqlens=(40, 17))
    inp = inputs.make_prefill_inputs(w, device="cuda")
    out, fin = kda.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta"], None,
                                 inp["cu_seqlens"])
    torch.cuda.synchronize()
    kda.check_device_status()
    assert torch.isfinite(out.float()).all() and torch.isfinite(fin).all()
