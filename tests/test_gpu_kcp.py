"""Sequence split across ranks (KCP, "Kimi K3：从三条信息流到完整系统",
§FlashKDA 与 KCP, eq. (17)) through the C ABI: each rank holds the next slice
of tokens of the same sequences; ranks 1.. run their tokens from a zero state
and as the transition, the ranks all-gather one (S0, Phi) pair per sequence
and head (gloo, through host memory), and each composes the state entering
its tokens and corrects its outputs.

The ranks are separate processes sharing this machine's one GPU: no kernel
waits on another rank (the exchange is a host-side all-gather between
launches).  The concatenated outputs and the last rank's final state are
compared with the fp64 oracle on the whole sequences (max|gpu - ref| <=
2e-2 x RMS, bf16 inputs, fp32 state).
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

from gated_delta_rule_11_gb300 import build as kbuild
from gated_delta_rule_11_gb300 import inputs, kda
from tests._parity import TOL, assert_close, oracle_heads

pytestmark = pytest.mark.gpu


def _workload(world, Tr, seed):
    return inputs.Workload("kcp", "prefill", H=2, dk=128, dv=128, dtype="bf16", z_std=2.0, s0_std=0.1,
                           seed=seed, B=2, T=world * Tr)


def _rank_main(rank, world, port, Tr, seed, outdir):
    import torch.distributed as dist

    from gated_delta_rule_11_gb300 import partition
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.cuda.set_device(0)
        kda.load_library()
        inp = inputs.make_prefill_inputs(_workload(world, Tr, seed), device="cuda")
        sl = slice(rank * Tr, (rank + 1) * Tr)
        part = [inp[n][:, sl].contiguous() for n in ("q", "k", "v", "g_raw", "beta")]
        out, fin = partition.kcp_prefill(*part, inp["init_state"] if rank == 0 else None)
        torch.cuda.synchronize()
        kda.check_device_status()
        torch.save({"out": out.cpu(), "fin": fin.cpu()}, os.path.join(outdir, f"rank{rank}.pt"))
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world,Tr", [(2, 300), (3, 160)])
def test_kcp_ranks_match_the_oracle(tmp_path, world, Tr):
    kbuild.build()
    seed = 50 + world
    mp.spawn(_rank_main, args=(world, _free_port(), Tr, seed, str(tmp_path)), nprocs=world, join=True)
    parts = [torch.load(os.path.join(tmp_path, f"rank{r}.pt")) for r in range(world)]
    out = torch.cat([p["out"] for p in parts], dim=1)
    # the ranks' inputs, drawn the same way on the GPU (the CPU generator differs)
    inp = inputs.make_prefill_inputs(_workload(world, Tr, seed), device="cuda")
    ro, rf = oracle_heads(inp, [0, 1])
    assert_close(f"KCP {world} ranks out", out, ro, TOL[torch.bfloat16])
    assert_close(f"KCP {world} ranks final_state", parts[-1]["fin"], rf, TOL[torch.bfloat16])


def test_kcp_arguments_are_checked():
    kbuild.build()
    lib = kda.load_library()
    assert lib.kda_chunk_fwd_kcp_workspace(1, 0, 2, 128, 128) == 0      # T >= 1
    assert lib.kda_chunk_fwd_kcp_workspace(1, 64, 2, 64, 64) == 0       # d = 128 only
    ws = torch.empty(kda.kcp_workspace_bytes(1, 64, 2, 128, 128), dtype=torch.uint8, device="cuda")
    x = torch.zeros((1, 64, 2, 128), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros((1, 64, 2), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        kda.kda_chunk_fwd_kcp_part(x, x, x, x, b, ws[:100])
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_chunk_fwd_kcp_finish(torch.zeros((1, 1, 2, 2, 128, 128), device="cuda"), 0, ws, 1, 64, 2)
    assert ei.value.status_name == "KDA_ERR_ARG"   # rank 0 never finishes
