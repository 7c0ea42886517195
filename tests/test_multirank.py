"""Multi-process paths on CPU (gloo, world size 2).

* The benchmark's replica timing: every rank reports its time and the
  maximum over ranks is taken (bench.reduce_max / barrier).
* Head partitioning of one workload (the benchmark's --partition heads):
  rank r runs heads [h0, h1) of every sequence, no exchange on the data
  path; gathering the ranks' slices reproduces the unsplit outputs exactly
  (the oracle stands in for the GPU path on these CPU ranks).
* Context parallelism over ranks ("Kimi K3：从三条信息流到完整系统",
  §FlashKDA 与 KCP, eq. 17): each rank owns a contiguous segment of one long
  sequence, computes its fragment (M, E) from zero state, one fixed-size
  all-gather exchanges the fragments, and each rank composes the fragments of
  the ranks before it into its entering state; running its segment from that
  state reproduces the unsplit sequence.  Fragments and segment runs use the
  fp64 oracle here (one GPU per box: the exchange is exercised on the host).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _bench_reduce(rank, world, port, q):
    _init(rank, world, port)
    import bench
    v = bench.reduce_max(10.0 + rank, world)
    bench.barrier(world)
    q.put((rank, v))
    dist.destroy_process_group()


def test_bench_max_over_ranks_gloo():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_bench_reduce, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 11.0, 1: 11.0}


def _inputs(T, dk, dv, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, T, 1, dk))
    k = rng.standard_normal((1, T, 1, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((1, T, 1, dv))
    z = rng.standard_normal((1, T, 1, dk)) * 2.0
    beta = rng.uniform(0, 1, (1, T, 1))
    S0 = rng.standard_normal((1, 1, dk, dv)) * 0.1
    return q, k, v, z, beta, S0


def _kcp_rank(rank, world, port, cuts, q_out):
    _init(rank, world, port)
    import oracle
    T, dk, dv = 96, 12, 7
    q, k, v, z, beta, S0 = _inputs(T, dk, dv, seed=5)
    a, b = cuts[rank], cuts[rank + 1]
    seg = lambda x: x[:, a:b]
    # local fragment: E = F(0) with the values, M = F(I) with zero values
    _, E = oracle.kda_oracle_fwd(seg(q), seg(k), seg(v), seg(z), seg(beta),
                                 np.zeros((1, 1, dk, dv)))
    _, M = oracle.kda_oracle_fwd(seg(q), seg(k), np.zeros((1, b - a, 1, dk)), seg(z), seg(beta),
                                 np.eye(dk)[None, None])
    frag = torch.from_numpy(np.concatenate([M[0, 0], E[0, 0]], axis=1))   # fixed size dk x (dk + dv)
    gathered = [torch.zeros_like(frag) for _ in range(world)]
    dist.all_gather(gathered, frag)                                          # the one exchange
    # entering state: S_in = M_{r-1} ... (M_0 S_0 + E_0) ... + E_{r-1}
    S_in = S0[0, 0].copy()
    for j in range(rank):
        Mj, Ej = gathered[j][:, :dk].numpy(), gathered[j][:, dk:].numpy()
        S_in = Mj @ S_in + Ej
    out, fin = oracle.kda_oracle_fwd(seg(q), seg(k), seg(v), seg(z), seg(beta), S_in[None, None])
    q_out.put((rank, out, fin))
    dist.destroy_process_group()


@pytest.mark.parametrize("cuts", [(0, 37, 96), (0, 1, 96), (0, 64, 96)])
def test_kcp_composition_over_two_ranks_gloo(cuts):
    import oracle
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_kcp_rank, args=(r, 2, port, cuts, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        r, out, fin = q.get(timeout=180)
        res[r] = (out, fin)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    qq, k, v, z, beta, S0 = _inputs(96, 12, 7, seed=5)
    ref_out, ref_fin = oracle.kda_oracle_fwd(qq, k, v, z, beta, S0)
    got = np.concatenate([res[0][0], res[1][0]], axis=1)
    np.testing.assert_allclose(got, ref_out, rtol=0, atol=1e-11)
    np.testing.assert_allclose(res[1][1], ref_fin, rtol=0, atol=1e-11)


def test_head_range_covers_every_head_once():
    from gated_delta_rule_11_gb300.partition import head_range
    for H, W in ((96, 1), (96, 2), (96, 8), (7, 3), (5, 5), (130, 8)):
        ranges = [head_range(r, W, H) for r in range(W)]
        assert ranges[0][0] == 0 and ranges[-1][1] == H
        for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
            assert a1 == b0
        sizes = [b - a for a, b in ranges]
        assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        head_range(0, 4, 3)
    with pytest.raises(ValueError):
        head_range(2, 2, 8)


def _heads_rank(rank, world, port, q_out):
    _init(rank, world, port)
    import oracle
    from gated_delta_rule_11_gb300 import inputs
    from gated_delta_rule_11_gb300.partition import shard_heads, unshard_heads
    w = inputs.Workload("heads", "prefill", H=5, dk=16, dv=8, dtype="f32", z_std=2.0, s0_std=0.1,
                        seed=11, seqlens=(9, 0, 23, 16))
    inp = inputs.make_prefill_inputs(w, device="cpu")
    sl = {n: shard_heads(inp[n], rank, world, axis=2) for n in ("q", "k", "v", "g_raw", "beta")}
    s0 = shard_heads(inp["init_state"], rank, world, axis=1)
    out, fin = oracle.kda_oracle_fwd(sl["q"], sl["k"], sl["v"], sl["g_raw"], sl["beta"], s0,
                                     inp["cu_seqlens"].numpy())
    outs = [None] * world
    fins = [None] * world
    dist.all_gather_object(outs, torch.from_numpy(out))      # reassembly only: no data-path exchange
    dist.all_gather_object(fins, torch.from_numpy(fin))
    if rank == 0:
        ref_out, ref_fin = oracle.kda_oracle_fwd(inp["q"], inp["k"], inp["v"], inp["g_raw"],
                                                 inp["beta"], inp["init_state"],
                                                 inp["cu_seqlens"].numpy())
        got_out = unshard_heads(outs, axis=2).numpy()
        got_fin = unshard_heads(fins, axis=1).numpy()
        q_out.put((bool((got_out == ref_out).all()), bool((got_fin == ref_fin).all()),
                   got_out.shape == ref_out.shape))
    dist.destroy_process_group()


def test_head_partition_reassembles_the_unsplit_run_gloo():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_heads_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    same_out, same_fin, same_shape = q.get(timeout=180)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert same_shape and same_out and same_fin
