"""Seeded synthetic inputs for the KDA operator (shared by the tests, the
benchmark and the smoke check).

This module only draws random numbers in the shapes and distributions of the
workloads; it holds none of the operator's arithmetic.  The recipe follows the
model's KDA layer shape (96 heads, head dimension 128; "Kimi K3：从三条信息流到
完整系统", §模型账本与公开边界) and the operator's input contract: q and k
arrive L2-normalised per token and head, beta already in (0, 1)
(§从投影到 Chunkwise 的完整接口, eq. (2) puts L2Norm and Sigmoid in the
projection chain before the operator).

Recipe (all draws in fp32 from one ``torch.Generator`` seeded per workload,
then cast to the input dtype):

* q, k ~ N(0, 1), each token/head vector divided by its L2 norm;
* v ~ N(0, 1);
* beta = sigmoid(N(0, 1));
* gate pre-activation z ~ N(0, z_std) (z_std = 1 or 2; the second argument
  of N(., .) is the standard deviation);
* initial state S_0 ~ N(0, s0_std) in fp32, or absent (zeros).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                  # "prefill" or "decode"
    H: int
    dk: int
    dv: int
    dtype: str                 # "f32" or "bf16" (state is always fp32)
    z_std: float
    s0_std: float              # 0 -> no initial state (zeros)
    seed: int
    B: int = 1
    T: int = 0
    seqlens: tuple = field(default=())   # packed sequences (varlen) if non-empty
    N: int = 0                 # decode: number of sequences
    steps: int = 0             # decode: consecutive steps
    drafts: int = 0            # speculative replay: tokens verified per sequence

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def total_tokens(self) -> int:
        if self.kind in ("decode", "spec"):
            return self.N
        return sum(self.seqlens) if self.seqlens else self.B * self.T

    @property
    def n_seqs(self) -> int:
        if self.kind in ("decode", "spec"):
            return self.N
        return len(self.seqlens) if self.seqlens else self.B


# The five workloads of the operator's specification, by what they are.
WORKLOADS = {
    "tiny_f32_T64_d32": Workload("tiny_f32_T64_d32", "prefill", H=1, dk=32, dv=32, dtype="f32",
                                 z_std=1.0, s0_std=0.0, seed=0, B=1, T=64),
    "small_bf16_B2_H4_T1024": Workload("small_bf16_B2_H4_T1024", "prefill", H=4, dk=128, dv=128,
                                       dtype="bf16", z_std=1.0, s0_std=0.1, seed=1, B=2, T=1024),
    "layer_bf16_H96_T8192": Workload("layer_bf16_H96_T8192", "prefill", H=96, dk=128, dv=128,
                                     dtype="bf16", z_std=2.0, s0_std=0.0, seed=2, B=1, T=8192),
    "varlen_bf16_H96_237568": Workload("varlen_bf16_H96_237568", "prefill", H=96, dk=128, dv=128,
                                       dtype="bf16", z_std=2.0, s0_std=0.0, seed=3,
                                       seqlens=(131072, 65536, 32768, 8192)),
    # The layer's 96 heads sharded 8 ways by head (12 per GPU), one
    # 131,072-token sequence: fewer chains than multiprocessors, the shape
    # the segment split is for.
    "tp8_bf16_H12_T131072": Workload("tp8_bf16_H12_T131072", "prefill", H=12, dk=128, dv=128,
                                     dtype="bf16", z_std=2.0, s0_std=0.0, seed=6, B=1, T=131072),
    "decode_bf16_N256_H96": Workload("decode_bf16_N256_H96", "decode", H=96, dk=128, dv=128,
                                     dtype="bf16", z_std=2.0, s0_std=0.1, seed=4, N=256, steps=100),
    # Speculative replay: 8 tokens verified per sequence (the last committed
    # token and 7 drafts), of which an accepted prefix of 1..8 is replayed.
    "spec_bf16_N256_H96_K8": Workload("spec_bf16_N256_H96_K8", "spec", H=96, dk=128, dv=128,
                                      dtype="bf16", z_std=2.0, s0_std=0.1, seed=5, N=256,
                                      steps=20, drafts=8),
}
WORKLOAD_ORDER = list(WORKLOADS)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def _draw(shape, g, device, std=1.0):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def make_prefill_inputs(w: Workload, device="cpu", seed: int | None = None, *,
                        B: int | None = None, T: int | None = None, seqlens=None,
                        H: int | None = None):
    """Draw one prefill batch.  Optional overrides shrink the shapes for tests.

    Returns a dict: q, k, g_raw [B, T, H, dk]; v [B, T, H, dv]; beta [B, T, H]
    (all in the workload dtype); init_state [N, H, dk, dv] fp32 or None;
    cu_seqlens int32 [N+1] (on ``device``) or None.
    """
    seed = w.seed if seed is None else seed
    H = w.H if H is None else H
    seqlens = w.seqlens if seqlens is None else tuple(seqlens)
    if seqlens:
        Bq, Tq, N = 1, int(sum(seqlens)), len(seqlens)
    else:
        Bq = w.B if B is None else B
        Tq = w.T if T is None else T
        N = Bq
    g = _gen(device, seed)
    dt = w.torch_dtype
    q = _unit_rows(_draw((Bq, Tq, H, w.dk), g, device)).to(dt)
    k = _unit_rows(_draw((Bq, Tq, H, w.dk), g, device)).to(dt)
    v = _draw((Bq, Tq, H, w.dv), g, device).to(dt)
    beta = torch.sigmoid(_draw((Bq, Tq, H), g, device)).to(dt)
    g_raw = _draw((Bq, Tq, H, w.dk), g, device, w.z_std).to(dt)
    init_state = _draw((N, H, w.dk, w.dv), g, device, w.s0_std) if w.s0_std > 0 else None
    cu = None
    if seqlens:
        c = [0]
        for L in seqlens:
            c.append(c[-1] + int(L))
        cu = torch.tensor(c, dtype=torch.int32, device=device)
    return dict(q=q, k=k, v=v, g_raw=g_raw, beta=beta, init_state=init_state, cu_seqlens=cu)


def make_decode_state(w: Workload, device="cpu", seed: int | None = None, *,
                      N: int | None = None, H: int | None = None):
    """The initial recurrent state [N, H, dk, dv] fp32 ~ N(0, s0_std)."""
    seed = w.seed if seed is None else seed
    N = w.N if N is None else N
    H = w.H if H is None else H
    g = _gen(device, seed * 1_000_003 + 7)
    return _draw((N, H, w.dk, w.dv), g, device, w.s0_std)


def make_decode_token(w: Workload, step: int, device="cpu", seed: int | None = None, *,
                      N: int | None = None, H: int | None = None):
    """One token per sequence for decode step ``step``.

    Returns q, k, g_raw [N, H, dk]; v [N, H, dv]; beta [N, H] in the workload dtype.
    """
    seed = w.seed if seed is None else seed
    N = w.N if N is None else N
    H = w.H if H is None else H
    g = _gen(device, seed * 1_000_003 + 1009 * (step + 1))
    dt = w.torch_dtype
    q = _unit_rows(_draw((N, H, w.dk), g, device)).to(dt)
    k = _unit_rows(_draw((N, H, w.dk), g, device)).to(dt)
    v = _draw((N, H, w.dv), g, device).to(dt)
    beta = torch.sigmoid(_draw((N, H), g, device)).to(dt)
    g_raw = _draw((N, H, w.dk), g, device, w.z_std).to(dt)
    return dict(q=q, k=k, v=v, g_raw=g_raw, beta=beta)


def make_decode_drafts(w: Workload, step: int, device="cpu", seed: int | None = None, *,
                       N: int | None = None, H: int | None = None, K: int | None = None,
                       min_accepted: int = 1):
    """One speculative-replay batch: K verified tokens per sequence and how
    many of them each sequence accepts.

    Returns q, k, g_raw [N, K, H, dk]; v [N, K, H, dv]; beta [N, K, H] in the
    workload dtype, and accepted int32 [N] drawn uniformly from
    [min_accepted, K].
    """
    seed = w.seed if seed is None else seed
    N = w.N if N is None else N
    H = w.H if H is None else H
    K = w.drafts if K is None else K
    g = _gen(device, seed * 1_000_003 + 7919 * (step + 1))
    dt = w.torch_dtype
    q = _unit_rows(_draw((N, K, H, w.dk), g, device)).to(dt)
    k = _unit_rows(_draw((N, K, H, w.dk), g, device)).to(dt)
    v = _draw((N, K, H, w.dv), g, device).to(dt)
    beta = torch.sigmoid(_draw((N, K, H), g, device)).to(dt)
    g_raw = _draw((N, K, H, w.dk), g, device, w.z_std).to(dt)
    accepted = torch.randint(min_accepted, K + 1, (N,), generator=g, device=device,
                             dtype=torch.int32)
    return dict(q=q, k=k, v=v, g_raw=g_raw, beta=beta, accepted=accepted)


def make_prep_inputs(T: int, H: int, d: int, dtype: str = "bf16", device="cpu", seed: int = 7,
                     N_state: int = 0):
    """Pre/post pass inputs: x_qkv [1, T, 3, H, d] ~ N(0, 1) (projection
    outputs), conv taps [3, H, d, 4] ~ N(0, 0.5) fp32, beta logits [1, T, H]
    ~ N(0, 1), and (N_state > 0) conv states [N_state, 3, 3, H, d] ~ N(0, 1)."""
    g = _gen(device, seed * 1_000_003 + 17)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    x = _draw((1, T, 3, H, d), g, device).to(dt)
    w = _draw((3, H, d, 4), g, device, 0.5)
    bl = _draw((1, T, H), g, device).to(dt)
    st = _draw((N_state, 3, 3, H, d), g, device).to(dt) if N_state else None
    return dict(x_qkv=x, conv_w=w, beta_logit=bl, conv_state=st)


def make_post_inputs(rows: int, d: int, dtype: str = "bf16", device="cpu", seed: int = 8):
    """Output-gate inputs: o [rows, d] ~ N(0, 0.3) (operator outputs), gate
    logits ~ N(0, 1), norm weight [d] ~ U(0.5, 1.5) fp32."""
    g = _gen(device, seed * 1_000_003 + 29)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    o = _draw((rows, d), g, device, 0.3).to(dt)
    gate = _draw((rows, d), g, device).to(dt)
    w = torch.rand((d,), generator=g, device=device, dtype=torch.float32) + 0.5
    return dict(o=o, gate=gate, norm_w=w)
