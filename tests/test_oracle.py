"""Pins for the fp64 oracle, against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: values the
pages print (tests/golden/), closed forms, invariants of eq. (1), a
brute-force product of the factored update matrices, the chunkwise form of
eqs. (3)-(4) derived independently, and the segment algebra of eq. (17).
Sources: "Kimi K3：从三条信息流到完整系统" (wineandchord.com).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng_global = np.random.default_rng(12345)


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def run(q, k, v, g, beta, S0=None, log_decay=True, **kw):
    """Single (sequence, head) chain: q,k,g [T,dk], v [T,dv], beta [T]."""
    T, dk = q.shape
    dv = v.shape[1]
    out, fin = oracle.kda_oracle_fwd(q[None, :, None], k[None, :, None], v[None, :, None],
                                     g[None, :, None], beta[None, :, None],
                                     init_state=None if S0 is None else S0[None, None],
                                     gate_is_log_decay=log_decay, **kw)
    return out[0, :, 0], fin[0, 0]


def rand_chain(rng, T, dk, dv, g_lo=-5.0, unit=True):
    q = rng.standard_normal((T, dk))
    k = rng.standard_normal((T, dk))
    if unit:
        q /= np.linalg.norm(q, axis=1, keepdims=True)
        k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, dv))
    g = rng.uniform(g_lo, 0.0, (T, dk))
    beta = rng.uniform(0.0, 1.0, T)
    return q, k, v, g, beta


# ----------------------------------------------------------------- page values

def test_worked_example_kda_step():
    """§KDA 是带逐通道遗忘的 delta rule: the printed kda_step example."""
    gd = _golden("kda_step_worked_example.json")
    S0 = np.array(gd["state"])
    k = np.array(gd["key"])[None]
    v = np.array(gd["value"])[None]
    q = np.array(gd["query"])[None]
    g = np.log(np.array(gd["alpha"]))[None]
    beta = np.array([gd["beta"]])
    out, fin = run(q, k, v, g, beta, S0)
    np.testing.assert_allclose(fin, np.array(gd["expected_state"]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(out[0], np.array(gd["expected_out"]), rtol=0, atol=1e-15)


def test_worked_example_through_gate():
    """Same example, with alpha reached through eq. (5) from the logit z."""
    gd = _golden("kda_step_worked_example.json")
    alpha = np.array(gd["alpha"])
    p = np.log(alpha) / -5.0             # sigmoid(z) = log(alpha) / g_min
    z = np.log(p / (1.0 - p))
    out, fin = run(np.array(gd["query"])[None], np.array(gd["key"])[None],
                   np.array(gd["value"])[None], z[None], np.array([gd["beta"]]),
                   np.array(gd["state"]), log_decay=False)
    np.testing.assert_allclose(fin, np.array(gd["expected_state"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(out[0], np.array(gd["expected_out"]), rtol=0, atol=1e-13)


def test_bounded_decay_example():
    """§下界 log-decay 是一个 kernel 设计: the bounded_decay asserts, eq. (5)."""
    gd = _golden("bounded_decay_example.json")
    g = oracle.kda_oracle_gate(np.array(gd["z"]), gd["A_log"], gd["g_min"])
    assert np.all((g >= gd["g_lower"]) & (g <= gd["g_upper"]))
    alpha = np.exp(g)
    assert np.all((alpha >= math.exp(gd["alpha_lower_log"])) & (alpha <= gd["alpha_upper"]))
    import torch
    assert math.exp(-gd["tile_log_decay_lower"]) < torch.finfo(torch.bfloat16).max
    # z = 0 sits at the sigmoid midpoint: g = g_min / 2 exactly
    assert g[1] == -2.5


def test_gate_closed_forms():
    """eq. (5) against identities of the sigmoid: tanh form and reflection."""
    z = np.linspace(-40, 40, 801)
    for A in (0.0, 0.7, -1.3):
        g = oracle.kda_oracle_gate(z, A, -5.0)
        x = math.exp(A) * z
        np.testing.assert_allclose(g, -5.0 * 0.5 * (1.0 + np.tanh(x / 2.0)), rtol=1e-13, atol=1e-15)
        g_neg = oracle.kda_oracle_gate(-z, A, -5.0)
        np.testing.assert_allclose(g + g_neg, -5.0, rtol=0, atol=1e-13)   # sigma(x)+sigma(-x)=1
        # the per-head log-scale only rescales the logit
        np.testing.assert_allclose(g, oracle.kda_oracle_gate(x, 0.0, -5.0), rtol=1e-15, atol=0)
    # a different floor scales g linearly
    np.testing.assert_allclose(oracle.kda_oracle_gate(z, 0.0, -3.0),
                               0.6 * oracle.kda_oracle_gate(z, 0.0, -5.0), rtol=1e-14)


def test_gate_bounds_and_tile_bound():
    """Every retention factor is above e^-5 (strictly for |z| <= 30), and a
    16-token tile's cumulative log-decay stays in (-80, 0]."""
    z = np.concatenate([np.linspace(-30, 30, 601), rng_global.standard_normal(4000) * 2.0])
    g = oracle.kda_oracle_gate(z, 0.0, -5.0)
    assert np.all(g > -5.0) and np.all(g < 0.0)
    assert np.all(np.exp(g) > math.exp(-5.0))
    tiles = oracle.kda_oracle_gate(rng_global.standard_normal((500, 16)) * 6.0, 0.0, -5.0)
    s = tiles.sum(axis=1)
    assert np.all(s > -80.0) and np.all(s < 0.0)
    # saturated inputs reach the bounds inclusively (floating point)
    sat = oracle.kda_oracle_gate(np.array([-1e4, 1e4, -np.inf, np.inf]), 0.0, -5.0)
    np.testing.assert_array_equal(sat, [-0.0, -5.0, -0.0, -5.0])


# ----------------------------------------------------------------- closed forms

@pytest.mark.parametrize("T,dk,dv", [(1, 4, 3), (37, 8, 5), (70, 16, 16)])
def test_beta_zero_is_pure_decay(T, dk, dv):
    """beta = 0: no write, so S_t = Diag(prod_{s<=t} alpha_s) S_0 and o_t = S_t^T q_t."""
    rng = np.random.default_rng(T)
    q, k, v, g, _ = rand_chain(rng, T, dk, dv)
    S0 = rng.standard_normal((dk, dv))
    out, fin = run(q, k, v, g, np.zeros(T), S0)
    cum = np.cumsum(g, axis=0)
    np.testing.assert_allclose(fin, np.exp(cum[-1])[:, None] * S0, rtol=1e-13, atol=1e-15)
    for t in range(T):
        St = np.exp(cum[t])[:, None] * S0
        np.testing.assert_allclose(out[t], St.T @ q[t], rtol=1e-12, atol=1e-14)


def test_orthonormal_keys_exact_recall():
    """alpha = 1, beta = 1, orthonormal keys from S_0 = 0: a query equal to an
    earlier key returns that key's value exactly; writing a key twice
    overwrites (the delta rule of P1 §The sequence axis / eq. (1))."""
    rng = np.random.default_rng(7)
    d, T = 24, 20
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    k = Qm[:T].copy()
    v = rng.standard_normal((T, d))
    q = np.stack([k[t // 2] for t in range(T)])
    out, fin = run(q, k, v, np.zeros((T, d)), np.ones(T))
    for t in range(T):
        np.testing.assert_allclose(out[t], v[t // 2], rtol=0, atol=1e-12)
    np.testing.assert_allclose(fin, k.T @ v, rtol=0, atol=1e-12)
    # same gate through eq. (5): z = -inf gives g = 0 exactly
    out2, fin2 = run(q, k, v, np.full((T, d), -np.inf), np.ones(T), log_decay=False)
    np.testing.assert_array_equal(out2, out)
    # overwrite: (k, v1) then (k, v2) leaves S = k v2^T
    kk = np.stack([k[0], k[0]])
    vv = rng.standard_normal((2, d))
    o3, f3 = run(kk, kk, vv, np.zeros((2, d)), np.ones(2))
    np.testing.assert_allclose(f3, np.outer(k[0], vv[1]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(o3[1], vv[1], rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_delta_invariant_any_decay(seed):
    """beta = 1 and ||k|| = 1 give k_t^T S_t = v_t^T for any alpha and S_0,
    so the read with q_t = k_t returns v_t exactly (the worked example is
    one instance)."""
    rng = np.random.default_rng(100 + seed)
    T, dk, dv = 50, 16, 9
    _, k, v, g, _ = rand_chain(rng, T, dk, dv)
    S0 = rng.standard_normal((dk, dv))
    out, _ = run(k, k, v, g, np.ones(T), S0)
    np.testing.assert_allclose(out, v, rtol=0, atol=1e-12)


# ----------------------------------------------------------------- brute force

def brute_force(q, k, v, g, beta, S0):
    """eq. (1) in its factored form: A_t = (I - beta_t k_t k_t^T) Diag(alpha_t),
    S_t = A_t S_{t-1} + beta_t k_t v_t^T; plus the unrolled product for S_T."""
    T, dk = q.shape
    I = np.eye(dk)
    As, S, outs = [], S0.copy(), []
    for t in range(T):
        A = (I - beta[t] * np.outer(k[t], k[t])) @ np.diag(np.exp(g[t]))
        As.append(A)
        S = A @ S + beta[t] * np.outer(k[t], v[t])
        outs.append(S.T @ q[t])
    P = I.copy()
    for A in As:
        P = A @ P
    S_unrolled = P @ S0
    for t in range(T):
        R = I.copy()
        for s in range(t + 1, T):
            R = As[s] @ R
        S_unrolled = S_unrolled + R @ (beta[t] * np.outer(k[t], v[t]))
    return np.array(outs), S, S_unrolled


@pytest.mark.parametrize("T,dk,dv,unit", [(1, 3, 2, True), (5, 3, 2, False), (8, 5, 4, True),
                                          (8, 6, 7, False)])
def test_brute_force_product(T, dk, dv, unit):
    rng = np.random.default_rng(T * 31 + dk)
    q, k, v, g, beta = rand_chain(rng, T, dk, dv, unit=unit)
    S0 = rng.standard_normal((dk, dv))
    out, fin = run(q, k, v, g, beta, S0)
    bo, bS, bU = brute_force(q, k, v, g, beta, S0)
    np.testing.assert_allclose(bS, bU, rtol=0, atol=1e-12)
    np.testing.assert_allclose(out, bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(fin, bS, rtol=0, atol=1e-12)


# ----------------------------------------------------------------- chunkwise form

def chunk_form(q, k, v, g, beta, S0, C):
    """eqs. (3)-(4) with the UT transform written out: per chunk,
    Gamma_r = prod_{s<=r} alpha_s; L = StrictTril[(K*Gamma)(K/Gamma)^T];
    T = (I + Diag(beta) L)^-1; U = T Diag(beta) V; W = T Diag(beta)(K*Gamma);
    Vt = U - W S; O = (Q*Gamma) S + Tril[(Q*Gamma)(K/Gamma)^T] Vt;
    S <- Diag(Gamma_C) S + (K*Gamma_C/Gamma)^T Vt."""
    Tn = q.shape[0]
    S = S0.copy()
    out = np.zeros((Tn, v.shape[1]))
    for s in range(0, Tn, C):
        e = min(s + C, Tn)
        Q, K, V, G, bt = q[s:e], k[s:e], v[s:e], g[s:e], beta[s:e]
        b = np.cumsum(G, axis=0)
        Gam = np.exp(b)
        Kg, Kinv, Qg = K * Gam, K / Gam, Q * Gam
        n = e - s
        L = np.tril(Kg @ Kinv.T, -1)
        A = np.tril(Qg @ Kinv.T, 0)
        Tm = np.linalg.inv(np.eye(n) + np.diag(bt) @ L)
        U = Tm @ (bt[:, None] * V)
        W = Tm @ (bt[:, None] * Kg)
        Vt = U - W @ S
        out[s:e] = Qg @ S + A @ Vt
        S = np.exp(b[-1])[:, None] * S + (K * np.exp(b[-1] - b)).T @ Vt
    return out, S


@pytest.mark.parametrize("C", [16, 4, 64])
def test_chunk_form_matches_recurrence(C):
    """Verification item of the pages (recurrent vs chunked KDA numerical
    alignment), in fp64: several chunks and a ragged tail."""
    rng = np.random.default_rng(C)
    T, dk, dv = 16 * 5 + 7, 12, 10
    q, k, v, g, beta = rand_chain(rng, T, dk, dv, g_lo=-5.0 if C <= 16 else -1.0)
    S0 = rng.standard_normal((dk, dv)) * 0.3
    out, fin = run(q, k, v, g, beta, S0)
    co, cS = chunk_form(q, k, v, g, beta, S0, C)
    np.testing.assert_allclose(out, co, rtol=0, atol=1e-10)
    np.testing.assert_allclose(fin, cS, rtol=0, atol=1e-10)


# ----------------------------------------------------------------- eq. (17)

def test_resume_from_final_state():
    """Splitting a sequence and resuming from final_state reproduces the unsplit run."""
    rng = np.random.default_rng(3)
    T, dk, dv = 90, 10, 6
    q, k, v, g, beta = rand_chain(rng, T, dk, dv)
    S0 = rng.standard_normal((dk, dv))
    out, fin = run(q, k, v, g, beta, S0)
    for p in (1, 17, 45, 89):
        o1, S1 = run(q[:p], k[:p], v[:p], g[:p], beta[:p], S0)
        o2, S2 = run(q[p:], k[p:], v[p:], g[p:], beta[p:], S1)
        np.testing.assert_allclose(np.concatenate([o1, o2]), out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(S2, fin, rtol=0, atol=1e-12)


def compose(right, left):
    """eq. (17): (M2, E2) o (M1, E1) = (M2 M1, M2 E1 + E2)."""
    (m2, e2), (m1, e1) = right, left
    return m2 @ m1, m2 @ e1 + e2


def segment_fragment(q, k, v, g, beta):
    """(M, E) of one segment, from the oracle alone: E = F(0) with the real
    values; M = F(I) with zero values (the state map is linear in S_0 and
    every value column evolves by the same M)."""
    dk = q.shape[1]
    _, E = run(q, k, v, g, beta, np.zeros((dk, v.shape[1])))
    _, M = run(q, k, np.zeros((len(q), dk)), g, beta, np.eye(dk))
    return M, E


def test_segment_transition_algebra():
    """§FlashKDA 与 KCP, eq. (17): per-segment fragments composed in order give
    every segment's entering state and the final state of the unsplit run."""
    rng = np.random.default_rng(11)
    T, dk, dv = 120, 8, 5
    q, k, v, g, beta = rand_chain(rng, T, dk, dv)
    S0 = rng.standard_normal((dk, dv))
    _, fin = run(q, k, v, g, beta, S0)
    cuts = [0, 13, 50, 51, 99, 120]
    frags = [segment_fragment(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b])
             for a, b in zip(cuts[:-1], cuts[1:])]
    # S_in^(i) = sum_{j<i} (prod_{l=j+1}^{i-1} M_l) E_j, with S_0 entering as E_{-1}
    acc = (np.eye(dk), S0)
    for i, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
        _, S_entering = run(q[:a], k[:a], v[:a], g[:a], beta[:a], S0) if a > 0 else (None, S0)
        np.testing.assert_allclose(acc[1], S_entering, rtol=0, atol=1e-11)
        acc = compose(frags[i], acc)
    np.testing.assert_allclose(acc[1], fin, rtol=0, atol=1e-11)
    # the printed associativity check, with random 2x2 fragments
    a, b, c = [(rng.standard_normal((2, 2)), rng.standard_normal((2, 1))) for _ in range(3)]
    l, r = compose(compose(c, b), a), compose(c, compose(b, a))
    np.testing.assert_allclose(l[0], r[0], rtol=1e-14)
    np.testing.assert_allclose(l[1], r[1], rtol=1e-14)


# ----------------------------------------------------------------- packing / options

def test_varlen_packing_is_independent_sequences():
    rng = np.random.default_rng(5)
    H, dk, dv = 3, 8, 6
    lens = [5, 0, 17, 1, 33]
    Tt = sum(lens)
    q = rng.standard_normal((1, Tt, H, dk))
    k = rng.standard_normal((1, Tt, H, dk))
    v = rng.standard_normal((1, Tt, H, dv))
    z = rng.standard_normal((1, Tt, H, dk)) * 2
    beta = rng.uniform(0, 1, (1, Tt, H))
    S0 = rng.standard_normal((len(lens), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    out, fin = oracle.kda_oracle_fwd(q, k, v, z, beta, S0, cu)
    for n, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        if b == a:
            np.testing.assert_array_equal(fin[n], S0[n])
            continue
        o1, f1 = oracle.kda_oracle_fwd(q[:, a:b], k[:, a:b], v[:, a:b], z[:, a:b],
                                       beta[:, a:b], S0[n:n + 1])
        np.testing.assert_array_equal(out[:, a:b], o1)
        np.testing.assert_array_equal(fin[n], f1[0])


def test_batch_equals_packed():
    rng = np.random.default_rng(6)
    B, T, H, dk, dv = 3, 21, 2, 8, 8
    args = [rng.standard_normal((B, T, H, d)) for d in (dk, dk, dv, dk)]
    beta = rng.uniform(0, 1, (B, T, H))
    o1, f1 = oracle.kda_oracle_fwd(*args, beta)
    packed = [a.reshape(1, B * T, H, -1) for a in args]
    cu = np.arange(B + 1, dtype=np.int32) * T
    o2, f2 = oracle.kda_oracle_fwd(*packed, beta.reshape(1, B * T, H), None, cu)
    np.testing.assert_array_equal(o1.reshape(1, B * T, H, dv), o2)
    np.testing.assert_array_equal(f1, f2)


def test_scale_and_head_log_scale():
    rng = np.random.default_rng(8)
    B, T, H, dk, dv = 1, 30, 2, 8, 4
    q, k, v, z = [rng.standard_normal((B, T, H, d)) for d in (dk, dk, dv, dk)]
    beta = rng.uniform(0, 1, (B, T, H))
    o1, f1 = oracle.kda_oracle_fwd(q, k, v, z, beta)
    o2, f2 = oracle.kda_oracle_fwd(q, k, v, z, beta, scale=0.125)
    np.testing.assert_allclose(o2, 0.125 * o1, rtol=1e-15, atol=0)
    np.testing.assert_array_equal(f1, f2)
    A = np.array([0.5, -0.25])
    o3, f3 = oracle.kda_oracle_fwd(q, k, v, z, beta, A_log=A)
    o4, f4 = oracle.kda_oracle_fwd(q, k, v, z * np.exp(A)[None, None, :, None], beta)
    np.testing.assert_allclose(o3, o4, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(f3, f4, rtol=1e-12, atol=1e-13)


def test_decode_is_prefill_one_token_at_a_time():
    rng = np.random.default_rng(9)
    N, H, dk, dv, steps = 3, 2, 8, 6, 5
    S = rng.standard_normal((N, H, dk, dv))
    toks = [[rng.standard_normal((N, H, d)) for d in (dk, dk, dv, dk)] +
            [rng.uniform(0, 1, (N, H))] for _ in range(steps)]
    outs = []
    S_dec = S
    for q, k, v, z, b in toks:
        o, S_dec = oracle.kda_oracle_decode(q, k, v, z, b, S_dec)
        outs.append(o)
    stack = lambda i: np.stack([t[i] for t in toks], axis=1)   # [N, steps, H, d]
    o_pf, S_pf = oracle.kda_oracle_fwd(stack(0), stack(1), stack(2), stack(3), stack(4), S)
    np.testing.assert_allclose(np.stack(outs, axis=1), o_pf, rtol=0, atol=1e-13)
    np.testing.assert_allclose(S_dec, S_pf, rtol=0, atol=1e-13)


def test_threads_are_deterministic():
    rng = np.random.default_rng(10)
    B, T, H, dk, dv = 2, 40, 5, 8, 8
    args = [rng.standard_normal((B, T, H, d)) for d in (dk, dk, dv, dk)]
    beta = rng.uniform(0, 1, (B, T, H))
    o1, f1 = oracle.kda_oracle_fwd(*args, beta, nthreads=1)
    o2, f2 = oracle.kda_oracle_fwd(*args, beta, nthreads=7)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(f1, f2)


def test_rejects_bad_cu_seqlens():
    z = np.zeros((1, 4, 1, 2))
    with pytest.raises(ValueError):
        oracle.kda_oracle_fwd(z, z, z, z, np.zeros((1, 4, 1)), None, np.array([0, 3, 2, 4]))


# ----------------------------------------------------------------- planted mistakes

def _mutant(kind):
    """Plausible wrong restatements of eq. (1), to show the pins catch them."""
    def step_all(q, k, v, g, beta, S0):
        S = S0.copy()
        outs = []
        for t in range(len(q)):
            a = np.exp(g[t])
            if kind == "decay_columns":
                D = S * a[None, : S.shape[1]] if S.shape[1] == len(a) else S * a[0]
            elif kind == "correct_before_decay":
                D = S
            else:
                D = a[:, None] * S
            e = v[t] - D.T @ k[t]
            if kind == "sign":
                e = v[t] + D.T @ k[t]
            Snew = D + beta[t] * np.outer(k[t], e)
            if kind == "correct_before_decay":
                Snew = a[:, None] * Snew
            outs.append((S if kind == "read_before_write" else Snew).T @ q[t])
            S = Snew
        return np.array(outs), S
    return step_all


@pytest.mark.parametrize("kind", ["decay_columns", "correct_before_decay", "sign",
                                  "read_before_write"])
def test_pins_catch_planted_mistakes(kind):
    """Each mutant of the recurrence fails the worked-example pin or the
    delta invariant, while the oracle passes both (tests above)."""
    gd = _golden("kda_step_worked_example.json")
    mut = _mutant(kind)
    o, S = mut(np.array(gd["query"])[None], np.array(gd["key"])[None],
               np.array(gd["value"])[None], np.log(np.array(gd["alpha"]))[None],
               np.array([gd["beta"]]), np.array(gd["state"]))
    ok_example = (np.allclose(S, gd["expected_state"]) and np.allclose(o[0], gd["expected_out"]))
    rng = np.random.default_rng(1)
    _, k, v, g, _ = rand_chain(rng, 12, 6, 6)
    S0 = rng.standard_normal((6, 6))
    o2, _ = mut(k, k, v, g, np.ones(12), S0)
    ok_invariant = np.allclose(o2, v)
    assert not (ok_example and ok_invariant)


# ----------------------------------------------------------------- gate variants

def _run_mode(q, k, v, z, beta, S0=None, mode="bounded", scalar=False, **kw):
    """Single chain with an explicit gate mode; z [T, dk] or [T] (scalar)."""
    out, fin = oracle.kda_oracle_fwd(q[None, :, None], k[None, :, None], v[None, :, None],
                                     None if z is None else z[None, :, None], beta[None, :, None],
                                     init_state=None if S0 is None else S0[None, None],
                                     gate_mode=mode, gate_scalar=scalar, **kw)
    return out[0, :, 0], fin[0, 0]


def test_neg_softplus_gate_closed_forms():
    """Kimi Linear's negative softplus: g(0) = -log 2, g -> -z for large z
    (unbounded below), g -> -e^z for very negative z, and the per-head scale
    multiplies the input as in eq. (5)."""
    g = oracle.kda_oracle_log_decay(np.array([0.0, 40.0, 100.0, -40.0, 2.0]), "neg_softplus")
    np.testing.assert_allclose(g[0], -math.log(2.0), rtol=1e-15)
    np.testing.assert_allclose(g[1], -40.0, rtol=1e-15)
    assert g[2] == -100.0                       # no floor: far below g_min = -5
    np.testing.assert_allclose(g[3], -math.exp(-40.0), rtol=1e-12)
    np.testing.assert_allclose(g[4], -math.log1p(math.exp(2.0)), rtol=1e-15)
    ga = oracle.kda_oracle_log_decay(np.array([1.5]), "neg_softplus", A_log=0.7)
    gb = oracle.kda_oracle_log_decay(np.array([1.5 * math.exp(0.7)]), "neg_softplus")
    np.testing.assert_allclose(ga, gb, rtol=1e-15)
    assert oracle.kda_oracle_log_decay(np.array([3.0]), "log_decay")[0] == 3.0
    assert oracle.kda_oracle_log_decay(np.array([3.0]), "none")[0] == 0.0


def test_no_gate_is_the_plain_delta_rule():
    """gate mode "none" (alpha = 1): orthonormal keys with beta = 1 from S_0 =
    0 recall every stored value exactly, the textbook delta-rule property;
    and it equals a log-decay gate of 0."""
    rng = np.random.default_rng(41)
    d, T = 16, 12
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    k = Qm[:T].copy()
    v = rng.standard_normal((T, d))
    out, fin = _run_mode(k, k, v, None, np.ones(T), mode="none")
    np.testing.assert_allclose(out, v, rtol=0, atol=1e-12)
    np.testing.assert_allclose(fin, k.T @ v, rtol=0, atol=1e-12)
    q = rng.standard_normal((T, d))
    beta = rng.uniform(0, 1, T)
    S0 = rng.standard_normal((d, d))
    a = _run_mode(q, k, v, None, beta, S0, mode="none")
    b = _run_mode(q, k, v, np.zeros((T, d)), beta, S0, mode="log_decay")
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("mode", ["bounded", "neg_softplus", "log_decay"])
def test_scalar_gate_is_the_channel_gate_broadcast(mode):
    """Gated delta: one gate per token shared by all key channels equals the
    per-channel gate with that value in every channel."""
    rng = np.random.default_rng(43)
    T, dk, dv = 9, 6, 5
    q, k, v, _, beta = rand_chain(rng, T, dk, dv)
    z = rng.uniform(-3, 3, T) if mode != "log_decay" else rng.uniform(-4, 0, T)
    S0 = rng.standard_normal((dk, dv))
    a = _run_mode(q, k, v, z, beta, S0, mode=mode, scalar=True, A_log=np.array([0.3]))
    b = _run_mode(q, k, v, np.repeat(z[:, None], dk, 1), beta, S0, mode=mode,
                  A_log=np.array([0.3]))
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_scalar_gated_delta_brute_force():
    """Gated delta in matrix form, S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1}
    + beta_t k_t v_t^T with a scalar alpha_t = exp(g_t), on tiny inputs."""
    rng = np.random.default_rng(44)
    T, dk, dv = 7, 4, 3
    q, k, v, _, beta = rand_chain(rng, T, dk, dv, unit=False)
    z = rng.uniform(-6, 6, T)
    S0 = rng.standard_normal((dk, dv))
    out, fin = _run_mode(q, k, v, z, beta, S0, mode="neg_softplus", scalar=True)
    S = S0.copy()
    for t in range(T):
        alpha = math.exp(-math.log1p(math.exp(z[t])))          # = 1 / (1 + e^z)
        S = alpha * (np.eye(dk) - beta[t] * np.outer(k[t], k[t])) @ S + beta[t] * np.outer(k[t], v[t])
        np.testing.assert_allclose(out[t], S.T @ q[t], rtol=0, atol=1e-12)
    np.testing.assert_allclose(fin, S, rtol=0, atol=1e-12)


def test_unbounded_decay_wipes_the_state():
    """A negative-softplus gate with z = 60 gives alpha = e^{-60} per step:
    every step forgets the past (the carried term is ~1e-26), so S_t = beta_t
    k_t v_t^T and o_t = beta_t (k_t . q_t) v_t up to rounding.  Over a 16-token tile the cumulative
    log-decay reaches -960, far past the bounded gate's -80."""
    rng = np.random.default_rng(45)
    T, dk, dv = 20, 8, 5
    q, k, v, _, beta = rand_chain(rng, T, dk, dv)
    S0 = rng.standard_normal((dk, dv))
    out, fin = _run_mode(q, k, v, np.full((T, dk), 60.0), beta, S0, mode="neg_softplus")
    for t in range(T):
        np.testing.assert_allclose(out[t], beta[t] * (k[t] @ q[t]) * v[t], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(fin, beta[-1] * np.outer(k[-1], v[-1]), rtol=1e-13, atol=1e-15)
