"""Pins of the fp64 oracle: checks against facts fixed by the pages and by mathematics, none of
which re-types the oracle's own loops.

Each ``pin_*`` function raises AssertionError when the oracle disagrees. They go through the
``oracle`` package, so ``oracle.use_library`` can point them at a deliberately broken build
(tests/test_oracle_mutants.py).

Sources: "【论文解读】 Qwen3.8 Flash Next" (wkq9411.github.io) §二.2 (HC, eq block: the widened
network equals Pre-Norm for static one-hot read/write), §二.4 (GatedNorm; GR eq rms, gate,
use_gate, s, write), §二.6 (eq rcv, eq auv; branches exchangeable at init);
"Qwen3.8-Flash-Next 架构笔记 · 06 / RESIDUAL" (cbphcr.github.io), two-branch example;
"Residual" (rainlin-net.pages.dev) §2.2 Pre-Norm.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as Fnn

import oracle
from oracle import dense

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _params(rng, nb, D, r, std=0.3, gamma_random=True):
    gamma = (1.0 + 0.3 * rng.standard_normal((nb, D))) if gamma_random else np.ones((nb, D))
    return {
        "gamma": gamma,
        "w_down": std * rng.standard_normal((r, nb * D)),
        "w_up": std * rng.standard_normal((nb * D, r)),
        "w_write": std * rng.standard_normal((nb, nb * D)),
    }


def _read(R, p, eps=1e-6, internals=False):
    return oracle.read(R, p["gamma"], p["w_down"], p["w_up"], p["w_write"], eps,
                       return_internals=internals)


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))


def _torch_rmsnorm(u, gamma, eps):
    """Textbook RMSNorm over the last axis (torch library routine)."""
    return Fnn.rms_norm(_t(u), (u.shape[-1],), weight=_t(gamma), eps=eps).numpy()


def _torch_gatednorm(u, gamma, W1, W2, eps):
    """GatedNorm(u) = RMSNorm(u) ⊙ σ(W2 SiLU(W1 RMSNorm(u))), Digest §二.4, from torch ops."""
    un = Fnn.rms_norm(_t(u), (u.shape[-1],), weight=_t(gamma), eps=eps)
    gate = torch.sigmoid(Fnn.linear(Fnn.silu(Fnn.linear(un, _t(W1))), _t(W2)))
    return (un * gate).numpy(), un.numpy()


# ---------------------------------------------------------------------------------------------

def pin_dense_bruteforce():
    """Loop formulation (C) == matrix formulation (numpy) on tiny shapes, incl. n_r != 4."""
    rng = np.random.default_rng(101)
    for (n, nb, D, r, eps) in [(1, 1, 1, 1, 1e-6), (3, 2, 3, 2, 1e-6), (4, 4, 8, 3, 0.3),
                               (2, 4, 17, 5, 1e-6), (5, 3, 16, 4, 1e-2), (2, 4, 32, 8, 0.0)]:
        R = rng.standard_normal((n, nb, D)) * rng.uniform(0.1, 10, size=(1, nb, 1))
        p = _params(rng, nb, D, r, std=0.5)
        x, s = _read(R, p, eps)
        x2, s2 = dense.read(R, p["gamma"], p["w_down"], p["w_up"], p["w_write"], eps)
        assert _rel(x, x2) < 1e-12 and _rel(s, s2) < 1e-12, (n, nb, D, r)
        y = rng.standard_normal((n, D))
        assert _rel(oracle.write(R, y, s), dense.write(R, y, s)) < 1e-14


def pin_zero_down_projection():
    """W_d = 0 ⇒ z = 0 ⇒ h = SiLU(0) = 0 ⇒ every gate is σ(0) = 1/2 exactly, so
    x = (1/(2 n_r)) Σ_i RMSNorm(R_i; γ_i) with RMSNorm from torch."""
    rng = np.random.default_rng(102)
    for nb in (4, 2):
        n, D, r, eps = 5, 24, 4, 1e-6
        R = rng.standard_normal((n, nb, D))
        p = _params(rng, nb, D, r)
        p["w_down"] = np.zeros_like(p["w_down"])
        x, s, G, inv = _read(R, p, eps, internals=True)
        assert np.all(G == 0.5)
        expect = sum(_torch_rmsnorm(R[:, i, :], p["gamma"][i], eps) for i in range(nb)) / (2 * nb)
        assert _rel(x, expect) < 1e-13


def pin_zero_up_projection():
    """W_u = 0 ⇒ G ≡ σ(0) = 1/2 whatever W_d does."""
    rng = np.random.default_rng(103)
    R = rng.standard_normal((3, 4, 16))
    p = _params(rng, 4, 16, 3, std=2.0)
    p["w_up"] = np.zeros_like(p["w_up"])
    _, _, G, _ = _read(R, p, internals=True)
    assert np.all(G == 0.5)


def pin_zero_write_projection():
    """W_w = 0 ⇒ s ≡ 2σ(0) = 1 exactly (eq s)."""
    rng = np.random.default_rng(104)
    R = rng.standard_normal((4, 4, 16))
    p = _params(rng, 4, 16, 3)
    p["w_write"] = np.zeros_like(p["w_write"])
    _, s = _read(R, p)
    assert np.all(s == 1.0)


def pin_gatednorm_single_branch():
    """n_r = 1: eq gate and eq use_gate collapse to GatedNorm (the 1/n_r factors are 1), and
    eq s to 2σ(W_w RMSNorm(u)). Compared with torch's rms_norm/linear/silu/sigmoid."""
    rng = np.random.default_rng(105)
    n, D, r, eps = 6, 20, 5, 1e-6
    u = rng.standard_normal((n, D)) * 3.0
    p = _params(rng, 1, D, r, std=0.5)
    x, s = _read(u[:, None, :], p, eps)
    gn, un = _torch_gatednorm(u, p["gamma"][0], p["w_down"], p["w_up"], eps)
    assert _rel(x, gn) < 1e-13
    s_t = (2.0 * torch.sigmoid(Fnn.linear(_t(un), _t(p["w_write"])))).numpy()
    assert _rel(s, s_t) < 1e-13


def pin_replicated_branches():
    """n_r = 4 copies of one stream u with equal gains and weights tiled over the branch
    blocks: (1/n_r) W_d vec R̂ = W_1 R̂, every G_i = σ(W_2 h), so x = GatedNorm(u) and
    s_j = 2σ(w_j · RMSNorm(u)). Fails if a 1/n_r is dropped or moved, or vec is mis-ordered."""
    rng = np.random.default_rng(106)
    n, D, r, eps, nb = 4, 12, 3, 1e-6, 4
    u = rng.standard_normal((n, D)) * 2.0
    gamma1 = 1.0 + 0.3 * rng.standard_normal(D)
    W1 = 0.6 * rng.standard_normal((r, D))
    W2 = 0.6 * rng.standard_normal((D, r))
    w = 0.6 * rng.standard_normal((nb, D))
    p = {"gamma": np.tile(gamma1, (nb, 1)), "w_down": np.tile(W1, (1, nb)),
         "w_up": np.tile(W2, (nb, 1)), "w_write": np.tile(w, (1, nb))}
    R = np.repeat(u[:, None, :], nb, axis=1)
    x, s = _read(R, p, eps)
    gn, un = _torch_gatednorm(u, gamma1, W1, W2, eps)
    assert _rel(x, gn) < 1e-13
    assert _rel(s, (2.0 * torch.sigmoid(Fnn.linear(_t(un), _t(w)))).numpy()) < 1e-13


def pin_prenorm_reduction():
    """One-hot read gates (G_0 = 1, others 0) with γ_0 = n_r·γ_pre and write strengths
    (1, 0, 0, 0) turn a GR stack into the Pre-Norm residual x ← x + F(RMSNorm(x)) on branch 0
    (Digest §二.2: static one-hot read, write e_0, identity mixing equals Pre-Norm; §二.4: GR
    replaces the pre-norm). The reference loop uses torch's rms_norm."""
    rng = np.random.default_rng(107)
    n, D, nb, L, eps = 3, 16, 4, 6, 1e-6
    gamma_pre = 1.0 + 0.2 * rng.standard_normal(D)
    Ms = [rng.standard_normal((D, D)) / math.sqrt(D) for _ in range(L)]
    x_pre = rng.standard_normal((n, D))
    R = rng.standard_normal((n, nb, D))
    R[:, 0, :] = x_pre
    others = R[:, 1:, :].copy()
    gamma = np.ones((nb, D))
    gamma[0] = nb * gamma_pre
    G = np.zeros((nb, D))
    G[0] = 1.0
    s = np.zeros((n, nb))
    s[:, 0] = 1.0
    for l in range(L):
        xin = oracle.read_fixed_gates(R, gamma, G, eps)
        R = oracle.write(R, xin @ Ms[l], s)
        x_pre = x_pre + _torch_rmsnorm(x_pre, gamma_pre, eps) @ Ms[l]
    assert _rel(R[:, 0, :], x_pre) < 1e-13
    assert np.array_equal(R[:, 1:, :], others)


def pin_two_branch_toy():
    """The two-branch example of the GR notes (tests/golden/two_branch_toy.json)."""
    with open(os.path.join(GOLDEN, "two_branch_toy.json")) as f:
        g = json.load(f)
    R = np.asarray(g["R"])[None]
    x = oracle.read_fixed_gates(R, np.asarray(g["gamma"]), np.asarray(g["G"]), g["eps"])
    exp = g["expected"]
    assert np.allclose(x[0], exp["x"], rtol=0, atol=1e-12)
    assert np.all(np.abs(x[0]) > 0.1)  # the sublayer input mixes both streams
    y = x @ np.asarray(g["F_matrix_rows_out"]).T
    assert np.allclose(y[0], exp["y"], rtol=0, atol=1e-12)
    Rp = oracle.write(R, y, np.asarray(g["s"])[None])
    assert np.allclose(Rp[0], exp["R_prime"], rtol=0, atol=1e-12)


def pin_two_branch_learned_gate():
    """The same two branches with a predicted gate, in closed form. r = 1, eps = 0,
    γ = 1/√2 (so R̂ = R), W_d = [2, 0, 0, 2]: z = (1/2)(2 + 2) = 2, h = SiLU(2) = 2σ(2).
    W_u = [1, -1, -1, 1]ᵀ: G_1 = (σ(h), σ(-h)), G_2 = (σ(-h), σ(h)) — branch 1 read mostly in
    dimension 1, branch 2 in dimension 2 — so x = (σ(h)/2, σ(h)/2).
    W_w = [[2,0,0,0],[0,0,0,-2]]: s = (2σ(1), 2σ(-1))."""
    sig = lambda a: 1.0 / (1.0 + math.exp(-a))  # noqa: E731
    R = np.array([[[1.0, 0.0], [0.0, 1.0]]])
    p = {"gamma": np.full((2, 2), 1.0 / math.sqrt(2.0)), "w_down": np.array([[2.0, 0, 0, 2.0]]),
         "w_up": np.array([[1.0], [-1.0], [-1.0], [1.0]]),
         "w_write": np.array([[2.0, 0, 0, 0], [0, 0, 0, -2.0]])}
    x, s, G, _ = _read(R, p, eps=0.0, internals=True)
    h = 2.0 * sig(2.0)
    assert np.allclose(G[0], [[sig(h), sig(-h)], [sig(-h), sig(h)]], rtol=0, atol=1e-14)
    assert np.allclose(x[0], [sig(h) / 2, sig(h) / 2], rtol=0, atol=1e-14)
    assert np.allclose(s[0], [2 * sig(1.0), 2 * sig(-1.0)], rtol=0, atol=1e-14)


def pin_chain_closed_form():
    """eq rcv: with no branch mixing, R_c^(v) = R_c^(0) + Σ_{u<v} s_c^(u) y^(u)."""
    rng = np.random.default_rng(108)
    n, nb, D, r, L = 3, 4, 16, 4, 7
    R0 = rng.standard_normal((n, nb, D))
    ys = [0.5 * rng.standard_normal((n, D)) for _ in range(L)]
    ps = [_params(rng, nb, D, r, std=0.4) for _ in range(L)]
    states, xs, ss = oracle.chain(R0, ys, ps)
    for v in range(L + 1):
        acc = R0.copy()
        for u in range(v):
            acc = acc + ss[u][:, :, None] * ys[u][:, None, :]
        assert _rel(states[v], acc) < 1e-13
    assert not np.allclose(ss[0], ss[1])  # strengths are data dependent


def pin_decomposition():
    """eq auv: x^(v) = a_{0→v} + Σ_{u<v} a_{u→v}, with
    a_{u→v} = (1/n_r) Σ_c G_c^(v) ⊙ γ_c ⊙ s_c^(u) y^(u) / rms(R_c^(v)) (and a_{0→v} the same
    with R_c^(0)); exact up to round-off, so the fractions π_uv sum to 1."""
    rng = np.random.default_rng(109)
    n, nb, D, r, L, eps = 2, 4, 16, 4, 5, 1e-6
    R0 = rng.standard_normal((n, nb, D))
    ys = [0.7 * rng.standard_normal((n, D)) for _ in range(L)]
    ps = [_params(rng, nb, D, r, std=0.4) for _ in range(L)]
    states, xs, ss = oracle.chain(R0, ys, ps, eps)
    v = L - 1
    p = ps[v]
    x, _, G, inv = _read(states[v], p, eps, internals=True)
    assert _rel(x, xs[v]) < 1e-14
    coef = G * p["gamma"][None] * inv[:, :, None]            # G_c γ_c / rms(R_c^(v))
    a0 = (coef * R0).sum(axis=1) / nb
    a = [(coef * (ss[u][:, :, None] * ys[u][:, None, :])).sum(axis=1) / nb for u in range(v)]
    assert _rel(a0 + sum(a), x) < 1e-13
    norms = np.array([np.linalg.norm(au, axis=1) for au in a])  # [v, n]
    pi = norms / norms.sum(axis=0, keepdims=True)
    assert np.allclose(pi.sum(axis=0), 1.0, atol=3e-8)


def pin_branch_permutation():
    """Branches are exchangeable (Digest §二.6): permuting branches together with γ rows, W_d
    column blocks, W_u row blocks and W_w rows and column blocks permutes s and leaves x."""
    rng = np.random.default_rng(110)
    n, nb, D, r = 4, 4, 12, 3
    R = rng.standard_normal((n, nb, D))
    p = _params(rng, nb, D, r, std=0.5)
    perm = np.array([2, 0, 3, 1])
    blocks = np.concatenate([np.arange(i * D, (i + 1) * D) for i in perm])
    q = {"gamma": p["gamma"][perm], "w_down": p["w_down"][:, blocks],
         "w_up": p["w_up"][blocks, :], "w_write": p["w_write"][perm][:, blocks]}
    x, s = _read(R, p)
    x2, s2 = _read(R[:, perm, :], q)
    assert _rel(x2, x) < 1e-13 and _rel(s2, s[:, perm]) < 1e-13


def pin_branch_scale_invariance():
    """With eps = 0, RMSNorm removes any positive per-branch scale: x and s are unchanged."""
    rng = np.random.default_rng(111)
    R = rng.standard_normal((3, 4, 16))
    p = _params(rng, 4, 16, 3, std=0.5)
    x, s = _read(R, p, eps=0.0)
    c = np.array([0.1, 1.0, 10.0, 100.0])[None, :, None]
    x2, s2 = _read(R * c, p, eps=0.0)
    assert _rel(x2, x) < 1e-13 and _rel(s2, s) < 1e-13


def pin_ranges_and_saturation():
    """G ∈ (0,1) and s ∈ (0,2) (bounded positive gates); huge logits stay finite."""
    rng = np.random.default_rng(112)
    R = rng.standard_normal((3, 4, 16))
    p = _params(rng, 4, 16, 3, std=0.5)
    x, s, G, _ = _read(R, p, internals=True)
    assert np.all((G > 0) & (G < 1)) and np.all((s > 0) & (s < 2))
    big = {k: (v * 1e4 if k != "gamma" else v) for k, v in p.items()}
    x, s, G, _ = _read(R, big, internals=True)
    assert np.all(np.isfinite(x)) and np.all(np.isfinite(s)) and np.all(np.isfinite(G))
    assert np.all((G >= 0) & (G <= 1)) and np.all((s >= 0) & (s <= 2))


def pin_residual_add():
    rng = np.random.default_rng(113)
    a, b = rng.standard_normal(1000), rng.standard_normal(1000)
    assert np.array_equal(oracle.residual_add(a, b), a + b)


# ---- backward -----------------------------------------------------------------------------------

def _fd_grad(f, A, h=1e-6):
    """Central finite differences of the scalar f() with respect to every entry of A."""
    G = np.zeros_like(A)
    for idx in np.ndindex(A.shape):
        o = A[idx]
        A[idx] = o + h
        a = f()
        A[idx] = o - h
        b = f()
        A[idx] = o
        G[idx] = (a - b) / (2 * h)
    return G


def pin_backward_finite_differences():
    """The read's gradients (state and all four parameters) equal central finite differences
    of L = Σ dx·x + Σ ds·s, for n_r = 4 and n_r = 2, eps > 0, random gains."""
    for nb, D, r, seed in ((4, 8, 3, 157), (2, 6, 2, 163)):
        rng = np.random.default_rng(seed)
        n, eps = 3, 1e-3
        R = rng.standard_normal((n, nb, D))
        p = _params(rng, nb, D, r, std=0.5)
        dx, ds = rng.standard_normal((n, D)), rng.standard_normal((n, nb))

        def L():
            x, s = _read(R, p, eps)
            return float((dx * x).sum() + (ds * s).sum())

        dR, g = oracle.read_backward(R, p, dx, ds, eps)
        assert _rel(_fd_grad(L, R), dR) < 1e-6
        for k in ("gamma", "w_down", "w_up", "w_write"):
            assert _rel(_fd_grad(L, p[k]), g[k]) < 1e-6, k


def pin_backward_torch_autograd():
    """The same gradients from torch's autograd (a library's reverse mode) through the read
    written in torch ops, on a few tokens."""
    import torch
    rng = np.random.default_rng(167)
    n, nb, D, r, eps = 5, 4, 16, 4, 1e-5
    R = rng.standard_normal((n, nb, D))
    p = _params(rng, nb, D, r, std=0.3)
    dx, ds = rng.standard_normal((n, D)), rng.standard_normal((n, nb))
    Rt = torch.tensor(R, requires_grad=True)
    pt = {k: torch.tensor(v, requires_grad=True) for k, v in p.items()}
    inv = torch.rsqrt((Rt * Rt).mean(-1, keepdim=True) + eps)
    Rh = Rt * inv * pt["gamma"]
    v = Rh.reshape(n, nb * D)
    z = v @ pt["w_down"].T / nb
    G = torch.sigmoid((z * torch.sigmoid(z)) @ pt["w_up"].T).reshape(n, nb, D)
    x = (G * Rh).sum(1) / nb
    s = 2 * torch.sigmoid(v @ pt["w_write"].T / nb)
    ((torch.tensor(dx) * x).sum() + (torch.tensor(ds) * s).sum()).backward()
    dR, g = oracle.read_backward(R, p, dx, ds, eps)
    assert _rel(dR, Rt.grad.numpy()) < 1e-12
    for k in g:
        assert _rel(g[k], pt[k].grad.numpy()) < 1e-12, k


def pin_write_backward():
    """eq write is linear: its gradients equal finite differences exactly enough, and dR = dR'."""
    rng = np.random.default_rng(173)
    n, nb, D = 3, 4, 5
    R, y, s = rng.standard_normal((n, nb, D)), rng.standard_normal((n, D)), rng.uniform(0, 2, (n, nb))
    dRp = rng.standard_normal((n, nb, D))

    def L():
        return float((dRp * oracle.write(R, y, s)).sum())

    dR, dy, dsv = oracle.write_backward(dRp, y, s)
    assert np.array_equal(dR, dRp)
    assert _rel(_fd_grad(L, y), dy) < 1e-8 and _rel(_fd_grad(L, s), dsv) < 1e-8


# ---- FP8 state (e4m3 codes, one power-of-two scale per 32-channel block) --------------------

def _torch_e4m3_values():
    """Value of every e4m3 code by torch's float8_e4m3fn (a library conversion)."""
    import torch
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def pin_fp8_codes_match_torch():
    """Every code decodes as torch's float8_e4m3fn does; rounding to the nearest code (ties to
    even) agrees with torch's conversion on random values, subnormals and every exact tie."""
    import torch
    t = _torch_e4m3_values()
    v = oracle.fp8_code_values()
    assert np.array_equal(np.isnan(v), np.isnan(t))
    assert np.array_equal(v[~np.isnan(v)], t[~np.isnan(t)])
    vals = np.unique(t[~np.isnan(t)])
    mids = (vals[:-1] + vals[1:]) / 2
    rng = np.random.default_rng(131)
    w = np.concatenate([rng.uniform(-448, 448, 20000), rng.uniform(-0.03, 0.03, 20000),
                        mids, -mids, vals]).astype(np.float32).astype(np.float64)
    ct = torch.from_numpy(w).float().to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.fp8_round_codes(w), ct)


def pin_fp8_block_scale():
    """The block exponent is the smallest e with amax <= 448·2^e (closed-form cases and the
    two defining inequalities on random blocks); an all-zero block gets the smallest scale."""
    cases = {448.0: 0, 449.0: 1, 1.0: -8, 1.75: -8, 1.7500001: -7, 0.875: -9, 2.0 ** -100: -108,
             3.0e38: 120}
    for amax, e in cases.items():
        V = np.zeros((1, 32))
        V[0, 5] = -amax
        _, b = oracle.fp8_encode(V)
        assert int(b[0, 0]) - 127 == e, (amax, int(b[0, 0]) - 127, e)
    _, b = oracle.fp8_encode(np.zeros((1, 64)))
    assert np.all(b == 0)
    rng = np.random.default_rng(137)
    V = (rng.standard_normal((64, 4, 256)) * np.exp(rng.uniform(-20, 20, (64, 4, 1)))
         ).astype(np.float32).astype(np.float64)
    _, b = oracle.fp8_encode(V)
    amax = np.abs(V).reshape(64, 4, 8, 32).max(-1)
    e = b.astype(np.float64) - 127
    assert np.all(amax <= 448 * 2.0 ** e) and np.all(amax > 448 * 2.0 ** (e - 1))


def pin_fp8_roundtrip():
    """Decoding an encoded block errs by at most half a code step: 2^-4 relative for values in
    the normal range of the scaled codes, 2^-10·scale absolute below it; encoding what a
    decode produced gives back the same values (the stored values are fixed points; the codes
    may differ where rounding brought a block's maximum down to 448·2^(e-1), which the smaller
    scale then represents exactly)."""
    rng = np.random.default_rng(139)
    V = (rng.standard_normal((32, 4, 512)) * np.exp(rng.uniform(-8, 8, (32, 4, 16, 1)))
         .repeat(32, axis=-1).reshape(32, 4, 512)).astype(np.float32).astype(np.float64)
    c, b = oracle.fp8_encode(V)
    W = oracle.fp8_decode(c, b)
    scale = (2.0 ** (b.astype(np.float64) - 127)).repeat(32, axis=-1)
    err = np.abs(W - V)
    normal = np.abs(V) >= scale * 2.0 ** -6
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(V[normal]))
    assert np.all(err[~normal] <= 2.0 ** -10 * scale[~normal])
    c2, b2 = oracle.fp8_encode(W)
    assert np.array_equal(oracle.fp8_decode(c2, b2), W)


def pin_fp8_blocks_independent():
    """A block's codes and scale depend on its own 32 channels only (blocks start at multiples
    of 32): scaling one block by 2^10 changes that block's scale by 10 and nothing else."""
    rng = np.random.default_rng(149)
    V = rng.standard_normal((3, 4, 128)).astype(np.float32).astype(np.float64)
    c, b = oracle.fp8_encode(V)
    V2 = V.copy()
    V2[1, 2, 64:96] *= 1024.0
    c2, b2 = oracle.fp8_encode(V2)
    mask = np.zeros(V.shape, bool)
    mask[1, 2, 64:96] = True
    assert np.array_equal(c2[~mask], c[~mask]) and np.array_equal(c2[mask], c[mask])
    bm = np.zeros(b.shape, bool)
    bm[1, 2, 2] = True
    assert np.array_equal(b2[~bm], b[~bm]) and int(b2[1, 2, 2]) == int(b[1, 2, 2]) + 10


def pin_fp8_write_then_read_error():
    """The FP8 fused step against the plain definition (fp64, no storage rounding) stays within
    the FP8 bounds: R' within 2^-4, x and s within 2^-3 (per-row relative L2)."""
    rng = np.random.default_rng(151)
    n, nb, D, r = 16, 4, 128, 8
    R0 = rng.standard_normal((n, nb, D)).astype(np.float32)
    c, b = oracle.fp8_encode(R0)
    R = oracle.fp8_decode(c, b)
    y = rng.standard_normal((n, D)).astype(np.float32) * 0.5
    sp = rng.uniform(0, 2, (n, nb))
    p = _params(rng, nb, D, r)
    c2, b2, x, s = oracle.write_then_read_fp8(c, b, y, sp, p)
    Rp, xp, sp2 = oracle.write_then_read(R, y, sp, p)
    assert _rel(oracle.fp8_decode(c2, b2).reshape(n * nb, D), Rp.reshape(n * nb, D)) <= 2.0 ** -4
    assert _rel(x, xp) <= 2.0 ** -3 and _rel(s, sp2) <= 2.0 ** -3


def pin_decompose_exact_split():
    """eq rcv + eq auv (Digest §二.6): on an fp64 chain the reader's input splits exactly into
    the initial state's share and the writers' shares, a_{0→v} + Σ_u a_{u→v} = x^(v), so the
    fractions π sum to 1 for every token; the norms are those of the returned vectors."""
    rng = np.random.default_rng(113)
    n, nb, D, r, L, eps = 3, 4, 24, 4, 6, 1e-6
    R0 = rng.standard_normal((n, nb, D))
    ys = [0.7 * rng.standard_normal((n, D)) for _ in range(L)]
    ps = [_params(rng, nb, D, r, std=0.4) for _ in range(L)]
    states, xs, ss = oracle.chain(R0, ys, ps, eps)
    for v in (1, L - 1):
        o = oracle.decompose(states[v], ps[v], np.stack(ys[:v]), np.stack(ss[:v]), eps, R0=R0,
                             vectors=True)
        assert _rel(o["A0"] + o["A"].sum(axis=1), xs[v]) < 1e-13
        assert np.allclose(o["pi"].sum(axis=1), 1.0, rtol=0, atol=1e-14)
        assert np.allclose(o["norm"], np.linalg.norm(o["A"], axis=2), rtol=1e-14, atol=0)
        assert np.allclose(o["a0_norm"], np.linalg.norm(o["A0"], axis=1), rtol=1e-14, atol=0)


def pin_decompose_closed_form():
    """With W_u = 0 every gate is exactly σ(0) = ½, and with a gain g_i constant over each branch
    a_{u→v,i} = (1/8) g_i s_i^(u) y^(u) / rms(R_i): every norm in closed form from the inputs
    (rms taken here with numpy from its definition, eps = 1e-3, signed s and gains)."""
    rng = np.random.default_rng(114)
    n, nb, D, r, U, eps = 5, 4, 16, 3, 7, 1e-3
    R = rng.standard_normal((n, nb, D)) * np.array([0.5, 1.0, 2.0, 4.0])[None, :, None]
    R0 = rng.standard_normal((n, nb, D))
    g = np.array([1.5, -0.7, 0.9, 2.0])
    p = _params(rng, nb, D, r, std=0.5)
    p["gamma"] = np.repeat(g[:, None], D, axis=1)
    p["w_up"] = np.zeros((nb * D, r))
    ys = rng.standard_normal((U, n, D))
    ss = rng.uniform(-2.0, 2.0, (U, n, nb))
    o = oracle.decompose(R, p, ys, ss, eps, R0=R0)
    inv = 1.0 / np.sqrt(np.mean(R * R, axis=2) + eps)                  # [n, nb]
    ynorm = np.linalg.norm(ys, axis=2).T                               # [n, U]
    coef = g[None, :] * inv                                            # [n, nb]
    bn = np.abs(coef[:, None, :] * ss.transpose(1, 0, 2)) * ynorm[:, :, None] / 8.0
    tot = np.abs((coef[:, None, :] * ss.transpose(1, 0, 2)).sum(axis=2)) * ynorm / 8.0
    a0 = np.linalg.norm((coef[:, :, None] * R0).sum(axis=1), axis=1) / 8.0
    assert np.allclose(o["bnorm"], bn, rtol=1e-13, atol=0)
    assert np.allclose(o["norm"], tot, rtol=1e-13, atol=0)
    assert np.allclose(o["pi"], tot / tot.sum(axis=1, keepdims=True), rtol=1e-13, atol=0)
    assert np.allclose(o["a0_norm"], a0, rtol=1e-13, atol=0)


def pin_decompose_branch_permutation():
    """Branches are exchangeable (Digest §二.6): permuting the branches of the state, the
    parameters, the write strengths and the initial state permutes the per-branch norms and
    leaves the per-writer norms, π and the initial state's share unchanged."""
    rng = np.random.default_rng(115)
    n, nb, D, r, U = 3, 4, 12, 3, 5
    R, R0 = rng.standard_normal((n, nb, D)), rng.standard_normal((n, nb, D))
    p = _params(rng, nb, D, r, std=0.5)
    ys, ss = rng.standard_normal((U, n, D)), rng.uniform(0, 2, (U, n, nb))
    perm = np.array([2, 0, 3, 1])
    blocks = np.concatenate([np.arange(i * D, (i + 1) * D) for i in perm])
    q = {"gamma": p["gamma"][perm], "w_down": p["w_down"][:, blocks],
         "w_up": p["w_up"][blocks, :], "w_write": p["w_write"][perm][:, blocks]}
    o = oracle.decompose(R, p, ys, ss, R0=R0)
    o2 = oracle.decompose(R[:, perm], q, ys, ss[:, :, perm], R0=R0[:, perm])
    assert _rel(o2["norm"], o["norm"]) < 1e-13 and _rel(o2["pi"], o["pi"]) < 1e-13
    assert _rel(o2["bnorm"], o["bnorm"][:, :, perm]) < 1e-13
    assert _rel(o2["a0_norm"], o["a0_norm"]) < 1e-13


def pin_decompose_degenerate():
    """No writers: empty outputs; writers that wrote zeros: zero norms and π = 0; one writer:
    π = 1."""
    rng = np.random.default_rng(116)
    n, nb, D, r = 2, 4, 8, 2
    R = rng.standard_normal((n, nb, D))
    p = _params(rng, nb, D, r)
    o = oracle.decompose(R, p, np.zeros((0, n, D)), np.zeros((0, n, nb)))
    assert o["norm"].shape == (n, 0) and o["pi"].shape == (n, 0)
    o = oracle.decompose(R, p, np.zeros((3, n, D)), np.ones((3, n, nb)))
    assert np.all(o["norm"] == 0) and np.all(o["pi"] == 0) and np.all(o["bnorm"] == 0)
    o = oracle.decompose(R, p, rng.standard_normal((1, n, D)), np.ones((1, n, nb)))
    assert np.all(o["pi"] == 1.0)


ALL_PINS = [pin_dense_bruteforce, pin_zero_down_projection, pin_zero_up_projection,
            pin_zero_write_projection, pin_gatednorm_single_branch, pin_replicated_branches,
            pin_prenorm_reduction, pin_two_branch_toy, pin_two_branch_learned_gate,
            pin_chain_closed_form, pin_decomposition, pin_branch_permutation,
            pin_branch_scale_invariance, pin_ranges_and_saturation, pin_residual_add,
            pin_fp8_codes_match_torch, pin_fp8_block_scale, pin_fp8_roundtrip,
            pin_fp8_blocks_independent, pin_fp8_write_then_read_error,
            pin_backward_finite_differences, pin_backward_torch_autograd, pin_write_backward,
            pin_decompose_exact_split, pin_decompose_closed_form, pin_decompose_branch_permutation,
            pin_decompose_degenerate]
