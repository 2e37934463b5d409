"""GPU parity: the CUDA library (through the C ABI) against the fp64 oracle, element by element
on seeded inputs, per-row relative L2 error within 1e-5 (fp32 states) / 2e-2 (bf16 states)."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from gr_testlib import TOL, TORCH_DTYPE, bf16_path_params, max_abs, params_to_torch, \
    path_params, rel_rows, to_f64, to_torch
from stream_gated_residual_gb300 import gr
from stream_gated_residual_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    gr.load()
    oracle.build()


def _pack(p: dict, dtype: str, eps: float):
    t = params_to_torch(p)
    return gr.pack_params(t["gamma"], t["w_down"], t["w_up"], t["w_write"], TORCH_DTYPE[dtype],
                          eps)


# Per-row tolerances against the oracle that models the library's storage (the write's sum is
# one fp32 fused multiply-add, then stored; the read sees the stored state; bf16-path weights
# are bf16 with gamma folded). R' then matches to the last bit; what is left for x and s is fp32
# accumulation order, the transcendental approximations, and the final rounding of x to the
# state dtype (at most 2^-9 relative per element for bf16, so 4e-3 leaves 2x for the rest).
MODELED_TOL = {"f32": {"R": 1e-7, "x": 1e-5, "s": 1e-5},
               "bf16": {"R": 1e-7, "x": 4e-3, "s": 1e-4}}


def fused_case(w: wl.Workload, n_tokens=None, weight_mult=1.0, random_gamma=False,
               rows=None, chunk=2048):
    """One fused write→read on the GPU against the oracle on `rows` (all rows if None).
    Returns (plain, modeled): per-row errors against the plain fp64 definition, and against the
    oracle run on the stored state with the weights the bf16 path uses."""
    N = w.n_tokens if n_tokens is None else n_tokens
    R = wl.make_state(w, N)
    y = wl.make_y(w, 0, N)
    s_prev = wl.make_s_prev(w, N)
    p = wl.make_params(w, 1, weight_mult)
    if random_gamma:
        p["gamma"] = wl.make_random_gamma(w, 1)
    if w.dtype == "bf16":
        pm = path_params(p, gr.kernel_path(N, w.d_model, w.rank, torch.bfloat16))
    else:
        pm = p
    Rt, yt, st = to_torch(R), to_torch(y), torch.from_numpy(s_prev).cuda()
    P = _pack(p, w.dtype, w.eps)
    x, s = gr.write_then_read(Rt, yt, st, P)
    torch.cuda.synchronize()
    rows = np.arange(N) if rows is None else rows
    plain = {"R": 0.0, "x": 0.0, "s": 0.0}
    modeled = {"R": 0.0, "x": 0.0, "s": 0.0}
    for a in range(0, len(rows), chunk):
        idx = rows[a:a + chunk]
        Rf, yf, sp = wl.to_f64(R[idx]), wl.to_f64(y[idx]), s_prev[idx]
        sel = torch.from_numpy(idx).cuda()
        got = {"R": to_f64(Rt[sel]), "x": to_f64(x[sel]), "s": to_f64(s[sel])}
        for ref, res in ((oracle.write_then_read(Rf, yf, sp, p, w.eps), plain),
                         (oracle.write_then_read(Rf, yf, sp, pm, w.eps, store=w.dtype), modeled)):
            for k, v in zip(("R", "x", "s"), ref):
                res[k] = max(res[k], rel_rows(got[k], v))
    assert torch.isfinite(x.float()).all() and torch.isfinite(Rt.float()).all()
    assert bool(((s >= 0) & (s <= 2)).all())  # 2σ(u) saturates to exactly 0 or 2 in fp32
    print(f"{w.name} N={N} D={w.d_model} r={w.rank} {w.dtype} x{weight_mult}: plain {plain} "
          f"modeled {modeled}")
    return plain, modeled


def check(w, plain, modeled, plain_too=True):
    tol = MODELED_TOL[w.dtype]
    assert all(modeled[k] < tol[k] for k in tol), modeled
    if plain_too:
        assert max(plain.values()) < TOL[w.dtype], plain


def test_tiny_fp32_read_then_write():
    """Tiny fp32 GR step: one read, then one write with the read's s (tol 1e-5)."""
    w = wl.WORKLOADS["tiny_fp32"]
    R = wl.make_state(w)
    y = wl.make_y(w)
    p = wl.make_params(w)
    Rt = to_torch(R)
    P = _pack(p, "f32", w.eps)
    x, s = gr.read(Rt, P)
    xo, so = oracle.read(wl.to_f64(R), p["gamma"], p["w_down"], p["w_up"], p["w_write"], w.eps)
    assert rel_rows(to_f64(x), xo) < TOL["f32"]
    assert rel_rows(to_f64(s), so) < TOL["f32"]
    gr.write(Rt, to_torch(y), s)
    Ro = oracle.write(wl.to_f64(R), wl.to_f64(y), to_f64(s))
    assert rel_rows(to_f64(Rt), Ro) < TOL["f32"]


def test_tiny_fp32_fused():
    w = wl.WORKLOADS["tiny_fp32"]
    check(w, *fused_case(w))


@pytest.mark.parametrize("N,D,r", [(1, 8, 1), (3, 8, 3), (17, 264, 5), (33, 520, 64),
                                   (5, 4104, 16)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_odd_shapes(N, D, r, dtype):
    w = wl.Workload("odd", N, D, r, dtype, y_std=0.5, seed=7)
    check(w, *fused_case(w, random_gamma=True))


def test_decode_full():
    """N=128, D=4096, r=16, bf16: all rows."""
    w = wl.WORKLOADS["decode"]
    check(w, *fused_case(w))


@pytest.mark.parametrize("mult", [10.0, 50.0])
def test_decode_sharp_gates_and_random_gamma(mult):
    """Weights x10 (gate logits spread over several units, G and s far from 1/2 and 1) and x50
    (gates saturated at 0 or 1), with non-unit gains. Against the plain definition, the bf16
    rounding of the stored state and of the folded weights moves each logit u by an absolute
    amount that grows with its spread, and where s = 2σ(u) is far from 1 it moves by that amount
    relative to itself: measured at x10, s is 2.8e-2 from the plain definition (R' 1.7e-3, x
    4.0e-3), past the 2e-2 bound, and more at x50. Only the storage-modelled comparison, which
    sees the same stored values and weights, bounds these cases; the x5 sweeps of the kernels
    below meet the plain bound as well (s up to 1.8e-2 at D = 7168)."""
    w = wl.WORKLOADS["decode"]
    check(w, *fused_case(w, weight_mult=mult, random_gamma=True), plain_too=False)


def test_prefill_full():
    """N=16384, D=4096, r=16, bf16: every row against the oracle (in chunks)."""
    w = wl.WORKLOADS["prefill"]
    check(w, *fused_case(w))


def test_large_skewed_subset():
    """The skewed distribution (branch scales 0.1/1/10/100, 1% outlier channels x50, y from
    Student-t(3)), D=7168, r=32, on the first 1024 tokens."""
    w = wl.WORKLOADS["large_skewed"]
    check(w, *fused_case(w, n_tokens=1024))


def test_large_skewed_full_size_sampled():
    """The large/skewed workload at its full size (N=65536, D=7168, r=32: a 3.8 GB state) in
    one call; every output row is finite and in range, and 512 seeded sampled rows (with the
    first and the last) are compared with the oracle."""
    w = wl.WORKLOADS["large_skewed"]
    rng = np.random.default_rng(17)
    rows = np.unique(np.concatenate([[0, w.n_tokens - 1],
                                     rng.choice(w.n_tokens, 510, replace=False)]))
    check(w, *fused_case(w, rows=rows))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fused_equals_write_then_read_separately(dtype):
    """The fused call reads the stored state, so it equals gr_write followed by gr_read."""
    w = wl.Workload("sep", 64, 512, 16, dtype, y_std=0.5, seed=3)
    R = wl.make_state(w)
    y = to_torch(wl.make_y(w))
    sp = torch.from_numpy(wl.make_s_prev(w)).cuda()
    P = _pack(wl.make_params(w, 1), dtype, w.eps)
    R1, R2 = to_torch(R), to_torch(R)
    x1, s1 = gr.write_then_read(R1, y, sp, P)
    gr.write(R2, y, sp)
    x2, s2 = gr.read(R2, P)
    assert torch.equal(R1, R2)
    tol = 0 if dtype == "f32" else 2e-3
    assert rel_rows(to_f64(x1), to_f64(x2)) <= tol and rel_rows(to_f64(s1), to_f64(s2)) <= tol


def test_empty_and_in_place_aliases():
    w = wl.Workload("alias", 8, 256, 8, "bf16", y_std=0.5, seed=5)
    P = _pack(wl.make_params(w), "bf16", w.eps)
    R0 = to_torch(wl.make_state(w))
    y = to_torch(wl.make_y(w))
    sp = torch.from_numpy(wl.make_s_prev(w)).cuda()
    # N = 0 is a valid no-op
    x0, s0 = gr.write_then_read(R0[:0], y[:0], sp[:0], P)
    assert x0.shape == (0, 256)
    # x may be y's buffer and s_next may be s_prev's buffer
    Ra, Rb = R0.clone(), R0.clone()
    xa, sa = gr.write_then_read(Ra, y.clone(), sp.clone(), P)
    yb, spb = y.clone(), sp.clone()
    gr.write_then_read(Rb, yb, spb, P, x=yb, s_next=spb)
    assert torch.equal(Ra, Rb) and torch.equal(xa, yb) and torch.equal(sa, spb)


@pytest.mark.parametrize("N,D,dtype", [(256, 1024, "bf16"), (5000, 512, "bf16"),
                                       (20000, 256, "bf16"), (3000, 256, "f32")])
def test_host_entry_matches_device_entry(N, D, dtype):
    """The host-buffer entry (pipelined over token chunks when N >= 2048, with a ragged last
    chunk) gives bit-for-bit the device entry's results."""
    w = wl.Workload("host", N, D, 16, dtype, y_std=0.5, seed=11)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    R, y, sp = wl.make_state(w), wl.make_y(w), wl.make_s_prev(w)
    P = _pack(wl.make_params(w, 1), dtype, w.eps)
    Rd = to_torch(R)
    xd, sd = gr.write_then_read(Rd, to_torch(y), torch.from_numpy(sp).cuda(), P)
    Rh = to_torch(R, "cpu").pin_memory()
    yh = to_torch(y, "cpu").pin_memory()
    sph = torch.from_numpy(sp).pin_memory()
    xh = torch.empty((w.n_tokens, w.d_model), dtype=tdt).pin_memory()
    sh = torch.empty((w.n_tokens, 4), dtype=torch.float32).pin_memory()
    nws = gr.host_workspace_size(w.n_tokens, w.d_model, tdt)
    buf = torch.empty(nws + 256, dtype=torch.uint8, device="cuda")
    ws = buf[(-buf.data_ptr()) % 256:][:nws]
    gr.write_then_read_host(Rh, yh, sph, P, xh, sh, ws)
    assert torch.equal(Rh, Rd.cpu()) and torch.equal(xh, xd.cpu()) and torch.equal(sh, sd.cpu())


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prenorm_reduction_on_gpu(dtype):
    """One-hot read gates with γ_0 = 4·γ_pre and writes (1,0,0,0): branch 0 follows the
    Pre-Norm residual x ← x + F(RMSNorm(x)) (Digest §二.2 and §二.4). F is a seeded linear map
    applied with torch; the reference loop runs in fp64 on the CPU."""
    rng = np.random.default_rng(21)
    N, D, L, eps = 64, 256, 8, 1e-6
    dt = TORCH_DTYPE[dtype]
    gamma_pre = (1.0 + 0.2 * rng.standard_normal(D))
    Ms = [rng.standard_normal((D, D)) / math.sqrt(D) for _ in range(L)]
    R0 = wl.make_state(wl.Workload("pn", N, D, 8, dtype, y_std=1.0, seed=21))
    R = to_torch(R0)
    gamma = np.ones((4, D))
    gamma[0] = 4 * gamma_pre
    G = np.zeros((4, D))
    G[0] = 1.0
    g_t = torch.tensor(gamma, dtype=torch.float32, device="cuda")
    G_t = torch.tensor(G, dtype=torch.float32, device="cuda")
    s = torch.zeros((N, 4), dtype=torch.float32, device="cuda")
    s[:, 0] = 1.0
    x_ref = wl.to_f64(R0)[:, 0, :].copy()
    others = R[:, 1:, :].clone()
    for l in range(L):
        xin = gr.read_fixed_gates(R, g_t, G_t, eps)
        y = (xin.float() @ torch.tensor(Ms[l], dtype=torch.float32, device="cuda")).to(dt)
        gr.write(R, y.contiguous(), s)
        rn = x_ref / np.sqrt(np.mean(x_ref ** 2, axis=1, keepdims=True) + eps) * gamma_pre
        x_ref = x_ref + rn @ Ms[l]
    tol = 1e-5 if dtype == "f32" else 5e-2
    assert rel_rows(to_f64(R[:, 0, :]), x_ref) < tol
    assert torch.equal(R[:, 1:, :], others)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_residual_add_reference(dtype):
    n = 1_000_003  # not a multiple of 8: vector body plus scalar tail
    rng = np.random.default_rng(4)
    xs = wl.to_storage(rng.standard_normal(n).astype(np.float32), dtype)
    ys = wl.to_storage(rng.standard_normal(n).astype(np.float32), dtype)
    x, y = to_torch(xs), to_torch(ys)
    gr.residual_add_ref(x, y)
    expect = oracle.residual_add(wl.to_f64(xs), wl.to_f64(ys))
    if dtype == "bf16":
        expect = wl.to_f64(wl.to_storage(expect.astype(np.float32), "bf16"))
        # fp32 sum of two bf16 values is exact; one rounding to bf16 on both sides
        assert np.array_equal(to_f64(x), expect)
    else:
        assert max_abs(to_f64(x), expect) <= 1e-6 * np.max(np.abs(expect))


def test_calls_reject_cpu_tensors():
    w = wl.Workload("cpu", 4, 64, 8, "bf16", y_std=0.5)
    P = _pack(wl.make_params(w), "bf16", w.eps)
    with pytest.raises(ValueError):
        gr.read(to_torch(wl.make_state(w), "cpu"), P)


@pytest.mark.parametrize("D,r,N", [(256, 8, 1), (256, 16, 17), (512, 16, 33), (1024, 12, 100),
                                   (2048, 16, 250), (4096, 16, 15), (4096, 1, 16),
                                   (4096, 4, 1000), (2048, 8, 4099)])
def test_fused_kernel_shapes(D, r, N):
    """Every cluster size (D = 256 … 4096 → 1 … 16 CTAs), ranks 1 … 16, ragged last tiles."""
    w = wl.Workload("fused", N, D, r, "bf16", y_std=0.5, seed=13)
    assert gr.kernel_path(N, D, r, torch.bfloat16) == "fused_bf16"
    check(w, *fused_case(w, random_gamma=True, weight_mult=5.0))
    assert gr.device_status(clear=True) == 0


@pytest.mark.parametrize("D,r,N", [(2048, 16, 77), (4096, 16, 300)])
def test_fused_read_only(D, r, N):
    """gr_read on the fused path: R untouched, x and s against the oracle's read."""
    w = wl.Workload("read", N, D, r, "bf16", y_std=0.5, seed=17)
    R = wl.make_state(w)
    p = wl.make_params(w, 1, weight_mult=5.0)
    p["gamma"] = wl.make_random_gamma(w, 1)
    Rt = to_torch(R)
    x, s = gr.read(Rt, _pack(p, "bf16", w.eps))
    torch.cuda.synchronize()
    assert torch.equal(Rt, to_torch(R))
    pm = bf16_path_params(p, "f16")
    xo, so = oracle.read(wl.to_f64(R), pm["gamma"], pm["w_down"], pm["w_up"], pm["w_write"],
                         w.eps)
    tol = MODELED_TOL["bf16"]
    assert rel_rows(to_f64(x), xo) < tol["x"] and rel_rows(to_f64(s), so) < tol["s"]
    assert gr.device_status(clear=True) == 0


@pytest.mark.parametrize("D,r,N", [(64, 1, 1), (192, 8, 31), (320, 12, 33), (448, 16, 65),
                                   (768, 20, 100), (1536, 32, 257), (4096, 32, 300),
                                   (6144, 24, 77), (7168, 32, 1000), (1536, 17, 10000)])
def test_tiled_kernel_shapes(D, r, N):
    """The two-pass kernel: D = 64 … 7168 (one to 112 channel chunks), both rank classes (up to
    16 and up to 32), ragged last tiles (including a single token and a tile whose second
    16-token half is empty), and more tiles than SMs (N = 10000)."""
    w = wl.Workload("tiled", N, D, r, "bf16", y_std=0.5, seed=29)
    assert gr.kernel_path(N, D, r, torch.bfloat16) == "tiled_bf16"
    check(w, *fused_case(w, random_gamma=True, weight_mult=5.0))
    assert gr.device_status(clear=True) == 0


@pytest.mark.parametrize("D,r,N", [(320, 8, 45), (7168, 32, 100)])
def test_tiled_read_only(D, r, N):
    """gr_read on the two-pass kernel: R untouched, x and s against the oracle's read."""
    w = wl.Workload("read", N, D, r, "bf16", y_std=0.5, seed=31)
    R = wl.make_state(w)
    p = wl.make_params(w, 1, weight_mult=5.0)
    p["gamma"] = wl.make_random_gamma(w, 1)
    Rt = to_torch(R)
    assert gr.kernel_path(N, D, r, torch.bfloat16) == "tiled_bf16"
    x, s = gr.read(Rt, _pack(p, "bf16", w.eps))
    torch.cuda.synchronize()
    assert torch.equal(Rt, to_torch(R))
    pm = bf16_path_params(p, "f16")
    xo, so = oracle.read(wl.to_f64(R), pm["gamma"], pm["w_down"], pm["w_up"], pm["w_write"],
                         w.eps)
    tol = MODELED_TOL["bf16"]
    assert rel_rows(to_f64(x), xo) < tol["x"] and rel_rows(to_f64(s), so) < tol["s"]
    assert gr.device_status(clear=True) == 0


@pytest.mark.parametrize("N,write", [(8192, True), (16384, False)])
def test_split_cluster_and_two_pass(N, write):
    """A large step on a cluster-kernel shape (D = 4096, r = 16) also runs a share of its tokens
    on the two-pass kernel, on the SMs the clusters leave idle (its programmatic dependent on the
    same stream): every row
    (both shares and the boundary between them) against the oracle, for the fused step and for
    the read alone, with sharp gates and random gains."""
    D, r = 4096, 16
    assert gr.kernel_path(N, D, r, torch.bfloat16) == "fused_bf16+tiled_bf16"
    w = wl.Workload("split", N, D, r, "bf16", y_std=0.5, seed=37)
    if write:
        check(w, *fused_case(w, random_gamma=True, weight_mult=5.0))
    else:
        R = wl.make_state(w)
        p = wl.make_params(w, 1, weight_mult=5.0)
        p["gamma"] = wl.make_random_gamma(w, 1)
        Rt = to_torch(R)
        x, s = gr.read(Rt, _pack(p, "bf16", w.eps))
        torch.cuda.synchronize()
        assert torch.equal(Rt, to_torch(R))
        pm = path_params(p, "fused_bf16+tiled_bf16")
        rows = np.arange(0, N, 7)
        xo, so = oracle.read(wl.to_f64(R[rows]), pm["gamma"], pm["w_down"], pm["w_up"],
                             pm["w_write"], w.eps)
        sel = torch.from_numpy(rows).cuda()
        tol = MODELED_TOL["bf16"]
        assert rel_rows(to_f64(x[sel]), xo) < tol["x"] and rel_rows(to_f64(s[sel]), so) < tol["s"]
    assert gr.device_status(clear=True) == 0


def test_deep_stack_chain():
    """96 chained sublayers (48 layers × token mixer, MLP) at N=8192, D=2048, r=16, bf16, fresh
    seeded y_l and weights per sublayer: gr_read, 95 fused steps, gr_write. Every sublayer's
    state, x and s are compared with the oracle's free-running fp64 chain on 256 sampled token
    rows (the whole chain of those rows: tokens are independent)."""
    w = wl.WORKLOADS["deep_stack"]
    L, N = w.n_sublayers, w.n_tokens
    rows = np.sort(np.random.default_rng(5).choice(N, 256, replace=False))
    sel = torch.from_numpy(rows).cuda()
    R0 = wl.make_state(w)
    R = to_torch(R0)
    ps = [wl.make_params(w, l) for l in range(L)]
    s_a = torch.empty((N, 4), dtype=torch.float32, device="cuda")
    s_b = torch.empty_like(s_a)
    x = torch.empty((N, w.d_model), dtype=torch.bfloat16, device="cuda")
    got = {"R": [], "x": [], "s": []}
    ys_rows = []
    P = _pack(ps[0], "bf16", w.eps)
    gr.read(R, P, x=x, s=s_a)
    got["R"].append(to_f64(R[sel]))
    got["x"].append(to_f64(x[sel]))
    got["s"].append(to_f64(s_a[sel]))
    for l in range(1, L + 1):
        y = wl.make_y(w, l - 1)
        ys_rows.append(wl.to_f64(y[rows]))
        yt = to_torch(y)
        if l < L:
            P = _pack(ps[l], "bf16", w.eps)
            gr.write_then_read(R, yt, s_a, P, x=x, s_next=s_b)
            s_a, s_b = s_b, s_a
            got["x"].append(to_f64(x[sel]))
            got["s"].append(to_f64(s_a[sel]))
        else:
            gr.write(R, yt, s_a)
        got["R"].append(to_f64(R[sel]))
    assert gr.device_status(clear=True) == 0
    states, xs, ss = oracle.chain(wl.to_f64(R0[rows]), ys_rows, ps, w.eps)
    curve = [max(rel_rows(got["R"][l], states[l]),
                 rel_rows(got["x"][l], xs[l]) if l < L else 0.0,
                 rel_rows(got["s"][l], ss[l]) if l < L else 0.0) for l in range(L + 1)]
    print("deep stack per-sublayer max per-row rel. error:",
          " ".join(f"{e:.2e}" for e in curve[::8]), "... final", f"{curve[-1]:.2e}")
    assert max(curve) < TOL["bf16"], curve
