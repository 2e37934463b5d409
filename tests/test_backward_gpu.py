"""GPU parity of the backward : gr_read_backward and gr_write_backward
through the C ABI against the fp64 oracle's chain-rule gradients (pinned by finite differences
and by torch autograd), on the same stored inputs. Per-row relative L2 ≤ 1e-4; rows of a
parameter gradient whose norm is below 1e-3 of the tensor's largest row are compared against
that floor instead (their relative error is rounding noise)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gr_testlib import to_f64, to_torch
from stream_gated_residual_gb300 import gr
from stream_gated_residual_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    gr.load()
    oracle.build()


def rel_rows_floor(a, b, floor_frac=1e-3):
    a = np.asarray(a, dtype=np.float64).reshape(-1, np.shape(a)[-1])
    b = np.asarray(b, dtype=np.float64).reshape(-1, np.shape(b)[-1])
    nb = np.linalg.norm(b, axis=1)
    den = np.maximum(nb, floor_frac * nb.max() + 1e-300)
    return float(np.max(np.linalg.norm(a - b, axis=1) / den))


@pytest.mark.parametrize("N,D,r,dtype", [(1, 64, 1, "f32"), (5, 64, 4, "f32"),
                                         (37, 256, 16, "bf16"), (100, 1032, 32, "f32"),
                                         (64, 4096, 16, "bf16"), (17, 520, 64, "f32"),
                                         (300, 2048, 20, "bf16"), (33, 512, 24, "bf16"),
                                         (9, 4096, 8, "f32"), (3, 12288, 40, "f32"),
                                         (7, 12288, 16, "bf16")])
def test_read_backward_matches_oracle(N, D, r, dtype):
    w = wl.Workload("bwd", N, D, r, dtype, y_std=0.5, seed=41)
    R = wl.make_state(w)
    p = wl.make_params(w, 1, weight_mult=5.0)
    p["gamma"] = wl.make_random_gamma(w, 1)
    rng = np.random.default_rng(43)
    dx = rng.standard_normal((N, D)).astype(np.float32)
    ds = rng.standard_normal((N, 4)).astype(np.float32)
    pt = {k: torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).cuda()
          for k, v in p.items()}
    dR, g = gr.read_backward(to_torch(R), pt["gamma"], pt["w_down"], pt["w_up"], pt["w_write"],
                             torch.from_numpy(dx).cuda(), torch.from_numpy(ds).cuda(), w.eps)
    torch.cuda.synchronize()
    dRo, go = oracle.read_backward(wl.to_f64(R), p, dx, ds, w.eps)
    errs = {"dR": rel_rows_floor(to_f64(dR), dRo, floor_frac=0.0)}
    for k in go:
        errs[k] = rel_rows_floor(to_f64(g[k]), go[k])
    print(f"backward N={N} D={D} r={r} {dtype}: {errs}")
    assert all(v < TOL for v in errs.values()), errs


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_write_backward_matches_oracle(dtype):
    N, D = 70, 384
    w = wl.Workload("wbwd", N, D, 8, dtype, y_std=0.5, seed=47)
    y = wl.make_y(w)
    s = wl.make_s_prev(w)
    rng = np.random.default_rng(53)
    dRp = rng.standard_normal((N, 4, D)).astype(np.float32)
    t = torch.from_numpy(dRp).cuda()
    dR, dy, dsv = gr.write_backward(t, to_torch(y), torch.from_numpy(s).cuda())
    torch.cuda.synchronize()
    dRo, dyo, dso = oracle.write_backward(dRp, wl.to_f64(y), s)
    assert np.array_equal(to_f64(dR), dRo)
    assert rel_rows_floor(to_f64(dy), dyo, 0.0) < 1e-5
    assert rel_rows_floor(to_f64(dsv), dso, 0.0) < 1e-5


def test_backward_of_a_fused_step_is_read_then_write_backward():
    """The fused step's gradient w.r.t. the state before it: the write's backward applied to the
    read's dL/dR' (plus a downstream dL/dR'), checked against the oracle's composition."""
    N, D, r = 48, 512, 16
    w = wl.Workload("fbwd", N, D, r, "f32", y_std=0.5, seed=59)
    R = wl.make_state(w)
    y = wl.make_y(w)
    sp = wl.make_s_prev(w)
    p = wl.make_params(w, 1, weight_mult=5.0)
    rng = np.random.default_rng(61)
    dx = rng.standard_normal((N, D)).astype(np.float32)
    ds = rng.standard_normal((N, 4)).astype(np.float32)
    dR_down = rng.standard_normal((N, 4, D)).astype(np.float32)
    Rp = oracle.round_to_storage(oracle.write(R, y, sp), "f32")   # the stored written state
    pt = {k: torch.from_numpy(v).cuda() for k, v in p.items()}
    dR_read, _ = gr.read_backward(torch.from_numpy(Rp.astype(np.float32)).cuda(), pt["gamma"],
                                  pt["w_down"], pt["w_up"], pt["w_write"],
                                  torch.from_numpy(dx).cuda(), torch.from_numpy(ds).cuda(),
                                  w.eps)
    dRp = dR_read + torch.from_numpy(dR_down).cuda()
    dR, dy, dsp = gr.write_backward(dRp, to_torch(y), torch.from_numpy(sp).cuda())
    torch.cuda.synchronize()
    dRo_read, _ = oracle.read_backward(Rp, p, dx, ds, w.eps)
    dRo, dyo, dspo = oracle.write_backward(dRo_read + dR_down, y, sp)
    assert rel_rows_floor(to_f64(dR), dRo, 0.0) < TOL
    assert rel_rows_floor(to_f64(dy), dyo, 0.0) < TOL
    assert rel_rows_floor(to_f64(dsp), dspo, 0.0) < TOL
