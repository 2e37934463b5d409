"""GPU parity of the contribution decomposition (eq auv and π, Digest §二.6):
gr_decompose through the C ABI against the fp64 oracle on the same stored inputs. Every norm,
per-branch norm, π and the initial state's share within 1e-4 relative, with an absolute floor of
1e-4 times the token's largest writer norm for terms far below it."""
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


def _close(got, ref, scale):
    """max over elements of |got − ref| / max(|ref|, 1e-4 · scale) (scale per token)."""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    den = np.maximum(np.abs(ref), 1e-4 * scale)
    return float(np.max(np.abs(got - ref) / den)) if ref.size else 0.0


def _case(N, D, r, dtype, U, seed=51, with_r0=True, zero_writer=None, weight_mult=5.0):
    w = wl.Workload("dec", N, D, r, dtype, y_std=0.5, seed=seed)
    R = wl.make_state(w)
    R0 = wl.make_state(wl.Workload("dec0", N, D, r, dtype, y_std=0.5, seed=seed + 1))
    p = wl.make_params(w, 1, weight_mult=weight_mult)
    p["gamma"] = wl.make_random_gamma(w, 1)
    rng = np.random.default_rng(seed + 2)
    ys = [wl.make_y(w, u) for u in range(U)]
    if zero_writer is not None and U:
        ys[zero_writer] = np.zeros_like(ys[zero_writer])
    Y = np.stack(ys) if U else np.zeros((0, N, D), dtype=R.dtype)
    S = rng.uniform(0.0, 2.0, (U, N, 4)).astype(np.float32)
    pt = {k: torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).cuda()
          for k, v in p.items()}
    Yt = to_torch(Y.reshape(U * N, D)).reshape(U, N, D) if U else None
    out = gr.decompose(to_torch(R), pt["gamma"], pt["w_down"], pt["w_up"], pt["w_write"], Yt,
                       torch.from_numpy(S).cuda() if U else None,
                       to_torch(R0) if with_r0 else None, w.eps)
    torch.cuda.synchronize()
    assert gr.device_status(clear=True) == 0
    ref = oracle.decompose(wl.to_f64(R), p, wl.to_f64(Y), S, w.eps,
                           R0=wl.to_f64(R0) if with_r0 else None)
    scale = (ref["norm"].max(axis=1, keepdims=True) if U else np.ones((N, 1)))
    errs = {"norm": _close(to_f64(out["norm"]), ref["norm"], scale),
            "branch_norm": _close(to_f64(out["branch_norm"]), ref["bnorm"], scale[:, :, None]),
            "pi": _close(to_f64(out["pi"]), ref["pi"], 1.0)}
    if with_r0:
        errs["a0"] = _close(to_f64(out["a0_norm"]), ref["a0_norm"], ref["a0_norm"].max())
    print(f"decompose N={N} D={D} r={r} {dtype} U={U}: {errs}")
    assert all(v < TOL for v in errs.values()), errs
    return out, ref


@pytest.mark.parametrize("N,D,r,dtype,U", [(1, 64, 1, "f32", 1), (5, 64, 4, "bf16", 6),
                                           (37, 256, 16, "bf16", 7), (100, 1032, 32, "f32", 13),
                                           (17, 520, 64, "f32", 3), (64, 4096, 16, "bf16", 12),
                                           (33, 2048, 20, "bf16", 40), (9, 4096, 8, "f32", 5),
                                           (7, 12288, 16, "bf16", 2), (3, 12288, 40, "f32", 4),
                                           (50, 256, 16, "bf16", 45), (70, 384, 32, "f32", 83)])
def test_decompose_matches_oracle(N, D, r, dtype, U):
    """Every rank class and tokens-per-CTA choice, ragged token tiles and writer groups (U not a
    multiple of 6, and U = 45 and 83), the widest D, both state types."""
    _case(N, D, r, dtype, U)


def test_no_writers_and_zero_writer():
    """U = 0 with the initial state (only its share); a writer that wrote zeros has norm 0 and
    π 0, the others' π still sum to 1."""
    _case(20, 512, 16, "bf16", 0)
    out, _ = _case(20, 512, 16, "bf16", 5, zero_writer=2)
    assert torch.all(out["norm"][:, 2] == 0) and torch.all(out["pi"][:, 2] == 0)
    assert torch.allclose(out["pi"].sum(dim=1), torch.ones(20, device="cuda"), atol=1e-5)


def test_without_optional_outputs():
    """No R0, no per-branch norms, no π: the norms alone, same values."""
    N, D, r, U = 40, 1024, 16, 8
    w = wl.Workload("dec", N, D, r, "bf16", y_std=0.5, seed=61)
    R = wl.make_state(w)
    p = wl.make_params(w, 1)
    Y = np.stack([wl.make_y(w, u) for u in range(U)])
    S = np.random.default_rng(62).uniform(0, 2, (U, N, 4)).astype(np.float32)
    pt = {k: torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).cuda()
          for k, v in p.items()}
    out = gr.decompose(to_torch(R), pt["gamma"], pt["w_down"], pt["w_up"], pt["w_write"],
                       to_torch(Y.reshape(U * N, D)).reshape(U, N, D),
                       torch.from_numpy(S).cuda(), None, w.eps, branch_norm=False, pi=False)
    torch.cuda.synchronize()
    ref = oracle.decompose(wl.to_f64(R), p, wl.to_f64(Y), S, w.eps)
    assert set(out) == {"norm"}
    assert _close(to_f64(out["norm"]), ref["norm"], ref["norm"].max(axis=1, keepdims=True)) < TOL


def test_stack_of_forty_blocks_sampled():
    """The pages' analysis shape: 40 GR blocks, the last reader and its 39 writers, on a
    deep-stack-width state (D = 2048, r = 16, bf16), 512 tokens."""
    _case(512, 2048, 16, "bf16", 39, seed=71, weight_mult=1.0)
