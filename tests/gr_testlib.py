"""Shared helpers of the tests: moving workload arrays to torch, per-row error metrics."""
from __future__ import annotations

import numpy as np
import torch

from stream_gated_residual_gb300 import workloads as wl

# tolerances on the per-row relative L2 error (max over rows): fp32 path, bf16 path
TOL = {"f32": 1e-5, "bf16": 2e-2}
TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}
# FP8 state against the storage-modelled oracle (the same stored state): x and s carry only the
# kernel's own arithmetic and the bf16 rounding of x, as on the bf16 path
MODELED_TOL_FP8 = {"x": 4e-3, "s": 1e-4}


def to_torch(a: np.ndarray, device="cuda") -> torch.Tensor:
    """Storage array (bf16 bits as uint16, or float32) -> torch tensor with the same bytes."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(
            device)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def params_to_torch(p: dict, device="cuda") -> dict:
    return {k: torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(device)
            for k, v in p.items()}


def rel_rows(a, b) -> float:
    """max over rows of ||a_row - b_row||_2 / ||b_row||_2 (rows = all but the last axis)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    a2 = a.reshape(-1, a.shape[-1])
    b2 = b.reshape(-1, b.shape[-1])
    num = np.linalg.norm(a2 - b2, axis=1)
    den = np.maximum(np.linalg.norm(b2, axis=1), 1e-30)
    return float(np.max(num / den)) if len(num) else 0.0


def max_abs(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b))) if a.size else 0.0


def bf16_path_params(p: dict, w_up: str = "bf16") -> dict:
    """The parameters the bf16 path computes with, written as oracle inputs: W_d and W_w with
    gamma folded in and rounded to bf16 (fp32 product, nearest even), divided back by gamma in
    fp64 so that the oracle's W·(γ ⊙ R) reproduces the folded weight; W_u rounded to bf16
    (w_up="bf16", the generic kernel) or, as ½·W_u, to fp16 (w_up="f16", the two tensor-core
    kernels, which pack ½·W_u as fp16 clamped to ±65504). Computed here from the fp32 inputs, never
    read back from the GPU."""
    K = p["w_down"].shape[1]
    g = np.asarray(p["gamma"], dtype=np.float32).reshape(-1)
    assert g.size == K and np.all(g != 0)

    def fold(W):
        Wf = wl.round_to_bf16((np.asarray(W, dtype=np.float32) * g[None, :]).astype(np.float32))
        return Wf.astype(np.float64) / g.astype(np.float64)[None, :]

    wu32 = np.asarray(p["w_up"], dtype=np.float32)
    if w_up == "bf16":
        wu = wl.round_to_bf16(wu32).astype(np.float64)
    elif w_up == "f16":
        half = np.clip(np.float32(0.5) * wu32, -65504.0, 65504.0).astype(np.float16)
        wu = 2.0 * half.astype(np.float64)
    else:
        raise ValueError(w_up)
    return {"gamma": np.asarray(p["gamma"], dtype=np.float64), "w_down": fold(p["w_down"]),
            "w_up": wu, "w_write": fold(p["w_write"])}


def path_params(p: dict, kernel_path: str) -> dict:
    """bf16_path_params for the kernel that serves a shape (gr.kernel_path's name): the cluster
    and two-pass kernels run the up projection in fp16, the generic kernel and the large-rank
    path keep bf16 W_u."""
    return bf16_path_params(p, "bf16" if kernel_path in ("generic", "tc_bf16") else "f16")


def sample_rows(n: int, k: int, seed: int = 0) -> np.ndarray:
    """A seeded sorted sample of k token rows, always including the first and last."""
    if n <= k:
        return np.arange(n)
    rng = np.random.default_rng([seed, 99])
    pick = rng.choice(np.arange(1, n - 1), size=k - 2, replace=False)
    return np.sort(np.concatenate([[0, n - 1], pick]))


__all__ = ["TOL", "TORCH_DTYPE", "MODELED_TOL_FP8", "to_torch", "to_f64", "params_to_torch", "rel_rows", "max_abs",
           "sample_rows", "bf16_path_params", "path_params", "wl"]
